"""GPU parity of the fused fp32-input calls (q8_1 quantization inside the GEMV).

The fused calls quantize x with the standalone quantizer's arithmetic while
staging it, so their outputs must equal qmv_quantize_q8_1 followed by the
q8_1-input call bit for bit (that path is itself pinned to the oracle:
q8_1 bytes bit-exact, y within 1e-4 of the L1 norm), and stay within the
oracle bound directly.
"""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4
FUSED_TYPES = (oracle.Q4_0, oracle.Q4_K, oracle.Q6_K)


@pytest.fixture(scope="module")
def q():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import quantized_decode_gemv_qmv_gb300 as qq

    torch.cuda.set_device(0)
    qq.set_pdl(True)
    for t in qq.WEIGHT_TYPES:
        qq.set_tuning(t)
    return qq


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


def check_l1(y, y_ref, l1, what):
    err = np.abs(np.asarray(y, dtype=np.float64) - y_ref)
    bad = err > TOL * l1
    assert not bad.any(), f"{what}: {bad.sum()} outputs off the oracle bound"


def weights(t, M, K, seed):
    return oracle.quantize_rows(t, synthetic.weights_f32(seed, M, K))


@pytest.mark.parametrize("t,M,K", [(oracle.Q4_0, 203, 4096), (oracle.Q4_0, 61, 256), (oracle.Q4_K, 203, 4096),
                                   (oracle.Q4_K, 130, 2304), (oracle.Q4_K, 37, 11264), (oracle.Q6_K, 203, 4096),
                                   (oracle.Q6_K, 45, 2048), (oracle.Q6_K, 21, 14336)])
@pytest.mark.parametrize("ncols", [1, 2, 3, 5, 8])
def test_fused_plain_equals_two_step(q, t, M, K, ncols):
    W = weights(t, M, K, 1100 + M + ncols)
    x = synthetic.activations_f32(1200 + K + ncols, ncols, K, outlier_frac=0.01)
    Wd, xd = dev(W), dev(x)
    y_fused = host(q.mul_mat_vec_f32(t, Wd, M, K, xd))
    y_two = host(q.mul_mat_vec(t, Wd, M, K, q.quantize_q8_1(xd), ncols))
    assert np.array_equal(y_fused, y_two)
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, oracle.quantize_q8_1(x), ncols)
    check_l1(y_fused, y_ref, l1, f"fused type {t} {M}x{K} ncols {ncols}")


@pytest.mark.parametrize("t", FUSED_TYPES)
def test_fused_strided_and_misaligned_x(q, t):
    import torch

    M, K, nc = 97, 2048, 3
    W = weights(t, M, K, 1300 + t)
    x = synthetic.activations_f32(1301, nc, K)
    Wd = dev(W)
    y_two = host(q.mul_mat_vec(t, Wd, M, K, q.quantize_q8_1(dev(x)), nc))
    # rows K + 5 floats apart (no 128-bit loads)
    big = torch.zeros((nc, K + 5), dtype=torch.float32, device="cuda")
    big[:, :K] = dev(x)
    assert np.array_equal(host(q.mul_mat_vec_f32(t, Wd, M, K, big[:, :K])), y_two)
    # base address 4 bytes past a 16-byte boundary
    flat = torch.zeros(nc * K + 1, dtype=torch.float32, device="cuda")
    flat[1:] = dev(x).reshape(-1)
    assert np.array_equal(host(q.mul_mat_vec_f32(t, Wd, M, K, flat[1:].view(nc, K))), y_two)


@pytest.mark.parametrize("t", FUSED_TYPES)
@pytest.mark.parametrize("ncols", [1, 2])
def test_fused_gate_up_equals_two_step(q, t, ncols):
    M, K = 150, 2048
    Wg, Wu = weights(t, M, K, 1400), weights(t, M, K, 1401)
    x = synthetic.activations_f32(1402, ncols, K)
    Wgd, Wud, xd = dev(Wg), dev(Wu), dev(x)
    y_fused = host(q.mul_mat_vec_gate_up_swiglu_f32(t, Wgd, Wud, M, K, xd))
    y_two = host(q.mul_mat_vec_gate_up_swiglu(t, Wgd, Wud, M, K, q.quantize_q8_1(xd), ncols))
    assert np.array_equal(y_fused, y_two)


@pytest.mark.parametrize("t", FUSED_TYPES)
def test_fused_moe_equals_two_step(q, t):
    import torch

    E, M, K = 8, 77, 2048
    W = weights(t, E * M, K, 1500 + t).reshape(E, -1)
    for ids in (synthetic.moe_ids(1501, 4, 2, E), np.array([[1, 9], [-1, 2], [2, 1]], dtype=np.int32)):
        T = ids.shape[0]
        x = synthetic.activations_f32(1502, T, K)
        Wd, xd, idd = dev(W), dev(x), dev(ids)
        s1 = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        s2 = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        y_fused = host(q.mul_mat_vec_id_f32(t, Wd, E, M, K, xd, idd, status=s1))
        y_two = host(q.mul_mat_vec_id(t, Wd, E, M, K, q.quantize_q8_1(xd), idd, status=s2))
        assert np.array_equal(y_fused, y_two)
        assert int(host(s1)[0]) == int(host(s2)[0]) == int(((ids < 0) | (ids >= E)).sum())


def test_fused_rejects_what_it_does_not_cover(q):
    import torch

    x = torch.zeros((1, 2304), dtype=torch.float32, device="cuda")
    W6 = torch.zeros((4, q.row_bytes(q.Q6_K, 2304)), dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmvError) as e:
        q.mul_mat_vec_f32(q.Q6_K, W6, 4, 2304, x)
    assert e.value.status == 3
    x96 = torch.zeros((1, 96), dtype=torch.float32, device="cuda")
    W0 = torch.zeros((4, q.row_bytes(q.Q4_0, 96)), dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmvError) as e:
        q.mul_mat_vec_f32(q.Q4_0, W0, 4, 96, x96)
    assert e.value.status == 3


def test_fused_chain_reads_the_previous_kernels_output(q):
    """y2 = W2 . (W1 . x) with both GEMVs fused, chained on one stream with
    programmatic dependent launch and inside a CUDA graph: the second kernel
    quantizes an input the first one writes."""
    import torch

    t = oracle.Q4_K
    M1, K1, M2 = 1024, 2048, 512
    W1, W2 = weights(t, M1, K1, 1600), weights(t, M2, M1, 1601)
    x = synthetic.activations_f32(1602, 1, K1)
    W1d, W2d, xd = dev(W1), dev(W2), dev(x)
    q.set_pdl(False)
    y1 = q.mul_mat_vec_f32(t, W1d, M1, K1, xd)
    y_ref = host(q.mul_mat_vec_f32(t, W2d, M2, M1, y1))
    q.set_pdl(True)
    s = torch.cuda.Stream()
    h = torch.empty((1, M1), dtype=torch.float32, device="cuda")
    y = torch.empty((1, M2), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        q.mul_mat_vec_f32(t, W1d, M1, K1, xd, out=h, stream=s)
        q.mul_mat_vec_f32(t, W2d, M2, M1, h, out=y, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(4):
            q.mul_mat_vec_f32(t, W1d, M1, K1, xd, out=h, stream=s)
            q.mul_mat_vec_f32(t, W2d, M2, M1, h, out=y, stream=s)
    h.zero_()
    y.zero_()
    g.replay()
    assert np.array_equal(host(y), y_ref)


@pytest.mark.parametrize("cl", [1, 2, 8])
@pytest.mark.parametrize("t,M,K,ncols", [(oracle.Q4_0, 5, 256, 3), (oracle.Q4_K, 203, 2304, 1),
                                         (oracle.Q4_K, 3, 256, 8), (oracle.Q6_K, 77, 2048, 2)])
def test_fused_cluster_sizes_bitwise(q, cl, t, M, K, ncols):
    """The CTAs of a cluster share the quantization (each stores its blocks in
    every CTA's shared memory): any cluster size, including more CTAs than row
    groups and one q8_1 block per CTA, gives the two-step result bit for bit."""
    W = weights(t, M, K, 1700 + M)
    Wg = weights(t, M, K, 1701 + M)
    x = synthetic.activations_f32(1702 + K, ncols, K, outlier_frac=0.01)
    Wd, Wgd, xd = dev(W), dev(Wg), dev(x)
    y_two = host(q.mul_mat_vec(t, Wd, M, K, q.quantize_q8_1(xd), ncols))
    g_two = host(q.mul_mat_vec_gate_up_swiglu(t, Wgd, Wd, M, K, q.quantize_q8_1(xd), ncols))
    q.set_tuning(t, cluster=cl)
    try:
        assert np.array_equal(host(q.mul_mat_vec_f32(t, Wd, M, K, xd)), y_two)
        assert np.array_equal(host(q.mul_mat_vec_gate_up_swiglu_f32(t, Wgd, Wd, M, K, xd)), g_two)
    finally:
        q.set_tuning(t)
