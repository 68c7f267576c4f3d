"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: q8_1 bytes, weight-quantizer bytes and per-sub-block integer sums are
bit-exact; fp32 outputs are within 1e-4 of the L1 norm of each row's scaled
block terms (the oracle's fp64 block formula).  Sizes span several pipeline
slices and row groups with ragged tails; full-size cases check sampled rows.
"""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4


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


def assert_close_l1(y, y_ref, l1, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bad = err > TOL * l1
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs off; first {tuple(i)}: gpu={y[tuple(i)]!r} "
                             f"ref={y_ref[tuple(i)]!r} l1={l1[tuple(i)]!r}")


def weights(t, M, K, seed):
    return oracle.quantize_rows(t, synthetic.weights_f32(seed, M, K))


# ---- q8_1 -----------------------------------------------------------------
@pytest.mark.parametrize("K,ncols,outl", [(32, 1, 0.0), (40, 2, 0.0), (513, 1, 0.0), (4096, 3, 0.01),
                                          (11008, 1, 0.01), (14336, 2, 0.0)])
def test_q8_1_bit_exact(q, K, ncols, outl):
    x = synthetic.activations_f32(7 + K, ncols, K, outlier_frac=outl)
    got = host(q.quantize_q8_1(dev(x)))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


def test_q8_1_bit_exact_special_values(q):
    K = 512
    x = np.zeros((6, K), dtype=np.float32)
    x[1] = 3.0                                               # constant
    x[2, :32] = np.arange(32) - 15.5                         # halfway cases at d = 1
    x[2, 0] = 127.0
    x[3, :8] = [1e-45, -2e-45, 3e-45, 1e-44, 0, 0, 0, 0]       # subnormal block
    x[4, :64] = synthetic.normal_f32(3, 64) * np.float32(1e-39)  # mixed subnormal / tiny normal
    x[5] = synthetic.normal_f32(4, K) * np.float32(1e30)     # huge
    got = host(q.quantize_q8_1(dev(x)))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


def test_q8_1_bit_exact_near_halfway_quotients(q):
    """Codes decided by the correctly rounded fp32 quotient x/d: values at and
    one ulp around (k + 0.5) * d for scales d that are not powers of two, and
    blocks with d near and beyond both ends of the fast-division range."""
    rng = np.random.default_rng(2024)
    nb = 2048
    x = np.zeros((nb, 32), dtype=np.float32)
    for b in range(nb):
        if b % 8 == 7:
            c = np.float32(2.0 ** rng.choice([-41, -40, -39, 39, 40, 41, -70, 70])) * np.float32(rng.uniform(0.6, 1.4))
        else:
            c = np.float32(10.0 ** rng.uniform(-6, 6))
        amax = np.float32(127) * c
        d = np.float32(amax) / np.float32(127)  # the quantizer's scale (IEEE division)
        x[b, 0] = amax
        k = rng.integers(-126, 126, size=31).astype(np.float32)
        v = (k + np.float32(0.5)) * d
        step = rng.integers(-1, 2, size=31)
        v = np.where(step > 0, np.nextafter(v, np.float32(np.inf)), np.where(step < 0, np.nextafter(v, np.float32(-np.inf)), v))
        x[b, 1:] = np.clip(v, -amax, amax).astype(np.float32)
    x = x.reshape(8, -1)  # 8 columns of 8192 values
    got = host(q.quantize_q8_1(dev(x)))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


# ---- weight quantizers ---------------------------------------------------------
@pytest.mark.parametrize("t,K", [(oracle.Q4_0, 96), (oracle.Q4_0, 4096), (oracle.Q4_K, 512), (oracle.Q4_K, 4096),
                                 (oracle.Q6_K, 768), (oracle.Q6_K, 4096)])
def test_weight_quantizer_bit_exact(q, t, K):
    M = 37
    w = synthetic.weights_f32(11 + K, M, K)
    w[0] = 0.0
    w[1] = 0.125
    w[2] = np.abs(w[2]) + 0.01
    w[3, : K // 2] *= 50.0
    w[4] = synthetic.normal_f32(5, K) * np.float32(1e-6)
    got = host(q.quantize_weights(t, dev(w)))
    assert np.array_equal(got, oracle.quantize_rows(t, w))


# ---- GEMV ------------------------------------------------------------------------
SHAPES = {
    oracle.Q4_0: [(203, 4096), (203, 96), (61, 256)],        # streaming, generic (K % 256), one unit
    oracle.Q4_K: [(203, 4096), (203, 2304), (61, 256)],      # 16 units, 9 units (ragged slice), 1 unit
    oracle.Q6_K: [(203, 4096), (61, 2048), (203, 512)],      # 2 units, 1 unit, generic (K % 2048)
}


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
@pytest.mark.parametrize("ncols", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemv_parity(q, t, ncols):
    for si, (M, K) in enumerate(SHAPES[t]):
        W = weights(t, M, K, 100 * t + si)
        x = synthetic.activations_f32(200 + ncols + si, ncols, K, outlier_frac=0.01)
        xq = oracle.quantize_q8_1(x)
        y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, ncols)
        y = host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), ncols))
        assert_close_l1(y, y_ref, l1, f"type {t} M={M} K={K} ncols={ncols}")


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
def test_gemv_random_blocks(q, t):
    # every code, every 6-bit scale/min and negative Q6_K scales
    for M, K in SHAPES[t]:
        W = oracle.random_blocks(t, M, K, seed=300 + K)
        for ncols in (1, 3):
            xq = oracle.quantize_q8_1(synthetic.activations_f32(301 + K, ncols, K))
            y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, ncols)
            y = host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), ncols))
            assert_close_l1(y, y_ref, l1, f"random type {t} K={K} ncols={ncols}")


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
@pytest.mark.parametrize("ncols", [1, 3, 8])
def test_subblock_sums_bit_exact(q, t, ncols):
    for si, (M, K) in enumerate(SHAPES[t]):
        W = oracle.random_blocks(t, M, K, seed=400 + si)
        xq = oracle.quantize_q8_1(synthetic.activations_f32(401 + si, ncols, K, outlier_frac=0.01))
        got = host(q.debug_subblock_sums(t, dev(W), M, K, dev(xq), ncols))
        assert np.array_equal(got, oracle.subblock_sums(t, W, M, K, xq, ncols)), (t, M, K, ncols)


def test_gemv_edge_shapes(q):
    # a single row; a single block; M = 1..9 around the row-group size
    for t in oracle.WEIGHT_TYPES:
        K = 256 if t != oracle.Q6_K else 2048
        for M in (1, 2, 3, 4, 5, 7, 8, 9):
            W = weights(t, M, K, 500 + M)
            xq = oracle.quantize_q8_1(synthetic.activations_f32(501, 2, K))
            y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, 2)
            y = host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), 2))
            assert_close_l1(y, y_ref, l1, f"type {t} M={M}")


def test_gemv_minimum_k(q):
    # K at one block of the format (Q4_0: 32, K-quants: one 256-weight super-block)
    for t, K in ((oracle.Q4_0, 32), (oracle.Q4_K, 256), (oracle.Q6_K, 256)):
        for M, ncols in ((5, 1), (37, 3)):
            W = weights(t, M, K, 550 + K + M)
            xq = oracle.quantize_q8_1(synthetic.activations_f32(551 + M, ncols, K))
            y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, ncols)
            y = host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), ncols))
            assert_close_l1(y, y_ref, l1, f"type {t} K={K} M={M} ncols={ncols}")


def test_zero_weights_and_activations_give_exact_zeros(q):
    for t in oracle.WEIGHT_TYPES:
        M, K = 33, 2048
        W = oracle.quantize_rows(t, np.zeros((M, K), dtype=np.float32))
        xq = oracle.quantize_q8_1(synthetic.activations_f32(1, 1, K))
        assert not host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), 1)).any()
        W = weights(t, M, K, 2)
        xq = oracle.quantize_q8_1(np.zeros((1, K), dtype=np.float32))
        assert not host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), 1)).any()


def test_generic_path_for_unaligned_weights(q):
    import torch

    for t in oracle.WEIGHT_TYPES:
        M, K = 45, 4096
        W = weights(t, M, K, 600 + t)
        xq = oracle.quantize_q8_1(synthetic.activations_f32(601, 2, K))
        y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, 2)
        buf = torch.zeros(W.size + 16, dtype=torch.uint8, device="cuda")
        buf[2:2 + W.size] = dev(W.reshape(-1))
        y = host(q.mul_mat_vec(t, buf[2:], M, K, dev(xq), 2))   # 2-byte aligned only
        assert_close_l1(y, y_ref, l1, f"unaligned type {t}")


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
@pytest.mark.parametrize("nc", [1, 3])
def test_tuning_variants_agree(q, t, nc):
    # geometry overrides (threads, units per tile row / slice, stages, CTAs per
    # SM, shared-memory share) change the launch, never the result
    M, K = 130, 4096
    W = weights(t, M, K, 700 + t)
    xq = oracle.quantize_q8_1(synthetic.activations_f32(701, nc, K))
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, nc)
    Wd, xd = dev(W), dev(xq)
    try:
        for tune in [(32, 1, 1, 1, 1), (64, 2, 3, 0, 2), (256, 8, 2, 0, 1), (128, 3, 6, 2, 0), (96, 16, 4, 0, 2),
                     (128, 4, 2, 3, 1), (384, 16, 1, 1, 4), (384, 4, 4, 2, 1), (256, 16, 3, 0, 0)]:
            q.set_tuning(t, *tune)
            y = host(q.mul_mat_vec(t, Wd, M, K, xd, nc))
            assert_close_l1(y, y_ref, l1, f"type {t} ncols {nc} tuning {tune}")
    finally:
        q.set_tuning(t)


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
def test_stream_tuning_variants_agree(q, t):
    # decoding warps and tiles requested before the dependency wait change the
    # launch, never the result (bitwise: rows never change warps' arithmetic order)
    M, K, nc = 517, 4096, 2
    W = weights(t, M, K, 710 + t)
    xq = oracle.quantize_q8_1(synthetic.activations_f32(711, nc, K))
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, nc)
    Wd, xd = dev(W), dev(xq)
    y0 = host(q.mul_mat_vec(t, Wd, M, K, xd, nc))
    assert_close_l1(y0, y_ref, l1, f"type {t} default")
    try:
        for dw, pre, st in [(1, 1, 2), (3, 1, 1), (5, 2, 2), (12, 1, 4), (7, 3, 3), (2, 4, 4)]:
            q.set_tuning(t, stages=st)
            q.set_stream_tuning(t, dec_warps=dw, pre_tiles=pre)
            y = host(q.mul_mat_vec(t, Wd, M, K, xd, nc))
            assert_close_l1(y, y_ref, l1, f"type {t} dec_warps {dw} pre {pre} stages {st}")
    finally:
        q.set_tuning(t)
        q.set_stream_tuning(t)



@pytest.mark.parametrize("t", [oracle.Q4_0, oracle.Q4_K])
def test_early_delay_changes_nothing(q, t):
    # a 4096x4096 launch requests its whole matrix before the dependency wait,
    # which the planner holds back by a short delay; no delay, the default and
    # a long one give bitwise-equal results, q8_1 and fp32 input alike
    M, K = 4096, 4096
    W = weights(t, M, K, 720 + t)
    x = synthetic.activations_f32(721, 1, K)
    xq = oracle.quantize_q8_1(x)
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, 1)
    Wd, xd, xfd = dev(W), dev(xq), dev(x)
    y0 = host(q.mul_mat_vec(t, Wd, M, K, xd, 1))
    assert_close_l1(y0, y_ref, l1, f"type {t} default delay")
    try:
        for ns in (-1, 5000, 0):
            q.set_early_delay(t, ns)
            assert np.array_equal(host(q.mul_mat_vec(t, Wd, M, K, xd, 1)), y0), f"type {t} delay {ns}"
            assert np.array_equal(host(q.mul_mat_vec_f32(t, Wd, M, K, xfd)), y0), f"type {t} delay {ns} fp32"
    finally:
        q.set_early_delay(t, 0)

# ---- fused gate/up + SwiGLU ------------------------------------------------------
def _swiglu_tol(g, u, l1g, l1u):
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    out = u * g * sig
    return np.abs(u) * np.abs(dsilu) * TOL * l1g + np.abs(g * sig) * TOL * l1u + 4e-7 * np.abs(out) + 1e-30


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
@pytest.mark.parametrize("ncols", [1, 2, 5])
def test_gate_up_swiglu_parity(q, t, ncols):
    M, K = 203, 4096 if t != oracle.Q4_0 else 1024
    Wg = weights(t, M, K, 800 + t)
    Wu = weights(t, M, K, 810 + t)
    xq = oracle.quantize_q8_1(synthetic.activations_f32(802, ncols, K))
    g, l1g = oracle.gemv_formula(t, Wg, M, K, xq, ncols)
    u, l1u = oracle.gemv_formula(t, Wu, M, K, xq, ncols)
    ref = oracle.swiglu(g, u)
    y = host(q.mul_mat_vec_gate_up_swiglu(t, dev(Wg), dev(Wu), M, K, dev(xq), ncols))
    err = np.abs(y.astype(np.float64) - ref)
    assert np.all(err <= _swiglu_tol(g, u, l1g, l1u)), err.max()


def test_gate_up_swiglu_generic_path(q):
    t, M, K = oracle.Q6_K, 70, 768
    Wg, Wu = weights(t, M, K, 820), weights(t, M, K, 821)
    xq = oracle.quantize_q8_1(synthetic.activations_f32(822, 1, K))
    g, l1g = oracle.gemv_formula(t, Wg, M, K, xq, 1)
    u, l1u = oracle.gemv_formula(t, Wu, M, K, xq, 1)
    y = host(q.mul_mat_vec_gate_up_swiglu(t, dev(Wg), dev(Wu), M, K, dev(xq), 1))
    assert np.all(np.abs(y - oracle.swiglu(g, u)) <= _swiglu_tol(g, u, l1g, l1u))


# ---- MoE ---------------------------------------------------------------------------
def _moe_case(q, t, E, M, K, ids, seed):
    import torch

    W = weights(t, E * M, K, seed).reshape(E, -1)
    T = ids.shape[0]
    xq = oracle.quantize_q8_1(synthetic.activations_f32(seed + 1, T, K))
    y_ref, l1, bad = oracle.moe_gemv(t, W, E, M, K, xq, ids)
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    y = host(q.mul_mat_vec_id(t, dev(W), E, M, K, dev(xq), dev(ids), status=status))
    assert_close_l1(y, y_ref, l1, f"moe type {t} ids {ids.tolist()}")
    assert int(host(status)[0]) == bad
    return y


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
def test_moe_parity_seeded_routing(q, t):
    K = 2048 if t == oracle.Q6_K else 1024
    ids = synthetic.moe_ids(900 + t, 4, 2, 8)
    _moe_case(q, t, 8, 203, K, ids, 910 + t)


def test_moe_edge_routings(q):
    t, E, M, K = oracle.Q4_K, 8, 77, 512
    _moe_case(q, t, E, M, K, np.array([[3, 3], [3, 3], [3, 3]], dtype=np.int32), 920)     # one expert for all
    _moe_case(q, t, E, M, K, np.array([[0, 7]], dtype=np.int32), 921)                     # one token
    y = _moe_case(q, t, E, M, K, np.array([[1, 9], [-1, 2], [2, 1]], dtype=np.int32), 922)  # invalid ids
    assert not y[0, 1].any() and not y[1, 0].any()
    ids8 = synthetic.moe_ids(923, 8, 4, E)
    _moe_case(q, t, E, M, K, ids8, 924)                                                   # 8 tokens, top-4
    _moe_case(q, oracle.Q6_K, E, M, 768, np.array([[0, 5], [5, 6]], dtype=np.int32), 925)  # generic path


# ---- execution modes --------------------------------------------------------------
def test_graph_capture_and_pdl_modes_agree(q):
    import torch

    t, M, K = oracle.Q4_K, 1000, 4096
    W = weights(t, M, K, 1000)
    x = synthetic.activations_f32(1001, 1, K)
    xq_ref = oracle.quantize_q8_1(x)
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq_ref, 1)
    Wd, xd = dev(W), dev(x)
    outs = []
    for pdl in (False, True):
        q.set_pdl(pdl)
        xq = q.quantize_q8_1(xd)
        outs.append(host(q.mul_mat_vec(t, Wd, M, K, xq, 1)))
    q.set_pdl(True)
    s = torch.cuda.Stream()
    xq = torch.empty((1, q.q8_1_bytes(K)), dtype=torch.uint8, device="cuda")
    y = torch.empty((1, M), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        q.quantize_q8_1(xd, out=xq)
        q.mul_mat_vec(t, Wd, M, K, xq, 1, out=y)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            q.quantize_q8_1(xd, out=xq)
            q.mul_mat_vec(t, Wd, M, K, xq, 1, out=y)
    y.zero_()
    g.replay()
    outs.append(host(y))
    for o in outs:
        assert_close_l1(o, y_ref, l1, "mode")
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_no_device_fault_recorded(q):
    assert q.device_fault() == 0
