"""GPU parity of the GEMV whose result is also written as q8_1 blocks
(qmv_mul_mat_vec_fused_q8_1), through the C ABI.

The q8_1 blocks are an integer encoding decided in fp32, so both sides take
the decision on the same floats: the blocks must equal, byte for byte, the
oracle's q8_1 quantization (mul_mat_vec_q page, section "激活的量化") of the
fp32 y that the GPU computes; that y must equal the fp32 result of
qmv_mul_mat_vec_fused bit for bit, and the ordinary fused call is already
held to the oracle's block formula within 1e-4 of each row's L1 norm.
Shapes cover a partial last block (M not a multiple of 32), fewer blocks than
CTAs, the 512-padding blocks, every format, plain and gate/up, q8_1 and fp32
activations, and the biases.
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
        qq.set_stream_tuning(t)
    return qq


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


def weights(t, M, K, seed):
    return oracle.quantize_rows(t, synthetic.weights_f32(seed, M, K))


def k_for(t):
    return 2048 if t == oracle.Q6_K else 1024


CASES = [(t, M, gate, f32) for t in oracle.WEIGHT_TYPES for M in (7, 1000, 4096 + 40)
         for gate in (False, True) for f32 in (False, True)]


@pytest.mark.parametrize("t,M,gate,f32", CASES,
                         ids=[f"t{c[0]}-M{c[1]}-{'gate' if c[2] else 'plain'}-{'f32' if c[3] else 'q8'}" for c in CASES])
def test_q8_1_output_matches_the_quantized_result(q, t, M, gate, f32):
    K = k_for(t)
    Wu = weights(t, M, K, 900 + t)
    Wg = weights(t, M, K, 910 + t) if gate else None
    x = synthetic.activations_f32(920 + M, 1, K, outlier_frac=0.01)
    xq = oracle.quantize_q8_1(x)
    act = {"x": dev(x)} if f32 else {"xq": dev(xq)}
    Wud, Wgd = dev(Wu), (dev(Wg) if gate else None)
    y_ref = host(q.mul_mat_vec_fused(t, Wud, M, K, W_gate=Wgd, **act))
    y, yq = q.mul_mat_vec_fused_q8_1(t, Wud, M, K, W_gate=Wgd, **act)
    y, yq = host(y), host(yq)
    assert np.array_equal(y, y_ref), "y equals the fused call's bit for bit"
    assert np.array_equal(yq, oracle.quantize_q8_1(y_ref)), "q8_1 blocks of y, byte for byte"
    # y itself against the oracle's block formula (the fused call's bound)
    if gate:
        g, l1g = oracle.gemv_formula(t, Wg, M, K, xq, 1)
        u, l1u = oracle.gemv_formula(t, Wu, M, K, xq, 1)
        ref = oracle.swiglu(g, u)
        sig = 1.0 / (1.0 + np.exp(-g))
        tol = (np.abs(u) * np.abs(sig * (1.0 + g * (1.0 - sig))) * TOL * l1g + np.abs(g * sig) * TOL * l1u
               + 4e-7 * np.abs(ref) + 1e-30)
    else:
        ref, l1 = oracle.gemv_formula(t, Wu, M, K, xq, 1)
        tol = TOL * l1 + 1e-30
    assert np.all(np.abs(y.astype(np.float64) - ref) <= tol)


@pytest.mark.parametrize("f32", [False, True])
def test_step_shape_with_biases_and_without_fp32_output(q, f32):
    # the decode step's gate/up launch (2 x 11008 x 4096, Q4_K), biases on, y
    # not written: the blocks still equal the quantized fused result, and the
    # down projection reading them equals the one reading quantize_q8_1(y)
    t, M, K = oracle.Q4_K, 11008, 4096
    Wu, Wg = weights(t, M, K, 930), weights(t, M, K, 931)
    x = synthetic.activations_f32(932, 1, K, outlier_frac=0.01)
    b = (0.5 * synthetic.activations_f32(933, 1, M)[0]).astype(np.float32)
    gb = (0.5 * synthetic.activations_f32(934, 1, M)[0]).astype(np.float32)
    act = {"x": dev(x)} if f32 else {"xq": dev(oracle.quantize_q8_1(x))}
    Wud, Wgd, bd, gbd = dev(Wu), dev(Wg), dev(b), dev(gb)
    y_ref = q.mul_mat_vec_fused(t, Wud, M, K, W_gate=Wgd, bias=bd, gate_bias=gbd, **act)
    y, yq = q.mul_mat_vec_fused_q8_1(t, Wud, M, K, W_gate=Wgd, bias=bd, gate_bias=gbd, want_y=False, **act)
    assert y is None
    assert np.array_equal(host(yq), oracle.quantize_q8_1(host(y_ref)))
    Wd = dev(weights(t, 4096, M, 935))
    d1 = host(q.mul_mat_vec(t, Wd, 4096, M, yq, 1))
    d2 = host(q.mul_mat_vec(t, Wd, 4096, M, q.quantize_q8_1(y_ref), 1))
    assert np.array_equal(d1, d2)


def test_two_calls_in_a_row_and_argument_errors(q):
    import torch

    t, M, K = oracle.Q4_K, 1000, 1024
    Wd = dev(weights(t, M, K, 940))
    xs = [synthetic.activations_f32(941 + i, 1, K) for i in range(2)]
    yqs = []
    for x in xs:
        y, yq = q.mul_mat_vec_fused_q8_1(t, Wd, M, K, x=dev(x))
        yqs.append((host(y), host(yq)))
    for y, yq in yqs:
        assert np.array_equal(yq, oracle.quantize_q8_1(y))
    with pytest.raises(ValueError):
        q.mul_mat_vec_fused_q8_1(t, Wd, M, K, x=dev(np.concatenate(xs)))  # two columns
    with pytest.raises(ValueError):
        q.mul_mat_vec_fused_q8_1(t, Wd, M, K, x=dev(xs[0]),
                                 out_q8_1=torch.empty(q.q8_1_bytes(M) - 1, dtype=torch.uint8, device="cuda"))
