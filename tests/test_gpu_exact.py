"""Exact-integer pins of the default (dp4a) decode for every format, through
the C ABI (mul_mat_vec_q page, "一次 vec_dot 的解剖": the block products).

With unit block scales (d = 1, and the K-quants' sub-block scales small
integers) and integer activations that quantize with d8 = 1 (each 32-value
block holds a +-127, the rest small), every block product, every partial sum
and y itself are integers below 2^24: the kernels' fp32 scaling must then
return the oracle's value bit for bit, on the tile kernel and the generic
kernel, from q8_1 and from fp32 input.  Q4_0 also needs the stored half
s = d8 * sum(q) exact, so the block sums stay within +-2048.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


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
        qq.set_mma_min_cols(t, 0)
    return qq


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


ONE = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)


def q4_0_rows(M, K, rng):
    """d = 1, random 4-bit codes: weights q - 8 in [-8, 7]."""
    blk = np.zeros((M, K // 32, 18), dtype=np.uint8)
    blk[:, :, 0:2] = ONE
    blk[:, :, 2:] = rng.integers(0, 256, size=(M, K // 32, 16), dtype=np.uint8)
    return blk.reshape(M, -1)


def q6_K_rows(M, K, rng):
    """d = 1, int8 sub-block scales in -3..3, random 6-bit codes (ql, qh)."""
    blk = np.zeros((M, K // 256, 210), dtype=np.uint8)
    blk[:, :, 0:192] = rng.integers(0, 256, size=(M, K // 256, 192), dtype=np.uint8)
    blk[:, :, 192:208] = rng.integers(-3, 4, size=(M, K // 256, 16)).astype(np.int8).view(np.uint8)
    blk[:, :, 208:210] = ONE
    return blk.reshape(M, -1)


def small_integer_activations(ncols, K, rng):
    """Integers in [-50, 50] with one +-127 per 32-value block: q8_1 gives
    d8 = 1, codes equal to the values, and |block sum| <= 127 + 31 * 50."""
    x = rng.integers(-50, 51, size=(ncols, K)).astype(np.float32)
    pos = rng.integers(0, 32, size=(ncols, K // 32))
    sign = np.where(rng.random((ncols, K // 32)) < 0.5, -127.0, 127.0).astype(np.float32)
    for c in range(ncols):
        x[c, np.arange(K // 32) * 32 + pos[c]] = sign[c]
    return x


# (type, M, K, rows builder, fp32 input possible): the tile kernel (Q4_0 K %
# 256 == 0, Q6_K K % 2048 == 0) and the generic kernel (other K)
CASES = [(oracle.Q4_0, 77, 1024, q4_0_rows, True), (oracle.Q4_0, 45, 96, q4_0_rows, False),
         (oracle.Q6_K, 61, 2048, q6_K_rows, True), (oracle.Q6_K, 29, 768, q6_K_rows, False)]


@pytest.mark.parametrize("t,M,K,rows,f32", CASES, ids=["q4_0-tile", "q4_0-generic", "q6_K-tile", "q6_K-generic"])
@pytest.mark.parametrize("ncols", [1, 3, 8])
def test_exact_integer_results(q, t, M, K, rows, f32, ncols):
    rng = np.random.default_rng(7000 + t * 10 + ncols)
    W = rows(M, K, rng)
    x = small_integer_activations(ncols, K, rng)
    xq = oracle.quantize_q8_1(x)
    assert np.array_equal(oracle.dequantize_q8_1(xq, K)[:, :K], x)
    w = oracle.dequantize_rows(t, W, K)
    assert np.array_equal(w, np.round(w))  # integer weights
    y_ref, _ = oracle.gemv_formula(t, W, M, K, xq, ncols)
    assert np.array_equal(y_ref, x.astype(np.float64) @ w.T)  # the block formula is the plain dot here
    assert np.all(np.abs(y_ref) < 2 ** 24)
    want = y_ref.astype(np.float32)
    Wd = dev(W)
    assert np.array_equal(host(q.mul_mat_vec(t, Wd, M, K, dev(xq), ncols)), want)
    if f32:
        assert np.array_equal(host(q.mul_mat_vec_f32(t, Wd, M, K, dev(x))), want)


@pytest.mark.parametrize("f32", [False, True], ids=["q8_1", "f32"])
def test_exact_integer_moe(q, f32):
    """The expert-indexed GEMV with integer experts: every valid slot is the
    exact integer W[ids[t][k]] x_t, a repeated expert serves its tokens in one
    pass, and an out-of-range id leaves its slot zero."""
    import torch

    t, E, M, K = oracle.Q4_0, 6, 33, 1024
    rng = np.random.default_rng(7100)
    W = q4_0_rows(E * M, K, rng).reshape(E, -1)
    ids = np.array([[2, 5], [2, 0], [7, 2], [5, 4]], dtype=np.int32)  # expert 2 three times; 7 is invalid
    T = ids.shape[0]
    x = small_integer_activations(T, K, rng)
    xq = oracle.quantize_q8_1(x)
    y_ref, _, bad = oracle.moe_gemv(t, W, E, M, K, xq, ids)
    assert bad == 1 and np.all(np.abs(y_ref) < 2 ** 24) and np.array_equal(y_ref, np.round(y_ref))
    w = oracle.dequantize_rows(t, W.reshape(E * M, -1), K).reshape(E, M, K)
    for tok in range(T):
        for k in range(2):
            e = ids[tok, k]
            exp = x[tok].astype(np.float64) @ w[e].T if e < E else np.zeros(M)
            assert np.array_equal(y_ref[tok, k], exp)
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    if f32:
        y = host(q.mul_mat_vec_id_f32(t, dev(W), E, M, K, dev(x), dev(ids), status=status))
    else:
        y = host(q.mul_mat_vec_id(t, dev(W), E, M, K, dev(xq), dev(ids), status=status))
    assert int(host(status)[0]) == 1
    assert np.array_equal(y, y_ref.astype(np.float32))


@pytest.mark.parametrize("f32", [False, True], ids=["q8_1", "f32"])
def test_exact_integer_fused_extras(q, f32):
    """The fused call's up bias and the MoE shared expert on integer data:
    y = W x + b and y_shared = W_shared x_t exactly."""
    import torch

    t, M, K, nc = oracle.Q4_0, 71, 1024, 3
    rng = np.random.default_rng(7200)
    W = q4_0_rows(M, K, rng)
    b = rng.integers(-1000, 1001, size=M).astype(np.float32)
    x = small_integer_activations(nc, K, rng)
    xq = oracle.quantize_q8_1(x)
    w = oracle.dequantize_rows(t, W, K)
    want = (x.astype(np.float64) @ w.T + b).astype(np.float32)
    kw = {"x": dev(x)} if f32 else {"xq": dev(xq)}
    assert np.array_equal(host(q.mul_mat_vec_fused(t, dev(W), M, K, bias=dev(b), **kw)), want)
    # MoE with a shared expert: the routed slots and the shared output, all exact
    E = 4
    We = q4_0_rows(E * M, K, rng).reshape(E, -1)
    Ws = q4_0_rows(M, K, rng)
    ids = np.array([[1, 3], [0, 1], [2, 2]], dtype=np.int32)
    T = ids.shape[0]
    xt = small_integer_activations(T, K, rng)
    xtq = oracle.quantize_q8_1(xt)
    kw = {"x": dev(xt)} if f32 else {"xq": dev(xtq)}
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    y, ys = q.mul_mat_vec_id_fused(t, dev(We), E, M, K, dev(ids), W_shared=dev(Ws), status=status, **kw)
    we = oracle.dequantize_rows(t, We.reshape(E * M, -1), K).reshape(E, M, K)
    ws = oracle.dequantize_rows(t, Ws, K)
    want_y = np.stack([np.stack([xt[i].astype(np.float64) @ we[ids[i, k]].T for k in range(2)]) for i in range(T)])
    assert int(host(status)[0]) == 0
    assert np.array_equal(host(y), want_y.astype(np.float32))
    assert np.array_equal(host(ys), (xt.astype(np.float64) @ ws.T).astype(np.float32))
