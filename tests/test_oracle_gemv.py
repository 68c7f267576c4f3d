"""Pins for the oracle's GEMV, block formula and integer sums.

The block formula and the plain dequantize-then-dot are two independent
computations of the same result; they agree exactly in exact arithmetic for
Q4_K and Q6_K and for Q4_0 whenever the q8_1 field s equals d*sum(q)
exactly.  Brute force against numpy's matmul and integer sums recomputed from
decoded codes pin the rest.
"""
import numpy as np
import pytest

import oracle
import synthetic

TYPES = [oracle.Q4_0, oracle.Q4_K, oracle.Q6_K]


def _xq(seed, ncols, K, outliers=0.0):
    return oracle.quantize_q8_1(synthetic.activations_f32(seed, ncols, K, outlier_frac=outliers))


@pytest.mark.parametrize("t", [oracle.Q4_K, oracle.Q6_K])
def test_formula_equals_plain_dot_for_k_quants(t):
    M, K, nc = 12, 1024, 3
    for W in (oracle.random_blocks(t, M, K, seed=21),
              oracle.quantize_rows(t, synthetic.weights_f32(22, M, K))):
        xq = _xq(23, nc, K, 0.01)
        yp = oracle.gemv_plain(t, W, M, K, xq, nc)
        yf, l1 = oracle.gemv_formula(t, W, M, K, xq, nc)
        assert np.all(np.abs(yp - yf) <= 1e-12 * l1 + 1e-300)
        assert np.all(l1 >= np.abs(yf))


def _q8_1_with_exact_s(seed, ncols, K):
    """q8_1 blocks with d = 2^-7 and random codes whose |sum| < 2048, so that
    s = d*sum(q) is exactly a half and equals d8*sum(q)."""
    nb = oracle.q8_1_padded_k(K) // 32
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.integers(-60, 61, size=(ncols, nb, 32))
    q[:, K // 32:, :] = 0
    b = np.zeros((ncols, nb, 36), dtype=np.uint8)
    dbits = np.uint16(0x2000)  # 2^-7
    sums = q.sum(axis=2)
    sbits = oracle.f32_to_f16_bits((sums * 2.0**-7).astype(np.float32))
    b[..., 0] = dbits & 0xFF
    b[..., 1] = dbits >> 8
    b[..., 2] = sbits & 0xFF
    b[..., 3] = sbits >> 8
    b[..., 4:] = q.astype(np.int8).view(np.uint8)
    return b.reshape(ncols, nb * 36)


def test_q4_0_formula_equals_plain_when_s_is_exact():
    M, K, nc = 10, 512, 2
    W = oracle.random_blocks(oracle.Q4_0, M, K, seed=31)
    xq = _q8_1_with_exact_s(32, nc, K)
    yp = oracle.gemv_plain(oracle.Q4_0, W, M, K, xq, nc)
    yf, l1 = oracle.gemv_formula(oracle.Q4_0, W, M, K, xq, nc)
    assert np.all(np.abs(yp - yf) <= 1e-12 * l1)


def test_q4_0_formula_differs_from_plain_only_through_s():
    # with real q8_1 blocks the gap is 8*d4*(s - d8*sum q) summed over blocks
    M, K = 6, 512
    W = oracle.random_blocks(oracle.Q4_0, M, K, seed=33)
    xq = _xq(34, 1, K)
    yp = oracle.gemv_plain(oracle.Q4_0, W, M, K, xq, 1)[0]
    yf, l1 = oracle.gemv_formula(oracle.Q4_0, W, M, K, xq, 1)
    nb = K // 32
    xb = xq.reshape(-1, 36)[:nb]
    d8 = oracle.f16_bits_to_f32(xb[:, 0:2].copy().view(np.uint16)[:, 0]).astype(np.float64)
    s8 = oracle.f16_bits_to_f32(xb[:, 2:4].copy().view(np.uint16)[:, 0]).astype(np.float64)
    sq = xb[:, 4:].view(np.int8).astype(np.int64).sum(axis=1)
    wb = W.reshape(M, nb, 18)
    d4 = oracle.f16_bits_to_f32(wb[:, :, 0:2].copy().view(np.uint16)[..., 0]).astype(np.float64)
    gap = (8 * d4 * (s8 - d8 * sq)[None]).sum(axis=1)
    assert np.allclose(yp - yf[0], gap, rtol=0, atol=1e-12 * l1[0].max())


@pytest.mark.parametrize("t", TYPES)
def test_plain_dot_matches_numpy_matmul(t):
    M, K, nc = 4, 256, 2
    W = oracle.random_blocks(t, M, K, seed=41)
    xq = _xq(42, nc, K)
    Wd = oracle.dequantize_rows(t, W, K)
    Xd = oracle.dequantize_q8_1(xq, K)
    ref = Xd @ Wd.T
    y = oracle.gemv_plain(t, W, M, K, xq, nc)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-300)


def _unit_scale_blocks(t, M, K, seed):
    """Random codes with unit scales (d = 1, dmin = 0, every sub-block scale 1,
    min 0), so the decoded weight equals the stored code (minus its offset)."""
    W = oracle.random_blocks(t, M, K, seed)
    nb = K // oracle.block_elems(t)
    b = W.reshape(M, nb, oracle.block_bytes(t))
    if t == oracle.Q4_0:
        b[:, :, 0:2] = [0x00, 0x3C]
    elif t == oracle.Q4_K:
        b[:, :, 0:4] = [0x00, 0x3C, 0x00, 0x00]
        b[:, :, 4:16] = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]
    else:
        b[:, :, 192:208] = 1
        b[:, :, 208:210] = [0x00, 0x3C]
    return np.ascontiguousarray(b.reshape(M, -1))


@pytest.mark.parametrize("t", TYPES)
def test_subblock_sums_match_codes_times_activations(t):
    M, K, nc = 5, 512, 3
    W = _unit_scale_blocks(t, M, K, seed=51)
    codes = oracle.dequantize_rows(t, W, K)          # exact small integers
    if t == oracle.Q4_0:
        codes = codes + 8                           # the sums use the raw nibble
    assert np.array_equal(codes, np.round(codes))
    xq = _xq(52, nc, K, 0.01)
    nb = oracle.q8_1_padded_k(K) // 32
    qy = xq.reshape(nc, nb, 36)[:, :K // 32, 4:].view(np.int8).astype(np.int64).reshape(nc, K)
    sums = oracle.subblock_sums(t, W, M, K, xq, nc)
    prod = codes[None].astype(np.int64) * qy[:, None, :]      # [nc][M][K]
    if t == oracle.Q4_0:
        exp = prod.reshape(nc, M, K // 32, 32).sum(axis=3)
    elif t == oracle.Q4_K:
        dot1 = prod.reshape(nc, M, K // 32, 32).sum(axis=3)
        dot2 = np.broadcast_to(qy.reshape(nc, 1, K // 32, 32).sum(axis=3), dot1.shape)
        exp = np.stack([dot1, dot2], axis=3).reshape(nc, M, K // 16)
    else:
        exp = prod.reshape(nc, M, K // 16, 16).sum(axis=3)
    assert np.array_equal(sums, exp)


@pytest.mark.parametrize("t", TYPES)
def test_row_subset_and_threads_agree(t):
    M, K, nc = 37, 512, 2
    W = oracle.random_blocks(t, M, K, seed=61)
    xq = _xq(62, nc, K)
    y, l1 = oracle.gemv_formula(t, W, M, K, xq, nc)
    rows = [36, 0, 17, 17]
    ys, l1s = oracle.gemv_formula(t, W, M, K, xq, nc, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(l1s, l1[:, rows])
    ym, l1m = oracle.gemv_formula_mt(t, W, M, K, xq, nc, nthreads=3)
    assert np.array_equal(ym, y) and np.array_equal(l1m, l1)
    ss = oracle.subblock_sums(t, W, M, K, xq, nc, rows=rows)
    assert np.array_equal(ss, oracle.subblock_sums(t, W, M, K, xq, nc)[:, rows])


def test_dropping_the_min_term_is_detected():
    # a plausible mistake (ignoring dmin*m) moves the result by far more than 1e-4*L1
    M, K = 8, 512
    W = oracle.quantize_rows(oracle.Q4_K, synthetic.weights_f32(71, M, K))
    xq = _xq(72, 1, K)
    yf, l1 = oracle.gemv_formula(oracle.Q4_K, W, M, K, xq, 1)
    W0 = W.reshape(M, 2, 144).copy()
    W0[:, :, 2:4] = 0                                 # dmin = 0
    y0, _ = oracle.gemv_formula(oracle.Q4_K, W0.reshape(M, -1), M, K, xq, 1)
    assert np.all(np.abs(y0 - yf) > 1e-4 * l1)


def test_swiglu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert np.isclose(oracle.silu(1.0), 1.0 / (1.0 + np.exp(-1.0)))
    assert np.isclose(oracle.silu(-50.0), -50.0 * np.exp(-50.0), rtol=1e-12)
    assert np.isclose(oracle.silu(50.0), 50.0, rtol=1e-15)
    assert np.allclose(oracle.swiglu([2.0, -3.0], [0.5, 4.0]),
                       [0.5 * 2 / (1 + np.exp(-2.0)), 4.0 * -3 / (1 + np.exp(3.0))])


def test_moe_routes_each_slot_to_its_expert():
    E, M, K, T, k = 4, 9, 256, 3, 2
    W = oracle.random_blocks(oracle.Q4_K, E * M, K, seed=81).reshape(E, -1)
    xq = _xq(82, T, K)
    ids = np.array([[2, 0], [2, 2], [3, 9]], dtype=np.int32)   # repeated and invalid ids
    y, l1, bad = oracle.moe_gemv(oracle.Q4_K, W, E, M, K, xq, ids)
    assert bad == 1
    for tok in range(T):
        xt = xq[tok:tok + 1]
        for s in range(k):
            e = ids[tok, s]
            if e >= E:
                assert not y[tok, s].any()
            else:
                ye, _ = oracle.gemv_formula(oracle.Q4_K, W[e], M, K, xt, 1)
                assert np.array_equal(y[tok, s], ye[0])
    assert np.array_equal(y[1, 0], y[1, 1])


def test_fused_epilogue_closed_forms():
    up = np.array([[1.0, 2.0, -3.0], [0.25, -1.0, 4.0]])
    gate = np.array([[0.0, 50.0, -2.0], [3.0, -60.0, 1.0]])
    b = np.array([0.5, -2.0, 3.0])
    gb = np.array([-0.0, 1.0, 2.0])
    # no extras: identity; bias only: a plain row-wise add, the same for every column
    assert np.array_equal(oracle.fused_epilogue(up), up)
    assert np.array_equal(oracle.fused_epilogue(up, bias=b), [[1.5, 0.0, 0.0], [0.75, -3.0, 7.0]])
    # no biases: exactly the SwiGLU epilogue
    assert np.array_equal(oracle.fused_epilogue(up, gate), oracle.swiglu(gate, up))
    # the gate bias moves the gate argument: gate + gate_bias = 0 gives silu(0) = 0
    z = oracle.fused_epilogue(up, np.array([[-1.0, -1.0, -1.0]]), b, np.array([1.0, 1.0, 1.0]))
    assert z.shape == (2, 3) and not z.any()
    # a large gate passes (up + bias) through, scaled by the gate argument itself
    r = oracle.fused_epilogue(up[:1, 1:2], gate[:1, 1:2], b[1:2], gb[1:2])
    assert np.isclose(r[0, 0], (2.0 - 2.0) * 51.0, atol=1e-12)
    r = oracle.fused_epilogue(np.array([[3.0]]), np.array([[40.0]]), np.array([1.0]), np.array([2.0]))
    assert np.isclose(r[0, 0], 4.0 * 42.0 * (1.0 / (1.0 + np.exp(-42.0))), rtol=1e-15)
    # a dropped gate bias or up bias is detected
    full = oracle.fused_epilogue(up, gate, b, gb)
    assert not np.allclose(full, oracle.fused_epilogue(up, gate, b, None))
    assert not np.allclose(full, oracle.fused_epilogue(up, gate, None, gb))
    assert np.allclose(full, (up + b) * ((gate + gb) / (1.0 + np.exp(-(gate + gb)))))


def test_shared_expert_is_every_token_routed_to_one_matrix():
    M, K, T = 11, 512, 3
    Ws = oracle.random_blocks(oracle.Q4_K, M, K, seed=91)
    xq = _xq(92, T, K)
    ys, l1 = oracle.shared_expert_gemv(oracle.Q4_K, Ws, M, K, xq, T)
    # the same as routing every token to expert 0 of a one-expert set
    ym, lm, bad = oracle.moe_gemv(oracle.Q4_K, Ws, 1, M, K, xq, np.zeros((T, 1), dtype=np.int32))
    assert bad == 0 and np.array_equal(ys, ym[:, 0, :]) and np.array_equal(l1, lm[:, 0, :])
    # and, for a K-quant, the fp64 dequantize-then-dot of each token's column
    Wd = oracle.dequantize_rows(oracle.Q4_K, Ws, K).astype(np.float64)
    xd = oracle.dequantize_q8_1(xq, K).astype(np.float64)
    assert np.allclose(ys, xd @ Wd.T, rtol=1e-12, atol=1e-12 * np.abs(l1).max())


# ---- the fp32 integer-formula GEMV (the second CPU baseline) -------------------
@pytest.mark.parametrize("t", TYPES)
def test_int_f32_formula_within_fp32_rounding_of_the_fp64_formula(t):
    M, K, nc = 24, 2048, 3
    for W in (oracle.random_blocks(t, M, K, seed=71),
              oracle.quantize_rows(t, synthetic.weights_f32(72, M, K))):
        xq = _xq(73, nc, K, 0.01)
        y64, l1 = oracle.gemv_formula(t, W, M, K, xq, nc)
        y32 = oracle.gemv_int_f32(t, W, M, K, xq, nc).astype(np.float64)
        # per row: K/16 scaled terms, each with at most four fp32 roundings,
        # summed in fp32: |error| <= (4 + K/16) * 2^-24 * L1 (first order)
        assert np.all(np.abs(y32 - y64) <= (4 + K / 16) * 2.0**-24 * l1 + 1e-30)


def _integer_q8_1(seed, ncols, K):
    """q8_1 blocks with d = 1 and codes in [-7, 7] (|sum| < 2048, so s = sum(q)
    is an exact half): every block product is an exact small integer."""
    nb = oracle.q8_1_padded_k(K) // 32
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.integers(-7, 8, size=(ncols, nb, 32))
    q[:, K // 32:, :] = 0
    b = np.zeros((ncols, nb, 36), dtype=np.uint8)
    b[..., 0:2] = [0x00, 0x3C]
    sbits = oracle.f32_to_f16_bits(q.sum(axis=2).astype(np.float32))
    b[..., 2] = sbits & 0xFF
    b[..., 3] = sbits >> 8
    b[..., 4:] = q.astype(np.int8).view(np.uint8)
    return b.reshape(ncols, nb * 36)


@pytest.mark.parametrize("t", TYPES)
def test_int_f32_formula_exact_on_integer_cases(t):
    # unit scales and integer activations: y is an integer below 2^24, which
    # fp32 holds exactly, so both formulas must give the same value exactly
    M, K, nc = 9, 1024, 2
    W = _unit_scale_blocks(t, M, K, seed=74)
    xq = _integer_q8_1(75, nc, K)
    y64, _ = oracle.gemv_formula(t, W, M, K, xq, nc)
    assert np.array_equal(y64, np.round(y64)) and np.all(np.abs(y64) < 2**24)
    assert np.array_equal(oracle.gemv_int_f32(t, W, M, K, xq, nc).astype(np.float64), y64)


@pytest.mark.parametrize("t", TYPES)
def test_int_f32_threads_agree(t):
    M, K, nc = 37, 512, 2
    W = oracle.random_blocks(t, M, K, seed=76)
    xq = _xq(77, nc, K)
    y1 = oracle.gemv_int_f32(t, W, M, K, xq, nc, nthreads=1)
    assert np.array_equal(oracle.gemv_int_f32(t, W, M, K, xq, nc, nthreads=5), y1)
