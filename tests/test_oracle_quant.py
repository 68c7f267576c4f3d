"""Pins for the oracle's quantizers (q8_1, Q4_0, Q4_K, Q6_K).

Checked against: the printed q8_1 kernel on a hand-worked block; closed forms
(inputs that are exact multiples of the scale quantize to known codes);
round-trip error bounds derived from the quantization rule; and brute force
(each stored code is the nearest representable one given the block's stored
scales).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synthetic

from conftest import GOLDEN

F32 = np.float32


def _fields_q8_1(xq, K):
    nb = oracle.q8_1_padded_k(K) // 32
    b = xq.reshape(-1, nb, 36)
    d = oracle.f16_bits_to_f32(b[..., 0:2].copy().view(np.uint16)[..., 0])
    s = oracle.f16_bits_to_f32(b[..., 2:4].copy().view(np.uint16)[..., 0])
    q = b[..., 4:].view(np.int8).astype(np.int64)
    return d, s, q


# ---- q8_1 ------------------------------------------------------------------
def test_q8_1_hand_block():
    g = json.load(open(os.path.join(GOLDEN, "q8_1_block.json")))
    xq = oracle.quantize_q8_1(np.asarray([g["x"]], dtype=F32))
    # K = 32 pads to 512: the first block is the fixture, the other 15 are zero
    assert xq.shape == (1, 16 * 36)
    assert xq[0, :36].tobytes().hex() == g["block_hex"]
    assert not xq[0, 36:].any()


def test_q8_1_integer_inputs_with_unit_scale():
    # amax = 127 makes d exactly 1, so integer inputs quantize to themselves
    rng = np.random.Generator(np.random.PCG64(5))
    x = rng.integers(-127, 128, size=(3, 512)).astype(F32)
    x[:, ::32] = 127.0
    d, s, q = _fields_q8_1(oracle.quantize_q8_1(x), 512)
    assert np.all(d == 1.0)
    assert np.array_equal(q.reshape(3, 512), x.astype(np.int64))


def test_q8_1_half_way_cases_round_away_from_zero():
    x = np.zeros((1, 32), dtype=F32)
    x[0, 0] = 127.0
    x[0, 1:9] = [0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 0.4999999, -126.5]
    _, _, q = _fields_q8_1(oracle.quantize_q8_1(x), 32)
    assert q[0, 0, :9].tolist() == [127, 1, -1, 2, -2, 3, -3, 0, -127]


def test_q8_1_zero_constant_and_padding():
    K = 40
    x = np.zeros((2, K), dtype=F32)
    x[1, :] = 3.0
    d, s, q = _fields_q8_1(oracle.quantize_q8_1(x), K)
    assert np.all(d[0] == 0) and np.all(s[0] == 0) and not q[0].any()
    # constant column: every real value maps to 127; tail of block 1 and blocks 2.. are zero
    assert np.all(q[1, 0] == 127) and np.all(q[1, 1, :8] == 127) and not q[1, 1, 8:].any()
    assert not q[1, 2:].any() and np.all(d[1, 2:] == 0)
    assert d[1, 0] == np.float32(np.float16(F32(3.0) / F32(127.0)))


def test_q8_1_subnormal_block_quantizes_to_zero():
    x = np.zeros((1, 32), dtype=F32)
    x[0, :4] = [1e-45, -2e-45, 3e-45, 0.0]   # amax/127 underflows to 0
    d, s, q = _fields_q8_1(oracle.quantize_q8_1(x), 32)
    assert d[0, 0] == 0 and s[0, 0] == 0 and not q.any()


def test_q8_1_error_bound_and_sum_field():
    x = synthetic.activations_f32(1, 4, 4096, outlier_frac=0.01)
    d, s, q = _fields_q8_1(oracle.quantize_q8_1(x), 4096)
    xb = x.reshape(4, 128, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    d32 = (amax.astype(F32) / F32(127)).astype(np.float64)
    err = np.abs(xb - d[..., None].astype(np.float64) * q)
    bound = d32 * (0.5 + 1e-5) + 127 * np.abs(d32 - d) + 1e-12
    assert np.all(err <= bound[..., None])
    assert np.all(np.abs(q) <= 127)
    # s holds d * sum(q) to half precision (relative 2^-11)
    sref = d32 * q.sum(axis=2)
    assert np.all(np.abs(s - sref) <= (2.0**-11 + 2.0**-23) * np.abs(sref) + 2.0**-25)


# ---- Q4_0 ------------------------------------------------------------------
def test_q4_0_integer_closed_form():
    # amax = 7 gives scale 1: integers in [-7, 7] store as value + 8
    rng = np.random.Generator(np.random.PCG64(9))
    v = rng.integers(-7, 8, size=(4, 64)).astype(F32)
    v[:, 0] = 7.0
    v[:, 32] = -7.0
    W = oracle.quantize_rows(oracle.Q4_0, v)
    blk = W.reshape(4, 2, 18)
    assert np.all(blk[:, :, 0] == 0x00) and np.all(blk[:, :, 1] == 0x3C)  # d = 1.0
    lo = blk[:, :, 2:] & 15
    hi = blk[:, :, 2:] >> 4
    codes = np.concatenate([lo, hi], axis=2).reshape(4, 64).astype(np.int64)
    assert np.array_equal(codes - 8, v.astype(np.int64))
    assert np.array_equal(oracle.dequantize_rows(oracle.Q4_0, W, 64), v.astype(np.float64))


def test_q4_0_zero_block_and_roundtrip_bound():
    w = synthetic.weights_f32(2, 16, 4096)
    w[0, :32] = 0.0
    W = oracle.quantize_rows(oracle.Q4_0, w)
    assert W[0, 0] == 0 and W[0, 1] == 0 and np.all(W[0, 2:18] == 0x88)
    deq = oracle.dequantize_rows(oracle.Q4_0, W, 4096)
    wb = w.reshape(16, 128, 32).astype(np.float64)
    amax = np.abs(wb).max(axis=2)
    d32 = (amax.astype(F32) / F32(7)).astype(np.float64)
    dh = np.float16(d32.astype(F32)).astype(np.float64)
    err = np.abs(deq.reshape(16, 128, 32) - wb)
    # rounding to the fp32 grid plus the half rounding of the stored scale
    bound = d32 * (0.5 + 1e-5) + 8 * np.abs(d32 - dh) + 1e-12
    assert np.all(err <= bound[..., None])


# ---- Q4_K ------------------------------------------------------------------
def _q4_K_fields(W, K):
    nb = K // 256
    b = W.reshape(-1, nb, 144)
    d = oracle.f16_bits_to_f32(b[..., 0:2].copy().view(np.uint16)[..., 0]).astype(np.float64)
    dmin = oracle.f16_bits_to_f32(b[..., 2:4].copy().view(np.uint16)[..., 0]).astype(np.float64)
    return b, d, dmin


def test_q4_K_roundtrip_bound():
    K = 4096
    w = synthetic.weights_f32(4, 32, K)
    w[1, :256] = 0.0                       # zero super-block
    w[2, :256] = np.abs(w[2, :256]) + 0.01  # all positive: min term 0
    W = oracle.quantize_rows(oracle.Q4_K, w)
    deq = oracle.dequantize_rows(oracle.Q4_K, W, K)
    b, d, dmin = _q4_K_fields(W, K)
    err = np.abs(deq - w).reshape(32, K // 256, 256)
    # per element: |x - xhat| <= d*sc/2 unrounded, and in the clamped cases
    # <= dmin/2 + 7.5 d, widened for the 6-bit clamp of sc and m against the
    # half-rounded d and dmin (at most 63 * 2^-11 of a step each), sc <= 63
    bound = np.maximum(d * 63 / 2, 0.55 * dmin + 8 * d) * (1 + 1e-5) + 1e-9
    assert np.all(err <= bound[..., None])
    assert not deq[1, :256].any()
    assert dmin[2, 0] == 0.0
    # typical accuracy: RMS error well under the 16-level step of N(0, 0.02)
    assert np.sqrt(np.mean((deq - w) ** 2)) < 0.004


def test_q4_K_codes_are_nearest_given_stored_fields():
    K = 512
    w = synthetic.weights_f32(6, 8, K, sigma=1.0)
    W = oracle.quantize_rows(oracle.Q4_K, w)
    # candidate values for every code 0..15 from the block's own stored fields
    one = np.zeros((1, 144), dtype=np.uint8)
    for r in range(8):
        for blkno in range(K // 256):
            blk = W[r, blkno * 144:(blkno + 1) * 144]
            cand = []
            for code in range(16):
                t = blk.copy()
                t[16:] = code | (code << 4)
                cand.append(oracle.dequantize_rows(oracle.Q4_K, t, 256)[0])
            cand = np.stack(cand)                       # [16][256]
            x = w[r, blkno * 256:(blkno + 1) * 256].astype(np.float64)
            got = oracle.dequantize_rows(oracle.Q4_K, blk, 256)[0]
            best = np.abs(cand - x[None]).min(axis=0)
            assert np.all(np.abs(got - x) <= best + 1e-6 * (np.abs(x) + 1e-3))


# ---- Q6_K ------------------------------------------------------------------
def test_q6_K_roundtrip_bound_and_zero():
    K = 4096
    w = synthetic.weights_f32(8, 16, K)
    w[3, :256] = 0.0
    W = oracle.quantize_rows(oracle.Q6_K, w)
    deq = oracle.dequantize_rows(oracle.Q6_K, W, K)
    blk = W.reshape(16, K // 256, 210)
    d = oracle.f16_bits_to_f32(blk[..., 208:210].copy().view(np.uint16)[..., 0]).astype(np.float64)
    sc = blk[..., 192:208].view(np.int8).astype(np.float64)          # [16][nb][16]
    step = np.abs(d[..., None] * sc)                                 # per sub-block
    err = np.abs(deq - w).reshape(16, K // 256, 16, 16)
    wb = np.abs(w.astype(np.float64)).reshape(16, K // 256, 16, 16).max(axis=3)
    bound = np.maximum(step / 2, wb - 31 * step) * (1 + 1e-5) + 1e-9
    assert np.all(err <= bound[..., None])
    assert not deq[3, :256].any()
    assert np.sqrt(np.mean((deq - w) ** 2)) < 0.001


def test_q6_K_codes_are_nearest_given_stored_fields():
    K = 256
    w = synthetic.weights_f32(10, 4, K, sigma=1.0)
    W = oracle.quantize_rows(oracle.Q6_K, w)
    for r in range(4):
        blk = W[r]
        d = float(oracle.f16_bits_to_f32(blk[208:210].copy().view(np.uint16))[0])
        sc = blk[192:208].view(np.int8).astype(np.float64)
        x = w[r].astype(np.float64)
        got = oracle.dequantize_rows(oracle.Q6_K, blk, 256)[0]
        levels = np.arange(-32, 32, dtype=np.float64)
        for e in range(256):
            best = np.abs(d * sc[e // 16] * levels - x[e]).min()
            assert abs(got[e] - x[e]) <= best + 1e-6 * (abs(x[e]) + 1e-3)


@pytest.mark.parametrize("t", [oracle.Q4_0, oracle.Q4_K, oracle.Q6_K])
def test_quantize_rejects_bad_shapes(t):
    with pytest.raises(ValueError):
        oracle.quantize_rows(t, np.zeros((2, 48), dtype=F32))
