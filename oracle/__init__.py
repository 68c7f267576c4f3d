"""CPU oracle for the quantized decode GEMV -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the repository's smoke check and the benchmark's
CPU-baseline / reference leg may import this package.  The GPU library never
imports, links or calls it, and the two share no code.

The arithmetic lives in plain C (``oracle.c``, ``half.c``), loaded here with
ctypes; this module only marshals numpy arrays.  The few Python-level
compositions (SwiGLU, expert routing) are written out in fp64 below, each
citing the passage it follows.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

Q4_0 = 2
Q8_1 = 9
Q4_K = 12
Q6_K = 14
WEIGHT_TYPES = (Q4_0, Q4_K, Q6_K)
TYPE_NAMES = {Q4_0: "q4_0", Q8_1: "q8_1", Q4_K: "q4_K", Q6_K: "q6_K"}

_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def lib():
    """The loaded liboracle (built on first use if missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_f32_to_f16.restype = ctypes.c_uint16
        L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.oracle_f16_to_f32.restype = ctypes.c_float
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f32_to_f16_array.argtypes = [_vp, _vp, _i64]
        L.oracle_f16_to_f32_array.argtypes = [_vp, _vp, _i64]
        for name in ("oracle_block_elems", "oracle_block_bytes"):
            getattr(L, name).restype = _i64
            getattr(L, name).argtypes = [ctypes.c_int]
        L.oracle_row_bytes.restype = _i64
        L.oracle_row_bytes.argtypes = [ctypes.c_int, _i64]
        L.oracle_q8_1_padded_k.restype = _i64
        L.oracle_q8_1_padded_k.argtypes = [_i64]
        L.oracle_subblock_count.restype = _i64
        L.oracle_subblock_count.argtypes = [ctypes.c_int, _i64]
        L.oracle_quantize_q8_1.argtypes = [_vp, _i64, _i64, _i64, _vp]
        L.oracle_quantize_rows.argtypes = [ctypes.c_int, _vp, _i64, _i64, _i64, _vp]
        L.oracle_dequantize_rows.argtypes = [ctypes.c_int, _vp, _i64, _i64, _vp]
        L.oracle_dequantize_q8_1.argtypes = [_vp, _i64, _i64, _vp]
        L.oracle_dequantize_row_q4_K_f32.argtypes = [_vp, _i64, _vp]
        L.oracle_gemv_plain.argtypes = [ctypes.c_int, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp]
        L.oracle_gemv_formula.argtypes = [ctypes.c_int, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp]
        L.oracle_gemv_formula_mt.argtypes = [ctypes.c_int, _vp, _i64, _i64, _vp, _i64, _vp, _vp, ctypes.c_int]
        L.oracle_gemv_int_f32.argtypes = [ctypes.c_int, _vp, _i64, _i64, _vp, _i64, _vp, ctypes.c_int]
        L.oracle_subblock_sums.argtypes = [ctypes.c_int, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp]
        for name in ("oracle_quantize_q8_1", "oracle_quantize_rows", "oracle_dequantize_rows",
                     "oracle_dequantize_q8_1", "oracle_dequantize_row_q4_K_f32", "oracle_gemv_plain",
                     "oracle_gemv_formula", "oracle_gemv_formula_mt", "oracle_gemv_int_f32",
                     "oracle_subblock_sums"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---- sizes -----------------------------------------------------------------
def block_elems(t: int) -> int:
    return int(lib().oracle_block_elems(t))


def block_bytes(t: int) -> int:
    return int(lib().oracle_block_bytes(t))


def row_bytes(t: int, K: int) -> int:
    r = int(lib().oracle_row_bytes(t, K))
    if r < 0:
        raise ValueError(f"K={K} is not a multiple of the {TYPE_NAMES.get(t, t)} block")
    return r


def q8_1_padded_k(K: int) -> int:
    return int(lib().oracle_q8_1_padded_k(K))


def q8_1_row_bytes(K: int) -> int:
    return q8_1_padded_k(K) // 32 * 36


def subblock_count(t: int, K: int) -> int:
    return int(lib().oracle_subblock_count(t, K))


# ---- fp16 -------------------------------------------------------------------
def f32_to_f16_bits(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(_p(a), _p(out), a.size)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
    out = np.empty(a.shape, dtype=np.float32)
    lib().oracle_f16_to_f32_array(_p(a), _p(out), a.size)
    return out


# ---- quantizers --------------------------------------------------------------
def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """x: fp32 [ncols][K] -> uint8 [ncols][padded_k/32*36] q8_1 blocks."""
    x = np.ascontiguousarray(np.atleast_2d(np.asarray(x, dtype=np.float32)))
    ncols, K = x.shape
    out = np.empty((ncols, q8_1_row_bytes(K)), dtype=np.uint8)
    _check(lib().oracle_quantize_q8_1(_p(x), K, ncols, K, _p(out)), "quantize_q8_1")
    return out


def quantize_rows(t: int, w: np.ndarray) -> np.ndarray:
    """w: fp32 [M][K] -> uint8 [M][row_bytes] blocks of type t."""
    w = np.ascontiguousarray(np.atleast_2d(np.asarray(w, dtype=np.float32)))
    M, K = w.shape
    out = np.empty((M, row_bytes(t, K)), dtype=np.uint8)
    _check(lib().oracle_quantize_rows(t, _p(w), M, K, K, _p(out)), "quantize_rows")
    return out


# ---- dequantizers ------------------------------------------------------------
def dequantize_rows(t: int, W: np.ndarray, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    M = W.size // row_bytes(t, K)
    out = np.empty((M, K), dtype=np.float64)
    _check(lib().oracle_dequantize_rows(t, _p(W), M, K, _p(out)), "dequantize_rows")
    return out


def dequantize_q8_1(xq: np.ndarray, K: int) -> np.ndarray:
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    ncols = xq.size // q8_1_row_bytes(K)
    out = np.empty((ncols, K), dtype=np.float64)
    _check(lib().oracle_dequantize_q8_1(_p(xq), K, ncols, _p(out)), "dequantize_q8_1")
    return out


def dequantize_row_q4_K_f32(W: np.ndarray, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    out = np.empty(K, dtype=np.float32)
    _check(lib().oracle_dequantize_row_q4_K_f32(_p(W), K, _p(out)), "dequantize_row_q4_K_f32")
    return out


# ---- GEMV ----------------------------------------------------------------------
def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, r.size


def gemv_plain(t: int, W: np.ndarray, M: int, K: int, xq: np.ndarray, ncols: int, rows=None):
    """fp64 dequantize-then-dot: y[ncols][nrows]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    r, n = _rows_arg(rows, M)
    y = np.empty((ncols, n), dtype=np.float64)
    _check(lib().oracle_gemv_plain(t, _p(W), M, K, _p(xq), ncols, None if r is None else _p(r), n, _p(y)),
           "gemv_plain")
    return y


def gemv_formula(t: int, W: np.ndarray, M: int, K: int, xq: np.ndarray, ncols: int, rows=None):
    """The method's block formula in fp64: (y, l1), each [ncols][nrows]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    r, n = _rows_arg(rows, M)
    y = np.empty((ncols, n), dtype=np.float64)
    l1 = np.empty((ncols, n), dtype=np.float64)
    _check(lib().oracle_gemv_formula(t, _p(W), M, K, _p(xq), ncols, None if r is None else _p(r), n,
                                     _p(y), _p(l1)), "gemv_formula")
    return y, l1


def gemv_formula_mt(t: int, W: np.ndarray, M: int, K: int, xq: np.ndarray, ncols: int, nthreads: int):
    """Threaded block-formula GEMV over all rows (CPU baseline)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    y = np.empty((ncols, M), dtype=np.float64)
    l1 = np.empty((ncols, M), dtype=np.float64)
    _check(lib().oracle_gemv_formula_mt(t, _p(W), M, K, _p(xq), ncols, _p(y), _p(l1), int(nthreads)),
           "gemv_formula_mt")
    return y, l1


def gemv_int_f32(t: int, W: np.ndarray, M: int, K: int, xq: np.ndarray, ncols: int, nthreads: int = 1):
    """The method's integer formula in fp32 over all rows (int32 block sums,
    fp32 scaling), threaded by rows: y float32 [ncols][M].  A CPU baseline."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    y = np.empty((ncols, M), dtype=np.float32)
    _check(lib().oracle_gemv_int_f32(t, _p(W), M, K, _p(xq), ncols, _p(y), int(nthreads)), "gemv_int_f32")
    return y


def subblock_sums(t: int, W: np.ndarray, M: int, K: int, xq: np.ndarray, ncols: int, rows=None):
    """Exact int32 per-sub-block sums, [ncols][nrows][subblock_count]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    r, n = _rows_arg(rows, M)
    out = np.empty((ncols, n, subblock_count(t, K)), dtype=np.int32)
    _check(lib().oracle_subblock_sums(t, _p(W), M, K, _p(xq), ncols, None if r is None else _p(r), n,
                                      _p(out)), "subblock_sums")
    return out


# ---- compositions ------------------------------------------------------------
def silu(g):
    """silu(g) = g / (1 + e^-g) in fp64 (the pages name ggml_cuda_op_silu_single
    in the fused epilogue of the mul_mat_vec_q page without defining it; this is
    the standard definition)."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def swiglu(gate, up):
    """Fused gate/up epilogue, mul_mat_vec_q page section "融合": result = up * silu(gate)."""
    return np.asarray(up, dtype=np.float64) * silu(gate)


def fused_epilogue(up, gate=None, bias=None, gate_bias=None):
    """The fused epilogue of the mul_mat_vec_q page, section "融合" (its
    SwiGLU case), in fp64: result = up + x_bias; with a gate, gate_value =
    gate + gate_bias and result *= silu(gate_value).  up and gate are
    [ncols][M]; bias and gate_bias are [M] vectors, the same for every column
    (the reading taken here: the page's epilogue adds the bias of the
    output row, and a layer's bias does not depend on the token)."""
    r = np.asarray(up, dtype=np.float64)
    if bias is not None:
        r = r + np.asarray(bias, dtype=np.float64)[None, :]
    if gate is None:
        return r
    g = np.asarray(gate, dtype=np.float64)
    if gate_bias is not None:
        g = g + np.asarray(gate_bias, dtype=np.float64)[None, :]
    return r * silu(g)


def shared_expert_gemv(t: int, W_shared: np.ndarray, M: int, K: int, xq: np.ndarray, n_tokens: int, rows=None):
    """MoE shared expert (mul_mat_vec_q page, section "融合", the extra grid
    slice after the routed experts): every token uses the same matrix, so
    y_shared[t] = W_shared . x[t]; returns (y, l1), each [n_tokens][nrows]."""
    return gemv_formula(t, W_shared, M, K, xq, n_tokens, rows)


def moe_gemv(t: int, W: np.ndarray, n_expert: int, M: int, K: int, xq: np.ndarray, ids: np.ndarray,
             rows=None):
    """Expert-indexed GEMV (mul_mat_vec_q page, "MoE" section): for token t and
    slot k, y[t][k] = W[ids[t][k]] . x[t].  Ids outside [0, n_expert) yield a
    zero output row (the reading taken here for invalid ids); returns
    (y, l1, n_invalid) with y, l1 of shape [n_tokens][top_k][nrows]."""
    W = np.ascontiguousarray(W, dtype=np.uint8).reshape(n_expert, -1)
    n_tokens, top_k = ids.shape
    xrow = q8_1_row_bytes(K)
    xq = np.ascontiguousarray(xq, dtype=np.uint8).reshape(-1)
    nrows = M if rows is None else len(rows)
    y = np.zeros((n_tokens, top_k, nrows))
    l1 = np.zeros((n_tokens, top_k, nrows))
    bad = 0
    for tok in range(n_tokens):
        for k in range(top_k):
            e = int(ids[tok, k])
            if e < 0 or e >= n_expert:
                bad += 1
                continue
            yy, ll = gemv_formula(t, W[e], M, K, xq[tok * xrow:(tok + 1) * xrow], 1, rows)
            y[tok, k] = yy[0]
            l1[tok, k] = ll[0]
    return y, l1, bad


def random_blocks(t: int, M: int, K: int, seed: int) -> np.ndarray:
    """Uniformly random block bytes of type t with the half-precision scale
    fields replaced by random finite positive halves in [2^-14, 2^-4).

    Exercises every code, every 6-bit scale/min and (for Q6_K) negative int8
    sub-block scales, none of which the quantizers above produce."""
    import synthetic

    rb = row_bytes(t, K)
    raw = synthetic.uniform_u8(seed, M * rb).reshape(M, rb)
    nb = K // block_elems(t)
    bs = block_bytes(t)
    if t == Q4_0:
        offs = [0]
    elif t == Q4_K:
        offs = [0, 2]
    else:
        offs = [208]
    # half exponent field 1..10 (2^-14 .. 2^-5 binades), random fraction, sign +
    halves = synthetic.uniform_int(seed + 1, (M, nb, len(offs)), 0, (10 << 10) - 1).astype(np.uint16) + (1 << 10)
    blk = raw.reshape(M, nb, bs)
    for j, o in enumerate(offs):
        blk[:, :, o] = (halves[:, :, j] & 0xFF).astype(np.uint8)
        blk[:, :, o + 1] = (halves[:, :, j] >> 8).astype(np.uint8)
    return np.ascontiguousarray(blk.reshape(M, rb))
