"""Python binding of libqmv, the GB300 quantized decode GEMV library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libqmv.so`` (built in-tree by ``build.build()``); this module
allocates outputs with PyTorch, passes raw device pointers and the current
CUDA stream through the C ABI declared in ``include/qmv.h``, and raises
:class:`QmvError` on any non-zero status.  There is no fallback: if the
library is missing, importing the functions fails loudly.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

Q4_0 = 2
Q8_1 = 9
Q4_K = 12
Q6_K = 14
WEIGHT_TYPES = (Q4_0, Q4_K, Q6_K)
TYPE_NAMES = {Q4_0: "q4_0", Q8_1: "q8_1", Q4_K: "q4_K", Q6_K: "q6_K"}
BLOCK_ELEMS = {Q4_0: 32, Q4_K: 256, Q6_K: 256}
MAX_COLS = 8

# Exported symbols of include/qmv.h (checked by the CPU test-suite).
EXPORTS = (
    "qmv_status_str", "qmv_version", "qmv_row_bytes", "qmv_q8_1_padded_k", "qmv_q8_1_bytes",
    "qmv_quantize_q8_1", "qmv_quantize_weights", "qmv_mul_mat_vec", "qmv_mul_mat_vec_gate_up_swiglu",
    "qmv_mul_mat_vec_id", "qmv_mul_mat_vec_f32", "qmv_mul_mat_vec_gate_up_swiglu_f32", "qmv_mul_mat_vec_id_f32",
    "qmv_mul_mat_vec_fused", "qmv_mul_mat_vec_id_fused",
    "qmv_debug_subblock_sums", "qmv_device_fault", "qmv_set_tuning", "qmv_set_stream_tuning", "qmv_set_pdl",
    "qmv_set_checked", "qmv_set_mma_min_cols", "qmv_describe_gemv", "qmv_read_bandwidth_probe",
    "qmv_set_early_warps",
)


class LaunchInfo(ctypes.Structure):
    """qmv_launch_info of include/qmv.h."""
    _fields_ = [(n, ctypes.c_int) for n in ("tile_kernel", "tensor_cores", "rows_per_tile", "grid", "block",
                                            "cluster", "stages", "dec_warps", "pre_tiles")] + \
               [("smem", ctypes.c_size_t)]


class QmvError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


_lib = None
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_int = ctypes.c_int


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libqmv (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libqmv is not built ({path} missing); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        L.qmv_status_str.restype = ctypes.c_char_p
        L.qmv_status_str.argtypes = [_int]
        L.qmv_version.restype = _int
        L.qmv_row_bytes.restype = ctypes.c_size_t
        L.qmv_row_bytes.argtypes = [_int, _i64]
        L.qmv_q8_1_padded_k.restype = _i64
        L.qmv_q8_1_padded_k.argtypes = [_i64]
        L.qmv_q8_1_bytes.restype = ctypes.c_size_t
        L.qmv_q8_1_bytes.argtypes = [_i64, _int]
        L.qmv_quantize_q8_1.argtypes = [_vp, _i64, _int, _i64, _vp, _vp]
        L.qmv_quantize_weights.argtypes = [_int, _vp, _i64, _i64, _i64, _vp, _vp]
        L.qmv_mul_mat_vec.argtypes = [_int, _vp, _i64, _i64, _vp, _int, _vp, _vp]
        L.qmv_mul_mat_vec_gate_up_swiglu.argtypes = [_int, _vp, _vp, _i64, _i64, _vp, _int, _vp, _vp]
        L.qmv_mul_mat_vec_id.argtypes = [_int, _vp, _i64, _i64, _i64, _vp, _vp, _int, _int, _vp, _vp, _vp]
        L.qmv_mul_mat_vec_f32.argtypes = [_int, _vp, _i64, _i64, _vp, _i64, _int, _vp, _vp]
        L.qmv_mul_mat_vec_gate_up_swiglu_f32.argtypes = [_int, _vp, _vp, _i64, _i64, _vp, _i64, _int, _vp, _vp]
        L.qmv_mul_mat_vec_id_f32.argtypes = [_int, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _int, _int, _vp, _vp,
                                             _vp]
        L.qmv_mul_mat_vec_fused.argtypes = [_int, _vp, _vp, _i64, _i64, _vp, _vp, _i64, _int, _vp, _vp, _vp, _vp]
        L.qmv_mul_mat_vec_id_fused.argtypes = [_int, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _int, _int,
                                               _vp, _vp, _vp, _vp, _vp, _vp]
        L.qmv_debug_subblock_sums.argtypes = [_int, _vp, _i64, _i64, _vp, _int, _vp, _vp]
        L.qmv_device_fault.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.qmv_set_tuning.argtypes = [_int, _int, _int, _int, _int, _int, _int]
        L.qmv_set_stream_tuning.argtypes = [_int, _int, _int]
        L.qmv_set_pdl.argtypes = [_int]
        L.qmv_set_checked.argtypes = [_int]
        L.qmv_set_mma_min_cols.argtypes = [_int, _int]
        L.qmv_set_early_warps.argtypes = [_int, _int]
        L.qmv_read_bandwidth_probe.argtypes = [_vp, ctypes.c_size_t, _vp, _vp]
        L.qmv_describe_gemv.argtypes = [_int, _int, _i64, _i64, _int, _int, ctypes.POINTER(LaunchInfo)]
        for name in ("qmv_quantize_q8_1", "qmv_quantize_weights", "qmv_mul_mat_vec",
                     "qmv_mul_mat_vec_gate_up_swiglu", "qmv_mul_mat_vec_id", "qmv_mul_mat_vec_f32",
                     "qmv_mul_mat_vec_gate_up_swiglu_f32", "qmv_mul_mat_vec_id_f32", "qmv_mul_mat_vec_fused",
                     "qmv_mul_mat_vec_id_fused", "qmv_debug_subblock_sums",
                     "qmv_device_fault", "qmv_set_tuning", "qmv_set_stream_tuning", "qmv_set_pdl",
                     "qmv_set_checked", "qmv_set_mma_min_cols", "qmv_describe_gemv",
                     "qmv_read_bandwidth_probe", "qmv_set_early_warps"):
            getattr(L, name).restype = _int
        _lib = L
    return _lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise QmvError(fn, rc, lib().qmv_status_str(rc).decode())


def _stream_handle(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return _vp(s.cuda_stream)


def _ptr(t):
    return _vp(t.data_ptr()) if t is not None else _vp(0)


def _need_cuda(t, name, dtype=None):
    import torch

    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


# ---- sizes --------------------------------------------------------------------
def row_bytes(qtype: int, K: int) -> int:
    return int(lib().qmv_row_bytes(qtype, K))


def q8_1_padded_k(K: int) -> int:
    return int(lib().qmv_q8_1_padded_k(K))


def q8_1_bytes(K: int, ncols: int = 1) -> int:
    return int(lib().qmv_q8_1_bytes(K, ncols))


# ---- quantization ------------------------------------------------------------
def quantize_q8_1(x, out=None, stream=None):
    """x: fp32 CUDA tensor [ncols][K] (or [K]) -> uint8 [ncols][q8_1_bytes(K)]."""
    import torch

    x2 = x.unsqueeze(0) if x.dim() == 1 else x
    _need_cuda(x2, "x", torch.float32)
    ncols, K = x2.shape
    if out is None:
        out = torch.empty((ncols, q8_1_bytes(K)), dtype=torch.uint8, device=x.device)
    _check("qmv_quantize_q8_1", lib().qmv_quantize_q8_1(_ptr(x2), K, ncols, K, _ptr(out), _stream_handle(stream)))
    return out


def quantize_weights(qtype: int, w, out=None, stream=None):
    """w: fp32 CUDA tensor [M][K] -> uint8 [M][row_bytes] blocks of qtype."""
    import torch

    _need_cuda(w, "w", torch.float32)
    M, K = w.shape
    if out is None:
        out = torch.empty((M, row_bytes(qtype, K)), dtype=torch.uint8, device=w.device)
    _check("qmv_quantize_weights",
           lib().qmv_quantize_weights(qtype, _ptr(w), M, K, K, _ptr(out), _stream_handle(stream)))
    return out


# ---- GEMV ------------------------------------------------------------------------
def mul_mat_vec(qtype: int, W, M: int, K: int, xq, ncols: int, out=None, stream=None):
    """y[ncols][M] = W . x for q8_1 activations xq (ncols rows)."""
    import torch

    if out is None:
        out = torch.empty((ncols, M), dtype=torch.float32, device=W.device)
    _check("qmv_mul_mat_vec", lib().qmv_mul_mat_vec(qtype, _ptr(W), M, K, _ptr(xq), ncols, _ptr(out),
                                                    _stream_handle(stream)))
    return out


def mul_mat_vec_gate_up_swiglu(qtype: int, W_gate, W_up, M: int, K: int, xq, ncols: int = 1, out=None,
                               stream=None):
    """y[ncols][M] = (W_up . x) * silu(W_gate . x)."""
    import torch

    if out is None:
        out = torch.empty((ncols, M), dtype=torch.float32, device=W_up.device)
    _check("qmv_mul_mat_vec_gate_up_swiglu",
           lib().qmv_mul_mat_vec_gate_up_swiglu(qtype, _ptr(W_gate), _ptr(W_up), M, K, _ptr(xq), ncols,
                                                _ptr(out), _stream_handle(stream)))
    return out


def mul_mat_vec_id(qtype: int, W, n_expert: int, M: int, K: int, xq, ids, out=None, status=None, stream=None):
    """Expert-indexed GEMV: y[t][k][M] = W[ids[t][k]] . x[t]; ids int32 [n_tokens][top_k]."""
    import torch

    _need_cuda(ids, "ids", torch.int32)
    n_tokens, top_k = ids.shape
    if out is None:
        out = torch.empty((n_tokens, top_k, M), dtype=torch.float32, device=W.device)
    _check("qmv_mul_mat_vec_id",
           lib().qmv_mul_mat_vec_id(qtype, _ptr(W), n_expert, M, K, _ptr(xq), _ptr(ids), n_tokens, top_k,
                                    _ptr(out), _ptr(status), _stream_handle(stream)))
    return out


# ---- GEMV with fp32 activations (quantization fused into the GEMV) ---------------
def _x2d(x):
    import torch

    x2 = x.unsqueeze(0) if x.dim() == 1 else x
    if not x2.is_cuda or x2.dtype != torch.float32:
        raise ValueError("x must be a float32 CUDA tensor")
    if x2.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    return x2


def mul_mat_vec_f32(qtype: int, W, M: int, K: int, x, out=None, stream=None):
    """y[ncols][M] = W . x for fp32 x [ncols][K] (rows may be strided)."""
    import torch

    x2 = _x2d(x)
    ncols = x2.shape[0]
    if out is None:
        out = torch.empty((ncols, M), dtype=torch.float32, device=W.device)
    _check("qmv_mul_mat_vec_f32", lib().qmv_mul_mat_vec_f32(qtype, _ptr(W), M, K, _ptr(x2), x2.stride(0), ncols,
                                                            _ptr(out), _stream_handle(stream)))
    return out


def mul_mat_vec_gate_up_swiglu_f32(qtype: int, W_gate, W_up, M: int, K: int, x, out=None, stream=None):
    """y[ncols][M] = (W_up . x) * silu(W_gate . x) for fp32 x [ncols][K]."""
    import torch

    x2 = _x2d(x)
    ncols = x2.shape[0]
    if out is None:
        out = torch.empty((ncols, M), dtype=torch.float32, device=W_up.device)
    _check("qmv_mul_mat_vec_gate_up_swiglu_f32",
           lib().qmv_mul_mat_vec_gate_up_swiglu_f32(qtype, _ptr(W_gate), _ptr(W_up), M, K, _ptr(x2), x2.stride(0),
                                                    ncols, _ptr(out), _stream_handle(stream)))
    return out


def mul_mat_vec_id_f32(qtype: int, W, n_expert: int, M: int, K: int, x, ids, out=None, status=None, stream=None):
    """Expert-indexed GEMV with fp32 tokens x [n_tokens][K]: y[t][k][M] = W[ids[t][k]] . x[t]."""
    import torch

    x2 = _x2d(x)
    _need_cuda(ids, "ids", torch.int32)
    n_tokens, top_k = ids.shape
    if out is None:
        out = torch.empty((n_tokens, top_k, M), dtype=torch.float32, device=W.device)
    _check("qmv_mul_mat_vec_id_f32",
           lib().qmv_mul_mat_vec_id_f32(qtype, _ptr(W), n_expert, M, K, _ptr(x2), x2.stride(0), _ptr(ids), n_tokens,
                                        top_k, _ptr(out), _ptr(status), _stream_handle(stream)))
    return out


def _activations(xq, x):
    """(xq pointer, x pointer, ldx, ncols) for exactly one of q8_1 rows xq [ncols][bytes] or fp32 x [ncols][K]."""
    import torch

    if (xq is None) == (x is None):
        raise ValueError("pass exactly one of xq (q8_1) and x (fp32)")
    if x is not None:
        x2 = _x2d(x)
        return _vp(0), _ptr(x2), x2.stride(0), x2.shape[0]
    xq2 = xq.unsqueeze(0) if xq.dim() == 1 else xq
    _need_cuda(xq2, "xq", torch.uint8)
    return _ptr(xq2), _vp(0), 0, xq2.shape[0]


def mul_mat_vec_fused(qtype: int, W_up, M: int, K: int, xq=None, x=None, W_gate=None, bias=None, gate_bias=None,
                      out=None, stream=None):
    """y = W_up.x (+ bias), or (W_up.x + bias) * silu(W_gate.x + gate_bias) with W_gate; q8_1 xq or fp32 x."""
    import torch

    pq, px, ldx, ncols = _activations(xq, x)
    for name, b in (("bias", bias), ("gate_bias", gate_bias)):
        if b is not None:
            _need_cuda(b, name, torch.float32)
    if out is None:
        out = torch.empty((ncols, M), dtype=torch.float32, device=W_up.device)
    _check("qmv_mul_mat_vec_fused",
           lib().qmv_mul_mat_vec_fused(qtype, _ptr(W_up), _ptr(W_gate), M, K, pq, px, ldx, ncols, _ptr(bias),
                                       _ptr(gate_bias), _ptr(out), _stream_handle(stream)))
    return out


def mul_mat_vec_id_fused(qtype: int, W, n_expert: int, M: int, K: int, ids, xq=None, x=None, W_gate=None,
                         W_shared=None, W_shared_gate=None, out=None, out_shared=None, status=None, stream=None):
    """Expert-indexed GEMV (q8_1 xq or fp32 x, one row per token), optionally gated
    ((W.x) * silu(W_gate.x) per routed slot) and with a shared expert (gated like
    the routed ones): returns (y [n_tokens][top_k][M], y_shared [n_tokens][M] or None)."""
    import torch

    pq, px, ldx, n_tok = _activations(xq, x)
    _need_cuda(ids, "ids", torch.int32)
    n_tokens, top_k = ids.shape
    if n_tok < n_tokens:
        raise ValueError("fewer activation rows than tokens")
    if out is None:
        out = torch.empty((n_tokens, top_k, M), dtype=torch.float32, device=W.device)
    if W_shared is not None and out_shared is None:
        out_shared = torch.empty((n_tokens, M), dtype=torch.float32, device=W.device)
    _check("qmv_mul_mat_vec_id_fused",
           lib().qmv_mul_mat_vec_id_fused(qtype, _ptr(W), _ptr(W_gate), n_expert, M, K, pq, px, ldx, _ptr(ids),
                                          n_tokens, top_k, _ptr(out), _ptr(W_shared), _ptr(W_shared_gate),
                                          _ptr(out_shared if W_shared is not None else None), _ptr(status),
                                          _stream_handle(stream)))
    return out, (out_shared if W_shared is not None else None)


def debug_subblock_sums(qtype: int, W, M: int, K: int, xq, ncols: int, stream=None):
    """Exact int32 per-sub-block sums [ncols][M][n] (see include/qmv.h)."""
    import torch

    n = K // 32 if qtype == Q4_0 else K // 16
    out = torch.empty((ncols, M, n), dtype=torch.int32, device=W.device)
    _check("qmv_debug_subblock_sums",
           lib().qmv_debug_subblock_sums(qtype, _ptr(W), M, K, _ptr(xq), ncols, _ptr(out), _stream_handle(stream)))
    return out


def device_fault() -> int:
    code = ctypes.c_uint(0)
    _check("qmv_device_fault", lib().qmv_device_fault(ctypes.byref(code)))
    return int(code.value)


def set_tuning(qtype: int, threads: int = 0, slice_units: int = 0, stages: int = 0, ctas_per_sm: int = 0,
               smem_share: int = 0, cluster: int = 0):
    """Launch-geometry override for sweeps (0 keeps the default; see include/qmv.h)."""
    _check("qmv_set_tuning",
           lib().qmv_set_tuning(qtype, threads, slice_units, stages, ctas_per_sm, smem_share, cluster))


def set_stream_tuning(qtype: int, dec_warps: int = 0, pre_tiles: int = 0):
    """Decoding warps per CTA and tiles per warp requested before the dependency wait (0: default)."""
    _check("qmv_set_stream_tuning", lib().qmv_set_stream_tuning(qtype, dec_warps, pre_tiles))


def read_bandwidth_probe(buf, sink, stream=None):
    """Diagnostic: read every 16-byte piece of the CUDA tensor buf once (see include/qmv.h)."""
    _need_cuda(buf, "buf")
    _check("qmv_read_bandwidth_probe", lib().qmv_read_bandwidth_probe(_ptr(buf), buf.numel() * buf.element_size(),
                                                                     _ptr(sink), _stream_handle(stream)))


def describe_gemv(qtype: int, M: int, K: int, ncols: int = 1, gate_up: bool = False, fp32_input: bool = False):
    """The launch geometry the library would use for this GEMV (nothing is launched), as a dict."""
    info = LaunchInfo()
    _check("qmv_describe_gemv", lib().qmv_describe_gemv(qtype, 1 if gate_up else 0, M, K, ncols,
                                                       1 if fp32_input else 0, ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in LaunchInfo._fields_}


def set_early_warps(qtype: int, early_warps: int = 0):
    """Decoding warps that request tiles before the dependency wait (0: all)."""
    _check("qmv_set_early_warps", lib().qmv_set_early_warps(qtype, early_warps))


def set_mma_min_cols(qtype: int, min_cols: int = 0):
    """Columns from which the plain Q4_K GEMV decodes with mma.sync (0: the default, never; 9: never)."""
    _check("qmv_set_mma_min_cols", lib().qmv_set_mma_min_cols(qtype, min_cols))


def set_pdl(enable: bool):
    _check("qmv_set_pdl", lib().qmv_set_pdl(1 if enable else 0))


def set_checked(enable: bool):
    """Checked mode: every call first verifies on the host that each argument's
    byte range lies inside one device allocation (QMV_ERR_RANGE otherwise)."""
    _check("qmv_set_checked", lib().qmv_set_checked(1 if enable else 0))
