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

# Exported symbols of include/qmv.h and include/qmv_debug.h (checked by the CPU test-suite).
EXPORTS = (
    "qmv_status_str", "qmv_version", "qmv_row_bytes", "qmv_q8_1_padded_k", "qmv_q8_1_bytes",
    "qmv_quantize_q8_1", "qmv_quantize_weights", "qmv_mul_mat_vec", "qmv_mul_mat_vec_gate_up_swiglu",
    "qmv_mul_mat_vec_id", "qmv_mul_mat_vec_f32", "qmv_mul_mat_vec_gate_up_swiglu_f32", "qmv_mul_mat_vec_id_f32",
    "qmv_mul_mat_vec_fused", "qmv_mul_mat_vec_fused_q8_1", "qmv_mul_mat_vec_id_fused",
    "qmv_debug_subblock_sums", "qmv_device_fault", "qmv_set_tuning", "qmv_set_stream_tuning", "qmv_set_pdl",
    "qmv_set_checked", "qmv_set_mma_min_cols", "qmv_describe_gemv", "qmv_read_bandwidth_probe",
    "qmv_set_early_warps", "qmv_set_early_delay", "qmv_debug_f32_withheld_share",
    "qmv_debug_f32_withheld_share_q8_1", "qmv_debug_trace",
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
        L.qmv_mul_mat_vec_fused_q8_1.argtypes = [_int, _vp, _vp, _i64, _i64, _vp, _vp, _i64, _int, _vp, _vp, _vp, _vp,
                                                 _vp]
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
        L.qmv_set_early_delay.argtypes = [_int, _int]
        L.qmv_read_bandwidth_probe.argtypes = [_vp, ctypes.c_size_t, _vp, _vp]
        L.qmv_describe_gemv.argtypes = [_int, _int, _i64, _i64, _int, _int, ctypes.POINTER(LaunchInfo)]
        L.qmv_debug_f32_withheld_share.argtypes = [_int, _vp, _i64, _i64, _vp, _i64, _int, _vp, ctypes.c_uint64, _vp]
        L.qmv_debug_f32_withheld_share_q8_1.argtypes = [_int, _vp, _i64, _i64, _vp, _vp, _vp, ctypes.c_uint64, _vp]
        L.qmv_debug_trace.argtypes = [_vp, _i64]
        for name in ("qmv_quantize_q8_1", "qmv_quantize_weights", "qmv_mul_mat_vec",
                     "qmv_mul_mat_vec_gate_up_swiglu", "qmv_mul_mat_vec_id", "qmv_mul_mat_vec_f32",
                     "qmv_mul_mat_vec_gate_up_swiglu_f32", "qmv_mul_mat_vec_id_f32", "qmv_mul_mat_vec_fused",
                     "qmv_mul_mat_vec_fused_q8_1",
                     "qmv_mul_mat_vec_id_fused", "qmv_debug_subblock_sums",
                     "qmv_device_fault", "qmv_set_tuning", "qmv_set_stream_tuning", "qmv_set_pdl",
                     "qmv_set_checked", "qmv_set_mma_min_cols", "qmv_describe_gemv",
                     "qmv_read_bandwidth_probe", "qmv_set_early_warps", "qmv_set_early_delay", "qmv_debug_f32_withheld_share",
                     "qmv_debug_f32_withheld_share_q8_1", "qmv_debug_trace"):
            getattr(L, name).restype = _int
        _lib = L
    return _lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise QmvError(fn, rc, lib().qmv_status_str(rc).decode())


def _ptr(t):
    return _vp(t.data_ptr()) if t is not None else _vp(0)


# ---- argument validation (host side, before any call into the library) ----------
# Every tensor a call reads or writes is checked here: its dtype, that it is
# contiguous where the call takes a flat buffer, and that it holds at least the
# bytes the call accesses; then that all of them are CUDA tensors on one device
# (and the stream, if given, on that device).  A failed check raises ValueError
# and nothing is launched.  The byte counts are those include/qmv.h states per
# argument, computed here in Python so that no check depends on the library.
BLOCK_BYTES = {Q4_0: 18, Q4_K: 144, Q6_K: 210}
_Q8_1_BLOCK, _Q8_1_PAD = 36, 512


def _shape_ok(qtype, M, K):
    return qtype in BLOCK_ELEMS and M > 0 and K > 0 and K % BLOCK_ELEMS[qtype] == 0


def _row_bytes(qtype, K):
    """Bytes of one weight row (the formula of qmv_row_bytes)."""
    return K // BLOCK_ELEMS[qtype] * BLOCK_BYTES[qtype]


def _q8_1_bytes(K, ncols):
    """Bytes of ncols q8_1 activation rows (the formula of qmv_q8_1_bytes)."""
    return ncols * ((K + _Q8_1_PAD - 1) // _Q8_1_PAD * _Q8_1_PAD) // 32 * _Q8_1_BLOCK


def _tensor(t, name, dtype=None, min_bytes=0, contiguous=True):
    import torch

    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    have = t.numel() * t.element_size()
    if have < min_bytes:
        raise ValueError(f"{name} holds {have} bytes; the call accesses {min_bytes}")
    return t


def _device_of(named, stream=None):
    """The one CUDA device of the named tensors (None entries are skipped)."""
    devs = set()
    for name, t in named:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        devs.add(t.device)
    if len(devs) != 1:
        raise ValueError("all tensor arguments must be on one CUDA device")
    dev = devs.pop()
    if stream is not None and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, the tensors on {dev}")
    return dev


def _call(fn, dev, stream, *args):
    """Calls lib().fn(*args, stream) with dev current; raises QmvError on a non-zero status."""
    import torch

    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = getattr(lib(), fn)(*args, _vp(s.cuda_stream))
    _check(fn, rc)


def _out(out, name, shape, device, nbytes):
    """The caller's float32 output (checked) or a new one of shape on device."""
    import torch

    if out is None:
        return torch.empty(shape, dtype=torch.float32, device=device)
    return _tensor(out, name, torch.float32, nbytes)


def _x2d(x, K=None, name="x"):
    """fp32 activations as [ncols][>= K] with unit stride along K; returns (x2d, ldx)."""
    import torch

    _tensor(x, name, torch.float32, contiguous=False)
    x2 = x.unsqueeze(0) if x.dim() == 1 else x
    if x2.dim() != 2:
        raise ValueError(f"{name} must be 1-D or 2-D")
    if x2.shape[1] > 1 and x2.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous")
    if K is not None and x2.shape[1] < K:
        raise ValueError(f"{name} rows hold {x2.shape[1]} values; the call reads K = {K}")
    ldx = x2.stride(0) if x2.shape[0] > 1 else max(x2.shape[1], 1)
    return x2, ldx


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

    _tensor(x, "x", torch.float32)
    x2 = x.unsqueeze(0) if x.dim() == 1 else x
    ncols, K = x2.shape
    if out is None:
        out = torch.empty((ncols, _q8_1_bytes(K, 1)), dtype=torch.uint8, device=x.device)
    else:
        _tensor(out, "out", torch.uint8, _q8_1_bytes(K, ncols))
    dev = _device_of((("x", x2), ("out", out)), stream)
    _call("qmv_quantize_q8_1", dev, stream, _ptr(x2), K, ncols, K, _ptr(out))
    return out


def quantize_weights(qtype: int, w, out=None, stream=None):
    """w: fp32 CUDA tensor [M][K] -> uint8 [M][row_bytes] blocks of qtype."""
    import torch

    _tensor(w, "w", torch.float32)
    if w.dim() != 2:
        raise ValueError("w must be 2-D [M][K]")
    M, K = w.shape
    ok = _shape_ok(qtype, M, K)
    if out is None:
        out = torch.empty((M, _row_bytes(qtype, K) if ok else 0), dtype=torch.uint8, device=w.device)
    else:
        _tensor(out, "out", torch.uint8, M * _row_bytes(qtype, K) if ok else 0)
    dev = _device_of((("w", w), ("out", out)), stream)
    _call("qmv_quantize_weights", dev, stream, qtype, _ptr(w), M, K, K, _ptr(out))
    return out


# ---- GEMV ------------------------------------------------------------------------
def _weights(W, name, qtype, M, K, n_mat=1):
    import torch

    return _tensor(W, name, torch.uint8, n_mat * M * _row_bytes(qtype, K) if _shape_ok(qtype, M, K) else 0)


def _q8_1(xq, K, ncols, name="xq"):
    import torch

    return _tensor(xq, name, torch.uint8, _q8_1_bytes(K, ncols) if K > 0 and ncols > 0 else 0)


def mul_mat_vec(qtype: int, W, M: int, K: int, xq, ncols: int, out=None, stream=None):
    """y[ncols][M] = W . x for q8_1 activations xq (ncols rows)."""
    _weights(W, "W", qtype, M, K)
    _q8_1(xq, K, ncols)
    out = _out(out, "out", (ncols, M), W.device, 4 * ncols * M)
    dev = _device_of((("W", W), ("xq", xq), ("out", out)), stream)
    _call("qmv_mul_mat_vec", dev, stream, qtype, _ptr(W), M, K, _ptr(xq), ncols, _ptr(out))
    return out


def mul_mat_vec_gate_up_swiglu(qtype: int, W_gate, W_up, M: int, K: int, xq, ncols: int = 1, out=None,
                               stream=None):
    """y[ncols][M] = (W_up . x) * silu(W_gate . x)."""
    _weights(W_gate, "W_gate", qtype, M, K)
    _weights(W_up, "W_up", qtype, M, K)
    _q8_1(xq, K, ncols)
    out = _out(out, "out", (ncols, M), W_up.device, 4 * ncols * M)
    dev = _device_of((("W_gate", W_gate), ("W_up", W_up), ("xq", xq), ("out", out)), stream)
    _call("qmv_mul_mat_vec_gate_up_swiglu", dev, stream, qtype, _ptr(W_gate), _ptr(W_up), M, K, _ptr(xq), ncols,
          _ptr(out))
    return out


def _ids(ids):
    import torch

    _tensor(ids, "ids", torch.int32)
    if ids.dim() != 2:
        raise ValueError("ids must be 2-D [n_tokens][top_k]")
    return ids.shape


def _status(status):
    import torch

    return None if status is None else _tensor(status, "status", torch.int32, 4)


def mul_mat_vec_id(qtype: int, W, n_expert: int, M: int, K: int, xq, ids, out=None, status=None, stream=None):
    """Expert-indexed GEMV: y[t][k][M] = W[ids[t][k]] . x[t]; ids int32 [n_tokens][top_k]."""
    n_tokens, top_k = _ids(ids)
    _weights(W, "W", qtype, M, K, max(n_expert, 0))
    _q8_1(xq, K, n_tokens)
    _status(status)
    out = _out(out, "out", (n_tokens, top_k, M), W.device, 4 * n_tokens * top_k * M)
    dev = _device_of((("W", W), ("xq", xq), ("ids", ids), ("out", out), ("status", status)), stream)
    _call("qmv_mul_mat_vec_id", dev, stream, qtype, _ptr(W), n_expert, M, K, _ptr(xq), _ptr(ids), n_tokens, top_k,
          _ptr(out), _ptr(status))
    return out


# ---- GEMV with fp32 activations (quantization fused into the GEMV) ---------------
def mul_mat_vec_f32(qtype: int, W, M: int, K: int, x, out=None, stream=None):
    """y[ncols][M] = W . x for fp32 x [ncols][K] (rows may be strided)."""
    x2, ldx = _x2d(x, K)
    ncols = x2.shape[0]
    _weights(W, "W", qtype, M, K)
    out = _out(out, "out", (ncols, M), W.device, 4 * ncols * M)
    dev = _device_of((("W", W), ("x", x2), ("out", out)), stream)
    _call("qmv_mul_mat_vec_f32", dev, stream, qtype, _ptr(W), M, K, _ptr(x2), ldx, ncols, _ptr(out))
    return out


def mul_mat_vec_gate_up_swiglu_f32(qtype: int, W_gate, W_up, M: int, K: int, x, out=None, stream=None):
    """y[ncols][M] = (W_up . x) * silu(W_gate . x) for fp32 x [ncols][K]."""
    x2, ldx = _x2d(x, K)
    ncols = x2.shape[0]
    _weights(W_gate, "W_gate", qtype, M, K)
    _weights(W_up, "W_up", qtype, M, K)
    out = _out(out, "out", (ncols, M), W_up.device, 4 * ncols * M)
    dev = _device_of((("W_gate", W_gate), ("W_up", W_up), ("x", x2), ("out", out)), stream)
    _call("qmv_mul_mat_vec_gate_up_swiglu_f32", dev, stream, qtype, _ptr(W_gate), _ptr(W_up), M, K, _ptr(x2), ldx,
          ncols, _ptr(out))
    return out


def mul_mat_vec_id_f32(qtype: int, W, n_expert: int, M: int, K: int, x, ids, out=None, status=None, stream=None):
    """Expert-indexed GEMV with fp32 tokens x [n_tokens][K]: y[t][k][M] = W[ids[t][k]] . x[t]."""
    n_tokens, top_k = _ids(ids)
    x2, ldx = _x2d(x, K)
    if x2.shape[0] < n_tokens:
        raise ValueError("fewer activation rows than tokens")
    _weights(W, "W", qtype, M, K, max(n_expert, 0))
    _status(status)
    out = _out(out, "out", (n_tokens, top_k, M), W.device, 4 * n_tokens * top_k * M)
    dev = _device_of((("W", W), ("x", x2), ("ids", ids), ("out", out), ("status", status)), stream)
    _call("qmv_mul_mat_vec_id_f32", dev, stream, qtype, _ptr(W), n_expert, M, K, _ptr(x2), ldx, _ptr(ids), n_tokens,
          top_k, _ptr(out), _ptr(status))
    return out


def _activations(xq, x, K, n_rows=None):
    """(named tensor, xq pointer, x pointer, ldx, rows) for exactly one of q8_1 rows
    xq [rows][bytes] or fp32 x [rows][K]; n_rows: the rows the call reads (default all)."""
    if (xq is None) == (x is None):
        raise ValueError("pass exactly one of xq (q8_1) and x (fp32)")
    if x is not None:
        x2, ldx = _x2d(x, K)
        if n_rows is not None and x2.shape[0] < n_rows:
            raise ValueError("fewer activation rows than tokens")
        return ("x", x2), _vp(0), _ptr(x2), ldx, x2.shape[0]
    import torch

    _tensor(xq, "xq", torch.uint8)
    xq2 = xq.unsqueeze(0) if xq.dim() == 1 else xq
    rows = xq2.shape[0]
    _q8_1(xq2, K, n_rows if n_rows is not None else rows)
    return ("xq", xq2), _ptr(xq2), _vp(0), 0, rows


def mul_mat_vec_fused(qtype: int, W_up, M: int, K: int, xq=None, x=None, W_gate=None, bias=None, gate_bias=None,
                      out=None, stream=None):
    """y = W_up.x (+ bias), or (W_up.x + bias) * silu(W_gate.x + gate_bias) with W_gate; q8_1 xq or fp32 x."""
    import torch

    act, pq, px, ldx, ncols = _activations(xq, x, K)
    _weights(W_up, "W_up", qtype, M, K)
    if W_gate is not None:
        _weights(W_gate, "W_gate", qtype, M, K)
    for name, b in (("bias", bias), ("gate_bias", gate_bias)):
        if b is not None:
            _tensor(b, name, torch.float32, 4 * M)
    out = _out(out, "out", (ncols, M), W_up.device, 4 * ncols * M)
    dev = _device_of((("W_up", W_up), ("W_gate", W_gate), act, ("bias", bias), ("gate_bias", gate_bias),
                      ("out", out)), stream)
    _call("qmv_mul_mat_vec_fused", dev, stream, qtype, _ptr(W_up), _ptr(W_gate), M, K, pq, px, ldx, ncols,
          _ptr(bias), _ptr(gate_bias), _ptr(out))
    return out


def mul_mat_vec_fused_q8_1(qtype: int, W_up, M: int, K: int, xq=None, x=None, W_gate=None, bias=None,
                           gate_bias=None, out=None, out_q8_1=None, want_y=True, stream=None):
    """mul_mat_vec_fused of one column whose result is also written as q8_1
    blocks (uint8 [q8_1_bytes(M)], the next GEMV's activations): returns
    (y [1][M] or None when want_y is False and out is None, yq)."""
    import torch

    act, pq, px, ldx, ncols = _activations(xq, x, K)
    if ncols != 1:
        raise ValueError("mul_mat_vec_fused_q8_1 takes one activation column")
    _weights(W_up, "W_up", qtype, M, K)
    if W_gate is not None:
        _weights(W_gate, "W_gate", qtype, M, K)
    for name, b in (("bias", bias), ("gate_bias", gate_bias)):
        if b is not None:
            _tensor(b, name, torch.float32, 4 * M)
    if out is not None or want_y:
        out = _out(out, "out", (1, M), W_up.device, 4 * M)
    nq = _q8_1_bytes(M, 1)
    if out_q8_1 is None:
        out_q8_1 = torch.empty((1, nq), dtype=torch.uint8, device=W_up.device)
    else:
        _tensor(out_q8_1, "out_q8_1", torch.uint8, nq)
    dev = _device_of((("W_up", W_up), ("W_gate", W_gate), act, ("bias", bias), ("gate_bias", gate_bias),
                      ("out", out), ("out_q8_1", out_q8_1)), stream)
    _call("qmv_mul_mat_vec_fused_q8_1", dev, stream, qtype, _ptr(W_up), _ptr(W_gate), M, K, pq, px, ldx, 1,
          _ptr(bias), _ptr(gate_bias), _ptr(out), _ptr(out_q8_1))
    return out, out_q8_1


def mul_mat_vec_id_fused(qtype: int, W, n_expert: int, M: int, K: int, ids, xq=None, x=None, W_gate=None,
                         W_shared=None, W_shared_gate=None, out=None, out_shared=None, status=None, stream=None):
    """Expert-indexed GEMV (q8_1 xq or fp32 x, one row per token), optionally gated
    ((W.x) * silu(W_gate.x) per routed slot) and with a shared expert (gated like
    the routed ones): returns (y [n_tokens][top_k][M], y_shared [n_tokens][M] or None)."""
    n_tokens, top_k = _ids(ids)
    act, pq, px, ldx, _ = _activations(xq, x, K, n_tokens)
    ne = max(n_expert, 0)
    _weights(W, "W", qtype, M, K, ne)
    if W_gate is not None:
        _weights(W_gate, "W_gate", qtype, M, K, ne)
    for name, Ws in (("W_shared", W_shared), ("W_shared_gate", W_shared_gate)):
        if Ws is not None:
            _weights(Ws, name, qtype, M, K)
    _status(status)
    out = _out(out, "out", (n_tokens, top_k, M), W.device, 4 * n_tokens * top_k * M)
    if W_shared is not None:
        out_shared = _out(out_shared, "out_shared", (n_tokens, M), W.device, 4 * n_tokens * M)
    else:
        out_shared = None
    dev = _device_of((("W", W), ("W_gate", W_gate), ("W_shared", W_shared), ("W_shared_gate", W_shared_gate), act,
                      ("ids", ids), ("out", out), ("out_shared", out_shared), ("status", status)), stream)
    _call("qmv_mul_mat_vec_id_fused", dev, stream, qtype, _ptr(W), _ptr(W_gate), n_expert, M, K, pq, px, ldx,
          _ptr(ids), n_tokens, top_k, _ptr(out), _ptr(W_shared), _ptr(W_shared_gate), _ptr(out_shared),
          _ptr(status))
    return out, out_shared


def debug_subblock_sums(qtype: int, W, M: int, K: int, xq, ncols: int, stream=None):
    """Exact int32 per-sub-block sums [ncols][M][n] (see include/qmv.h)."""
    import torch

    _weights(W, "W", qtype, M, K)
    _q8_1(xq, K, ncols)
    n = K // 32 if qtype == Q4_0 else K // 16
    out = torch.empty((max(ncols, 0), max(M, 0), max(n, 0)), dtype=torch.int32, device=W.device)
    dev = _device_of((("W", W), ("xq", xq)), stream)
    _call("qmv_debug_subblock_sums", dev, stream, qtype, _ptr(W), M, K, _ptr(xq), ncols, _ptr(out))
    return out


def debug_f32_withheld_share(qtype: int, W, M: int, K: int, x, wait_ns: int, out=None, stream=None):
    """Test only: mul_mat_vec_f32 with one CTA of every cluster withholding its
    share of the quantized activations, so that its partner's bounded wait
    (wait_ns) runs out; that partner's rows come back NaN and the device fault
    word gets code 2 (see include/qmv_debug.h).  One or two columns."""
    x2, ldx = _x2d(x, K)
    ncols = x2.shape[0]
    _weights(W, "W", qtype, M, K)
    out = _out(out, "out", (ncols, M), W.device, 4 * ncols * M)
    dev = _device_of((("W", W), ("x", x2), ("out", out)), stream)
    _call("qmv_debug_f32_withheld_share", dev, stream, qtype, _ptr(W), M, K, _ptr(x2), ldx, ncols, _ptr(out),
          ctypes.c_uint64(wait_ns))
    return out


def debug_f32_withheld_share_q8_1(qtype: int, W, M: int, K: int, x, wait_ns: int, stream=None):
    """Test only: mul_mat_vec_fused_q8_1 (plain, one column, fp32 x) with the
    withheld share of debug_f32_withheld_share; returns (y, yq).  The rows of
    the warps that give up come back NaN, and their q8_1 blocks with a NaN
    scale (see include/qmv_debug.h)."""
    import torch

    x2, _ = _x2d(x, K)
    if x2.shape[0] != 1 or not x2.is_contiguous():
        raise ValueError("x must be one contiguous column")
    _weights(W, "W", qtype, M, K)
    y = torch.empty((1, M), dtype=torch.float32, device=W.device)
    yq = torch.empty((1, _q8_1_bytes(M, 1)), dtype=torch.uint8, device=W.device)
    dev = _device_of((("W", W), ("x", x2)), stream)
    _call("qmv_debug_f32_withheld_share_q8_1", dev, stream, qtype, _ptr(W), M, K, _ptr(x2), _ptr(y), _ptr(yq),
          ctypes.c_uint64(wait_ns))
    return y, yq


TRACE_MAX_CTAS = 1024
TRACE_WORDS = 6  # stamps per CTA: entry, wait returned, first loads, own staging, staged, done


def debug_trace(buf=None, slots: int = 0):
    """Diagnostics: per-CTA timestamps of the next `slots` GEMV launches that
    have an instrumented twin (plain, 1-2 columns; gate/up, 1 column) into buf
    (int64 CUDA tensor of slots*1024*6, zeroed); None stops (see
    include/qmv_debug.h, qmv_debug_trace)."""
    import torch

    if buf is None:
        _check("qmv_debug_trace", lib().qmv_debug_trace(None, 0))
        return
    _tensor(buf, "buf", torch.int64, slots * TRACE_MAX_CTAS * TRACE_WORDS * 8)
    _device_of((("buf", buf),))
    _check("qmv_debug_trace", lib().qmv_debug_trace(_ptr(buf), slots))


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
    import torch

    _tensor(buf, "buf")
    _tensor(sink, "sink", torch.int32, 4)
    dev = _device_of((("buf", buf), ("sink", sink)), stream)
    _call("qmv_read_bandwidth_probe", dev, stream, _ptr(buf), buf.numel() * buf.element_size(), _ptr(sink))


def describe_gemv(qtype: int, M: int, K: int, ncols: int = 1, gate_up: bool = False, fp32_input: bool = False):
    """The launch geometry the library would use for this GEMV (nothing is launched), as a dict."""
    info = LaunchInfo()
    _check("qmv_describe_gemv", lib().qmv_describe_gemv(qtype, 1 if gate_up else 0, M, K, ncols,
                                                       1 if fp32_input else 0, ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in LaunchInfo._fields_}


def set_early_warps(qtype: int, early_warps: int = 0):
    """Decoding warps that request tiles before the dependency wait (0: all)."""
    _check("qmv_set_early_warps", lib().qmv_set_early_warps(qtype, early_warps))


def set_early_delay(qtype: int, ns: int = 0):
    """Delay in ns of the early weight requests of launches that request their
    whole matrix early (0: the default, -1: none; see include/qmv.h)."""
    _check("qmv_set_early_delay", lib().qmv_set_early_delay(qtype, ns))


def set_mma_min_cols(qtype: int, min_cols: int = 0):
    """Columns from which the plain Q4_K GEMV decodes with mma.sync (0: the default, never; 9: never)."""
    _check("qmv_set_mma_min_cols", lib().qmv_set_mma_min_cols(qtype, min_cols))


def set_pdl(enable: bool):
    _check("qmv_set_pdl", lib().qmv_set_pdl(1 if enable else 0))


def set_checked(enable: bool):
    """Checked mode: every call first verifies on the host that each argument's
    byte range lies inside one device allocation (QMV_ERR_RANGE otherwise)."""
    _check("qmv_set_checked", lib().qmv_set_checked(1 if enable else 0))
