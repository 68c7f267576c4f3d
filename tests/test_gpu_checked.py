"""Checked mode on the GPU (qmv_set_checked / QMV_CHECKED).

With the mode on, every call gives the same bits as without it.  At the edge
of a device allocation, each pointer argument whose byte range ends exactly at
the allocation's end is accepted, and the same range moved one element (one
row for weights) further is rejected with QMV_ERR_RANGE.

The boundary calls run inside a CUDA graph capture that is never replayed: a
call the check lets through is only recorded, never executed, so no kernel
ever runs on a range outside its allocation, whatever the check returns.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, RANGE = 0, 9


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
    yield qq
    qq.set_checked(False)


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint32)


def segment_of(ptr):
    """(base, size) of the driver allocation the caching allocator placed ptr in."""
    import torch

    for seg in torch.cuda.memory_snapshot():
        a, n = seg["address"], seg["total_size"]
        if a <= ptr < a + n:
            return a, n
    raise AssertionError("pointer not in any allocator segment")


def captured(calls):
    """Run each call (a function of the stream handle returning a status)
    inside one graph capture that is discarded without being replayed."""
    import torch

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rcs = [fn(st) for fn in calls]
    del g
    torch.cuda.synchronize()
    return rcs


def test_checked_calls_match_unchecked(q):
    t, M, K = oracle.Q4_K, 300, 4096
    W = dev(oracle.quantize_rows(t, synthetic.weights_f32(1600, M, K)))
    Wg = dev(oracle.quantize_rows(t, synthetic.weights_f32(1601, M, K)))
    x = dev(synthetic.activations_f32(1602, 2, K))
    ids = dev(synthetic.moe_ids(1603, 2, 2, 3))
    W3 = dev(oracle.quantize_rows(t, synthetic.weights_f32(1604, 3 * M, K)).reshape(3, -1))
    b = dev(synthetic.activations_f32(1605, 1, M)[0])

    def run():
        xq = q.quantize_q8_1(x)
        outs = [xq, q.mul_mat_vec(t, W, M, K, xq, 2), q.mul_mat_vec_gate_up_swiglu(t, Wg, W, M, K, xq, 2),
                q.mul_mat_vec_id(t, W3, 3, M, K, xq, ids), q.mul_mat_vec_f32(t, W, M, K, x),
                q.mul_mat_vec_fused(t, W, M, K, x=x, W_gate=Wg, bias=b, gate_bias=b),
                q.debug_subblock_sums(t, W, M, K, xq, 2), q.quantize_weights(t, x)]
        y, ys = q.mul_mat_vec_id_fused(t, W3, 3, M, K, ids, x=x, W_shared=W)
        return [bits(o) for o in outs + [y, ys]]

    q.set_checked(False)
    ref = run()
    q.set_checked(True)
    try:
        got = run()
    finally:
        q.set_checked(False)
    for i, (a, b_) in enumerate(zip(ref, got)):
        assert np.array_equal(a, b_), i


def test_ranges_at_the_end_of_an_allocation(q):
    import torch

    L = q.lib()
    buf = torch.zeros(24 << 20, dtype=torch.uint8, device="cuda")   # a 24 MiB allocation of its own
    a, n = segment_of(buf.data_ptr())
    end = a + n
    lo = ctypes.c_void_p(a)          # room for every argument that is not under test
    nul = ctypes.c_void_p(0)

    def at(nbytes, past=0):
        """The range of nbytes ending at the allocation's end, moved `past` bytes further."""
        return ctypes.c_void_p(end - nbytes + past)

    t, M, K, rb = oracle.Q4_K, 16, 4096, 2304      # Q4_K rows of 4096 weights: 16 blocks of 144 bytes
    E, T, k, nc, ldx = 4, 2, 2, 2, 4160
    qb = q.q8_1_bytes(K, nc)
    xb = ((nc - 1) * ldx + K) * 4
    per_row = K // 16
    cases = {
        # name: (call given a pointer, bytes the argument covers, one element past)
        "W": (lambda p, s: L.qmv_mul_mat_vec(t, p, M, K, lo, nc, lo, s), M * rb, rb),
        "xq": (lambda p, s: L.qmv_mul_mat_vec(t, lo, M, K, p, nc, lo, s), qb, 4),
        "y": (lambda p, s: L.qmv_mul_mat_vec(t, lo, M, K, lo, nc, p, s), nc * M * 4, 4),
        "W_gate": (lambda p, s: L.qmv_mul_mat_vec_gate_up_swiglu(t, p, lo, M, K, lo, nc, lo, s), M * rb, rb),
        "W_experts": (lambda p, s: L.qmv_mul_mat_vec_id(t, p, E, M, K, lo, lo, T, k, lo, lo, s), E * M * rb, rb),
        "ids": (lambda p, s: L.qmv_mul_mat_vec_id(t, lo, E, M, K, lo, p, T, k, lo, lo, s), T * k * 4, 4),
        "y_moe": (lambda p, s: L.qmv_mul_mat_vec_id(t, lo, E, M, K, lo, lo, T, k, p, lo, s), T * k * M * 4, 4),
        "x": (lambda p, s: L.qmv_mul_mat_vec_f32(t, lo, M, K, p, ldx, nc, lo, s), xb, 4),
        "x_gate": (lambda p, s: L.qmv_mul_mat_vec_gate_up_swiglu_f32(t, lo, lo, M, K, p, ldx, nc, lo, s), xb, 4),
        "x_moe": (lambda p, s: L.qmv_mul_mat_vec_id_f32(t, lo, E, M, K, p, ldx, lo, T, k, lo, lo, s), xb, 4),
        "bias": (lambda p, s: L.qmv_mul_mat_vec_fused(t, lo, lo, M, K, lo, nul, 0, nc, p, lo, lo, s), M * 4, 4),
        "gate_bias": (lambda p, s: L.qmv_mul_mat_vec_fused(t, lo, lo, M, K, lo, nul, 0, nc, lo, p, lo, s),
                      M * 4, 4),
        "W_shared": (lambda p, s: L.qmv_mul_mat_vec_id_fused(t, lo, nul, E, M, K, lo, nul, 0, lo, T, k, lo,
                                                             p, nul, lo, lo, s), M * rb, rb),
        "W_shared_gate": (lambda p, s: L.qmv_mul_mat_vec_id_fused(t, lo, lo, E, M, K, lo, nul, 0, lo, T, k, lo,
                                                                  lo, p, lo, lo, s), M * rb, rb),
        "y_shared": (lambda p, s: L.qmv_mul_mat_vec_id_fused(t, lo, nul, E, M, K, lo, nul, 0, lo, T, k, lo,
                                                             lo, nul, p, lo, s), T * M * 4, 4),
        "quantize_x": (lambda p, s: L.qmv_quantize_q8_1(p, K, nc, ldx, lo, s), xb, 4),
        "quantize_xq": (lambda p, s: L.qmv_quantize_q8_1(lo, K, nc, ldx, p, s), qb, 4),
        "weights_w": (lambda p, s: L.qmv_quantize_weights(t, p, M, K, ldx, lo, s), ((M - 1) * ldx + K) * 4, 4),
        "weights_W": (lambda p, s: L.qmv_quantize_weights(t, lo, M, K, ldx, p, s), M * rb, rb),
        "debug_out": (lambda p, s: L.qmv_debug_subblock_sums(t, lo, M, K, lo, nc, p, s), nc * M * per_row * 4, 4),
        # (the 4-byte sink cannot straddle an allocation end without breaking
        # its alignment first, so only the buffer's range is probed here)
        "probe_buf": (lambda p, s: L.qmv_read_bandwidth_probe(p, 4096, lo, s), 4096, 16),
    }
    names = list(cases)
    # every call once for real with all its pointers at the allocation's start, where every range
    # fits (zeros: valid blocks, expert id 0), so that each kernel is loaded before the capture
    st0 = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for name in names:
        assert cases[name][0](lo, st0) == OK, name
    torch.cuda.synchronize()
    calls = []
    for name in names:
        fn, nbytes, step = cases[name]
        assert nbytes <= n // 2
        calls.append(lambda s, fn=fn, nbytes=nbytes: fn(at(nbytes), s))
        calls.append(lambda s, fn=fn, nbytes=nbytes, step=step: fn(at(nbytes, step), s))
    q.set_checked(True)
    try:
        rcs = captured(calls)
    finally:
        q.set_checked(False)
    for i, name in enumerate(names):
        assert (rcs[2 * i], rcs[2 * i + 1]) == (OK, RANGE), name
    # the same out-of-range calls without the mode are accepted (the mode is what rejects them)
    fn, nbytes, step = cases["W"]
    assert captured([lambda s: fn(at(nbytes, step), s)]) == [OK]
    del buf


def test_host_memory_and_huge_shapes_are_rejected(q):
    import torch

    L = q.lib()
    t, M, K = oracle.Q4_K, 16, 4096
    W = torch.zeros((M, q.row_bytes(t, K)), dtype=torch.uint8, device="cuda")
    xq = torch.zeros(q.q8_1_bytes(K, 1), dtype=torch.uint8, device="cuda")
    y = torch.zeros(M, dtype=torch.float32, device="cuda")
    host_y = np.zeros(M, dtype=np.float32)            # pageable host memory
    p = lambda tt: ctypes.c_void_p(tt.data_ptr())
    st0 = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.qmv_mul_mat_vec(t, p(W), M, K, p(xq), 1, p(y), st0) == OK     # loads the kernel
    torch.cuda.synchronize()
    calls = [
        lambda s: L.qmv_mul_mat_vec(t, p(W), M, K, p(xq), 1, p(y), s),
        lambda s: L.qmv_mul_mat_vec(t, p(W), M, K, p(xq), 1, ctypes.c_void_p(host_y.ctypes.data), s),
        lambda s: L.qmv_mul_mat_vec(t, p(W), 1 << 30, K, p(xq), 1, p(y), s),
        lambda s: L.qmv_mul_mat_vec_id(t, p(W), 60000, M, K, p(xq), p(y), 1, 1, p(y), ctypes.c_void_p(0), s),
    ]
    q.set_checked(True)
    try:
        assert captured(calls) == [OK, RANGE, RANGE, RANGE]
    finally:
        q.set_checked(False)


def test_environment_variable_turns_the_mode_on(q):
    """QMV_CHECKED=1 in a fresh process turns the check on; QMV_CHECKED=0 leaves it off."""
    code = (
        "import ctypes, torch, numpy as np\n"
        "import quantized_decode_gemv_qmv_gb300 as q\n"
        "L = q.lib()\n"
        "W = torch.zeros((16, q.row_bytes(12, 4096)), dtype=torch.uint8, device='cuda')\n"
        "xq = torch.zeros(q.q8_1_bytes(4096, 1), dtype=torch.uint8, device='cuda')\n"
        "y = torch.zeros(16, dtype=torch.float32, device='cuda')\n"
        "P = lambda t: ctypes.c_void_p(t.data_ptr())\n"
        "s0 = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)\n"
        "assert L.qmv_mul_mat_vec(12, P(W), 16, 4096, P(xq), 1, P(y), s0) == 0\n"
        "torch.cuda.synchronize()\n"
        "g = torch.cuda.CUDAGraph()\n"
        "with torch.cuda.graph(g, stream=torch.cuda.Stream(), capture_error_mode='relaxed'):\n"
        "    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)\n"
        "    rc = L.qmv_mul_mat_vec(12, P(W), 1 << 20, 4096, P(xq), 1, P(y), s)\n"
        "del g\n"
        "print('rc', rc)\n"
    )
    for val, want in (("1", RANGE), ("0", OK)):
        env = dict(os.environ, QMV_CHECKED=val, PYTHONPATH=ROOT)
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                             timeout=300)
        assert out.returncode == 0, out.stderr[-2000:]
        assert f"rc {want}" in out.stdout, (val, out.stdout)
