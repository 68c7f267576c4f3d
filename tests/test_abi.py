"""The C-ABI library builds, loads, exports every symbol include/qmv.h
declares, agrees with the oracle on sizes, and rejects bad arguments on the
host before launching anything (no GPU needed: no compute call is made)."""
import ctypes
import os
import re
import shutil

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qlib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__

    __graft_entry__.build()
    import quantized_decode_gemv_qmv_gb300 as q

    return q


def _declared_symbols():
    inc = os.path.join(ROOT, "include")
    text = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports(qlib):
    assert _declared_symbols() == sorted(qlib.EXPORTS)


def test_library_exports_every_declared_symbol(qlib):
    L = ctypes.CDLL(qlib.library_path())
    for name in _declared_symbols():
        assert hasattr(L, name), name


@pytest.mark.parametrize("t", oracle.WEIGHT_TYPES)
@pytest.mark.parametrize("K", [32, 256, 4096, 11008, 14336, 2048 + 256])
def test_sizes_agree_with_oracle(qlib, t, K):
    qk = oracle.block_elems(t)
    exp = oracle.row_bytes(t, K) if K % qk == 0 else 0
    assert qlib.row_bytes(t, K) == exp
    assert qlib.q8_1_padded_k(K) == oracle.q8_1_padded_k(K)
    assert qlib.q8_1_bytes(K, 3) == 3 * oracle.q8_1_row_bytes(K)


def test_status_strings_and_version(qlib):
    L = qlib.lib()
    assert L.qmv_status_str(0) == b"ok"
    assert L.qmv_status_str(3) == b"bad shape"
    assert L.qmv_status_str(9) == b"argument outside its device allocation"
    assert L.qmv_status_str(11) == b"unknown status"
    assert L.qmv_version() >= 10000


def test_host_validation_rejects_bad_arguments(qlib):
    L = qlib.lib()
    p = ctypes.c_void_p(0x1000)      # never dereferenced: validation fails first
    nul = ctypes.c_void_p(0)
    # bad type, null pointers, bad shapes and column counts
    assert L.qmv_mul_mat_vec(5, p, 16, 256, p, 1, p, nul) == 2
    assert L.qmv_mul_mat_vec(12, nul, 16, 256, p, 1, p, nul) == 1
    assert L.qmv_mul_mat_vec(12, p, 16, 250, p, 1, p, nul) == 3
    assert L.qmv_mul_mat_vec(12, p, 0, 256, p, 1, p, nul) == 3
    assert L.qmv_mul_mat_vec(12, p, 16, 256, p, 0, p, nul) == 4
    assert L.qmv_mul_mat_vec(12, p, 16, 256, p, 9, p, nul) == 4
    assert L.qmv_mul_mat_vec(2, p, 16, 48, p, 1, p, nul) == 3
    # misaligned pointers
    assert L.qmv_mul_mat_vec(12, ctypes.c_void_p(0x1001), 16, 256, p, 1, p, nul) == 5
    assert L.qmv_mul_mat_vec(12, p, 16, 256, ctypes.c_void_p(0x1002), 1, p, nul) == 5
    # gate/up and MoE specifics
    assert L.qmv_mul_mat_vec_gate_up_swiglu(12, nul, p, 16, 256, p, 1, p, nul) == 1
    assert L.qmv_mul_mat_vec_id(12, p, 8, 16, 256, p, nul, 4, 2, p, nul, nul) == 1
    assert L.qmv_mul_mat_vec_id(12, p, 8, 16, 256, p, p, 9, 2, p, nul, nul) == 4
    assert L.qmv_mul_mat_vec_id(12, p, 0, 16, 256, p, p, 4, 2, p, nul, nul) == 3
    assert L.qmv_mul_mat_vec_id(12, p, 8, 16, 256, p, p, 4, 33, p, nul, nul) == 3
    assert L.qmv_mul_mat_vec_id(12, p, 65535, 16, 256, p, p, 4, 2, p, nul, nul) == 3  # grid rows: at most 65534
    # quantizers
    assert L.qmv_quantize_q8_1(nul, 256, 1, 256, p, nul) == 1
    assert L.qmv_quantize_q8_1(p, 256, 1, 100, p, nul) == 3
    assert L.qmv_quantize_weights(12, p, 4, 100, 100, p, nul) == 3
    assert L.qmv_quantize_weights(9, p, 4, 256, 256, p, nul) == 2
    assert L.qmv_debug_subblock_sums(14, p, 4, 256, p, 0, p, nul) == 4
    # the withheld-share test entry: the fp32 call's checks, and a wait limit of 1 ns .. 1 s
    wh = L.qmv_debug_f32_withheld_share
    assert wh(12, p, 16, 4096, p, 4096, 1, p, 0, nul) == 3
    assert wh(12, p, 16, 4096, p, 4096, 1, p, 1000000001, nul) == 3
    assert wh(14, p, 16, 2304, p, 2304, 1, p, 1000, nul) == 3
    assert wh(12, p, 16, 4096, p, 4096, 9, p, 1000, nul) == 4
    assert wh(12, ctypes.c_void_p(0x1008), 16, 4096, p, 4096, 1, p, 1000, nul) == 5
    whq = L.qmv_debug_f32_withheld_share_q8_1
    assert whq(12, p, 16, 4096, p, p, p, 0, nul) == 3
    assert whq(12, p, 16, 4096, p, p, nul, 1000, nul) == 1
    assert whq(12, p, 16, 4096, p, nul, nul, 1000, nul) == 1
    assert whq(12, p, 16, 4096, p, p, ctypes.c_void_p(0x1002), 1000, nul) == 5
    assert whq(14, p, 16, 2304, p, p, p, 1000, nul) == 3
    assert whq(12, ctypes.c_void_p(0x1008), 16, 4096, p, p, p, 1000, nul) == 5
    # fused fp32-input calls: the tile kernel's shapes (Q4_0/Q4_K: K % 256, Q6_K: K % 2048), 16-byte aligned W
    assert L.qmv_mul_mat_vec_f32(14, p, 16, 2304, p, 2304, 1, p, nul) == 3
    assert L.qmv_mul_mat_vec_f32(2, p, 16, 96, p, 96, 1, p, nul) == 3
    assert L.qmv_mul_mat_vec_f32(12, p, 16, 4096, p, 4000, 1, p, nul) == 3
    assert L.qmv_mul_mat_vec_f32(12, ctypes.c_void_p(0x1008), 16, 4096, p, 4096, 1, p, nul) == 5
    assert L.qmv_mul_mat_vec_f32(12, p, 16, 4096, nul, 4096, 1, p, nul) == 1
    assert L.qmv_mul_mat_vec_f32(12, p, 16, 4096, p, 4096, 9, p, nul) == 4
    assert L.qmv_mul_mat_vec_gate_up_swiglu_f32(12, nul, p, 16, 4096, p, 4096, 1, p, nul) == 1
    assert L.qmv_mul_mat_vec_gate_up_swiglu_f32(12, ctypes.c_void_p(0x1008), p, 16, 4096, p, 4096, 1, p, nul) == 5
    assert L.qmv_mul_mat_vec_id_f32(12, p, 8, 16, 4096, p, 4096, nul, 4, 2, p, nul, nul) == 1
    assert L.qmv_mul_mat_vec_id_f32(14, p, 8, 16, 2304, p, 2304, p, 4, 2, p, nul, nul) == 3
    # fused epilogue extras: one activation kind, gate bias needs a gate, tile shapes, aligned biases
    fm = L.qmv_mul_mat_vec_fused
    assert fm(12, p, nul, 16, 4096, nul, nul, 0, 1, nul, nul, p, nul) == 1
    assert fm(12, p, nul, 16, 4096, p, p, 4096, 1, nul, nul, p, nul) == 3
    assert fm(12, p, nul, 16, 4096, p, nul, 0, 1, nul, p, p, nul) == 3
    assert fm(12, p, p, 16, 4096, p, nul, 0, 1, ctypes.c_void_p(0x1002), nul, p, nul) == 5
    assert fm(14, p, nul, 16, 2304, p, nul, 0, 1, nul, nul, p, nul) == 3
    assert fm(12, p, nul, 16, 4096, nul, p, 4000, 1, nul, nul, p, nul) == 3
    assert fm(12, p, nul, 16, 4096, p, nul, 0, 0, nul, nul, p, nul) == 4
    assert fm(12, p, ctypes.c_void_p(0x1008), 16, 4096, p, nul, 0, 1, nul, nul, p, nul) == 5
    assert fm(9, p, nul, 16, 4096, p, nul, 0, 1, nul, nul, p, nul) == 2
    # the q8_1-output form: yq required and 4-byte aligned, y optional, one column
    fq = L.qmv_mul_mat_vec_fused_q8_1  # (type, W_up, W_gate, M, K, xq, x, ldx, ncols, b, gb, y, yq, s)
    assert fq(12, p, nul, 16, 4096, p, nul, 0, 1, nul, nul, p, nul, nul) == 1
    assert fq(12, p, nul, 16, 4096, nul, nul, 0, 1, nul, nul, nul, p, nul) == 1
    assert fq(12, p, nul, 16, 4096, p, p, 4096, 1, nul, nul, nul, p, nul) == 3
    assert fq(12, p, nul, 16, 4096, p, nul, 0, 1, nul, nul, nul, ctypes.c_void_p(0x1002), nul) == 5
    assert fq(12, p, nul, 16, 4096, p, nul, 0, 2, nul, nul, nul, p, nul) == 4
    assert fq(12, p, nul, 16, 4096, p, nul, 0, 1, nul, p, nul, p, nul) == 3
    assert fq(14, p, nul, 16, 2304, p, nul, 0, 1, nul, nul, nul, p, nul) == 3
    assert fq(9, p, nul, 16, 4096, p, nul, 0, 1, nul, nul, nul, p, nul) == 2
    im = L.qmv_mul_mat_vec_id_fused   # (type, W, W_gate, E, M, K, xq, x, ldx, ids, T, k, y, Ws, Wsg, ys, st, s)
    assert im(12, p, nul, 8, 16, 4096, nul, nul, 0, p, 4, 2, p, nul, nul, nul, nul, nul) == 1
    assert im(12, p, nul, 8, 16, 4096, p, p, 4096, p, 4, 2, p, nul, nul, nul, nul, nul) == 3
    assert im(12, p, nul, 8, 16, 4096, p, nul, 0, p, 4, 2, p, p, nul, nul, nul, nul) == 1    # Ws without ys
    assert im(12, p, nul, 8, 16, 4096, p, nul, 0, p, 4, 2, p, nul, nul, p, nul, nul) == 1    # ys without Ws
    assert im(12, p, p, 8, 16, 4096, p, nul, 0, p, 4, 2, p, p, nul, p, nul, nul) == 1        # gated, no shared gate
    assert im(12, p, nul, 8, 16, 4096, p, nul, 0, p, 4, 2, p, p, p, p, nul, nul) == 1        # shared gate, not gated
    assert im(12, p, nul, 8, 16, 4096, p, nul, 0, p, 4, 2, p, nul, p, nul, nul, nul) == 3    # shared gate alone
    assert im(12, p, nul, 8, 16, 4096, p, nul, 0, p, 4, 2, p, ctypes.c_void_p(0x1008), nul, p, nul, nul) == 5
    assert im(12, p, ctypes.c_void_p(0x1008), 8, 16, 4096, p, nul, 0, p, 4, 2, p, nul, nul, nul, nul, nul) == 5
    assert im(12, p, nul, 8, 16, 4096, p, nul, 0, p, 9, 2, p, p, nul, p, nul, nul) == 4
    assert im(12, p, nul, 8, 16, 4096, p, nul, 0, nul, 4, 2, p, p, nul, p, nul, nul) == 1
    assert im(14, p, nul, 8, 16, 2304, p, nul, 0, p, 4, 2, p, p, nul, p, nul, nul) == 3
    # tuning knobs validate too
    assert L.qmv_set_tuning(12, 100, 0, 0, 0, 0, 0) == 3
    assert L.qmv_set_tuning(12, 544, 0, 0, 0, 0, 0) == 3
    assert L.qmv_set_tuning(12, 0, 0, 0, 0, 5, 0) == 3
    assert L.qmv_set_tuning(12, 0, 0, 0, 0, 0, 9) == 3
    assert L.qmv_set_tuning(12, 0, 0, 0, 0, 0, -1) == 3
    assert L.qmv_set_tuning(3, 0, 0, 0, 0, 0, 0) == 2
    assert L.qmv_set_tuning(12, 0, 0, 0, 0, 0, 0) == 0
    assert L.qmv_set_stream_tuning(12, 13, 0) == 3
    assert L.qmv_set_stream_tuning(12, 0, 5) == 3
    assert L.qmv_set_stream_tuning(12, -1, 0) == 3
    assert L.qmv_set_stream_tuning(9, 0, 0) == 2
    assert L.qmv_set_stream_tuning(12, 0, 0) == 0
    assert L.qmv_set_mma_min_cols(12, 10) == 3
    assert L.qmv_set_mma_min_cols(12, -1) == 3
    assert L.qmv_set_mma_min_cols(9, 0) == 2
    assert L.qmv_set_mma_min_cols(12, 0) == 0
    assert L.qmv_set_early_warps(12, 13) == 3 and L.qmv_set_early_warps(12, -1) == 3
    assert L.qmv_set_early_warps(2, 0) == 0 and L.qmv_set_early_warps(9, 0) == 2
    assert L.qmv_set_early_delay(12, -2) == 3 and L.qmv_set_early_delay(12, 100001) == 3
    assert L.qmv_set_early_delay(9, 0) == 2 and L.qmv_set_early_delay(12, -1) == 0
    assert L.qmv_set_early_delay(12, 0) == 0
    assert L.qmv_debug_trace(p, -1) == 3 and L.qmv_debug_trace(ctypes.c_void_p(0x1004), 1) == 5
    assert L.qmv_debug_trace(nul, 0) == 0
    rp = L.qmv_read_bandwidth_probe
    assert rp(nul, 16, p, nul) == 1 and rp(p, 16, nul, nul) == 1
    assert rp(p, 0, p, nul) == 3 and rp(p, 17, p, nul) == 3
    assert rp(ctypes.c_void_p(0x1008), 16, p, nul) == 5
    info = qlib.LaunchInfo()
    assert L.qmv_describe_gemv(12, 0, 16, 4096, 1, 0, None) == 1
    assert L.qmv_describe_gemv(12, 0, 16, 250, 1, 0, ctypes.byref(info)) == 3
    assert L.qmv_describe_gemv(12, 0, 16, 4096, 9, 0, ctypes.byref(info)) == 4
    assert L.qmv_describe_gemv(5, 0, 16, 4096, 1, 0, ctypes.byref(info)) == 2
    assert L.qmv_describe_gemv(14, 0, 16, 2304, 1, 1, ctypes.byref(info)) == 3  # fp32 input: Q6_K K % 2048


def test_checked_mode_runs_after_the_argument_checks(qlib):
    """Checked mode only adds the byte-range check; every argument error is
    still reported with its own status before any range is queried."""
    L = qlib.lib()
    assert L.qmv_set_checked(1) == 0
    try:
        test_host_validation_rejects_bad_arguments(qlib)
    finally:
        assert L.qmv_set_checked(0) == 0


GEOM_PROBE = """
import ctypes, sys
sys.path.insert(0, sys.argv[1])
import quantized_decode_gemv_qmv_gb300 as q
L = q.lib()
p = ctypes.c_void_p(0x1000)
# a call whose arguments pass the host checks, so the environment override is
# read next; with a malformed spec it fails before any CUDA call
print('rc', L.qmv_mul_mat_vec(12, p, 16, 256, p, 1, p, ctypes.c_void_p(0)))
"""


@pytest.mark.parametrize("spec,want", [
    ("q4_K:threads=256,stages=3;q6_K:cluster=1", None),   # valid: the call goes on to the device query
    ("q4_K:threads=544", 10),                             # out of range (at most 384 threads)
    ("q4_K:stages=x", 10),                                # not a number
    ("q5_K:stages=2", 10),                                # unknown type
    ("q4_K:warps=4", 10),                                 # unknown key
    ("q4_K", 10),                                         # no key list
])
def test_geometry_environment_override(qlib, spec, want):
    """QMV_GEOM is parsed once, through the setters' range checks; a bad spec
    fails every GEMV call with QMV_ERR_CONFIG before anything reaches CUDA."""
    import subprocess
    import sys

    import torch

    if want is None and torch.cuda.is_available():
        pytest.skip("a valid spec would launch on the placeholder pointers")
    env = dict(os.environ, QMV_GEOM=spec)
    out = subprocess.run([sys.executable, "-c", GEOM_PROBE, ROOT], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr[-2000:]
    rc = int(out.stdout.split()[-1])
    if want is None:
        assert rc == 6  # no device here: past the override, the device query fails
    else:
        assert rc == want
    assert qlib.lib().qmv_status_str(10) == b"malformed or out-of-range QMV_GEOM override"


def test_header_is_plain_c99(tmp_path):
    """include/qmv.h and qmv_debug.h are C headers: they compile as C99 with every warning an
    error, and a C program declares and calls through it."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use_header.c"
    src.write_text('#include "qmv.h"\n#include "qmv_debug.h"\n'
                   "int main(void) { qmv_launch_info info; (void)info;\n"
                   "  return qmv_status_str(QMV_OK) != 0 && qmv_version() > 0 ? 0 : 1; }\n")
    import subprocess

    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_calls_the_library(qlib, tmp_path):
    """A C program linked against libqmv.so (no Python involved) gets the
    sizes and the host-validation statuses the header documents."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    import subprocess

    libdir = os.path.dirname(qlib.library_path())
    src = tmp_path / "prog.c"
    src.write_text(
        '#include <stdio.h>\n#include "qmv.h"\n'
        "int main(void) {\n"
        "  void *p = (void *)0x1000;\n"
        '  printf("%zu %zu %lld %d %d %d\\n", qmv_row_bytes(QMV_TYPE_Q4_K, 4096), qmv_q8_1_bytes(11008, 1),\n'
        "         (long long)qmv_q8_1_padded_k(11008), qmv_mul_mat_vec(5, p, 16, 256, p, 1, (float *)p, 0),\n"
        "         qmv_mul_mat_vec(QMV_TYPE_Q4_K, p, 16, 250, p, 1, (float *)p, 0),\n"
        "         qmv_mul_mat_vec(QMV_TYPE_Q4_K, p, 16, 256, p, 9, (float *)p, 0));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "prog"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-L", libdir, "-lqmv", "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["2304", "12672", "11264", "2", "3", "4"]
