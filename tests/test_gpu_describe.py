"""The launch geometry the planner picks (qmv_describe_gemv), on the GPU:
plausible for every benchmark shape, shared by fp32 and q8_1 input (their
outputs are bit-identical because of it), and moved by the tuning setters
and by the QMV_GEOM environment override (no GEMV is launched).  Also the
diagnostic read-bandwidth probe.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import quantized_decode_gemv_qmv_gb300 as qq

    torch.cuda.set_device(0)
    for t in qq.WEIGHT_TYPES:
        qq.set_tuning(t)
        qq.set_stream_tuning(t)
        qq.set_mma_min_cols(t, 0)
    yield qq
    for t in qq.WEIGHT_TYPES:
        qq.set_tuning(t)
        qq.set_stream_tuning(t)
        qq.set_mma_min_cols(t, 0)


SHAPES = [("q4_K", 12, 12288, 4096, False), ("q4_K", 12, 4096, 4096, False), ("q4_K", 12, 11008, 4096, True),
          ("q4_K", 12, 4096, 11008, False), ("q6_K", 14, 32000, 4096, False), ("q6_K", 14, 4096, 14336, False),
          ("q4_0", 2, 4096, 4096, False), ("q4_K", 12, 14336, 4096, False)]


@pytest.mark.parametrize("name,t,M,K,gate", SHAPES, ids=[f"{s[0]}-{s[2]}x{s[3]}{'-gate' if s[4] else ''}"
                                                          for s in SHAPES])
@pytest.mark.parametrize("ncols", [1, 4, 8])
def test_geometry_is_plausible_and_shared_by_both_inputs(q, name, t, M, K, gate, ncols):
    import torch

    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    a = q.describe_gemv(t, M, K, ncols, gate_up=gate)
    assert a["tile_kernel"] == 1 and a["tensor_cores"] == 0 and a["rows_per_tile"] == 4
    assert a["grid"] % n_sm == 0 or a["grid"] < n_sm
    assert 1 <= a["stages"] <= 4 and 1 <= a["dec_warps"] <= a["block"] // 32 <= 12
    assert 1 <= a["pre_tiles"] <= a["stages"] and a["cluster"] == 1
    assert 0 < a["smem"] <= 227 * 1024
    b = q.describe_gemv(t, M, K, ncols, gate_up=gate, fp32_input=True)
    for k in ("tile_kernel", "rows_per_tile", "block", "stages", "dec_warps"):
        assert a[k] == b[k], k
    # how many tiles are requested before the dependency wait changes no result:
    # an fp32-input launch held back requests its whole ring
    assert b["pre_tiles"] in (a["pre_tiles"], b["stages"])
    assert b["cluster"] in (1, 2) and b["grid"] % b["cluster"] == 0


def test_half_sm_budget_is_exact_for_q6_K_4096x14336(q):
    """This shape fills half an SM's shared memory exactly with 7 decoding
    warps of 2 stages (activations 20,608 B + 7 x 2 x 6,784 B + 128 B); any
    static shared memory in the plain kernel would cost it a warp."""
    g = q.describe_gemv(14, 4096, 14336, 1)
    assert (g["dec_warps"], g["stages"]) == (7, 2), g


def test_tuning_and_tensor_core_choice_show_in_the_geometry(q):
    q.set_tuning(12, stages=1, threads=256)
    try:
        g = q.describe_gemv(12, 14336, 4096, 1)
        assert g["stages"] == 1 and g["block"] == 256
    finally:
        q.set_tuning(12)
    q.set_mma_min_cols(12, 3)
    try:
        assert q.describe_gemv(12, 14336, 4096, 2)["tensor_cores"] == 0
        g = q.describe_gemv(12, 14336, 4096, 3)
        assert g["tensor_cores"] == 1 and g["rows_per_tile"] == 8
        assert g == q.describe_gemv(12, 14336, 4096, 3, fp32_input=True)
    finally:
        q.set_mma_min_cols(12, 0)
    # shapes the tile kernel does not take go to the generic kernel
    assert q.describe_gemv(14, 77, 2304, 2)["tile_kernel"] == 0


def test_environment_override_reaches_the_planner(q):
    code = ("import sys; sys.path.insert(0, sys.argv[1])\n"
            "import quantized_decode_gemv_qmv_gb300 as q\n"
            "g = q.describe_gemv(12, 14336, 4096, 1)\n"
            "print(g['stages'], g['block'], g['pre_tiles'])\n")
    env = dict(os.environ, QMV_GEOM="q4_K:stages=3,threads=320,pre_tiles=2")
    out = subprocess.run([sys.executable, "-c", code, ROOT], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.split()[-3:] == ["3", "320", "2"], out.stdout


def test_read_bandwidth_probe(q):
    """The diagnostic read probe runs over a buffer with a ragged piece count;
    its sink is written only when one thread's XOR of the words it read is
    0x9E3779B9, which words below 2^21 cannot produce."""
    import torch

    buf = torch.arange(0, (1 << 20) + 12, dtype=torch.int32, device="cuda")  # 4 MiB + 48 bytes
    sink = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    q.read_bandwidth_probe(buf, sink)
    torch.cuda.synchronize()
    assert int(sink.item()) == 7
    assert q.device_fault() == 0
