"""The launch timeline (qmv_debug_trace) and its instrumented kernels.

While the timeline is on, launches that have an instrumented twin run it and
write six timestamps per CTA; other launches are not recorded and take no
slot.  Checked: a traced launch's outputs are bit for bit the ordinary
launch's; every CTA of a recorded launch has its six stamps in order (entry,
dependency wait returned, first activation loads returned, its own part of the
staging done, all activations in shared memory, last warp done) and no CTA
past the grid has any; a launch without a twin leaves its slot free; nothing is
written past the enabled slots; with programmatic dependent launch, a
dependent launch's wait returns no earlier than its predecessor's last CTA
finished.
"""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

SLOT = 1024 * 6  # int64 words per slot: 1024 CTAs x 6 stamps
CLOCK_SLACK_NS = 1000  # globaltimer ticks and SM-to-SM skew, generously


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
    qq.debug_trace(None)


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


def stamps(buf, k, grid):
    """Slot k as [grid][6], and whether every CTA past the grid is blank."""
    s = host(buf)[k * SLOT:(k + 1) * SLOT].reshape(1024, 6)
    return s[:grid], not s[grid:].any()


def test_timeline_of_instrumented_launches(q):
    import torch

    t, M, K, F = oracle.Q4_K, 4096, 4096, 2048
    W = dev(oracle.quantize_rows(t, synthetic.weights_f32(2400, M, K)))
    Wg = dev(oracle.quantize_rows(t, synthetic.weights_f32(2401, F, K)))
    Wu = dev(oracle.quantize_rows(t, synthetic.weights_f32(2402, F, K)))
    x1 = dev(synthetic.activations_f32(2403, 1, K))
    x3 = dev(synthetic.activations_f32(2404, 3, K))
    s = torch.cuda.Stream()

    def run():
        with torch.cuda.stream(s):
            y3 = q.mul_mat_vec_f32(t, W, M, K, x3, stream=s)  # three columns: no twin
            y1 = q.mul_mat_vec_f32(t, W, M, K, x1, stream=s)
            yg = q.mul_mat_vec_gate_up_swiglu_f32(t, Wg, Wu, F, K, x1, stream=s)
            y1b = q.mul_mat_vec_f32(t, W, M, K, x1, stream=s)  # past the slots
        s.synchronize()
        return [host(v) for v in (y3, y1, yg, y1b)]

    ref = run()
    buf = torch.zeros(3 * SLOT, dtype=torch.int64, device="cuda")
    q.debug_trace(buf, 2)
    try:
        got = run()
    finally:
        q.debug_trace(None)
    for a, b in zip(got, ref):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))

    g1 = q.describe_gemv(t, M, K, 1, fp32_input=True)["grid"]
    gg = q.describe_gemv(t, F, K, 1, gate_up=True, fp32_input=True)["grid"]
    s0, blank0 = stamps(buf, 0, g1)
    s1, blank1 = stamps(buf, 1, gg)
    assert blank0 and blank1
    for s_ in (s0, s1):
        assert np.all(s_ > 0), "every CTA of a recorded launch writes all six stamps"
        assert np.all(np.diff(s_, axis=1) >= 0), "entry <= wait <= loads <= own part <= staged <= done"
    assert not host(buf)[2 * SLOT:].any(), "nothing is written past the enabled slots"
    # the gate/up launch depends on the plain one: its wait returns after the plain one's last CTA
    assert s1[:, 1].min() >= s0[:, 5].max() - CLOCK_SLACK_NS


def test_launch_without_twin_takes_no_slot(q):
    import torch

    t, M, K = oracle.Q6_K, 1024, 4096
    W = dev(oracle.quantize_rows(t, synthetic.weights_f32(2410, M, K)))
    x4 = dev(synthetic.activations_f32(2411, 4, K))
    x2 = dev(synthetic.activations_f32(2412, 2, K))
    buf = torch.zeros(2 * SLOT, dtype=torch.int64, device="cuda")
    q.debug_trace(buf, 1)
    try:
        q.mul_mat_vec_f32(t, W, M, K, x4)
        assert not host(buf).any(), "four columns have no twin"
        y2 = host(q.mul_mat_vec_f32(t, W, M, K, x2))  # the first recorded launch
    finally:
        q.debug_trace(None)
    s0, blank0 = stamps(buf, 0, q.describe_gemv(t, M, K, 2, fp32_input=True)["grid"])
    assert blank0 and np.all(s0 > 0) and np.all(np.diff(s0, axis=1) >= 0)
    assert not host(buf)[SLOT:].any()
    xq = oracle.quantize_q8_1(host(x2))
    y_ref, l1 = oracle.gemv_formula(t, host(W), M, K, xq, 2)
    assert np.all(np.abs(y2.astype(np.float64) - y_ref) <= 1e-4 * l1)
