"""The one bounded device wait, made to run out on purpose.

The fp32-input GEMV shares the quantization of x among the CTAs of a cluster;
each CTA waits, with a time limit, for its partners' shares.  The test-only
entry qmv_debug_f32_withheld_share has the rank-1 CTA of every cluster keep
its share, so the rank-0 CTA's wait (1 ms here) runs out.  Checked: the call
returns; the device fault word reads code 2; the rows of the warps that gave up
are NaN in every column, and every other output is bit for bit the ordinary
call's; the next ordinary call finds the fault word clear, matches the oracle
and leaves the word clear.  No kernel hangs or faults: the withholding CTA still
receives its partner's share and finishes normally.
"""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4


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
    qq.device_fault()  # start from a clear word
    return qq


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.mark.parametrize("t,M,K,ncols", [(oracle.Q4_K, 4096, 4096, 1), (oracle.Q4_K, 1003, 2048, 2),
                                         (oracle.Q6_K, 517, 4096, 2), (oracle.Q4_0, 700, 1024, 1)])
def test_withheld_share_runs_the_wait_out(q, t, M, K, ncols):
    W = oracle.quantize_rows(t, synthetic.weights_f32(2200 + M, M, K))
    x = synthetic.activations_f32(2201 + M, ncols, K, outlier_frac=0.01)
    Wd, xd = dev(W), dev(x)
    assert q.describe_gemv(t, M, K, ncols, fp32_input=True)["cluster"] >= 2
    assert q.device_fault() == 0
    y_ok = host(q.mul_mat_vec_f32(t, Wd, M, K, xd))
    assert q.device_fault() == 0

    y = host(q.debug_f32_withheld_share(t, Wd, M, K, xd, 1_000_000))
    assert q.device_fault() == 2
    nan = np.isnan(y)
    assert nan.any() and not nan.all()
    assert np.array_equal(nan, np.broadcast_to(nan[0], nan.shape)), "a row is NaN in every column or in none"
    assert np.array_equal(y[~nan].view(np.uint32), y_ok[~nan].view(np.uint32))
    assert q.device_fault() == 0  # read and cleared

    # the context is intact: the next ordinary call is clean and right
    y2 = host(q.mul_mat_vec_f32(t, Wd, M, K, xd))
    assert q.device_fault() == 0
    assert np.array_equal(y2.view(np.uint32), y_ok.view(np.uint32))
    xq = oracle.quantize_q8_1(x)
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, ncols)
    assert np.all(np.abs(y2.astype(np.float64) - y_ref) <= TOL * l1)


def test_withheld_share_needs_an_instrumented_kernel(q):
    """Three columns have no instrumented twin: refused before any launch."""
    t, M, K = oracle.Q4_K, 512, 2048
    W = oracle.quantize_rows(t, synthetic.weights_f32(2300, M, K))
    x = synthetic.activations_f32(2301, 3, K)
    y = dev(np.full((3, M), 7.0, np.float32))
    with pytest.raises(q.QmvError) as e:
        q.debug_f32_withheld_share(t, dev(W), M, K, dev(x), 1_000_000, out=y)
    assert e.value.status == 10
    assert np.all(host(y) == 7.0) and q.device_fault() == 0
