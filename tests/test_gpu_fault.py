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
                                         (oracle.Q6_K, 517, 4096, 2), (oracle.Q4_0, 700, 1024, 1),
                                         # long rows (the step's down projection has K = 11008)
                                         (oracle.Q4_K, 1024, 11008, 1), (oracle.Q4_K, 777, 8192, 2)])
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


@pytest.mark.parametrize("t,M,K", [(oracle.Q4_K, 4096, 4096), (oracle.Q4_K, 1000, 2048), (oracle.Q6_K, 777, 2048),
                                   (oracle.Q4_K, 1024, 11008)])
def test_withheld_share_with_q8_1_output(q, t, M, K):
    """The q8_1-output GEMV with the wait run out: NaN rows in y, a NaN scale
    on every block holding one (the quantizer's amax alone would pass over
    them), every other row and block as the ordinary call gives them, and the
    next ordinary calls exact."""
    W = oracle.quantize_rows(t, synthetic.weights_f32(2400 + M, M, K))
    x = synthetic.activations_f32(2401 + M, 1, K, outlier_frac=0.01)
    Wd, xd = dev(W), dev(x)
    assert q.device_fault() == 0
    y_ok, yq_ok = q.mul_mat_vec_fused_q8_1(t, Wd, M, K, x=xd)
    y_ok, yq_ok = host(y_ok)[0], host(yq_ok)[0]
    assert q.device_fault() == 0

    y, yq = q.debug_f32_withheld_share_q8_1(t, Wd, M, K, xd, 1_000_000)
    y, yq = host(y)[0], host(yq)[0]
    assert q.device_fault() == 2
    nan = np.isnan(y)
    assert nan.any() and not nan.all()
    assert np.array_equal(y[~nan].view(np.uint32), y_ok[~nan].view(np.uint32))
    nb = (M + 31) // 32
    blocks, blocks_ok = yq[: nb * 36].reshape(nb, 36), yq_ok[: nb * 36].reshape(nb, 36)
    bad = np.zeros(nb, bool)
    np.logical_or.at(bad, np.arange(M) // 32, nan)
    assert np.array_equal(blocks[~bad], blocks_ok[~bad])
    d = blocks[bad, 0:2].copy().view(np.float16)[:, 0]
    assert np.all(np.isnan(d)), "a block holding a NaN row has a NaN scale"
    assert np.array_equal(yq[nb * 36:], yq_ok[nb * 36:])  # the padding blocks
    assert q.device_fault() == 0

    for _ in range(2):
        y2, yq2 = q.mul_mat_vec_fused_q8_1(t, Wd, M, K, x=xd)
        assert np.array_equal(host(y2)[0].view(np.uint32), y_ok.view(np.uint32))
        assert np.array_equal(host(yq2)[0], yq_ok)
    assert q.device_fault() == 0
    assert np.array_equal(yq_ok, oracle.quantize_q8_1(y_ok[None])[0])
