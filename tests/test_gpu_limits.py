"""The GEMV at the edges of what it takes (GPU, through the C ABI):

* activations too large to stage in shared memory (8 columns of K = 65536):
  the q8_1 call takes the generic kernel and still matches the oracle; the
  fp32-input call, which has no generic path, returns QMV_ERR_SHAPE without
  launching;
* the largest K whose 8 staged columns still fit the tile kernel;
* a half-million-row ragged M (2^19 + 3 rows), checked on sampled rows.
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
        qq.set_mma_min_cols(t, 0)
    return qq


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


def test_activations_beyond_shared_memory(q):
    t, M, K, nc = oracle.Q4_K, 64, 65536, 8
    g = q.describe_gemv(t, M, K, nc)
    assert g["tile_kernel"] == 0, g  # 8 columns x 256 units x 352 B do not fit: generic kernel
    W = oracle.quantize_rows(t, synthetic.weights_f32(2100, M, K))
    x = synthetic.activations_f32(2101, nc, K, outlier_frac=0.01)
    xq = oracle.quantize_q8_1(x)
    y = host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), nc))
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, nc)
    assert np.all(np.abs(y - y_ref) <= TOL * l1)
    with pytest.raises(q.QmvError) as e:
        q.mul_mat_vec_f32(t, dev(W), M, K, dev(x))
    assert e.value.status == 3
    assert q.device_fault() == 0


def test_largest_staged_k_at_eight_columns(q):
    # the largest multiple of 256 whose 8 columns of packed activations fit
    # beside at least one tile ring: found through the planner, then checked
    t, M, nc = oracle.Q4_K, 40, 8
    K = 256
    while q.describe_gemv(t, M, K + 256, nc)["tile_kernel"] == 1:
        K += 256
    assert 16384 <= K <= 32768, K
    W = oracle.quantize_rows(t, synthetic.weights_f32(2200, M, K))
    x = synthetic.activations_f32(2201, nc, K)
    xq = oracle.quantize_q8_1(x)
    y = host(q.mul_mat_vec(t, dev(W), M, K, dev(xq), nc))
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, nc)
    assert np.all(np.abs(y - y_ref) <= TOL * l1), K
    assert np.array_equal(host(q.mul_mat_vec_f32(t, dev(W), M, K, dev(x))).view(np.uint32), y.view(np.uint32))


def test_half_million_row_ragged_m(q):
    t, M, K = oracle.Q4_0, (1 << 19) + 3, 256
    w = synthetic.weights_f32(2300, M, K)
    W = oracle.quantize_rows(t, w)
    x = synthetic.activations_f32(2301, 2, K)
    xq = oracle.quantize_q8_1(x)
    Wd = q.quantize_weights(t, dev(w))
    assert np.array_equal(host(Wd), W)
    y = host(q.mul_mat_vec(t, Wd, M, K, dev(xq), 2))
    rows = np.unique(np.concatenate([np.arange(4), np.arange(M - 4, M),
                                     synthetic.host_rng(2302).choice(M, 200, replace=False)]))
    y_ref, l1 = oracle.gemv_formula(t, W, M, K, xq, 2, rows=rows)
    assert np.all(np.abs(y[:, rows] - y_ref) <= TOL * l1)
    assert np.all(np.isfinite(y))
