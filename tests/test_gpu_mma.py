"""GPU parity of the tensor-core decode of the plain Q4_K GEMV (mma.sync on
8-row tiles, opt-in through set_mma_min_cols; mul_mat_vec_q page, "一次
vec_dot 的解剖" for the block products) through the C ABI.

* Against the oracle at every column count, forced on (from one column) and
  forced off, on shapes with ragged row groups (M not a multiple of 8), one
  and odd numbers of super-blocks per row, and a row long enough that only a
  few warps fit beside the staged activations.  The bound is the GEMV's usual
  1e-4 of the L1 norm of the row's scaled terms.
* Exact integers: with d = dmin = d8 = 1 every block product is an integer and
  so is y (below 2^24), so both decodes must return the oracle's value bit for
  bit.  A tensor-core accumulation that dropped or rounded any bit of a block
  dot would show here.
* fp32 input equals q8_1 input bit for bit on this decode too.
"""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4
T = oracle.Q4_K


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
    qq.set_mma_min_cols(T, 0)


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


def run_both(q, W, M, K, x, xq, ncols, min_cols):
    """(q8_1-input y, fp32-input y) with the decode choice min_cols."""
    q.set_mma_min_cols(T, min_cols)
    try:
        Wd = dev(W)
        y8 = host(q.mul_mat_vec(T, Wd, M, K, dev(xq), ncols))
        yf = host(q.mul_mat_vec_f32(T, Wd, M, K, dev(x)))
    finally:
        q.set_mma_min_cols(T, 0)
    return y8, yf


SHAPES = [(1, 256), (17, 256), (45, 2304), (203, 4096), (517, 1024), (37, 11264)]


@pytest.mark.parametrize("M,K", SHAPES, ids=[f"{m}x{k}" for m, k in SHAPES])
@pytest.mark.parametrize("ncols", [1, 2, 3, 5, 8])
def test_mma_decode_matches_oracle(q, M, K, ncols):
    W = oracle.quantize_rows(T, synthetic.weights_f32(1800 + M, M, K))
    x = synthetic.activations_f32(1801 + K + ncols, ncols, K, outlier_frac=0.01)
    xq = oracle.quantize_q8_1(x)
    y_ref, l1 = oracle.gemv_formula(T, W, M, K, xq, ncols)
    for min_cols in (1, 9):  # tensor cores at every column count; never
        y8, yf = run_both(q, W, M, K, x, xq, ncols, min_cols)
        err = np.abs(y8.astype(np.float64) - y_ref)
        assert np.all(err <= TOL * l1), (min_cols, (err / (TOL * l1)).max())
        assert np.array_equal(y8.view(np.uint32), yf.view(np.uint32)), min_cols


def exact_q4_K_rows(M, K, seed):
    """Q4_K rows with d = dmin = 1 and scales / mins in 0..3 (so every weight
    d*sc*q - dmin*m is a small integer), random 4-bit codes."""
    rng = np.random.default_rng(seed)
    U = K // 256
    blk = np.zeros((M, U, 144), dtype=np.uint8)
    one = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)
    blk[:, :, 0:2] = one
    blk[:, :, 2:4] = one
    sc = rng.integers(0, 4, size=(M, U, 8), dtype=np.uint8)
    m = rng.integers(0, 4, size=(M, U, 8), dtype=np.uint8)
    # 6-bit packing of the format: sub-blocks 0..3 in bytes 0..3 / 4..7, 4..7 in
    # the nibbles of bytes 8..11 (values below 16: no high bits)
    blk[:, :, 4:8] = sc[:, :, 0:4]
    blk[:, :, 8:12] = m[:, :, 0:4]
    blk[:, :, 12:16] = sc[:, :, 4:8] | (m[:, :, 4:8] << 4)
    blk[:, :, 16:144] = rng.integers(0, 256, size=(M, U, 128), dtype=np.uint8)
    return blk.reshape(M, U * 144), sc, m


def exact_activations(ncols, K, seed):
    """Integer activations in [-127, 127] with a +-127 in every 32-value block:
    q8_1 gives d = 1 and codes equal to the values."""
    rng = np.random.default_rng(seed)
    x = rng.integers(-127, 128, size=(ncols, K)).astype(np.float32)
    pos = rng.integers(0, 32, size=(ncols, K // 32))
    sign = np.where(rng.random((ncols, K // 32)) < 0.5, -127.0, 127.0).astype(np.float32)
    for c in range(ncols):
        x[c, np.arange(K // 32) * 32 + pos[c]] = sign[c]
    return x


@pytest.mark.parametrize("M,K", [(45, 1024), (16, 256), (130, 2304)])
def test_exact_integer_block_dots(q, M, K):
    W, sc, m = exact_q4_K_rows(M, K, 1900 + M)
    # the packing above is the format's: the oracle's dequantization gives sc*q - m
    w = oracle.dequantize_rows(T, W, K).reshape(M, K // 32, 32)
    codes = np.stack([W.reshape(M, K // 256, 144)[:, :, 16:144] & 15, W.reshape(M, K // 256, 144)[:, :, 16:144] >> 4],
                     axis=2)  # [M][U][lo/hi][128]
    q0 = codes.reshape(M, K // 256, 2, 4, 32).transpose(0, 1, 3, 2, 4).reshape(M, K // 32, 32)
    scs = sc.reshape(M, K // 32, 1).astype(np.float64)
    ms = m.reshape(M, K // 32, 1).astype(np.float64)
    assert np.array_equal(w, scs * q0 - ms)
    for ncols in (1, 3, 8):
        x = exact_activations(ncols, K, 1901 + ncols)
        xq = oracle.quantize_q8_1(x)
        assert np.array_equal(oracle.dequantize_q8_1(xq, K)[:, :K], x)
        y_ref, _ = oracle.gemv_formula(T, W, M, K, xq, ncols)
        assert np.all(np.abs(y_ref) < 2 ** 24) and np.array_equal(y_ref, np.round(y_ref))
        for min_cols in (1, 9):
            y8, yf = run_both(q, W, M, K, x, xq, ncols, min_cols)
            assert np.array_equal(y8, y_ref.astype(np.float32)), (ncols, min_cols)
            assert np.array_equal(yf, y_ref.astype(np.float32)), (ncols, min_cols)


def test_mma_bias_and_default_choice(q):
    """The fused call's bias on the default decode and on the tensor-core decode
    (forced from one column); without a bias the fused call equals the plain
    call bit for bit on either."""
    M, K = 301, 4096
    W = oracle.quantize_rows(T, synthetic.weights_f32(1950, M, K))
    b = (0.5 * synthetic.activations_f32(1951, 1, M)[0]).astype(np.float32)
    for min_cols in (0, 1):
        q.set_mma_min_cols(T, min_cols)
        try:
            for ncols in (2, 3, 4, 8):
                x = synthetic.activations_f32(1952 + ncols, ncols, K)
                xq = oracle.quantize_q8_1(x)
                up, l1 = oracle.gemv_formula(T, W, M, K, xq, ncols)
                ref = oracle.fused_epilogue(up, bias=b)
                y = host(q.mul_mat_vec_fused(T, dev(W), M, K, xq=dev(xq), bias=dev(b)))
                err = np.abs(y.astype(np.float64) - ref)
                assert np.all(err <= TOL * l1 + 2.0 ** -23 * np.abs(ref)), (min_cols, ncols)
                y0 = host(q.mul_mat_vec_fused(T, dev(W), M, K, xq=dev(xq)))
                y1 = host(q.mul_mat_vec(T, dev(W), M, K, dev(xq), ncols))
                assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32)), (min_cols, ncols)
        finally:
            q.set_mma_min_cols(T, 0)
