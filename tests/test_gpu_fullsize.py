"""Full-size parity at the benchmark shapes, in the launch configuration the
benchmark times (default geometry, programmatic dependent launch on).

Weights are the seeded N(0, 0.02) matrices quantized by the oracle; the GPU
weight quantizer must reproduce those bytes exactly at full size.  Every
output -- every row, every column, every MoE slot and every shared-expert
token -- is checked against the oracle's block formula (computed over all
host cores), within 1e-4 of each output's L1 norm of scaled terms, so a
fault confined to some rows of the full-size geometry (a CTA's range edge, a
warp's last row group, a cluster partner's half) cannot pass.
"""
import os
import zlib

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
    return qq


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch

    torch.cuda.synchronize()
    return t.cpu().numpy()


def reference(t, W, M, K, xq, ncols):
    """The oracle's block formula over every row: (y, l1), each [ncols][M]."""
    return oracle.gemv_formula_mt(t, W, M, K, xq, ncols, os.cpu_count() or 1)


def glu_bound(g, u, l1g, l1u):
    """Bound of u * silu(g) when g and u each carry TOL * l1 (first order)."""
    sig = 1.0 / (1.0 + np.exp(-g))
    return np.abs(u) * np.abs(sig * (1 + g * (1 - sig))) * TOL * l1g + np.abs(g * sig) * TOL * l1u + \
        1e-6 * np.abs(u * g * sig)


def quantized(q, t, M, K, seed):
    """(oracle bytes, device bytes): the device copy comes from the GPU
    quantizer, which must match the oracle bit for bit."""
    w = synthetic.weights_f32(seed, M, K)
    W = oracle.quantize_rows(t, w)
    Wd = q.quantize_weights(t, dev(w))
    assert np.array_equal(host(Wd), W), "GPU weight quantizer differs from the oracle"
    return W, Wd


CONFIGS = [
    ("q4_0 4096x4096", oracle.Q4_0, 4096, 4096, 0.0),
    ("q4_K 4096x4096", oracle.Q4_K, 4096, 4096, 0.01),
    ("q4_K 11008x4096", oracle.Q4_K, 11008, 4096, 0.01),
    ("q4_K 4096x11008", oracle.Q4_K, 4096, 11008, 0.01),
    ("q6_K 32000x4096", oracle.Q6_K, 32000, 4096, 0.0),
    ("q6_K 4096x14336", oracle.Q6_K, 4096, 14336, 0.0),
]


@pytest.mark.parametrize("name,t,M,K,outl", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_fullsize_gemv_ncols1(q, name, t, M, K, outl):
    W, Wd = quantized(q, t, M, K, seed=zlib.crc32(name.encode()) % 100000)
    x = synthetic.activations_f32(17, 1, K, outlier_frac=outl)
    xq_ref = oracle.quantize_q8_1(x)
    xq = q.quantize_q8_1(dev(x))
    assert np.array_equal(host(xq), xq_ref)
    y = host(q.mul_mat_vec(t, Wd, M, K, xq, 1))
    y_ref, l1 = reference(t, W, M, K, xq_ref, 1)
    err = np.abs(y - y_ref)
    assert np.all(err <= TOL * l1), (err / l1).max()
    assert np.all(np.isfinite(y))


def test_fullsize_q4_K_small_batch_sweep(q):
    """The column sweep the benchmark times, with both decodes: per-column
    dp4a (the default) and the tensor-core decode (forced from one column)."""
    t, M, K = oracle.Q4_K, 14336, 4096
    W, Wd = quantized(q, t, M, K, seed=4141)
    for ncols in range(1, 9):
        x = synthetic.activations_f32(20 + ncols, ncols, K)
        xq_ref = oracle.quantize_q8_1(x)
        y_ref, l1 = reference(t, W, M, K, xq_ref, ncols)
        for min_cols in (0, 1):
            q.set_mma_min_cols(t, min_cols)
            try:
                y = host(q.mul_mat_vec(t, Wd, M, K, dev(xq_ref), ncols))
            finally:
                q.set_mma_min_cols(t, 0)
            assert np.all(np.abs(y - y_ref) <= TOL * l1), (ncols, min_cols)


def test_fullsize_fused_gate_up(q):
    t, M, K = oracle.Q4_K, 14336, 4096
    Wg, Wgd = quantized(q, t, M, K, seed=5151)
    Wu, Wud = quantized(q, t, M, K, seed=5152)
    xq_ref = oracle.quantize_q8_1(synthetic.activations_f32(53, 1, K))
    y = host(q.mul_mat_vec_gate_up_swiglu(t, Wgd, Wud, M, K, dev(xq_ref), 1))
    g, l1g = reference(t, Wg, M, K, xq_ref, 1)
    u, l1u = reference(t, Wu, M, K, xq_ref, 1)
    assert np.all(np.abs(y - oracle.swiglu(g, u)) <= glu_bound(g, u, l1g, l1u))


def test_fullsize_moe(q):
    import torch

    t, E, M, K, T, k = oracle.Q4_K, 8, 14336, 4096, 4, 2
    rb = oracle.row_bytes(t, K)
    W = np.empty((E, M * rb), dtype=np.uint8)
    Wd = torch.empty((E, M * rb), dtype=torch.uint8, device="cuda")
    for e in range(E):
        We, Wed = quantized(q, t, M, K, seed=6000 + e)
        W[e] = We.reshape(-1)
        Wd[e] = Wed.reshape(-1)
    ids = synthetic.moe_ids(61, T, k, E)
    xq_ref = oracle.quantize_q8_1(synthetic.activations_f32(62, T, K))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = host(q.mul_mat_vec_id(t, Wd, E, M, K, dev(xq_ref), dev(ids), status=status))
    assert int(host(status)[0]) == 0
    y_ref, l1, bad = oracle.moe_gemv(t, W, E, M, K, xq_ref, ids)
    assert bad == 0
    assert np.all(np.abs(y - y_ref) <= TOL * l1)


def test_fullsize_fused_gate_up_biases(q):
    # the bench's "gate+up 2x14336x4096 swiglu + up/gate biases" call (q8_1 input)
    t, M, K = oracle.Q4_K, 14336, 4096
    Wg, Wgd = quantized(q, t, M, K, seed=5251)
    Wu, Wud = quantized(q, t, M, K, seed=5252)
    xq_ref = oracle.quantize_q8_1(synthetic.activations_f32(55, 1, K))
    b = synthetic.activations_f32(56, 1, M)[0]
    gb = synthetic.activations_f32(57, 1, M)[0]
    y = host(q.mul_mat_vec_fused(t, Wud, M, K, xq=dev(xq_ref), W_gate=Wgd, bias=dev(b), gate_bias=dev(gb)))
    g, l1g = reference(t, Wg, M, K, xq_ref, 1)
    u, l1u = reference(t, Wu, M, K, xq_ref, 1)
    ref = oracle.fused_epilogue(u, g, b, gb)
    gs, us = g + gb[None, :], u + b[None, :]
    sig = 1.0 / (1.0 + np.exp(-gs))
    eg = TOL * l1g + 2 ** -22 * np.abs(gs)
    eu = TOL * l1u + 2 ** -22 * np.abs(us)
    tol = np.abs(us) * np.abs(sig * (1 + gs * (1 - sig))) * eg + np.abs(gs * sig) * eu + 1e-6 * np.abs(ref)
    assert np.all(np.abs(y - ref) <= tol)


def test_fullsize_moe_shared_expert(q):
    # the bench's MoE call plus a shared 14336x4096 expert, one launch
    import torch

    t, E, M, K, T, k = oracle.Q4_K, 8, 14336, 4096, 4, 2
    rb = oracle.row_bytes(t, K)
    W = np.empty((E, M * rb), dtype=np.uint8)
    Wd = torch.empty((E, M * rb), dtype=torch.uint8, device="cuda")
    for e in range(E):
        We, Wed = quantized(q, t, M, K, seed=6100 + e)
        W[e] = We.reshape(-1)
        Wd[e] = Wed.reshape(-1)
    Ws, Wsd = quantized(q, t, M, K, seed=6199)
    ids = synthetic.moe_ids(64, T, k, E)
    xq_ref = oracle.quantize_q8_1(synthetic.activations_f32(65, T, K))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y, ys = q.mul_mat_vec_id_fused(t, Wd, E, M, K, dev(ids), xq=dev(xq_ref), W_shared=Wsd, status=status)
    y, ys = host(y), host(ys)
    assert int(host(status)[0]) == 0
    y_ref, l1, bad = oracle.moe_gemv(t, W, E, M, K, xq_ref, ids)
    assert bad == 0
    assert np.all(np.abs(y - y_ref) <= TOL * l1)
    ys_ref, l1s = oracle.shared_expert_gemv(t, Ws, M, K, xq_ref, T)
    assert np.all(np.abs(ys - ys_ref) <= TOL * l1s)


def test_fullsize_moe_gated_shared_expert(q):
    # the bench's gated MoE call: 8 experts x (up + gate) 14336x4096, 4 tokens
    # top-2, plus a gated shared expert, one launch
    import torch

    t, E, M, K, T, k = oracle.Q4_K, 8, 14336, 4096, 4, 2
    rb = oracle.row_bytes(t, K)
    W = {n: np.empty((E, M * rb), dtype=np.uint8) for n in ("up", "gate")}
    Wd = {n: torch.empty((E, M * rb), dtype=torch.uint8, device="cuda") for n in ("up", "gate")}
    for n, base in (("up", 6300), ("gate", 6400)):
        for e in range(E):
            We, Wed = quantized(q, t, M, K, seed=base + e)
            W[n][e] = We.reshape(-1)
            Wd[n][e] = Wed.reshape(-1)
    Wsu, Wsud = quantized(q, t, M, K, seed=6498)
    Wsg, Wsgd = quantized(q, t, M, K, seed=6499)
    ids = synthetic.moe_ids(67, T, k, E)
    xq_ref = oracle.quantize_q8_1(synthetic.activations_f32(68, T, K))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y, ys = q.mul_mat_vec_id_fused(t, Wd["up"], E, M, K, dev(ids), xq=dev(xq_ref), W_gate=Wd["gate"],
                                   W_shared=Wsud, W_shared_gate=Wsgd, status=status)
    y, ys = host(y), host(ys)
    assert int(host(status)[0]) == 0
    u, l1u, _ = oracle.moe_gemv(t, W["up"], E, M, K, xq_ref, ids)
    g, l1g, _ = oracle.moe_gemv(t, W["gate"], E, M, K, xq_ref, ids)
    assert np.all(np.abs(y - oracle.swiglu(g, u)) <= glu_bound(g, u, l1g, l1u))
    su, l1su = oracle.shared_expert_gemv(t, Wsu, M, K, xq_ref, T)
    sg, l1sg = oracle.shared_expert_gemv(t, Wsg, M, K, xq_ref, T)
    assert np.all(np.abs(ys - oracle.swiglu(sg, su)) <= glu_bound(sg, su, l1sg, l1su))


def test_fullsize_q6_K_small_batch_sweep(q):
    # the bench's Q6_K column sweep (4096x14336, the down projection of an
    # 8B-class FFN), 1..8 columns, including the single-tile-ring geometry at 7-8
    t, M, K = oracle.Q6_K, 4096, 14336
    W, Wd = quantized(q, t, M, K, seed=4646)
    for ncols in range(1, 9):
        xq_ref = oracle.quantize_q8_1(synthetic.activations_f32(48 + ncols, ncols, K))
        y = host(q.mul_mat_vec(t, Wd, M, K, dev(xq_ref), ncols))
        y_ref, l1 = reference(t, W, M, K, xq_ref, ncols)
        assert np.all(np.abs(y - y_ref) <= TOL * l1), ncols


STEP_KINDS = [("qkv", 12288, 4096, False), ("o", 4096, 4096, False), ("gate_up", 11008, 4096, True),
              ("down", 4096, 11008, False)]


@pytest.mark.parametrize("name,M,K,gate", STEP_KINDS, ids=[s[0] for s in STEP_KINDS])
def test_fullsize_step_launches_fp32_input(q, name, M, K, gate):
    """The benchmark step's launches as it times them: fp32 activations
    quantized inside the GEMV by clusters of CTAs, bit-identical to quantizing
    first and running the q8_1 GEMV, and within the bound of the oracle."""
    t = oracle.Q4_K
    W, Wd = quantized(q, t, M, K, seed=zlib.crc32(name.encode()) % 100000)
    x = synthetic.activations_f32(70 + K, 1, K, outlier_frac=0.01)
    xq_ref = oracle.quantize_q8_1(x)
    xd = dev(x)
    if gate:
        Wg, Wgd = quantized(q, t, M, K, seed=zlib.crc32(b"gate") % 100000)
        y = host(q.mul_mat_vec_gate_up_swiglu_f32(t, Wgd, Wd, M, K, xd))
        y2 = host(q.mul_mat_vec_gate_up_swiglu(t, Wgd, Wd, M, K, q.quantize_q8_1(xd), 1))
        g, l1g = reference(t, Wg, M, K, xq_ref, 1)
        u, l1u = reference(t, W, M, K, xq_ref, 1)
        assert np.all(np.abs(y - oracle.swiglu(g, u)) <= glu_bound(g, u, l1g, l1u))
    else:
        y = host(q.mul_mat_vec_f32(t, Wd, M, K, xd))
        y2 = host(q.mul_mat_vec(t, Wd, M, K, q.quantize_q8_1(xd), 1))
        y_ref, l1 = reference(t, W, M, K, xq_ref, 1)
        assert np.all(np.abs(y - y_ref) <= TOL * l1)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
    assert q.describe_gemv(t, M, K, 1, gate_up=gate, fp32_input=True)["cluster"] == 2
