"""GPU parity of the fused epilogue extras through the C ABI: the up and gate
biases of the fused launch and the MoE shared expert (mul_mat_vec_q page,
section "融合:把 gate、bias 和 SwiGLU 塞进同一个 kernel").

The bias add is one fp32 rounding after the GEMV, so the bound is the GEMV's
(1e-4 of the L1 norm of the row's scaled terms) plus half an ulp of the
result; through silu the bound is propagated as for the plain SwiGLU.  Calls
without extras must equal the existing calls bit for bit.
"""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4
ULP = 2.0 ** -23


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


def weights(t, M, K, seed):
    return oracle.quantize_rows(t, synthetic.weights_f32(seed, M, K))


def bias_vec(seed, M, scale=0.5):
    return (scale * synthetic.activations_f32(seed, 1, M)[0]).astype(np.float32)


def glu_tol(g, u, l1g, l1u):
    """Bound of (u) * silu(g) when g and u each carry TOL * l1 (plus the bias
    roundings, a few ulps of each) -- first-order propagation."""
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    eg = TOL * l1g + 2 * ULP * np.abs(g)
    eu = TOL * l1u + 2 * ULP * np.abs(u)
    return np.abs(u) * np.abs(dsilu) * eg + np.abs(g * sig) * eu + 4 * ULP * np.abs(u * g * sig) + 1e-30


SHAPES = [(oracle.Q4_0, 517, 1024), (oracle.Q4_K, 517, 4096), (oracle.Q6_K, 517, 4096)]


@pytest.mark.parametrize("t,M,K", SHAPES, ids=["q4_0", "q4_K", "q6_K"])
@pytest.mark.parametrize("ncols", [1, 3])
@pytest.mark.parametrize("inp", ["q8_1", "f32"])
def test_bias_plain(q, t, M, K, ncols, inp):
    W = weights(t, M, K, 1200 + t)
    x = synthetic.activations_f32(1201 + ncols, ncols, K)
    xq = oracle.quantize_q8_1(x)
    b = bias_vec(1202, M)
    up, l1 = oracle.gemv_formula(t, W, M, K, xq, ncols)
    ref = oracle.fused_epilogue(up, bias=b)
    Wd = dev(W)
    kw = {"xq": dev(xq)} if inp == "q8_1" else {"x": dev(x)}
    y = host(q.mul_mat_vec_fused(t, Wd, M, K, bias=dev(b), **kw))
    err = np.abs(y.astype(np.float64) - ref)
    assert np.all(err <= TOL * l1 + ULP * np.abs(ref)), (err / (TOL * l1)).max()
    # without extras: the plain calls, bit for bit
    y0 = host(q.mul_mat_vec_fused(t, Wd, M, K, **kw))
    y1 = host(q.mul_mat_vec(t, Wd, M, K, dev(xq), ncols) if inp == "q8_1"
              else q.mul_mat_vec_f32(t, Wd, M, K, dev(x)))
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))


@pytest.mark.parametrize("t,M,K", SHAPES, ids=["q4_0", "q4_K", "q6_K"])
@pytest.mark.parametrize("ncols", [1, 2])
@pytest.mark.parametrize("inp", ["q8_1", "f32"])
def test_bias_gate_up(q, t, M, K, ncols, inp):
    Wg, Wu = weights(t, M, K, 1300 + t), weights(t, M, K, 1310 + t)
    x = synthetic.activations_f32(1301 + ncols, ncols, K)
    xq = oracle.quantize_q8_1(x)
    b, gb = bias_vec(1302, M), bias_vec(1303, M)
    g, l1g = oracle.gemv_formula(t, Wg, M, K, xq, ncols)
    u, l1u = oracle.gemv_formula(t, Wu, M, K, xq, ncols)
    Wgd, Wud = dev(Wg), dev(Wu)
    kw = {"xq": dev(xq)} if inp == "q8_1" else {"x": dev(x)}
    for bb, gg in ((b, gb), (None, gb), (b, None)):
        ref = oracle.fused_epilogue(u, g, bb, gg)
        y = host(q.mul_mat_vec_fused(t, Wud, M, K, W_gate=Wgd, bias=None if bb is None else dev(bb),
                                     gate_bias=None if gg is None else dev(gg), **kw))
        gs = g + (0.0 if gg is None else gg[None, :])
        us = u + (0.0 if bb is None else bb[None, :])
        err = np.abs(y.astype(np.float64) - ref)
        assert np.all(err <= glu_tol(gs, us, l1g, l1u)), (bb is None, gg is None)
    y0 = host(q.mul_mat_vec_fused(t, Wud, M, K, W_gate=Wgd, **kw))
    y1 = host(q.mul_mat_vec_gate_up_swiglu(t, Wgd, Wud, M, K, dev(xq), ncols) if inp == "q8_1"
              else q.mul_mat_vec_gate_up_swiglu_f32(t, Wgd, Wud, M, K, dev(x)))
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))


def _moe_shared_case(q, t, E, M, K, ids, seed, inp):
    import torch

    W = weights(t, E * M, K, seed).reshape(E, -1)
    Ws = weights(t, M, K, seed + 5)
    T = ids.shape[0]
    x = synthetic.activations_f32(seed + 1, T, K)
    xq = oracle.quantize_q8_1(x)
    y_ref, l1, bad = oracle.moe_gemv(t, W, E, M, K, xq, ids)
    ys_ref, l1s = oracle.shared_expert_gemv(t, Ws, M, K, xq, T)
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    Wd, idd = dev(W), dev(ids)
    kw = {"xq": dev(xq)} if inp == "q8_1" else {"x": dev(x)}
    y, ys = q.mul_mat_vec_id_fused(t, Wd, E, M, K, idd, W_shared=dev(Ws), status=status, **kw)
    y, ys = host(y), host(ys)
    assert int(host(status)[0]) == bad
    assert np.all(np.abs(y - y_ref) <= TOL * l1), f"routed, ids {ids.tolist()}"
    assert np.all(np.abs(ys - ys_ref) <= TOL * l1s), "shared expert"
    # the routed outputs do not depend on the shared slice: the plain MoE call, bit for bit
    y_plain = host(q.mul_mat_vec_id(t, Wd, E, M, K, dev(xq), idd) if inp == "q8_1"
                   else q.mul_mat_vec_id_f32(t, Wd, E, M, K, dev(x), idd))
    assert np.array_equal(y.view(np.uint32), y_plain.view(np.uint32))
    # without a shared expert the fused call is the plain one
    y2, ys2 = q.mul_mat_vec_id_fused(t, Wd, E, M, K, idd, **kw)
    assert ys2 is None and np.array_equal(host(y2).view(np.uint32), y_plain.view(np.uint32))
    return y, ys


@pytest.mark.parametrize("t", [oracle.Q4_0, oracle.Q4_K, oracle.Q6_K])
@pytest.mark.parametrize("inp", ["q8_1", "f32"])
def test_moe_shared_expert(q, t, inp):
    K = 2048 if t == oracle.Q6_K else 1024
    ids = synthetic.moe_ids(1400 + t, 4, 2, 8)
    _moe_shared_case(q, t, 8, 203, K, ids, 1410 + t, inp)


def test_moe_shared_expert_edge_routings(q):
    t, E, M, K = oracle.Q4_K, 8, 77, 512
    # invalid ids: their slots are zero, the shared expert still serves every token
    y, ys = _moe_shared_case(q, t, E, M, K, np.array([[1, 9], [-1, 2], [2, 1]], dtype=np.int32), 1420, "q8_1")
    assert not y[0, 1].any() and not y[1, 0].any() and ys.any()
    # no valid id at all: only the shared expert works
    y, ys = _moe_shared_case(q, t, E, M, K, np.array([[-3, 8]], dtype=np.int32), 1421, "f32")
    assert not y.any() and ys.any()
    # eight tokens picking 256 distinct experts, plus the shared one
    E2 = 300
    rng = np.random.default_rng(1422)
    ids = rng.permutation(E2)[:256].astype(np.int32).reshape(8, 32)
    _moe_shared_case(q, t, E2, 20, 256, ids, 1423, "q8_1")


def _moe_gated_case(q, t, E, M, K, ids, seed, inp, shared=True):
    import torch

    Wu = weights(t, E * M, K, seed).reshape(E, -1)
    Wg = weights(t, E * M, K, seed + 2).reshape(E, -1)
    Wsu, Wsg = weights(t, M, K, seed + 5), weights(t, M, K, seed + 6)
    T = ids.shape[0]
    x = synthetic.activations_f32(seed + 1, T, K)
    xq = oracle.quantize_q8_1(x)
    u, l1u, bad = oracle.moe_gemv(t, Wu, E, M, K, xq, ids)
    g, l1g, _ = oracle.moe_gemv(t, Wg, E, M, K, xq, ids)
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    kw = {"xq": dev(xq)} if inp == "q8_1" else {"x": dev(x)}
    if shared:
        kw.update(W_shared=dev(Wsu), W_shared_gate=dev(Wsg))
    y, ys = q.mul_mat_vec_id_fused(t, dev(Wu), E, M, K, dev(ids), W_gate=dev(Wg), status=status, **kw)
    y = host(y)
    assert int(host(status)[0]) == bad
    ref = oracle.swiglu(g, u)
    assert np.all(np.abs(y - ref) <= glu_tol(g, u, l1g, l1u)), f"routed, ids {ids.tolist()}"
    if shared:
        ys = host(ys)
        su, l1su = oracle.shared_expert_gemv(t, Wsu, M, K, xq, T)
        sg, l1sg = oracle.shared_expert_gemv(t, Wsg, M, K, xq, T)
        assert np.all(np.abs(ys - oracle.swiglu(sg, su)) <= glu_tol(sg, su, l1sg, l1su)), "shared expert"
    else:
        assert ys is None
    return y


@pytest.mark.parametrize("t", [oracle.Q4_0, oracle.Q4_K, oracle.Q6_K])
@pytest.mark.parametrize("inp", ["q8_1", "f32"])
def test_moe_gated(q, t, inp):
    # the MoE form of the fused gate/up: y[t][k] = (W_up[e] x_t) * silu(W_gate[e] x_t)
    K = 2048 if t == oracle.Q6_K else 1024
    ids = synthetic.moe_ids(1500 + t, 4, 2, 8)
    _moe_gated_case(q, t, 8, 203, K, ids, 1510 + t, inp)


def test_moe_gated_edge_routings(q):
    t, E, M, K = oracle.Q4_K, 8, 77, 512
    y = _moe_gated_case(q, t, E, M, K, np.array([[1, 9], [-1, 2], [2, 1]], dtype=np.int32), 1520, "q8_1")
    assert not y[0, 1].any() and not y[1, 0].any()
    _moe_gated_case(q, t, E, M, K, synthetic.moe_ids(1521, 8, 4, E), 1522, "f32", shared=False)
    _moe_gated_case(q, t, E, M, K, np.array([[3, 3]], dtype=np.int32), 1523, "q8_1")
