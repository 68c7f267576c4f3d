"""The Python binding checks every tensor argument before it calls the library.

For each call: arguments of the right sizes and dtypes but on the CPU, each
tensor argument in turn with a wrong dtype, and each buffer in turn one
element too short, all raise ValueError, and the library is never reached (a
stand-in that fails the test replaces it).  On a GPU the same short buffers
are rejected with CUDA tensors, before anything is launched.
"""
import pytest

torch = pytest.importorskip("torch")

import quantized_decode_gemv_qmv_gb300 as q  # noqa: E402

T, M, K, NC, E, TOPK = q.Q4_K, 8, 512, 2, 3, 2
RB = K // 256 * 144
Q8 = NC * 512 // 32 * 36  # q8_1 bytes of NC columns of K = 512


def u8(n, dev="cpu"):
    return torch.zeros(n, dtype=torch.uint8, device=dev)


def f32(*shape, dev="cpu"):
    return torch.zeros(*shape, dtype=torch.float32, device=dev)


def i32(*shape, dev="cpu"):
    return torch.zeros(*shape, dtype=torch.int32, device=dev)


def specs(dev="cpu"):
    """name -> (argument factory, call); the factory gives fresh valid tensors."""
    return {
        "mul_mat_vec": (lambda: dict(W=u8(M * RB, dev), xq=u8(Q8, dev), out=f32(NC * M, dev=dev)),
                        lambda a: q.mul_mat_vec(T, a["W"], M, K, a["xq"], NC, out=a["out"])),
        "gate_up_swiglu": (lambda: dict(W_gate=u8(M * RB, dev), W_up=u8(M * RB, dev), xq=u8(Q8, dev),
                                        out=f32(NC * M, dev=dev)),
                           lambda a: q.mul_mat_vec_gate_up_swiglu(T, a["W_gate"], a["W_up"], M, K, a["xq"], NC,
                                                                  out=a["out"])),
        "id": (lambda: dict(W=u8(E * M * RB, dev), xq=u8(Q8, dev), ids=i32(NC, TOPK, dev=dev),
                            out=f32(NC * TOPK * M, dev=dev), status=i32(1, dev=dev)),
               lambda a: q.mul_mat_vec_id(T, a["W"], E, M, K, a["xq"], a["ids"], out=a["out"], status=a["status"])),
        "f32": (lambda: dict(W=u8(M * RB, dev), x=f32(NC, K, dev=dev), out=f32(NC * M, dev=dev)),
                lambda a: q.mul_mat_vec_f32(T, a["W"], M, K, a["x"], out=a["out"])),
        "gate_up_swiglu_f32": (lambda: dict(W_gate=u8(M * RB, dev), W_up=u8(M * RB, dev), x=f32(NC, K, dev=dev),
                                            out=f32(NC * M, dev=dev)),
                               lambda a: q.mul_mat_vec_gate_up_swiglu_f32(T, a["W_gate"], a["W_up"], M, K, a["x"],
                                                                          out=a["out"])),
        "id_f32": (lambda: dict(W=u8(E * M * RB, dev), x=f32(NC, K, dev=dev), ids=i32(NC, TOPK, dev=dev),
                                out=f32(NC * TOPK * M, dev=dev), status=i32(1, dev=dev)),
                   lambda a: q.mul_mat_vec_id_f32(T, a["W"], E, M, K, a["x"], a["ids"], out=a["out"],
                                                  status=a["status"])),
        "fused": (lambda: dict(W_up=u8(M * RB, dev), W_gate=u8(M * RB, dev), x=f32(NC, K, dev=dev),
                               bias=f32(M, dev=dev), gate_bias=f32(M, dev=dev), out=f32(NC * M, dev=dev)),
                  lambda a: q.mul_mat_vec_fused(T, a["W_up"], M, K, x=a["x"], W_gate=a["W_gate"], bias=a["bias"],
                                                gate_bias=a["gate_bias"], out=a["out"])),
        "fused_q8_1": (lambda: dict(W_up=u8(M * RB, dev), xq=u8(Q8, dev).view(NC, -1), out=f32(NC * M, dev=dev)),
                       lambda a: q.mul_mat_vec_fused(T, a["W_up"], M, K, xq=a["xq"], out=a["out"])),
        "id_fused": (lambda: dict(W=u8(E * M * RB, dev), W_gate=u8(E * M * RB, dev), W_shared=u8(M * RB, dev),
                                  W_shared_gate=u8(M * RB, dev), x=f32(NC, K, dev=dev), ids=i32(NC, TOPK, dev=dev),
                                  out=f32(NC * TOPK * M, dev=dev), out_shared=f32(NC * M, dev=dev),
                                  status=i32(1, dev=dev)),
                     lambda a: q.mul_mat_vec_id_fused(T, a["W"], E, M, K, a["ids"], x=a["x"], W_gate=a["W_gate"],
                                                      W_shared=a["W_shared"], W_shared_gate=a["W_shared_gate"],
                                                      out=a["out"], out_shared=a["out_shared"],
                                                      status=a["status"])),
        "quantize_q8_1": (lambda: dict(x=f32(NC, K, dev=dev), out=u8(Q8, dev)),
                          lambda a: q.quantize_q8_1(a["x"], out=a["out"])),
        "quantize_weights": (lambda: dict(w=f32(M, K, dev=dev), out=u8(M * RB, dev)),
                             lambda a: q.quantize_weights(T, a["w"], out=a["out"])),
        "debug_subblock_sums": (lambda: dict(W=u8(M * RB, dev), xq=u8(Q8, dev)),
                                lambda a: q.debug_subblock_sums(T, a["W"], M, K, a["xq"], NC)),
        "read_bandwidth_probe": (lambda: dict(buf=u8(64, dev), sink=i32(1, dev=dev)),
                                 lambda a: q.read_bandwidth_probe(a["buf"], a["sink"])),
    }


WRONG = {torch.uint8: torch.int8, torch.float32: torch.float64, torch.int32: torch.int64}
# arguments whose size the call does not read from the tensor's length
NOT_SIZED = {"ids", "x", "w", "buf"}


@pytest.fixture
def no_library(monkeypatch):
    def reached():
        raise AssertionError("the library was called")

    monkeypatch.setattr(q, "lib", reached)


def _cases():
    out = []
    for name, (make, _) in specs("cpu").items():
        args = make()
        out.append((name, None, "cpu"))
        for arg in args:
            out.append((name, arg, "dtype"))
            if arg not in NOT_SIZED:
                out.append((name, arg, "short"))
    return out


def _apply(args, arg, kind):
    t = args[arg]
    if kind == "dtype":
        args[arg] = t.to(WRONG[t.dtype])
    elif kind == "short" and t.dim() > 1:
        args[arg] = t[..., :-1].contiguous()  # every row one element short
    elif kind == "short":
        args[arg] = t[: t.numel() - 1]
    return args


@pytest.mark.parametrize("name,arg,kind", _cases(), ids=lambda v: str(v))
def test_rejected_before_any_call(no_library, name, arg, kind):
    make, call = specs("cpu")[name]
    args = make()
    if kind != "cpu":
        _apply(args, arg, kind)
    with pytest.raises(ValueError) as e:
        call(args)
    msg = str(e.value)
    if kind == "cpu":
        assert "CUDA" in msg, msg
    elif kind == "dtype":
        assert arg in msg and "must be" in msg, msg
    else:
        assert arg in msg and "bytes" in msg, msg


def test_short_activation_rows_rejected(no_library):
    with pytest.raises(ValueError, match="rows hold"):
        q.mul_mat_vec_f32(T, u8(M * RB), M, K, f32(NC, K - 1))
    with pytest.raises(ValueError, match="fewer activation rows"):
        q.mul_mat_vec_id_f32(T, u8(E * M * RB), E, M, K, f32(1, K), i32(NC, TOPK))


def test_sizes_match_the_library_formulas():
    # the Python byte counts the checks use are the C ABI's size helpers
    import __graft_entry__

    __graft_entry__.build()
    for t in q.WEIGHT_TYPES:
        for k in (q.BLOCK_ELEMS[t], 4096, 11008 if t != q.Q6_K else 11264):
            assert q._row_bytes(t, k) == q.row_bytes(t, k)
    for k in (1, 32, 512, 513, 4096, 11008):
        for nc in (1, 3, 8):
            assert q._q8_1_bytes(k, nc) == q.q8_1_bytes(k, nc)


@pytest.mark.gpu
@pytest.mark.parametrize("name,arg,kind", [c for c in _cases() if c[2] == "short"], ids=lambda v: str(v))
def test_short_cuda_buffers_rejected(name, arg, kind):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    make, call = specs("cuda")[name]
    args = _apply(make(), arg, kind)
    with pytest.raises(ValueError, match="bytes"):
        call(args)
    call(make())  # the same call with full-size buffers goes through
    torch.cuda.synchronize()
