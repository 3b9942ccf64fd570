"""The torch layer checks every caller-provided tensor before it reaches the C
ABI, which takes raw pointers and trusts their sizes. Runs on the CPU: shape
and dtype errors are raised before the device check, and well-formed tensors
on the CPU are refused by the device check, so nothing is launched."""
import pytest

torch = pytest.importorskip("torch")
ops = pytest.importorskip("causal_head_attention_fwd_gb300.ops")

B, T, C, NH = 2, 16, 128, 2
bf, f32 = torch.bfloat16, torch.float32


def _qkv(dtype=bf):
    return torch.zeros((B, T, 3 * C), dtype=dtype)


@pytest.mark.parametrize("kw,msg", [
    (dict(out=torch.zeros((B, T, C - 1), dtype=bf)), "out has shape"),
    (dict(out=torch.zeros((B, T, C), dtype=f32)), "out has dtype"),
    (dict(lse=torch.zeros((B, T, NH), dtype=f32)), "lse has shape"),
    (dict(lse=torch.zeros((B, NH, T), dtype=bf)), "lse has dtype"),
    (dict(out=torch.zeros((B, C, T), dtype=bf).transpose(1, 2)), "contiguous"),
    (dict(), "CUDA device"),
])
def test_forward_checks_tensors(kw, msg):
    with pytest.raises(ValueError, match=msg):
        ops.attention_forward(_qkv(), NH, True, **kw)


def test_forward_checks_qkv():
    with pytest.raises(ValueError, match="dtype"):
        ops.attention_forward(_qkv(torch.float16), NH)
    with pytest.raises(ValueError, match=r"\(B, T, 3C\)"):
        ops.attention_forward(torch.zeros((B, T, 3 * C + 1), dtype=bf), NH)
    with pytest.raises(ValueError, match="does not divide"):
        ops.attention_forward(_qkv(), 3)
    with pytest.raises(ValueError, match="contiguous"):
        ops.attention_forward(torch.zeros((B, 3 * C, T), dtype=bf).transpose(1, 2), NH)


def _bwd_args():
    return dict(dout=torch.zeros((B, T, C), dtype=bf), qkv=_qkv(), out=torch.zeros((B, T, C), dtype=bf),
                lse=torch.zeros((B, NH, T), dtype=f32))


@pytest.mark.parametrize("name,bad,msg", [
    ("dout", torch.zeros((B, T, 3 * C), dtype=bf), "dout has shape"),
    ("out", torch.zeros((B, T, C), dtype=f32), "out has dtype"),
    ("lse", torch.zeros((B, NH, T + 1), dtype=f32), "lse has shape"),
    ("dqkv", torch.zeros((B, T, C), dtype=bf), "dqkv has shape"),
    ("lse", None, "required"),
])
def test_backward_checks_tensors(name, bad, msg):
    a = _bwd_args()
    dqkv = None
    if name == "dqkv":
        dqkv = bad
    else:
        a[name] = bad
    with pytest.raises(ValueError, match=msg):
        ops.attention_backward(a["dout"], a["qkv"], a["out"], a["lse"], NH, True, dqkv=dqkv)


def test_backward_on_cpu_is_refused():
    a = _bwd_args()
    with pytest.raises(ValueError, match="CUDA device"):
        ops.attention_backward(a["dout"], a["qkv"], a["out"], a["lse"], NH, True)


def test_linear_checks_tensors():
    x = torch.zeros((4, 64), dtype=bf)
    w = torch.zeros((32, 64), dtype=bf)
    with pytest.raises(ValueError, match="weight has shape"):
        ops.linear(x, torch.zeros((32, 48), dtype=bf))
    with pytest.raises(ValueError, match="bias has shape"):
        ops.linear(x, w, torch.zeros((31,), dtype=bf))
    with pytest.raises(ValueError, match="inp has dtype"):
        ops.linear(x.float(), w)
    with pytest.raises(ValueError, match="out has shape"):
        ops.linear(x, w, out=torch.zeros((4, 33), dtype=bf))
    with pytest.raises(ValueError, match="CUDA device"):
        ops.linear(x, w)


def test_fp8_decode_and_matrices_check_tensors():
    codes = torch.zeros((B, T, 3 * C), dtype=torch.uint8)
    with pytest.raises(ValueError, match="dtype"):
        ops.attention_forward_fp8(_qkv(), torch.ones(3), NH)
    with pytest.raises(ValueError, match="descale has shape"):
        ops.attention_forward_fp8(codes, torch.ones(2), NH)
    with pytest.raises(ValueError, match="out has shape"):
        ops.attention_decode(_qkv(), NH, 3, out=torch.zeros((B, 2, C), dtype=bf))
    with pytest.raises(ValueError, match="lse has shape"):
        ops.attention_matrices(_qkv(), torch.zeros((B, NH), dtype=f32), NH)
    with pytest.raises(ValueError, match="att has shape"):
        ops.attention_matrices(_qkv(), torch.zeros((B, NH, T), dtype=f32), NH, att=torch.zeros((B, NH, T, T - 1)))
