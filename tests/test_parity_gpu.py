"""GPU parity: the CUDA path (through the C ABI) against the float64 CPU oracle.

Both sides receive the same seeded inputs (bf16 values widened exactly for the
oracle). Tolerance rule, applied to the whole tensor:
    max |gpu - oracle| <= tol * max |oracle|
with tol = 2e-2 for bf16 inputs (out and dqkv), and for fp32 inputs 2e-3 (out)
and 1e-2 (dqkv).

lse is an fp32 row statistic, lse = (m*c + log2 l) * ln 2 with c = scale*log2 e.
With bf16 inputs its absolute error is bounded by:
  - the score: exact bf16 products summed in fp32 over hs terms, |ds| <= hs 2^-24
    sum_i |q_i k_i| (about 4e-5 for N(0, 0.5^2) inputs at hs = 64, worst case),
    times the scale: <= 1e-5;
  - the row sum l: ex2.approx (relative error below 2^-22) of each term, fp32
    partial sums of at most 16 terms per tile and one running sum per key tile
    (at most T/128 = 64 additions at T = 8192): relative <= (16 + 64) 2^-24 + 2^-22,
    about 5e-6 in ln l;
  - lg2.approx (absolute error below 2^-22) and the final products: < 1e-6.
So the error stays below about 2e-5; the test allows 1e-4 (measured: ~1e-6).
A wrong scale, base, mask or key range moves lse by >= 1e-2. With fp32
inputs the tensor core reads q and k as tf32 (8 + 10 bits: each operand loses
less than 2^-10 of its magnitude), so every score moves by at most
2^-9 * sum_i |q_i k_i| and lse, a log-sum-exp of scale * scores, by at most
scale times the largest such bound of the head; the test uses that bound, plus
1e-5 for the fp32 sums.

Coverage: every head of small shapes (one tile, several tiles, ragged tails,
hs 32 and 64, causal and not); every head of shapes whose persistent kernels
give each CTA several work items (the forward's causal deal table, its snake
order without the mask, the backward's snake order, the Q double buffer and the
K/V rings running on across items), also with more causal items than the deal
table holds (both kernels in the snake order); and every head of the full GPT-2 small
(fp32 and bf16), GPT-2 XL-width and ViT-B/16 workloads, with four heads over
both sequences of the long-context one, in the benchmark's launch configuration.
"""
import numpy as np
import pytest

import oracle
from causal_head_attention_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-2), "f32": (2e-3, 1e-2)}     # (out, dqkv)
LSE_ABS = 1e-4


def _lse_tol(qkv, C, NH, dtype, heads=None):
    """Absolute lse tolerance: 1e-4 for bf16 inputs; for fp32 inputs the tf32
    operand bound described in the module docstring (over the given heads)."""
    if dtype == "bf16":
        return LSE_ABS
    hs = C // NH
    x = np.abs(np.asarray(qkv, dtype=np.float64))
    worst = 0.0
    for h in (range(NH) if heads is None else heads):
        for b in range(x.shape[0]):
            q = x[b, :, h * hs:(h + 1) * hs]
            k = x[b, :, C + h * hs:C + (h + 1) * hs]
            worst = max(worst, float(np.max(q @ k.T)))
    return 2.0 ** -9 * worst / np.sqrt(hs) + 1e-5


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_head_attention_fwd_gb300 import build
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    return torch, api, ops


def _rel(a, ref):
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(a - ref)) / (den if den > 0 else 1.0))


def _run(env, B, T, C, NH, causal, dtype="bf16", sq=0.5, sd=1e-2, seed=0):
    torch, api, ops = env
    host = inputs.make_inputs(B, T, C, NH, dtype, sq, sd, 100 + seed, 200 + seed)
    qkv = ops.upload(host.qkv_dev, dtype)
    dout = ops.upload(host.dout_dev, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.full((B, T, C), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((B, NH, T), float("nan"), dtype=torch.float32, device="cuda")
    dqkv = torch.full((B, T, 3 * C), float("nan"), dtype=tdt, device="cuda")
    ops.attention_forward(qkv, NH, bool(causal), out=out, lse=lse)
    ops.attention_backward(dout, qkv, out, lse, NH, bool(causal), dqkv=dqkv)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    return host, ops.download_f64(out), ops.download_f64(lse), ops.download_f64(dqkv)


SHAPES = [
    # B, T, C, NH, causal         (hs = C/NH; T spans one tile, several tiles, ragged tails)
    (1, 1, 128, 2, 1), (1, 1, 128, 2, 0), (2, 2, 128, 2, 1),
    (2, 17, 128, 2, 1), (2, 64, 128, 4, 1), (2, 127, 64, 1, 0),
    (1, 128, 128, 2, 1), (1, 129, 128, 4, 1), (2, 196, 128, 2, 0),
    (1, 255, 64, 1, 1), (1, 256, 64, 1, 0), (1, 257, 64, 1, 1),
    (1, 600, 64, 2, 1), (1, 1000, 128, 2, 1), (1, 1000, 128, 2, 0),
    (2, 300, 128, 4, 0), (1, 1000, 64, 2, 0),          # hs = 32 without the mask
]

# Shapes with more work items than the GPU has SMs, so every persistent CTA
# runs several items: (forward items = B*NH*ceil(T/256), backward items =
# B*NH*ceil(T/128); 152 CTAs on a GB300).
MULTI_ITEM = [
    (8, 1024, 768, 12, 1),      # hs 64, causal: 384 forward / 768 backward items (deal table)
    (16, 1024, 256, 4, 1),      # hs 64, causal: 256 / 512
    (16, 512, 256, 8, 1),       # hs 32, causal: 256 / 512
    (8, 600, 256, 8, 0),        # hs 32, no mask: 192 / 320 (snake order)
    (6, 1000, 768, 12, 0),      # hs 64, no mask, ragged tail: 288 / 576
    (6, 1100, 768, 12, 1),      # hs 64, causal, the last pair's second tile past T: 360 / 648
]


def _check(host, out, lse, dqkv, B, T, C, NH, causal, dtype):
    tol_out, tol_d = TOL[dtype]
    ref_out, ref_lse = oracle.forward(host.qkv, B, T, C, NH, bool(causal))
    ref_dqkv = oracle.backward(host.dout, host.qkv, B, T, C, NH, bool(causal))
    assert np.isfinite(out).all() and np.isfinite(lse).all() and np.isfinite(dqkv).all()
    e_out = _rel(out, ref_out)
    assert e_out <= tol_out, f"out rel err {e_out:.3e}"
    e_lse = np.max(np.abs(lse - ref_lse))
    assert e_lse <= _lse_tol(host.qkv, C, NH, dtype), f"lse abs err {e_lse:.3e}"
    for name, sl in (("dq", slice(0, C)), ("dk", slice(C, 2 * C)), ("dv", slice(2 * C, 3 * C))):
        e = _rel(dqkv[:, :, sl], ref_dqkv[:, :, sl])
        assert e <= tol_d, f"{name} rel err {e:.3e}"
    assert _rel(dqkv, ref_dqkv) <= tol_d


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,C,NH,causal", SHAPES)
def test_parity_all_heads(env, B, T, C, NH, causal, dtype):
    host, out, lse, dqkv = _run(env, B, T, C, NH, causal, dtype=dtype, seed=T + C)
    _check(host, out, lse, dqkv, B, T, C, NH, causal, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,C,NH,causal", MULTI_ITEM)
def test_parity_all_heads_several_items_per_cta(env, B, T, C, NH, causal, dtype):
    """Every head against the oracle where each persistent CTA walks several
    work items (checked: the items outnumber the SMs)."""
    torch = env[0]
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * NH * ((T + 255) // 256) > n_sm
    host, out, lse, dqkv = _run(env, B, T, C, NH, causal, dtype=dtype, seed=3 * T + NH)
    _check(host, out, lse, dqkv, B, T, C, NH, causal, dtype)


def test_parity_causal_beyond_the_deal_table(env):
    """Causal items of unequal length, more than the 2048 the host's deal
    table holds: both persistent kernels fall back to the snake order
    (hs 32: 2080 forward items of 1 and 2 key steps per query tile, 4160
    backward items of 1 to 4 steps). Every head against the oracle."""
    B, T, C, NH = 260, 512, 128, 4
    assert B * NH * ((T + 255) // 256) > 2048 and B * NH * ((T + 127) // 128) > 2048
    host, out, lse, dqkv = _run(env, B, T, C, NH, 1, seed=5 * B + T)
    _check(host, out, lse, dqkv, B, T, C, NH, 1, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_parity_unit_variance_hs32(env, dtype):
    """The tiny workload's shape and distribution (N(0,1) qkv and dout); with
    fp32 inputs this is the tiny workload itself."""
    B, T, C, NH = 2, 64, 128, 4
    host, out, lse, dqkv = _run(env, B, T, C, NH, 1, dtype=dtype, sq=1.0, sd=1.0, seed=5)
    _check(host, out, lse, dqkv, B, T, C, NH, 1, dtype)


def test_tiny_workload_f32(env):
    """The tiny workload exactly as defined (its seeds and distribution)."""
    w = inputs.WORKLOADS["tiny"]
    torch, api, ops = env
    host = inputs.workload_inputs(w)
    qkv = ops.upload(host.qkv_dev, w.dtype)
    dout = ops.upload(host.dout_dev, w.dtype)
    out, lse = ops.attention_forward(qkv, w.NH, bool(w.causal))
    dqkv = ops.attention_backward(dout, qkv, out, lse, w.NH, bool(w.causal))
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    _check(host, ops.download_f64(out), ops.download_f64(lse), ops.download_f64(dqkv),
           w.B, w.T, w.C, w.NH, w.causal, w.dtype)


def test_first_row_is_v0_and_dq0_small(env):
    """Causal row 0 attends only to key 0: out = v_0 exactly (bf16), dq_0 ~ 0."""
    B, T, C, NH = 2, 300, 128, 2
    host, out, _, dqkv = _run(env, B, T, C, NH, 1, seed=9)
    np.testing.assert_array_equal(out[:, 0, :], host.qkv[:, 0, 2 * C:].astype(np.float64))
    assert np.max(np.abs(dqkv[:, 0, :C])) <= 1e-3 * np.max(np.abs(dqkv[:, :, :C]))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_outputs_fully_overwritten_and_no_out_of_bounds_writes(env, dtype):
    """Outputs live inside larger buffers pre-filled with a sentinel: the region
    must be fully written (no NaN left) and the guard bands untouched."""
    torch, api, ops = env
    B, T, C, NH, G = 2, 333, 128, 2, 4096
    host = inputs.make_inputs(B, T, C, NH, dtype, 0.5, 1e-2, 77, 78)
    qkv = ops.upload(host.qkv_dev, dtype)
    dout = ops.upload(host.dout_dev, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    n_out, n_lse, n_d = B * T * C, B * NH * T, B * T * 3 * C
    big_out = torch.full((n_out + 2 * G,), float("nan"), dtype=tdt, device="cuda")
    big_lse = torch.full((n_lse + 2 * G,), float("nan"), dtype=torch.float32, device="cuda")
    big_d = torch.full((n_d + 2 * G,), float("nan"), dtype=tdt, device="cuda")
    out = big_out[G:G + n_out].view(B, T, C)
    lse = big_lse[G:G + n_lse].view(B, NH, T)
    dqkv = big_d[G:G + n_d].view(B, T, 3 * C)
    ops.attention_forward(qkv, NH, True, out=out, lse=lse)
    ops.attention_backward(dout, qkv, out, lse, NH, True, dqkv=dqkv)
    torch.cuda.synchronize()
    for big, n in ((big_out, n_out), (big_lse, n_lse), (big_d, n_d)):
        assert not torch.isnan(big[G:G + n]).any()
        assert torch.isnan(big[:G]).all() and torch.isnan(big[G + n:]).all()


def test_repeat_runs_deterministic_where_designed(env):
    """Forward and dK/dV have a fixed summation order: bit-identical reruns.
    dQ is reduced with atomics: reruns agree within the tolerance only."""
    torch, api, ops = env
    B, T, C, NH = 2, 700, 128, 2
    host = inputs.make_inputs(B, T, C, NH, "bf16", 0.5, 1e-2, 31, 32)
    qkv = ops.upload(host.qkv_dev, "bf16")
    dout = ops.upload(host.dout_dev, "bf16")
    o1, l1 = ops.attention_forward(qkv, NH, True)
    o2, l2 = ops.attention_forward(qkv, NH, True)
    d1 = ops.attention_backward(dout, qkv, o1, l1, NH, True)
    d2 = ops.attention_backward(dout, qkv, o1, l1, NH, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(d1[:, :, C:], d2[:, :, C:])
    dq1, dq2 = d1[:, :, :C].float(), d2[:, :, :C].float()
    assert (dq1 - dq2).abs().max().item() <= 1e-2 * dq1.abs().max().item()


def test_repeat_runs_bit_identical_f32(env):
    """The fp32 path has no atomics anywhere: every output reruns bit-identically."""
    torch, api, ops = env
    B, T, C, NH = 2, 700, 128, 2
    host = inputs.make_inputs(B, T, C, NH, "f32", 0.5, 1e-2, 33, 34)
    qkv = ops.upload(host.qkv_dev, "f32")
    dout = ops.upload(host.dout_dev, "f32")
    o1, l1 = ops.attention_forward(qkv, NH, True)
    o2, l2 = ops.attention_forward(qkv, NH, True)
    d1 = ops.attention_backward(dout, qkv, o1, l1, NH, True)
    d2 = ops.attention_backward(dout, qkv, o1, l1, NH, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(d1, d2)


FULL = ["gpt2s_f32", "gpt2s_bf16", "xl_bf16", "vit_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_all_heads(env, name):
    """Full workload sizes, in the launch configuration the benchmark times;
    every (b, h) head against the oracle, whole-tensor tolerance rule."""
    torch, api, ops = env
    w = inputs.WORKLOADS[name]
    host = inputs.workload_inputs(w)
    qkv = ops.upload(host.qkv_dev, w.dtype)
    dout = ops.upload(host.dout_dev, w.dtype)
    out, lse = ops.attention_forward(qkv, w.NH, bool(w.causal))
    dqkv = ops.attention_backward(dout, qkv, out, lse, w.NH, bool(w.causal))
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    g_out, g_lse, g_d = ops.download_f64(out), ops.download_f64(lse), ops.download_f64(dqkv)
    del out, lse, dqkv, qkv, dout
    _check(host, g_out, g_lse, g_d, w.B, w.T, w.C, w.NH, w.causal, w.dtype)


def test_long_context_heads_of_both_sequences(env):
    """The long-context workload (B=2, T=8192): four heads, two of each
    sequence, against the oracle (each head is an exact check of that head);
    every output finite."""
    torch, api, ops = env
    w = inputs.WORKLOADS["long_bf16"]
    host = inputs.workload_inputs(w)
    qkv = ops.upload(host.qkv_dev, w.dtype)
    dout = ops.upload(host.dout_dev, w.dtype)
    out, lse = ops.attention_forward(qkv, w.NH, bool(w.causal))
    dqkv = ops.attention_backward(dout, qkv, out, lse, w.NH, bool(w.causal))
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    heads = [(0, 0), (0, 7), (1, 4), (1, 11)]
    hs, C = w.hs, w.C
    tol_out, tol_d = TOL[w.dtype]
    for b, h in heads:
        x = host.qkv[b:b + 1].astype(np.float64)
        d = host.dout[b:b + 1].astype(np.float64)
        ref_out, ref_lse = oracle.forward(x, 1, w.T, C, w.NH, bool(w.causal), heads=[(0, h)])
        ref_d = oracle.backward(d, x, 1, w.T, C, w.NH, bool(w.causal), heads=[(0, h)])
        cols = slice(h * hs, (h + 1) * hs)
        g_out = ops.download_f64(out[b, :, cols])
        assert _rel(g_out, ref_out[0, :, cols]) <= tol_out, (b, h)
        assert np.max(np.abs(ops.download_f64(lse[b, h]) - ref_lse[0, h])) <= LSE_ABS, (b, h)
        for off in (0, C, 2 * C):
            sl = slice(off + h * hs, off + (h + 1) * hs)
            assert _rel(ops.download_f64(dqkv[b, :, sl]), ref_d[0, :, sl]) <= tol_d, (b, h, off)
    assert torch.isfinite(out.float()).all() and torch.isfinite(dqkv.float()).all()
