"""FP8 (e4m3) forward and backward against the oracle on the dequantised inputs.

The e4m3 codes stand for exact values (code * the descale of the code's
128-row tile of its head's q, k or v), so the oracle runs the plain float64
forward on those values. The kernel's only coarse rounding is the
probabilities entering P.V as e4m3 codes (relative error <= 2^-4 each); the
scores are exact sums of e4m3 products in fp32, the row sums and lse use the
fp32 probabilities, and out is rounded to bf16 (2^-9). Hence, per output:
  |err| <= 2^-4 * sum_j att_tj |v_j| + 2^-9 |out_t|  <=  (2^-4 + 2^-9) max|v|   (bound)
and, rounding errors of independent probabilities having standard deviation at
most 2^-4/sqrt(3) of the value, the error of out_t,d has standard deviation at
most sigma_t,d = sqrt((2^-4/sqrt 3)^2 sum_j att_tj^2 v_jd^2 + (2^-9/sqrt 3)^2 out_t,d^2).
The tests check the bound and that the RMS of err / sigma stays below 1.5 (a
misplaced code or a wrong descale gives values far above 1). lse: 1e-4 absolute.

The backward (attn_bwd_fp8: the codes expanded to bf16, then the bf16 backward)
is checked given the exact forward (bf16 rule, 2e-2 * max|ref| per q/k/v) and
chained behind attn_fwd_fp8, where the forward's rounding reaches dq and dk
through D = rowsum(dout * out); that test widens the rule by the propagated
error of D, computed from the forward's measured error.
"""
import math

import numpy as np
import pytest

import oracle
from causal_head_attention_fwd_gb300 import inputs

U4 = 2.0 ** -4
U9 = 2.0 ** -9


# ----------------------------------------------------------------------------- e4m3 codec pins
def test_e4m3_codes_of_the_format_definition():
    # 1 = 2^0 (exponent field 7): 0x38; 448 = 1.75 * 2^8: 0x7E; 2^-6 (first normal): 0x08;
    # 2^-9 (smallest subnormal): 0x01; -2: 0xC0; 0.875 * 2^-6 (largest subnormal): 0x07
    vals = np.array([1.0, 448.0, 2.0 ** -6, 2.0 ** -9, -2.0, 7 * 2.0 ** -9])
    codes = np.array([0x38, 0x7E, 0x08, 0x01, 0xC0, 0x07], dtype=np.uint8)
    assert np.array_equal(inputs.e4m3_encode(vals), codes)
    assert np.array_equal(inputs.e4m3_decode(codes), vals)


def test_e4m3_round_trip_and_rounding():
    c = np.arange(256, dtype=np.uint8)
    c = c[(c & 0x7F) != 0x7F]                                  # drop the two NaN codes
    v = inputs.e4m3_decode(c)
    nz = v != 0
    assert np.array_equal(inputs.e4m3_encode(v[nz]), c[nz])
    # ties to even: 1 + 1/16 lies between codes 0x38 (1) and 0x39 (1.125) -> 0x38;
    # 1 + 3/16 between 0x39 and 0x3A -> 0x3A; saturation beyond 448
    assert list(inputs.e4m3_encode(np.array([1.0625, 1.1875, 1000.0, -1000.0]))) == [0x38, 0x3A, 0x7E, 0xFE]
    # every finite value within half a spacing of its code
    x = np.linspace(-400, 400, 20001)
    r = inputs.e4m3_decode(inputs.e4m3_encode(x))
    spacing = np.where(np.abs(x) < 2 ** -6, 2 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 1e-30))) - 3))
    assert np.all(np.abs(r - x) <= spacing / 2 + 1e-12)


def test_fp8_inputs_dequantise_to_the_codes():
    B, T, C, NH = 2, 300, 128, 2
    for gain in (False, True):
        f = inputs.make_fp8_inputs(B, T, C, sigma=0.5, seed=7, NH=NH, tile_gain=gain)
        assert f.descale.shape == (3, B, NH, 3)
        for part in range(3):
            for b, h, k, sl in inputs.fp8_tile_view(f.codes, C, NH, part):
                d = float(f.descale[part, b, h, k])
                assert np.array_equal(inputs.e4m3_decode(f.codes[sl]) * d, f.qkv[sl])
                assert np.max(f.codes[sl] & 0x7F) == 0x7E          # each tile uses the full range
    # the gains make the tiles' scales differ
    g = inputs.make_fp8_inputs(B, T, C, sigma=0.5, seed=7, NH=NH, tile_gain=True).descale
    assert g.max() / g.min() > 2.0


# ----------------------------------------------------------------------------- ABI
def test_fp8_rejects_bad_arguments():
    from causal_head_attention_fwd_gb300 import api
    A, S = 1 << 32, 1 << 30

    def call(**kw):
        a = dict(qkv=A, d=A + S, out=A + 2 * S, lse=A + 3 * S, B=2, T=64, C=128, NH=2, causal=1)
        a.update(kw)
        return api.attn_fwd_fp8(a["qkv"], a["d"], a["out"], a["lse"], a["B"], a["T"], a["C"], a["NH"],
                                a["causal"], 0, check=False)
    assert call(d=0) == api.ATTN_ERR_INVALID_ARG
    assert call(qkv=0) == api.ATTN_ERR_INVALID_ARG
    assert call(d=A + S + 2) == api.ATTN_ERR_MISALIGNED
    assert call(out=A + 2 * S + 8) == api.ATTN_ERR_MISALIGNED
    assert call(C=96) == api.ATTN_ERR_UNSUPPORTED
    assert call(causal=3) == api.ATTN_ERR_INVALID_ARG
    assert call(out=A + 1024) == api.ATTN_ERR_INVALID_ARG          # out overlaps qkv
    assert call(d=A + 2 * S + 64) == api.ATTN_ERR_INVALID_ARG      # descale inside out
    # the descale array spans 3 * B * NH * ceil(T/128) floats (48 bytes here):
    # one that starts 32 bytes before out runs into it
    assert call(d=A + 2 * S - 32) == api.ATTN_ERR_INVALID_ARG


# ----------------------------------------------------------------------------- GPU parity
@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    from causal_head_attention_fwd_gb300 import build
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    return torch, api, ops


def _run(env, f, B, T, C, NH, causal):
    torch, api, ops = env
    codes = torch.from_numpy(f.codes).cuda()
    descale = torch.from_numpy(f.descale).cuda()
    out = torch.full((B, T, C), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, NH, T), float("nan"), dtype=torch.float32, device="cuda")
    ops.attention_forward_fp8(codes, descale, NH, causal, out=out, lse=lse)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    return ops.download_f64(out), ops.download_f64(lse)


def _check_head(g_out, g_lse, qkv, b, h, T, C, NH, causal):
    hs = C // NH
    q, k, v = oracle.split_heads(qkv[b:b + 1], C, NH)
    o, l, att, _ = oracle.head_forward(q[0, h], k[0, h], v[0, h], causal, return_att=True)
    got = g_out[b, :, h * hs:(h + 1) * hs]
    err = got - o
    vmax = np.max(np.abs(v[0, h]))
    assert np.isfinite(got).all()
    assert np.max(np.abs(err)) <= (U4 + U9) * vmax + 1e-6, "worst-case rounding bound exceeded"
    sigma = np.sqrt((U4 / math.sqrt(3)) ** 2 * ((att ** 2) @ (v[0, h] ** 2)) + (U9 / math.sqrt(3) * o) ** 2)
    z = err / np.maximum(sigma, 1e-12)
    assert math.sqrt(np.mean(z ** 2)) <= 1.5, "error larger than e4m3 rounding of the probabilities explains"
    assert np.max(np.abs(g_lse[b, h] - l)) <= 1e-4


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,C,NH,causal", [
    (2, 64, 128, 4, 1),       # hs 32
    (1, 300, 128, 2, 1),      # hs 64, ragged tail, several tiles
    (2, 256, 128, 2, 0),      # non-causal
    (1, 1, 128, 2, 1),        # one token
    (1, 700, 128, 2, 0),      # non-causal ragged
    (1, 1000, 64, 1, 1),      # one head, eight tiles
])
@pytest.mark.parametrize("gain", [False, True])
def test_fp8_forward_matches_oracle(env, B, T, C, NH, causal, gain):
    f = inputs.make_fp8_inputs(B, T, C, sigma=0.5, seed=77 + T, NH=NH, tile_gain=gain)
    g_out, g_lse = _run(env, f, B, T, C, NH, causal)
    for b in range(B):
        for h in range(NH):
            _check_head(g_out, g_lse, f.qkv, b, h, T, C, NH, bool(causal))


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,C,NH", [
    (8, 600, 768, 12),        # hs 64: 288 items for 152 CTAs, the last pair's second tile past T
    (16, 300, 256, 8),        # hs 32: 256 items
])
def test_fp8_noncausal_several_items_per_cta_all_heads(env, B, T, C, NH):
    """Without the mask the two softmax warpgroups take turns at the
    exponentials; every head against the oracle where each persistent CTA walks
    several items, some with one tile past T (that warpgroup's turns idle)."""
    f = inputs.make_fp8_inputs(B, T, C, sigma=0.5, seed=91 + T, NH=NH)
    g_out, g_lse = _run(env, f, B, T, C, NH, 0)
    for b in range(B):
        for h in range(NH):
            _check_head(g_out, g_lse, f.qkv, b, h, T, C, NH, False)


@pytest.mark.gpu
def test_fp8_gpt2s_workload_all_heads(env):
    """The FP8 benchmark's shape (B=16, T=1024, C=768, NH=12): every head against
    the oracle on the dequantised inputs, and the whole output written."""
    w = inputs.FP8_WORKLOADS["gpt2s_fp8"]
    B, T, C, NH = w["B"], w["T"], w["C"], w["NH"]
    f = inputs.make_fp8_inputs(B, T, C, sigma=w["sigma"], seed=w["seed"], NH=NH)
    g_out, g_lse = _run(env, f, B, T, C, NH, w["causal"])
    assert np.isfinite(g_out).all() and np.isfinite(g_lse).all()
    for b in range(B):
        for h in range(NH):
            _check_head(g_out, g_lse, f.qkv, b, h, T, C, NH, w["causal"])


# ----------------------------------------------------------------------------- FP8 backward
def test_fp8_bwd_rejects_bad_arguments():
    from causal_head_attention_fwd_gb300 import api
    A, S = 1 << 32, 1 << 30
    B, T, C, NH = 2, 64, 128, 2
    n = api.attn_bwd_fp8_workspace_size(B, T, C, NH, 1)
    assert n >= B * T * 3 * C * 2 + B * NH * T * 4

    def call(**kw):
        a = dict(dout=A, qkv=A + S, d=A + 2 * S, out=A + 3 * S, lse=A + 4 * S, dqkv=A + 5 * S, ws=A + 6 * S, n=n)
        a.update(kw)
        return api.attn_bwd_fp8(a["dout"], a["qkv"], a["d"], a["out"], a["lse"], a["dqkv"], B, T, C, NH, 1,
                                a["ws"], a["n"], 0, check=False)
    assert call(d=0) == api.ATTN_ERR_INVALID_ARG
    assert call(n=n - 1) == api.ATTN_ERR_WORKSPACE
    assert call(ws=0) == api.ATTN_ERR_WORKSPACE
    assert call(ws=A + 6 * S + 16) == api.ATTN_ERR_MISALIGNED
    assert call(dqkv=A + S + 64) == api.ATTN_ERR_INVALID_ARG         # dqkv overlaps qkv
    assert call(ws=A + 5 * S) == api.ATTN_ERR_INVALID_ARG            # workspace overlaps dqkv


def _bwd_fp8(env, f, out_bits, lse_f32, dout_bits, B, T, C, NH):
    torch, api, ops = env
    codes = torch.from_numpy(f.codes).cuda()
    descale = torch.from_numpy(f.descale).cuda()
    out = out_bits if isinstance(out_bits, torch.Tensor) else ops.upload(out_bits, "bf16")
    lse = lse_f32 if isinstance(lse_f32, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(lse_f32, np.float32)).cuda()
    dout = ops.upload(dout_bits, "bf16")
    dqkv = torch.full((B, T, 3 * C), float("nan"), dtype=torch.bfloat16, device="cuda")
    nws = api.attn_bwd_fp8_workspace_size(B, T, C, NH, 1)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    api.attn_bwd_fp8(dout, codes, descale, out, lse, dqkv, B, T, C, NH, 1, ws, nws)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    return ops.download_f64(dqkv)


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,C,NH", [(2, 64, 128, 4), (1, 300, 128, 2), (1, 1000, 64, 1)])
def test_fp8_backward_given_exact_forward(env, B, T, C, NH):
    """out and lse from the oracle: the GPU backward must meet the bf16 rule (2e-2 * max|ref| per q/k/v)."""
    f = inputs.make_fp8_inputs(B, T, C, sigma=0.5, seed=91 + T, NH=NH, tile_gain=True)
    r_out, r_lse = oracle.forward(f.qkv, B, T, C, NH, True)
    dout, dout_bits = inputs.draw((B, T, C), 1e-2, 92 + T, "bf16")
    out_bits = inputs.f32_to_bf16_bits(r_out.astype(np.float32))
    g = _bwd_fp8(env, f, out_bits, r_lse, dout_bits, B, T, C, NH)
    assert np.isfinite(g).all()
    ref = oracle.backward(dout.astype(np.float64), f.qkv, B, T, C, NH, True)
    for sl in (slice(0, C), slice(C, 2 * C), slice(2 * C, 3 * C)):
        assert np.max(np.abs(g[:, :, sl] - ref[:, :, sl])) <= 2e-2 * np.max(np.abs(ref[:, :, sl]))


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,C,NH", [(1, 300, 128, 2), (2, 256, 64, 1)])
def test_fp8_forward_then_backward(env, B, T, C, NH):
    """The chain attn_fwd_fp8 -> attn_bwd_fp8. dv does not see the forward's rounding: bf16 rule.
    dq, dk see it through D_t = dout_t . out_t: with dD_t the error of that sum (known here from
    the forward's measured error), |err dq_t| <= 2e-2 max|dq| + scale |dD_t| sum_j att_tj |k_j| and
    |err dk_j| <= 2e-2 max|dk| + scale sum_t att_tj |dD_t| |q_t|."""
    torch, api, ops = env
    f = inputs.make_fp8_inputs(B, T, C, sigma=0.5, seed=93 + T, NH=NH, tile_gain=True)
    g_out, g_lse = _run(env, f, B, T, C, NH, 1)
    dout, dout_bits = inputs.draw((B, T, C), 1e-2, 94 + T, "bf16")
    out_bits = inputs.f32_to_bf16_bits(g_out.astype(np.float32))   # exact: g_out holds bf16 values
    g = _bwd_fp8(env, f, out_bits, g_lse, dout_bits, B, T, C, NH)
    ref = oracle.backward(dout.astype(np.float64), f.qkv, B, T, C, NH, True)
    r_out, _ = oracle.forward(f.qkv, B, T, C, NH, True)
    hs = C // NH
    scale = 1.0 / math.sqrt(hs)
    q, k, v = oracle.split_heads(f.qkv, C, NH)
    lim = {s: 2e-2 * np.max(np.abs(ref[:, :, s * C:(s + 1) * C])) for s in range(3)}
    for b in range(B):
        for h in range(NH):
            cols = slice(h * hs, (h + 1) * hs)
            _, _, att, _ = oracle.head_forward(q[b, h], k[b, h], v[b, h], True, return_att=True)
            dD = np.sum(dout[b, :, cols].astype(np.float64) * (g_out[b, :, cols] - r_out[b, :, cols]), axis=1)
            tol_q = lim[0] + scale * np.abs(dD)[:, None] * (att @ np.abs(k[b, h]))
            tol_k = lim[1] + scale * (att.T @ (np.abs(dD)[:, None] * np.abs(q[b, h])))
            e_q = np.abs(g[b, :, cols] - ref[b, :, cols])
            e_k = np.abs(g[b, :, C + h * hs:C + (h + 1) * hs] - ref[b, :, C + h * hs:C + (h + 1) * hs])
            e_v = np.abs(g[b, :, 2 * C + h * hs:2 * C + (h + 1) * hs] - ref[b, :, 2 * C + h * hs:2 * C + (h + 1) * hs])
            assert np.all(e_q <= tol_q) and np.all(e_k <= tol_k) and np.max(e_v) <= lim[2]
