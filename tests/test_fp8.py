"""FP8 (e4m3) forward: attn_fwd_fp8 against the oracle on the dequantised inputs.

The e4m3 codes stand for exact values (code * descale), so the oracle runs the
plain float64 forward on those values. The kernel's only coarse rounding is the
probabilities entering P.V as e4m3 codes (relative error <= 2^-4 each); the
scores are exact sums of e4m3 products in fp32, the row sums and lse use the
fp32 probabilities, and out is rounded to bf16 (2^-9). Hence, per output:
  |err| <= 2^-4 * sum_j att_tj |v_j| + 2^-9 |out_t|  <=  (2^-4 + 2^-9) max|v|   (bound)
and, rounding errors of independent probabilities having standard deviation at
most 2^-4/sqrt(3) of the value, the error of out_t,d has standard deviation at
most sigma_t,d = sqrt((2^-4/sqrt 3)^2 sum_j att_tj^2 v_jd^2 + (2^-9/sqrt 3)^2 out_t,d^2).
The tests check the bound and that the RMS of err / sigma stays below 1.5 (a
misplaced code or a wrong descale gives values far above 1). lse: 1e-4 absolute.
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
    f = inputs.make_fp8_inputs(2, 8, 64, sigma=0.5, seed=7)
    for i in range(3):
        part = inputs.e4m3_decode(f.codes[:, :, i * 64:(i + 1) * 64]) * float(f.descale[i])
        assert np.array_equal(part, f.qkv[:, :, i * 64:(i + 1) * 64])
        assert np.max(np.abs(f.codes[:, :, i * 64:(i + 1) * 64] & 0x7F)) == 0x7E   # full range used


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
def test_fp8_forward_matches_oracle(env, B, T, C, NH, causal):
    f = inputs.make_fp8_inputs(B, T, C, sigma=0.5, seed=77 + T)
    g_out, g_lse = _run(env, f, B, T, C, NH, causal)
    for b in range(B):
        for h in range(NH):
            _check_head(g_out, g_lse, f.qkv, b, h, T, C, NH, bool(causal))


@pytest.mark.gpu
def test_fp8_gpt2s_workload_sampled_heads(env):
    """The FP8 benchmark's shape (B=16, T=1024, C=768, NH=12); the oracle checks sampled heads,
    and the whole output must be written."""
    w = inputs.FP8_WORKLOADS["gpt2s_fp8"]
    B, T, C, NH = w["B"], w["T"], w["C"], w["NH"]
    f = inputs.make_fp8_inputs(B, T, C, sigma=w["sigma"], seed=w["seed"])
    g_out, g_lse = _run(env, f, B, T, C, NH, w["causal"])
    assert np.isfinite(g_out).all() and np.isfinite(g_lse).all()
    rng = np.random.default_rng(w["seed"])
    for _ in range(3):
        b, h = int(rng.integers(B)), int(rng.integers(NH))
        _check_head(g_out, g_lse, f.qkv, b, h, T, C, NH, w["causal"])
