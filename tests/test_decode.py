"""Decode forward (attn_decode) against the oracle.

The oracle computes the full causal forward over all L positions; the decode
step's outputs must equal its last Tq rows (out and lse), since query i sits
at position L-Tq+i and sees keys 0..L-Tq+i. The decode kernels compute in fp32
from the stored inputs (no reduced-precision products), so fp32 inputs match
to 2e-3 of max|out| (the fp32 parity rule; observed ~1e-6) and bf16 inputs to
2e-2 (the bf16 output rounding dominates); lse to 1e-4 absolute.
"""
import numpy as np
import pytest

import oracle
from causal_head_attention_fwd_gb300 import inputs


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    from causal_head_attention_fwd_gb300 import build
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    return torch, api, ops


def _rel(a, r):
    return float(np.max(np.abs(a - r)) / max(np.max(np.abs(r)), 1e-30))


TOL = {"bf16": 2e-2, "f32": 2e-3}


def test_decode_rejects_bad_arguments(env):
    _, api, _ = env
    A, S = 1 << 32, 1 << 30
    def call(**kw):
        a = dict(qkv=A, out=A + S, lse=A + 2 * S, B=2, L=64, C=128, NH=2, Tq=1, ws=A + 3 * S, n=1 << 20)
        a.update(kw)
        return api.attn_decode(a["qkv"], a["out"], a["lse"], a["B"], a["L"], a["C"], a["NH"], a["Tq"], 1,
                               a["ws"], a["n"], 0, check=False)
    assert call(Tq=0) == api.ATTN_ERR_INVALID_ARG
    assert call(Tq=9) == api.ATTN_ERR_INVALID_ARG                 # more than 8 new tokens
    assert call(L=3, Tq=4) == api.ATTN_ERR_INVALID_ARG            # more new tokens than positions
    assert call(n=16) == api.ATTN_ERR_WORKSPACE
    assert call(ws=0) == api.ATTN_ERR_WORKSPACE
    assert call(out=A + S + 8) == api.ATTN_ERR_MISALIGNED
    assert call(C=96) == api.ATTN_ERR_UNSUPPORTED
    assert api.attn_decode_workspace_size(2, 64, 128, 2, 0, 1) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,L,C,NH,Tq", [
    (1, 1, 128, 2, 1), (2, 17, 128, 2, 1), (2, 300, 128, 4, 3), (1, 257, 64, 1, 8),
    (1, 512, 128, 2, 5), (3, 1000, 128, 2, 2), (1, 256, 128, 2, 1),
    # caches shorter than the 16 query rows the tensor-core form loads
    (1, 5, 128, 2, 4), (2, 3, 128, 4, 3),
    # hs 32, one to four query tokens: the combine's one-record-per-lane form, one column per lane
    (2, 300, 128, 4, 1), (1, 4100, 64, 2, 1), (1, 2100, 64, 2, 4),
    # hs 32 with more than four query tokens (the 8-query instantiation)
    (1, 700, 128, 4, 7),
])
def test_decode_matches_last_rows_of_the_full_forward(env, dtype, B, L, C, NH, Tq):
    torch, api, ops = env
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    host = inputs.make_inputs(B, L, C, NH, dtype, 0.5, 1e-2, 90 + L, 91 + L)
    qkv = ops.upload(host.qkv_dev, dtype)
    out, lse = ops.attention_decode(qkv, NH, Tq)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    ref_out, ref_lse = oracle.forward(host.qkv, B, L, C, NH, True)
    g_out, g_lse = ops.download_f64(out), ops.download_f64(lse)
    assert np.isfinite(g_out).all() and np.isfinite(g_lse).all()
    assert _rel(g_out, ref_out[:, L - Tq:, :]) <= TOL[dtype]
    assert np.max(np.abs(g_lse - ref_lse[:, :, L - Tq:])) <= 1e-4


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["gpt2s_decode", "gpt2s_decode4"])
def test_decode_workload_sampled_heads(env, name):
    """The decode benchmark's shapes; the oracle checks sampled (b, h) heads."""
    torch, api, ops = env
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = inputs.DECODE_WORKLOADS[name]
    qkv_h, qkv_dev = inputs.draw((w.B, w.L, 3 * w.C), w.sigma_qkv, w.seed_qkv, w.dtype)
    qkv = ops.upload(qkv_dev, w.dtype)
    out, lse = ops.attention_decode(qkv, w.NH, w.Tq)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    rng = np.random.default_rng(w.seed_qkv)
    hs, C = w.hs, w.C
    for _ in range(2):
        b, h = int(rng.integers(w.B)), int(rng.integers(w.NH))
        ref_out, ref_lse = oracle.forward(qkv_h[b:b + 1].astype(np.float64), 1, w.L, C, w.NH, True, heads=[(0, h)])
        cols = slice(h * hs, (h + 1) * hs)
        g = ops.download_f64(out[b, :, cols])
        assert _rel(g, ref_out[0, w.L - w.Tq:, cols]) <= TOL[w.dtype]
        assert np.max(np.abs(ops.download_f64(lse[b, h]) - ref_lse[0, h, w.L - w.Tq:])) <= 1e-4


@pytest.mark.gpu
def test_decode_output_fully_written_no_out_of_bounds(env):
    torch, api, ops = env
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, L, C, NH, Tq, G = 2, 700, 128, 2, 3, 512
    host = inputs.make_inputs(B, L, C, NH, "bf16", 0.5, 1e-2, 5, 6)
    qkv = ops.upload(host.qkv_dev, "bf16")
    n = B * Tq * C
    big = torch.full((n + 2 * G,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = big[G:G + n].view(B, Tq, C)
    ops.attention_decode(qkv, NH, Tq, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(big[G:G + n]).any()
    assert torch.isnan(big[:G]).all() and torch.isnan(big[G + n:]).all()
