"""attn_linear_fwd (GEMM with fused bias) and the attention block forward
(c_attn -> attention -> c_proj) against the oracle.

Linear tolerance: the kernel accumulates exact bf16 products in fp32 and
rounds once to bf16, so per element |err| <= 2^-9 |ref| + K 2^-24 sum_k
|a_mk w_ok| (rounding of the result, worst-case fp32 summation); the tests
allow 2^-8 |ref| + 2^-14 sum_k |a_mk w_ok|. The block is checked stage by
stage, each stage fed the GPU's own bf16 input (linear bound for c_attn and
c_proj, the bf16 attention rule 2e-2 * max|ref| for the attention), and end
to end against the exact block at 2e-2 * max|y|.
"""
import numpy as np
import pytest

import oracle
from causal_head_attention_fwd_gb300 import inputs


def _lin_tol(a, w, ref):
    return 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * (np.abs(a) @ np.abs(w).T)


def test_linear_rejects_bad_arguments():
    from causal_head_attention_fwd_gb300 import api
    A, S = 1 << 32, 1 << 30

    def call(**kw):
        a = dict(inp=A, w=A + S, b=A + 2 * S, out=A + 3 * S, M=64, N=256, K=64)
        a.update(kw)
        return api.attn_linear_fwd(a["inp"], a["w"], a["b"], a["out"], a["M"], a["N"], a["K"], 0, check=False)
    assert call(M=0) == api.ATTN_ERR_INVALID_ARG
    assert call(N=100) == api.ATTN_ERR_UNSUPPORTED
    assert call(K=20) == api.ATTN_ERR_UNSUPPORTED
    assert call(inp=0) == api.ATTN_ERR_INVALID_ARG
    assert call(out=A + 3 * S + 8) == api.ATTN_ERR_MISALIGNED
    assert call(b=A + 2 * S + 2) == api.ATTN_ERR_MISALIGNED
    assert call(out=A + 64) == api.ATTN_ERR_INVALID_ARG            # out overlaps inp


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    from causal_head_attention_fwd_gb300 import build
    build.build()
    from causal_head_attention_fwd_gb300 import api, ops
    return torch, api, ops


def _dev(torch, ops, bits):
    return ops.upload(bits, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,bias", [
    (128, 256, 64, True),       # one tile, one k-block
    (300, 520, 200, True),      # ragged M, N and K
    (1, 8, 8, True),            # smallest
    (1000, 768, 768, False),    # c_proj shape, no bias, several tiles per CTA
    (513, 2304, 128, True),     # 9 column tiles
])
def test_linear_matches_oracle(env, M, N, K, bias):
    torch, api, ops = env
    a, ab = inputs.draw((M, K), 1.0, 600 + M, "bf16")
    w, wb = inputs.draw((N, K), 0.05, 601 + N, "bf16")
    b, bb = inputs.draw((N,), 0.05, 602 + K, "bf16")
    big = torch.full((M * N + 2048,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = big[1024:1024 + M * N].view(M, N)
    ops.linear(_dev(torch, ops, ab), _dev(torch, ops, wb), _dev(torch, ops, bb) if bias else None, out=out)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    ref = oracle.linear(a, w, b if bias else None)
    got = ops.download_f64(out)
    assert np.all(np.abs(got - ref) <= _lin_tol(a.astype(np.float64), w.astype(np.float64), ref))
    assert torch.isnan(big[:1024].float()).all() and torch.isnan(big[1024 + M * N:].float()).all()


@pytest.mark.gpu
def test_linear_gpt2s_c_attn_sampled_rows(env):
    """The block benchmark's c_attn GEMM (M = 16384, N = 2304, K = 768): sampled rows, whole output finite."""
    torch, api, ops = env
    M, N, K = 16 * 1024, 2304, 768
    a, ab = inputs.draw((M, K), 1.0, 700, "bf16")
    w, wb = inputs.draw((N, K), 0.02, 701, "bf16")
    b, bb = inputs.draw((N,), 0.02, 702, "bf16")
    out = ops.linear(_dev(torch, ops, ab), _dev(torch, ops, wb), _dev(torch, ops, bb))
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    assert torch.isfinite(out.float()).all()
    rows = np.random.default_rng(7).choice(M, 64, replace=False)
    ref = oracle.linear(a[rows], w, b)
    got = ops.download_f64(out[torch.from_numpy(rows).cuda()])
    assert np.all(np.abs(got - ref) <= _lin_tol(a[rows].astype(np.float64), w.astype(np.float64), ref))


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,C,NH", [(2, 300, 128, 2), (1, 129, 256, 4)])
def test_block_forward_stage_by_stage(env, B, T, C, NH):
    torch, api, ops = env
    bi = inputs.make_block_inputs(B, T, C, seed=800 + T)
    d = {k: _dev(torch, ops, v) for k, v in bi.bits.items()}
    y, qkv, out, lse = ops.attention_block_forward(d["x"], d["w_attn"], d["b_attn"], d["w_proj"], d["b_proj"], NH)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    g_qkv, g_out, g_y = ops.download_f64(qkv), ops.download_f64(out), ops.download_f64(y)
    x64 = bi.x.astype(np.float64).reshape(B * T, C)
    # c_attn on x
    r_qkv = oracle.linear(x64, bi.w_attn, bi.b_attn).reshape(B, T, 3 * C)
    tol = _lin_tol(x64, bi.w_attn.astype(np.float64), r_qkv.reshape(B * T, 3 * C)).reshape(B, T, 3 * C)
    assert np.all(np.abs(g_qkv - r_qkv) <= tol)
    # attention on the GPU's qkv
    r_out, r_lse = oracle.forward(g_qkv, B, T, C, NH, True)
    assert np.max(np.abs(g_out - r_out)) <= 2e-2 * np.max(np.abs(r_out))
    assert np.max(np.abs(ops.download_f64(lse) - r_lse)) <= 1e-3
    # c_proj on the GPU's out
    o64 = g_out.reshape(B * T, C)
    r_y = oracle.linear(o64, bi.w_proj, bi.b_proj)
    assert np.all(np.abs(g_y.reshape(B * T, C) - r_y) <= _lin_tol(o64, bi.w_proj.astype(np.float64), r_y))
    # end to end against the exact block
    e_y = oracle.block_forward(bi.x, bi.w_attn, bi.b_attn, bi.w_proj, bi.b_proj, NH, True)[0]
    assert np.max(np.abs(g_y - e_y)) <= 2e-2 * np.max(np.abs(e_y))
