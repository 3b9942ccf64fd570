"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a plug-in whose host framework owns all device allocations, or a
loop that must not call cudaMalloc after start-up) get the same result as
attn_bwd without passing a workspace: the library uses a fixed scratch array
of its own instead. This test calls the new entry point through the C ABI
twice in a row and compares each result with attn_bwd's, within the tolerance
the parity tests use for dqkv (max|diff| <= tol * max|reference|, tol = 2e-2
for bf16 and 1e-2 for fp32 inputs). Both dtypes are covered: the bf16 backward
keeps D and an fp32 dq accumulator in the scratch, the fp32 backward only D.
This file is named so that pytest collects it after every other test file.
"""
import numpy as np
import pytest

from causal_head_attention_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-2}


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
    a = a.float()
    ref = ref.float()
    return float((a - ref).abs().max().item() / max(ref.abs().max().item(), 1e-30))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,C,NH,causal", [(2, 300, 128, 2, 1), (1, 257, 128, 4, 0)])
def test_noalloc_matches_attn_bwd_on_two_calls(env, B, T, C, NH, causal, dtype):
    torch, api, ops = env
    adt = api.ATTN_BF16 if dtype == "bf16" else api.ATTN_F32
    host = inputs.make_inputs(B, T, C, NH, dtype, 0.5, 1e-2, 900 + T, 901 + T)
    qkv = ops.upload(host.qkv_dev, dtype)
    dout = ops.upload(host.dout_dev, dtype)
    out, lse = ops.attention_forward(qkv, NH, bool(causal))
    # existing entry point, with a caller-provided workspace
    ref = ops.attention_backward(dout, qkv, out, lse, NH, bool(causal))
    assert api.attn_bwd_workspace_size(B, T, C, NH, causal, adt) <= api.NOALLOC_SCRATCH_BYTES
    for call in range(2):
        dqkv = torch.full_like(qkv, float("nan"))
        api.attn_bwd_noalloc(dout, qkv, out, lse, dqkv, B, T, C, NH, causal, adt)
        torch.cuda.synchronize()
        assert api.attn_last_device_error() == api.ATTN_OK
        assert not torch.isnan(dqkv.float()).any(), f"call {call}: dqkv not fully written"
        for sl in (slice(0, C), slice(C, 2 * C), slice(2 * C, 3 * C)):
            e = _rel(dqkv[:, :, sl], ref[:, :, sl])
            assert e <= TOL[dtype], f"call {call}: rel err {e:.3e}"


def test_noalloc_rejects_problems_larger_than_its_scratch(env):
    torch, api, ops = env
    B, T, C, NH = 16, 1024, 768, 12          # needs ~51 MB > the fixed scratch
    assert api.attn_bwd_workspace_size(B, T, C, NH, 1, api.ATTN_BF16) > api.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")   # never touched: rejected first
    st = api.attn_bwd_noalloc(t, t, t, t, t, B, T, C, NH, 1, api.ATTN_BF16, check=False)
    assert st == api.ATTN_ERR_WORKSPACE
