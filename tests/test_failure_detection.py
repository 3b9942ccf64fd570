"""Failure detection without a GPU fault.

Every wait in the library's kernels is bounded: when it runs out it records
ATTN_ERR_TIMEOUT in the device error word and the kernel returns. The
self-test entry point runs that mechanism on a barrier nothing completes (a
limit of a few milliseconds); the host must see the timeout through
attn_last_device_error, the word must be cleared by that read, and the
context must stay usable for real work afterwards.
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


def test_selftest_rejects_bad_limits(env):
    _, api, _ = env
    assert api.attn_selftest_wait_timeout(0, 0) == api.ATTN_ERR_INVALID_ARG
    assert api.attn_selftest_wait_timeout(10_000_001, 0) == api.ATTN_ERR_INVALID_ARG


@pytest.mark.gpu
def test_expired_wait_is_reported_and_the_context_survives(env):
    torch, api, ops = env
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert api.attn_last_device_error() == api.ATTN_OK            # clean start
    assert api.attn_selftest_wait_timeout(5000) == api.ATTN_OK    # 5 ms limit
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_ERR_TIMEOUT
    assert api.attn_last_device_error() == api.ATTN_OK            # cleared by the read
    # the context still runs the real kernels correctly
    B, T, C, NH = 1, 200, 128, 2
    host = inputs.make_inputs(B, T, C, NH, "bf16", 0.5, 1e-2, 11, 12)
    qkv = ops.upload(host.qkv_dev, "bf16")
    dout = ops.upload(host.dout_dev, "bf16")
    out, lse = ops.attention_forward(qkv, NH, True)
    dqkv = ops.attention_backward(dout, qkv, out, lse, NH, True)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    ref_out, _ = oracle.forward(host.qkv, B, T, C, NH, True)
    ref_d = oracle.backward(host.dout, host.qkv, B, T, C, NH, True)
    got_out, got_d = ops.download_f64(out), ops.download_f64(dqkv)
    assert np.max(np.abs(got_out - ref_out)) <= 2e-2 * np.max(np.abs(ref_out))
    assert np.max(np.abs(got_d - ref_d)) <= 2e-2 * np.max(np.abs(ref_d))
