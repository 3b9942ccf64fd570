"""Failure detection without a GPU fault.

Every wait in the library's kernels is bounded: when it runs out it records
ATTN_ERR_TIMEOUT in the device error word and the kernel returns. The
self-test entry point runs that mechanism on a barrier nothing completes (a
limit of a few milliseconds); the host must see the timeout through
attn_last_device_error, the word must be cleared by that read, and the
context must stay usable for real work afterwards.

The real forward and backward kernels are made to give up too: a copy of the
library is built with a wait limit of zero (ATTN_WAIT_NS=0), a clock read at
every poll and non-blocking polls (mbarrier.test_wait; the product build's
try_wait may suspend until the phase completes), so their first wait that is
not over within about a microsecond runs out, in whichever role it happens.
In a child process that copy runs a forward and a backward with several work
items per CTA, an fp32-input forward and a non-causal FP8 forward; each must
return, the host must read ATTN_ERR_TIMEOUT once per call, and no CUDA error
may follow. The parent then runs the normal library
on the same GPU and checks its results against the oracle.
"""
import json
import pathlib
import subprocess
import sys

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


_CHILD = r"""
import ctypes, json, sys
import torch
lib = ctypes.CDLL(sys.argv[1])
vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
lib.attn_fwd.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
lib.attn_fwd.restype = i
lib.attn_bwd_workspace_size.argtypes = [i] * 6
lib.attn_bwd_workspace_size.restype = sz
lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]
lib.attn_bwd.restype = i
lib.attn_last_device_error.argtypes = [vp]
lib.attn_last_device_error.restype = i
B, T, C, NH = 8, 1024, 768, 12            # 384 forward and 768 backward work items
g = torch.Generator(device="cuda").manual_seed(0)
qkv = (torch.randn(B, T, 3 * C, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
dout = (torch.randn(B, T, C, device="cuda", generator=g) * 0.01).to(torch.bfloat16)
out = torch.empty(B, T, C, dtype=torch.bfloat16, device="cuda")
lse = torch.empty(B, NH, T, dtype=torch.float32, device="cuda")
dqkv = torch.empty_like(qkv)
n = lib.attn_bwd_workspace_size(B, T, C, NH, 1, 1)
ws = torch.empty(n, dtype=torch.uint8, device="cuda")
s = torch.cuda.current_stream().cuda_stream
r = {}
r["fwd_status"] = lib.attn_fwd(qkv.data_ptr(), out.data_ptr(), lse.data_ptr(), B, T, C, NH, 1, 1, s)
torch.cuda.synchronize()
r["fwd_error"] = lib.attn_last_device_error(s)
r["bwd_status"] = lib.attn_bwd(dout.data_ptr(), qkv.data_ptr(), out.data_ptr(), lse.data_ptr(), dqkv.data_ptr(),
                               B, T, C, NH, 1, 1, ws.data_ptr(), n, s)
torch.cuda.synchronize()
r["bwd_error"] = lib.attn_last_device_error(s)
r["after"] = lib.attn_last_device_error(s)
# the fp32-input forward and the non-causal FP8 forward (their softmax
# warpgroups take turns through named barriers, which must pair up however
# the waits give up)
q32 = torch.randn(B, T, 3 * C, device="cuda", generator=g) * 0.5
o32 = torch.empty(B, T, C, device="cuda")
r["f32_status"] = lib.attn_fwd(q32.data_ptr(), o32.data_ptr(), lse.data_ptr(), B, T, C, NH, 1, 0, s)
torch.cuda.synchronize()
r["f32_error"] = lib.attn_last_device_error(s)
lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
lib.attn_fwd_fp8.restype = i
nT = (T + 127) // 128
codes = torch.randn(B, T, 3 * C, device="cuda", generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
desc = (torch.rand(3, B, NH, nT, device="cuda", generator=g) + 0.5) * 0.25
r["fp8_status"] = lib.attn_fwd_fp8(codes.data_ptr(), desc.data_ptr(), out.data_ptr(), lse.data_ptr(), B, T, C, NH, 0, s)
torch.cuda.synchronize()
r["fp8_error"] = lib.attn_last_device_error(s)
print(json.dumps(r))
"""


@pytest.mark.gpu
def test_real_kernels_wind_down_when_their_waits_run_out(env):
    torch, api, ops = env
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_head_attention_fwd_gb300 import build
    root = pathlib.Path(__file__).resolve().parents[1]
    lib = build.build(extra_flags=["-DATTN_WAIT_NS=0ull", "-DATTN_WAIT_POLLS_PER_CHECK=1",
                                                  "-DATTN_WAIT_NONBLOCKING=1"], lib=root / "_build" / "zero_wait" / "libattn_zero_wait.so",
                      build_dir=root / "_build" / "zero_wait")
    r = subprocess.run([sys.executable, "-c", _CHILD, str(lib)], capture_output=True, text=True, timeout=180)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["fwd_status"] == api.ATTN_OK and res["bwd_status"] == api.ATTN_OK     # launched
    assert res["fwd_error"] == api.ATTN_ERR_TIMEOUT                                  # gave up, reported
    assert res["bwd_error"] == api.ATTN_ERR_TIMEOUT
    assert res["after"] == api.ATTN_OK                                               # the read cleared it
    assert res["f32_status"] == api.ATTN_OK and res["f32_error"] == api.ATTN_ERR_TIMEOUT
    assert res["fp8_status"] == api.ATTN_OK and res["fp8_error"] == api.ATTN_ERR_TIMEOUT
    # the GPU still runs the normal library's kernels correctly
    assert api.attn_last_device_error() == api.ATTN_OK
    B, T, C, NH = 2, 300, 128, 2
    host = inputs.make_inputs(B, T, C, NH, "bf16", 0.5, 1e-2, 13, 14)
    qkv = ops.upload(host.qkv_dev, "bf16")
    dout = ops.upload(host.dout_dev, "bf16")
    out, lse = ops.attention_forward(qkv, NH, True)
    dqkv = ops.attention_backward(dout, qkv, out, lse, NH, True)
    torch.cuda.synchronize()
    assert api.attn_last_device_error() == api.ATTN_OK
    ref_out, _ = oracle.forward(host.qkv, B, T, C, NH, True)
    ref_d = oracle.backward(host.dout, host.qkv, B, T, C, NH, True)
    assert np.max(np.abs(ops.download_f64(out) - ref_out)) <= 2e-2 * np.max(np.abs(ref_out))
    assert np.max(np.abs(ops.download_f64(dqkv) - ref_d)) <= 2e-2 * np.max(np.abs(ref_d))
