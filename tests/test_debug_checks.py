"""The debug build (compiled with -DATTN_CHECK): every kernel tests the index of
each plain global load and store against its buffer's extent and records
ATTN_ERR_BOUNDS instead of touching memory outside it.

The GPU test builds that library apart from the normal one, runs every entry
point of both builds on the same small ragged shapes in a child process, and
checks that the checked build reports no out-of-range index and computes what
the normal build computes. The CPU test checks that the checks compile away
in a normal build and that the status code is declared and named.
"""
import json
import pathlib
import re
import subprocess
import sys

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]


def test_bounds_status_is_declared():
    from causal_head_attention_fwd_gb300 import api
    header = (ROOT / "include" / "attn.h").read_text()
    assert re.search(r"ATTN_ERR_BOUNDS\s*=\s*7", header)
    assert api.ATTN_ERR_BOUNDS == 7
    assert api.attn_status_string(api.ATTN_ERR_BOUNDS).startswith("ATTN_ERR_BOUNDS")


def test_checks_compile_away_in_a_normal_build():
    ptx = (ROOT / "causal_head_attention_fwd_gb300" / "csrc" / "ptx.cuh").read_text()
    # the normal build's macro is the constant true, so no test and no branch remain
    normal = re.search(r"#else\s*\n#define ATTN_IN_RANGE\(cond, err\) \(true\)", ptx)
    assert normal, "ATTN_IN_RANGE must expand to (true) without ATTN_CHECK"


_CHILD = r"""
import ctypes, json, sys
import torch
from causal_head_attention_fwd_gb300 import api
norm = api.configure(ctypes.CDLL(api.library_path()))
chk = api.configure(ctypes.CDLL(sys.argv[1]))
dev = torch.device("cuda", 0)
s = torch.cuda.current_stream().cuda_stream
res = {"status": [], "device_error": [], "maxdiff": {}}

def gen(shape, scale, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(*shape, device=dev, generator=g) * scale).to(dtype)

def run(lib, fn):
    outs = fn(lib)
    torch.cuda.synchronize()
    res["device_error"].append(lib.attn_last_device_error(s))
    return outs

def both(name, fn, exact=True):
    a = run(norm, fn)
    b = run(chk, fn)
    d = 0.0
    for x, y in zip(a, b):
        x, y = x.float(), y.float()
        d = max(d, float((x - y).abs().max()) / max(float(x.abs().max()), 1e-30))
    res["maxdiff"][name] = d

def att_case(B, T, C, NH, causal, dt):
    tdt = torch.bfloat16 if dt == 1 else torch.float32
    qkv = gen((B, T, 3 * C), 0.5, 1, tdt)
    dout = gen((B, T, C), 0.01, 2, tdt)
    def fn(lib):
        out = torch.empty(B, T, C, dtype=tdt, device=dev); lse = torch.empty(B, NH, T, device=dev)
        dqkv = torch.empty_like(qkv)
        n = lib.attn_bwd_workspace_size(B, T, C, NH, causal, dt)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        res["status"].append(lib.attn_fwd(qkv.data_ptr(), out.data_ptr(), lse.data_ptr(), B, T, C, NH, causal, dt, s))
        res["status"].append(lib.attn_bwd(dout.data_ptr(), qkv.data_ptr(), out.data_ptr(), lse.data_ptr(), dqkv.data_ptr(),
                                          B, T, C, NH, causal, dt, ws.data_ptr(), n, s))
        d2 = torch.empty_like(qkv)
        res["status"].append(lib.attn_bwd_noalloc(dout.data_ptr(), qkv.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                                  d2.data_ptr(), B, T, C, NH, causal, dt, s))
        pre = torch.empty(B, NH, T, T, device=dev); att = torch.empty(B, NH, T, T, device=dev)
        res["status"].append(lib.attn_fwd_att(qkv.data_ptr(), lse.data_ptr(), pre.data_ptr(), att.data_ptr(),
                                              B, T, C, NH, causal, dt, s))
        return out, lse, dqkv, d2, pre, att
    both(f"attention B{B} T{T} C{C} NH{NH} causal{causal} dtype{dt}", fn)

att_case(2, 300, 128, 2, 1, 1)
att_case(1, 200, 256, 8, 0, 1)
att_case(2, 200, 128, 2, 1, 0)

# decode
B, L, C, NH, Tq = 2, 300, 128, 2, 3
qkv = gen((B, L, 3 * C), 0.5, 3)
def dec(lib):
    out = torch.empty(B, Tq, C, dtype=torch.bfloat16, device=dev); lse = torch.empty(B, NH, Tq, device=dev)
    n = lib.attn_decode_workspace_size(B, L, C, NH, Tq, 1)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    res["status"].append(lib.attn_decode(qkv.data_ptr(), out.data_ptr(), lse.data_ptr(), B, L, C, NH, Tq, 1,
                                         ws.data_ptr(), n, s))
    return out, lse
both("decode", dec)
Tq = 1
both("decode one token", dec)

# FP8 forward and backward
B, T, C, NH = 2, 300, 128, 2
nT = (T + 127) // 128
codes = gen((B, T, 3 * C), 1.0, 4, torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)
desc = (torch.rand(3, B, NH, nT, device=dev, generator=torch.Generator(device="cuda").manual_seed(5)) + 0.5) * 0.25
dout = gen((B, T, C), 0.01, 6)
def fp8(lib):
    out = torch.empty(B, T, C, dtype=torch.bfloat16, device=dev); lse = torch.empty(B, NH, T, device=dev)
    res["status"].append(lib.attn_fwd_fp8(codes.data_ptr(), desc.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                          B, T, C, NH, 1, s))
    out_nc = torch.empty_like(out); lse_nc = torch.empty_like(lse)          # no mask: turns at the exponentials
    res["status"].append(lib.attn_fwd_fp8(codes.data_ptr(), desc.data_ptr(), out_nc.data_ptr(), lse_nc.data_ptr(),
                                          B, T, C, NH, 0, s))
    dqkv = torch.empty(B, T, 3 * C, dtype=torch.bfloat16, device=dev)
    n = lib.attn_bwd_fp8_workspace_size(B, T, C, NH, 1)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    res["status"].append(lib.attn_bwd_fp8(dout.data_ptr(), codes.data_ptr(), desc.data_ptr(), out.data_ptr(),
                                          lse.data_ptr(), dqkv.data_ptr(), B, T, C, NH, 1, ws.data_ptr(), n, s))
    return out, lse, dqkv, out_nc, lse_nc
both("fp8", fp8)

# linear
M, N, K = 300, 520, 200
x = gen((M, K), 1.0, 7); w = gen((N, K), 0.05, 8); bias = gen((N,), 0.1, 9)
def lin(lib):
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    res["status"].append(lib.attn_linear_fwd(x.data_ptr(), w.data_ptr(), bias.data_ptr(), y.data_ptr(), M, N, K, s))
    return (y,)
both("linear", lin)
print(json.dumps(res))
"""


@pytest.mark.gpu
def test_checked_build_reports_no_out_of_range_index():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_head_attention_fwd_gb300 import api, build
    build.build()
    lib = build.build(extra_flags=["-DATTN_CHECK"], lib=ROOT / "_build" / "check" / "libattn_check.so",
                      build_dir=ROOT / "_build" / "check")
    r = subprocess.run([sys.executable, "-c", _CHILD, str(lib)], capture_output=True, text=True, timeout=300,
                       cwd=str(ROOT))
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert all(st == api.ATTN_OK for st in res["status"]), res["status"]
    assert all(e == api.ATTN_OK for e in res["device_error"]), res["device_error"]
    # the checks change no arithmetic; only the order of the fp32 dq reductions
    # (atomic adds) may differ between runs
    for name, d in res["maxdiff"].items():
        assert d <= 1e-5, (name, d)
