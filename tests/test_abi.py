"""Host-side tests of the C ABI (no GPU needed).

The library must load and export every function include/attn.h declares, and
reject bad arguments on the host before anything is launched. These calls use
fake, never-dereferenced device addresses and stop at the argument checks.
"""
import ctypes
import pathlib
import re

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def api():
    from causal_head_attention_fwd_gb300 import build
    try:
        build.build()
    except RuntimeError as e:  # no nvcc in this environment
        pytest.skip(str(e))
    from causal_head_attention_fwd_gb300 import api as a
    return a


def _declared():
    text = (ROOT / "include" / "attn.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_status_string",
              "attn_last_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(api):
    lib = ctypes.CDLL(api.library_path())
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in include/attn.h but not exported"
    assert set(api.EXPORTED) <= set(_declared())


def _header_constants():
    """Enumerators and #define values of include/attn.h, by name."""
    text = (ROOT / "include" / "attn.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    vals = {}
    for body in re.findall(r"typedef\s+enum\s*\{(.*?)\}", text, flags=re.S):
        for name, v in re.findall(r"\b(ATTN_[A-Z0-9_]+)\s*=\s*(\d+)", body):
            vals[name] = int(v)
    for name, expr in re.findall(r"#define[ \t]+(ATTN_[A-Z0-9_]+)[ \t]+([^\n]+)", text):
        m = re.fullmatch(r"\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", expr.strip())
        vals[name] = int(m.group(1)) << int(m.group(2)) if m else int(expr.strip())
    return vals


def test_python_constants_match_the_header(api):
    """The binding mirrors the header's constants by hand; they must agree."""
    h = _header_constants()
    for name in ("ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_MISALIGNED",
                 "ATTN_ERR_WORKSPACE", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "ATTN_ERR_BOUNDS", "ATTN_F32",
                 "ATTN_BF16"):
        assert getattr(api, name) == h[name], name
    assert api.NOALLOC_SCRATCH_BYTES == h["ATTN_NOALLOC_SCRATCH_BYTES"]
    ids = {"K_FWD": "ATTN_PROFILE_FWD", "K_BWD_PRE": "ATTN_PROFILE_BWD_PRE", "K_BWD_MAIN": "ATTN_PROFILE_BWD_MAIN",
           "K_BWD_DQ": "ATTN_PROFILE_BWD_DQ", "K_LINEAR": "ATTN_PROFILE_LINEAR"}
    for py, c in ids.items():
        assert getattr(api, py) == h[c], py
    assert len(ids) == h["ATTN_PROFILE_NUM_KERNELS"]
    # the binding covers every entry point the header declares
    assert set(api.EXPORTED) == set(_declared())


def test_status_strings(api):
    for s in range(8):
        assert api.attn_status_string(s).startswith("ATTN_")
    assert "UNKNOWN" in api.attn_status_string(99)


A = 1 << 32          # fake, 16-byte aligned, never dereferenced addresses
S = 1 << 30          # spacing so fake buffers never overlap


def _fwd(api, qkv=A, out=A + S, lse=A + 2 * S, B=2, T=64, C=128, NH=2, causal=1, dt=1):
    return api.attn_fwd(qkv, out, lse, B, T, C, NH, causal, dt, 0, check=False)


def _bwd(api, dout=A, qkv=A + S, out=A + 2 * S, lse=A + 3 * S, dqkv=A + 4 * S, B=2, T=64, C=128,
         NH=2, causal=1, dt=1, ws=A + 5 * S, wsb=None):
    if wsb is None:
        wsb = api.attn_bwd_workspace_size(B, T, C, NH, causal, dt)
    return api.attn_bwd(dout, qkv, out, lse, dqkv, B, T, C, NH, causal, dt, ws, wsb, 0, check=False)


@pytest.mark.parametrize("kw,expect", [
    (dict(B=0), "INVALID_ARG"), (dict(T=0), "INVALID_ARG"), (dict(NH=0), "INVALID_ARG"),
    (dict(C=0), "INVALID_ARG"), (dict(C=130, NH=4), "INVALID_ARG"), (dict(causal=2), "INVALID_ARG"),
    (dict(dt=7), "INVALID_ARG"), (dict(C=384, NH=3), "UNSUPPORTED"), (dict(C=16, NH=1), "UNSUPPORTED"),
    (dict(qkv=0), "INVALID_ARG"), (dict(out=0), "INVALID_ARG"), (dict(lse=0), "INVALID_ARG"),
    (dict(qkv=A + 8), "MISALIGNED"), (dict(out=A + S + 2), "MISALIGNED"),
    (dict(lse=A + 2 * S + 4), "MISALIGNED"), (dict(out=A + 16), "INVALID_ARG"),
])
def test_fwd_rejects_bad_arguments(api, kw, expect):
    st = _fwd(api, **kw)
    assert st == getattr(api, "ATTN_ERR_" + expect), api.attn_status_string(st)


@pytest.mark.parametrize("kw,expect", [
    (dict(B=-1), "INVALID_ARG"), (dict(C=96, NH=2), "UNSUPPORTED"), (dict(dout=0), "INVALID_ARG"),
    (dict(dqkv=0), "INVALID_ARG"), (dict(dqkv=A + 4 * S + 8), "MISALIGNED"),
    (dict(ws=0), "WORKSPACE"), (dict(wsb=1024), "WORKSPACE"), (dict(ws=A + 5 * S + 128), "MISALIGNED"),
    (dict(dqkv=A + S + 4096), "INVALID_ARG"), (dict(dqkv=A), "INVALID_ARG"),
    # the workspace is written, so it may not overlap any input or dqkv
    (dict(ws=A + 4 * S), "INVALID_ARG"), (dict(ws=A + 256), "INVALID_ARG"), (dict(ws=A + S), "INVALID_ARG"),
    (dict(ws=A + 2 * S + 256), "INVALID_ARG"), (dict(ws=A + 3 * S), "INVALID_ARG"),
])
def test_bwd_rejects_bad_arguments(api, kw, expect):
    st = _bwd(api, **kw)
    assert st == getattr(api, "ATTN_ERR_" + expect), api.attn_status_string(st)


def test_workspace_size(api):
    B, T, C, NH = 3, 100, 128, 2
    n = api.attn_bwd_workspace_size(B, T, C, NH, 1, 1)
    d = (B * NH * T * 4 + 255) // 256 * 256
    assert n == d + B * T * C * 4
    assert api.attn_bwd_workspace_size(B, T, 100, NH, 1, 1) == 0      # rejected shape


def test_binding_refuses_unknown_dtype(api):
    with pytest.raises(ValueError):
        api._dtype("fp8")


def test_product_path_has_no_oracle_or_fallback():
    """The package must not import the oracle, and must fail loudly without its library."""
    pkg = ROOT / "causal_head_attention_fwd_gb300"
    for f in pkg.rglob("*.py"):
        src = f.read_text()
        assert "import oracle" not in src and "from oracle" not in src, f
    assert "raise ImportError" in (pkg / "api.py").read_text()


def test_att_rejects_bad_arguments(api):
    ok = dict(qkv=A, lse=A + S, pre=A + 2 * S, att=A + 3 * S)
    def call(**kw):
        a = dict(ok, **kw)
        return api.attn_fwd_att(a["qkv"], a["lse"], a["pre"], a["att"], 2, 64, 128, 2, 1, 1, 0, check=False)
    assert call(qkv=0) == api.ATTN_ERR_INVALID_ARG
    assert call(pre=0, att=0) == api.ATTN_ERR_INVALID_ARG
    assert call(att=A + 3 * S + 4) == api.ATTN_ERR_MISALIGNED
    assert call(att=A + 2 * S) == api.ATTN_ERR_INVALID_ARG        # preatt and att overlap
    assert api.attn_fwd_att(A, A + S, A + 2 * S, None, 2, 64, 96, 2, 1, 1, 0, check=False) == \
        api.ATTN_ERR_UNSUPPORTED                                    # hs = 48
