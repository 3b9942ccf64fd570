"""Python binding of libattn.so (include/attn.h): argument marshalling only.

Every function here has the name and argument order of its C counterpart.
Tensor arguments may be torch tensors (their data_ptr() is passed) or plain
integer device addresses; `stream` may be a torch.cuda.Stream, a raw
cudaStream_t integer, or None for torch's current stream. All computation
happens in the CUDA kernels behind the C ABI; there is no fallback path: if
the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import pathlib

_LIB_PATH = pathlib.Path(__file__).resolve().parent / "libattn.so"

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_WORKSPACE = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_TIMEOUT = 6
ATTN_ERR_BOUNDS = 7

ATTN_F32 = 0
ATTN_BF16 = 1

EXPORTED = ("attn_fwd", "attn_bwd_workspace_size", "attn_bwd", "attn_status_string",
            "attn_last_device_error", "attn_profile_enable", "attn_profile_reset",
            "attn_profile_read", "attn_bwd_noalloc", "attn_selftest_wait_timeout", "attn_fwd_att",
            "attn_decode_workspace_size", "attn_decode", "attn_fwd_fp8", "attn_linear_fwd",
            "attn_bwd_fp8_workspace_size", "attn_bwd_fp8", "attn_fwd_schedule")

# size of the fixed scratch array attn_bwd_noalloc uses (ATTN_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 32 << 20

# kernel ids of attn_profile_read
K_FWD, K_BWD_PRE, K_BWD_MAIN, K_BWD_DQ, K_LINEAR = 0, 1, 2, 3, 4
KERNEL_NAMES = {K_FWD: "attn_fwd_kernel", K_BWD_PRE: "attn_bwd_pre",
                K_BWD_MAIN: "attn_bwd_kernel", K_BWD_DQ: "attn_bwd_dq_out"}
# The same four profiling slots hold the fp32 path's kernels.
KERNEL_NAMES_F32 = {K_FWD: "attn_fwd_f32_kernel", K_BWD_PRE: "attn_bwd_pre_f32",
                    K_BWD_MAIN: "attn_bwd_dkdv_f32", K_BWD_DQ: "attn_bwd_dq_f32"}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


def _load() -> ctypes.CDLL:
    if not _LIB_PATH.exists():
        raise ImportError(f"libattn.so not built at {_LIB_PATH}; run "
                          "`python -m causal_head_attention_fwd_gb300.build` (needs nvcc)")
    return configure(ctypes.CDLL(str(_LIB_PATH)))


def configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the argument and result types of every entry point on a loaded
    build of the library (this package's, or another build of the same
    sources, e.g. with different compile flags)."""
    vp, i, f_p, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, f_p, i, i, i, i, i, i, vp]
    lib.attn_fwd.restype = i
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.attn_bwd_workspace_size.restype = sz
    lib.attn_bwd.argtypes = [vp, vp, vp, f_p, vp, i, i, i, i, i, i, vp, sz, vp]
    lib.attn_bwd.restype = i
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_last_device_error.argtypes = [vp]
    lib.attn_last_device_error.restype = i
    lib.attn_profile_enable.argtypes = [i]
    lib.attn_profile_enable.restype = i
    lib.attn_profile_reset.argtypes = []
    lib.attn_profile_reset.restype = i
    lib.attn_profile_read.argtypes = [i, ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_longlong)]
    lib.attn_profile_read.restype = i
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, f_p, vp, i, i, i, i, i, i, vp]
    lib.attn_bwd_noalloc.restype = i
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
    lib.attn_selftest_wait_timeout.restype = i
    lib.attn_fwd_att.argtypes = [vp, f_p, f_p, f_p, i, i, i, i, i, i, vp]
    lib.attn_fwd_att.restype = i
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_decode.argtypes = [vp, vp, f_p, i, i, i, i, i, i, vp, sz, vp]
    lib.attn_decode.restype = i
    lib.attn_fwd_fp8.argtypes = [vp, f_p, vp, f_p, i, i, i, i, i, vp]
    lib.attn_fwd_fp8.restype = i
    lib.attn_linear_fwd.argtypes = [vp, vp, vp, vp, i, i, i, vp]
    lib.attn_linear_fwd.restype = i
    lib.attn_bwd_fp8_workspace_size.argtypes = [i, i, i, i, i]
    lib.attn_bwd_fp8_workspace_size.restype = sz
    lib.attn_bwd_fp8.argtypes = [vp, vp, f_p, vp, f_p, vp, i, i, i, i, i, vp, sz, vp]
    lib.attn_bwd_fp8.restype = i
    lib.attn_fwd_schedule.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int), i]
    lib.attn_fwd_schedule.restype = i
    return lib


_lib = _load()


def library_path() -> str:
    return str(_LIB_PATH)


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _dtype(d) -> int:
    if isinstance(d, int):
        return d
    name = str(d)
    if name in ("bf16", "torch.bfloat16"):
        return ATTN_BF16
    if name in ("f32", "torch.float32"):
        return ATTN_F32
    raise ValueError(f"unsupported dtype {d!r}")


def attn_status_string(status: int) -> str:
    return _lib.attn_status_string(int(status)).decode()


def attn_fwd(qkv, out, lse, B, T, C, NH, causal, dtype, stream=None, check=True) -> int:
    st = _lib.attn_fwd(_ptr(qkv), _ptr(out), _ptr(lse), B, T, C, NH, int(causal), _dtype(dtype),
                       _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_fwd")
    return st


def attn_bwd_workspace_size(B, T, C, NH, causal, dtype) -> int:
    return int(_lib.attn_bwd_workspace_size(B, T, C, NH, int(causal), _dtype(dtype)))


def attn_bwd(dout, qkv, out, lse, dqkv, B, T, C, NH, causal, dtype, workspace, workspace_bytes,
             stream=None, check=True) -> int:
    st = _lib.attn_bwd(_ptr(dout), _ptr(qkv), _ptr(out), _ptr(lse), _ptr(dqkv), B, T, C, NH,
                       int(causal), _dtype(dtype), _ptr(workspace), int(workspace_bytes),
                       _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return st


def attn_last_device_error(stream=None) -> int:
    return int(_lib.attn_last_device_error(_stream(stream)))


def attn_fwd_att(qkv, lse, preatt, att, B, T, C, NH, causal, dtype, stream=None, check=True) -> int:
    st = _lib.attn_fwd_att(_ptr(qkv), _ptr(lse), _ptr(preatt), _ptr(att), B, T, C, NH, int(causal),
                           _dtype(dtype), _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_fwd_att")
    return st


def attn_decode_workspace_size(B, L, C, NH, Tq, dtype) -> int:
    return int(_lib.attn_decode_workspace_size(B, L, C, NH, Tq, _dtype(dtype)))


def attn_decode(qkv, out, lse, B, L, C, NH, Tq, dtype, workspace, workspace_bytes, stream=None,
                check=True) -> int:
    st = _lib.attn_decode(_ptr(qkv), _ptr(out), _ptr(lse), B, L, C, NH, Tq, _dtype(dtype), _ptr(workspace),
                          int(workspace_bytes), _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_decode")
    return st


def attn_fwd_fp8(qkv, descale, out, lse, B, T, C, NH, causal, stream=None, check=True) -> int:
    """e4m3 qkv codes with per-tile descales (device, (3, B, NH, ceil(T/128)) fp32)
    -> bf16 out, fp32 lse."""
    st = _lib.attn_fwd_fp8(_ptr(qkv), _ptr(descale), _ptr(out), _ptr(lse), B, T, C, NH, int(causal),
                           _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8")
    return st


def attn_bwd_fp8_workspace_size(B, T, C, NH, causal) -> int:
    return int(_lib.attn_bwd_fp8_workspace_size(B, T, C, NH, int(causal)))


def attn_bwd_fp8(dout, qkv, descale, out, lse, dqkv, B, T, C, NH, causal, workspace, workspace_bytes,
                 stream=None, check=True) -> int:
    st = _lib.attn_bwd_fp8(_ptr(dout), _ptr(qkv), _ptr(descale), _ptr(out), _ptr(lse), _ptr(dqkv), B, T, C, NH,
                           int(causal), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_bwd_fp8")
    return st


def attn_linear_fwd(inp, weight, bias, out, M, N, K, stream=None, check=True) -> int:
    """out (M, N) = inp (M, K) . weight (N, K)^T + bias (N), bf16; bias may be None."""
    st = _lib.attn_linear_fwd(_ptr(inp), _ptr(weight), _ptr(bias), _ptr(out), M, N, K, _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_linear_fwd")
    return st


def attn_fwd_schedule(B, T, C, NH, n_cta):
    """The forward's causal deal of work items over min(items, n_cta) CTAs:
    (off, items) int lists, CTA c running items[off[c]:off[c+1]]; None when the
    forward uses its snake order for this shape."""
    n_items = B * NH * ((T + 255) // 256)
    grid = min(n_items, n_cta)
    off = (ctypes.c_int * (grid + 1))()
    items = (ctypes.c_int * max(n_items, 1))()
    n = _lib.attn_fwd_schedule(B, T, C, NH, n_cta, off, items, n_items)
    if n < 0:
        raise AttnError(ATTN_ERR_INVALID_ARG, "attn_fwd_schedule")
    if n == 0:
        return None
    return list(off), list(items)[:n]


def attn_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return int(_lib.attn_selftest_wait_timeout(int(limit_us), _stream(stream)))


def attn_profile_enable(enable: bool) -> None:
    st = _lib.attn_profile_enable(int(bool(enable)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_profile_enable")


def attn_profile_reset() -> None:
    st = _lib.attn_profile_reset()
    if st != ATTN_OK:
        raise AttnError(st, "attn_profile_reset")


def attn_profile_read(kernel_id: int):
    """(total device ms, launch count) of one kernel since the last reset."""
    ms, n = ctypes.c_double(), ctypes.c_longlong()
    st = _lib.attn_profile_read(int(kernel_id), ctypes.byref(ms), ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_profile_read")
    return ms.value, n.value


def attn_bwd_noalloc(dout, qkv, out, lse, dqkv, B, T, C, NH, causal, dtype, stream=None,
                     check=True) -> int:
    """attn_bwd without a workspace argument: for callers that cannot allocate
    device memory; the library's fixed scratch array is used instead."""
    st = _lib.attn_bwd_noalloc(_ptr(dout), _ptr(qkv), _ptr(out), _ptr(lse), _ptr(dqkv), B, T, C, NH,
                               int(causal), _dtype(dtype), _stream(stream))
    if check and st != ATTN_OK:
        raise AttnError(st, "attn_bwd_noalloc")
    return st
