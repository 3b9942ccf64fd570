"""Torch-facing convenience layer over the C ABI.

Allocates outputs and workspace with torch (device memory and streams only)
and calls attn_fwd / attn_bwd; the arithmetic runs in the library's kernels.
The C ABI takes raw pointers and trusts their sizes, so every tensor a caller
passes in is checked here first (shape, dtype, contiguity, one CUDA device):
a mismatch raises ValueError before anything is launched.
"""
from __future__ import annotations

import torch

from . import api

_DT = {torch.bfloat16: api.ATTN_BF16, torch.float32: api.ATTN_F32}


def upload(arr, dtype: str, device="cuda", pin: bool = False) -> torch.Tensor:
    """Host array in device representation (float32, or uint16 bf16 bits) -> torch tensor."""
    import numpy as np
    a = np.ascontiguousarray(arr)
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif dtype == "f32":
        t = torch.from_numpy(a.astype(np.float32, copy=False))
    else:
        raise ValueError(dtype)
    if pin:
        return t.pin_memory()
    return t.to(device)


def download_f64(t: torch.Tensor):
    """Device tensor -> float64 numpy array (exact widening of bf16/fp32)."""
    return t.detach().float().cpu().double().numpy()


def _shape(qkv: torch.Tensor, n_head: int, dtypes=tuple(_DT)):
    if not isinstance(qkv, torch.Tensor):
        raise TypeError("qkv must be a torch.Tensor")
    if qkv.dim() != 3 or qkv.shape[2] % 3 != 0:
        raise ValueError("qkv must have shape (B, T, 3C)")
    if qkv.dtype not in dtypes:
        raise ValueError(f"qkv has dtype {qkv.dtype}; supported: {', '.join(str(d) for d in dtypes)}")
    if not qkv.is_contiguous():
        raise ValueError("qkv must be contiguous")
    B, T, C3 = qkv.shape
    C = C3 // 3
    if int(n_head) < 1 or C % int(n_head) != 0:
        raise ValueError(f"n_head={n_head} does not divide C={C}")
    return B, T, C, int(n_head)


def _expect(t, name: str, shape, dtype):
    """A caller-provided tensor must match the shape and dtype the kernels assume."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_device(ref: torch.Tensor, **tensors):
    """Every tensor on the reference tensor's CUDA device (the kernels dereference them all)."""
    if ref.device.type != "cuda":
        raise ValueError(f"tensors must be on a CUDA device, got {ref.device}")
    for name, t in tensors.items():
        if t is not None and t.device != ref.device:
            raise ValueError(f"{name} is on {t.device}, expected {ref.device}")


def attention_forward(qkv: torch.Tensor, n_head: int, causal: bool = True, out=None, lse=None,
                      stream=None):
    """out (B, T, C) in qkv's dtype and lse (B, NH, T) fp32."""
    B, T, C, NH = _shape(qkv, n_head)
    _expect(out, "out", (B, T, C), qkv.dtype)
    _expect(lse, "lse", (B, NH, T), torch.float32)
    _on_device(qkv, out=out, lse=lse)
    if out is None:
        out = torch.empty((B, T, C), dtype=qkv.dtype, device=qkv.device)
    if lse is None:
        lse = torch.empty((B, NH, T), dtype=torch.float32, device=qkv.device)
    api.attn_fwd(qkv, out, lse, B, T, C, NH, int(causal), _DT[qkv.dtype], stream)
    return out, lse


def attention_forward_fp8(qkv_e4m3: torch.Tensor, descale: torch.Tensor, n_head: int, causal: bool = True,
                          out=None, lse=None, stream=None):
    """e4m3 qkv codes (uint8, (B, T, 3C)) and per-tile descales ((3, B, NH,
    ceil(T/128)) fp32 on the device: q, k, v of each head's 128-row tiles)
    -> out (B, T, C) bf16 and lse (B, NH, T) fp32."""
    B, T, C, NH = _shape(qkv_e4m3, n_head, dtypes=(torch.uint8,))
    _expect(descale, "descale", (3, B, NH, (T + 127) // 128), torch.float32)
    _expect(out, "out", (B, T, C), torch.bfloat16)
    _expect(lse, "lse", (B, NH, T), torch.float32)
    _on_device(qkv_e4m3, descale=descale, out=out, lse=lse)
    if out is None:
        out = torch.empty((B, T, C), dtype=torch.bfloat16, device=qkv_e4m3.device)
    if lse is None:
        lse = torch.empty((B, NH, T), dtype=torch.float32, device=qkv_e4m3.device)
    api.attn_fwd_fp8(qkv_e4m3, descale, out, lse, B, T, C, NH, int(causal), stream)
    return out, lse


def linear(inp: torch.Tensor, weight: torch.Tensor, bias=None, out=None, stream=None):
    """out (..., N) = inp (..., K) . weight (N, K)^T + bias (N), bf16 (fused bias epilogue)."""
    if not isinstance(inp, torch.Tensor) or inp.dim() < 1:
        raise ValueError("inp must be a tensor of shape (..., K)")
    if not isinstance(weight, torch.Tensor) or weight.dim() != 2:
        raise ValueError("weight must have shape (N, K)")
    K = inp.shape[-1]
    N = weight.shape[0]
    M = inp.numel() // K if K else 0
    _expect(inp, "inp", inp.shape, torch.bfloat16)
    _expect(weight, "weight", (N, K), torch.bfloat16)
    _expect(bias, "bias", (N,), torch.bfloat16)
    _expect(out, "out", (*inp.shape[:-1], N), torch.bfloat16)
    _on_device(inp, weight=weight, bias=bias, out=out)
    if out is None:
        out = torch.empty((*inp.shape[:-1], N), dtype=torch.bfloat16, device=inp.device)
    api.attn_linear_fwd(inp, weight, bias, out, M, N, K, stream)
    return out


def attention_block_forward(x: torch.Tensor, w_attn, b_attn, w_proj, b_proj, n_head: int, causal: bool = True,
                            stream=None):
    """GPT-2 attention block forward: qkv = c_attn(x) -> attention -> y = c_proj(out).
    Returns (y, qkv, out, lse); three launches on one stream."""
    qkv = linear(x, w_attn, b_attn, stream=stream)
    out, lse = attention_forward(qkv, n_head, causal, stream=stream)
    y = linear(out, w_proj, b_proj, stream=stream)
    return y, qkv, out, lse


def attention_matrices(qkv: torch.Tensor, lse: torch.Tensor, n_head: int, causal: bool = True,
                       preatt=True, att=True, stream=None):
    """llm.c drop-in mode: (preatt, att), each (B, NH, T, T) fp32 or None.
    preatt = q.k without the scale (full matrix); att = the softmax with the
    masked entries set to zero. lse is the forward's row statistic."""
    B, T, C, NH = _shape(qkv, n_head)
    _expect(lse, "lse", (B, NH, T), torch.float32)
    for name, m in (("preatt", preatt), ("att", att)):
        if not isinstance(m, bool):
            _expect(m, name, (B, NH, T, T), torch.float32)
    _on_device(qkv, lse=lse, preatt=None if isinstance(preatt, bool) else preatt,
               att=None if isinstance(att, bool) else att)
    pa = torch.empty((B, NH, T, T), dtype=torch.float32, device=qkv.device) if preatt is True else preatt
    at = torch.empty((B, NH, T, T), dtype=torch.float32, device=qkv.device) if att is True else att
    pa = pa if pa is not False else None
    at = at if at is not False else None
    api.attn_fwd_att(qkv, lse, pa, at, B, T, C, NH, int(causal), _DT[qkv.dtype], stream)
    return pa, at


def attention_decode(qkv: torch.Tensor, n_head: int, n_new: int, out=None, lse=None, workspace=None,
                     stream=None):
    """Decode forward: the last n_new rows of qkv (B, L, 3C) attend to every
    key up to their own position. Returns out (B, n_new, C), lse (B, NH, n_new)."""
    B, L, C, NH = _shape(qkv, n_head)
    _expect(out, "out", (B, n_new, C), qkv.dtype)
    _expect(lse, "lse", (B, NH, n_new), torch.float32)
    _on_device(qkv, out=out, lse=lse)
    if out is None:
        out = torch.empty((B, n_new, C), dtype=qkv.dtype, device=qkv.device)
    if lse is None:
        lse = torch.empty((B, NH, n_new), dtype=torch.float32, device=qkv.device)
    dt = _DT[qkv.dtype]
    nbytes = api.attn_decode_workspace_size(B, L, C, NH, n_new, dt)
    ws = (workspace or _decode_ws).get(nbytes, qkv.device)
    api.attn_decode(qkv, out, lse, B, L, C, NH, n_new, dt, ws, nbytes, stream)
    return out, lse


class Workspace:
    """Reusable device scratch buffer for attn_bwd (grown on demand).

    One buffer serves one stream at a time: calls that may run concurrently on
    different streams each need their own Workspace (the module-level default
    is shared by every call that passes none)."""

    def __init__(self):
        self.buf = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != torch.device(device):
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        return self.buf


_default_ws = Workspace()
_decode_ws = Workspace()


def attention_backward(dout, qkv, out, lse, n_head: int, causal: bool = True, dqkv=None,
                       workspace: Workspace | None = None, stream=None):
    """dqkv (B, T, 3C) in qkv's dtype, written with =."""
    B, T, C, NH = _shape(qkv, n_head)
    _expect(dout, "dout", (B, T, C), qkv.dtype)
    _expect(out, "out", (B, T, C), qkv.dtype)
    _expect(lse, "lse", (B, NH, T), torch.float32)
    _expect(dqkv, "dqkv", (B, T, 3 * C), qkv.dtype)
    if dout is None or out is None or lse is None:
        raise ValueError("dout, out and lse are required")
    _on_device(qkv, dout=dout, out=out, lse=lse, dqkv=dqkv)
    if dqkv is None:
        dqkv = torch.empty_like(qkv)
    dt = _DT[qkv.dtype]
    nbytes = api.attn_bwd_workspace_size(B, T, C, NH, int(causal), dt)
    ws = (workspace or _default_ws).get(nbytes, qkv.device)
    api.attn_bwd(dout, qkv, out, lse, dqkv, B, T, C, NH, int(causal), dt, ws, nbytes, stream)
    return dqkv
