"""CPU oracle for the linear layers around the attention (c_attn, c_proj) and
the attention block forward they form. TEST INFRASTRUCTURE ONLY (see the
package docstring); float64 numpy, numpy matmul as the only library step.

  Sources:
    [LSQ]   "LLM Systems 10 & 11: Accelerating Transformer Training and
            Inference", §1.1 / §1.1.1: the MHA layer is GEMMs plus non-GEMM
            ops; the non-GEMM ops (here the bias add) are fused into their
            neighbours. The pages do not print the GEMM itself.
    [LLMC]  llm.c layout conventions (qkv (B, T, 3C), out (B, T, C)).

  Reading (the pages are silent on the linear layer's definition): the
  GPT-2 linear layer out = inp . weight^T + bias, weight stored (OC, C) as in
  llm.c, the same definition for c_attn (OC = 3C) and c_proj (OC = C).
"""
from __future__ import annotations

import numpy as np

from .attention import forward as attention_forward


def linear(inp: np.ndarray, weight: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """out[..., o] = bias[o] + sum_k inp[..., k] * weight[o, k], float64."""
    x = np.asarray(inp, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    out = x @ w.T
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float64)
    return out


def block_forward(x: np.ndarray, w_attn, b_attn, w_proj, b_proj, NH: int, causal: bool = True):
    """x (B, T, C) -> qkv = linear(x, w_attn, b_attn) -> attention -> y = linear(out, w_proj, b_proj).

    Returns (y, qkv, out, lse). `qkv` and `out` are the exact intermediates;
    a caller comparing against a bf16 pipeline may re-enter with rounded ones.
    """
    B, T, C = x.shape
    qkv = linear(x, w_attn, b_attn)
    out, lse = attention_forward(qkv, B, T, C, NH, causal)
    y = linear(out, w_proj, b_proj)
    return y, qkv, out, lse
