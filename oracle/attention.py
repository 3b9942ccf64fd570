"""CPU oracle for GPT-2-style multi-head self-attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the product imports this module; only the
tests, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg call it.
It shares no code with the CUDA path.

What it computes is the plain definition, in float64, one (batch, head) pair at
a time, with numpy matmuls as the only library steps:

  Sources (web pages):
    [LLMC]  llm.c ``dev/cuda/attention_backward.cu`` (gitea mirror), the CPU
            reference functions ``attention_forward_cpu`` (passes 1-4) and
            ``attention_backward_cpu`` (backward passes 4, 2&3, 1), and the
            softmax-backward ``kernel7`` simplification.
    [ANNO]  "llm.c 的中文注解-20240423" (aqwu.net), section 1.1 (activation
            gradients are written with = rather than +=).
    [VIT]   "Umakini wa kujitegemea, kerneli za CUDA na FlashAttention",
            section 1 (Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V, heads in
            parallel) and section 3 (only small normalisation statistics are
            kept between the passes).

  Layout [LLMC, attention_forward_cpu]: qkv is (B, T, 3C); for head h the query
  of token t is qkv[b, t, h*hs : (h+1)*hs], its key sits at offset +C and its
  value at +2C. out is (B, T, C) with head h at columns h*hs..(h+1)*hs.

Readings where the pages are silent or disagree (each listed in the design notes):
  * row max: taken over the allowed keys J(t) (the CPU reference scans all keys,
    the GPU softmax only j <= t; the result is the same real number).
  * lse (not defined on the pages): lse = scale*m + ln(sum_j exp(scale*(s_j - m))),
    natural log, one value per (b, h, t).
  * dqkv is written with = (activation gradient) [ANNO 1.1].
  * scale = 1/sqrt(hs) [LLMC, attention_forward_cpu].
"""
from __future__ import annotations

import math

import numpy as np


def _allowed(T: int, causal: bool) -> np.ndarray:
    """J(t) as a boolean (T, T) matrix: key j is visible to query t."""
    if causal:
        return np.tril(np.ones((T, T), dtype=bool))
    return np.ones((T, T), dtype=bool)


def split_heads(qkv: np.ndarray, C: int, NH: int):
    """(B, T, 3C) -> q, k, v each (B, NH, T, hs) float64 [LLMC layout]."""
    B, T, C3 = qkv.shape
    assert C3 == 3 * C and C % NH == 0
    hs = C // NH
    x = np.asarray(qkv, dtype=np.float64).reshape(B, T, 3, NH, hs)
    q = np.ascontiguousarray(x[:, :, 0].transpose(0, 2, 1, 3))
    k = np.ascontiguousarray(x[:, :, 1].transpose(0, 2, 1, 3))
    v = np.ascontiguousarray(x[:, :, 2].transpose(0, 2, 1, 3))
    return q, k, v


def head_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                 return_att: bool = False):
    """One head. q, k, v: (T, hs) float64. Returns out (T, hs), lse (T,) [, att, preatt].

    [LLMC attention_forward_cpu]: pass 1 preatt = q.k (no scale); pass 2
    exp(scale*(preatt - max)) and its sum over visible keys; pass 3 normalise
    and zero the masked entries; pass 4 out = att @ v.
    """
    T, hs = q.shape
    scale = 1.0 / math.sqrt(hs)
    allowed = _allowed(T, causal)
    preatt = q @ k.T                                   # pass 1 (unscaled)
    m = np.where(allowed, preatt, -np.inf).max(axis=1)  # max over J(t)
    e = np.where(allowed, np.exp(scale * (preatt - m[:, None])), 0.0)  # pass 2
    l = e.sum(axis=1)
    assert np.all(l > 0.0), "the expsum==0 guard of the page must never fire"
    att = e / l[:, None]                               # pass 3 (zeros above the diagonal)
    out = att @ v                                      # pass 4
    lse = scale * m + np.log(l)
    if return_att:
        return out, lse, att, preatt
    return out, lse


def head_backward(q, k, v, dout_h, causal: bool, return_parts: bool = False):
    """One head. dout_h: (T, hs). Returns dq, dk, dv (T, hs).

    [LLMC attention_backward_cpu] with the softmax step in the row-sum form of
    [LLMC kernel7]: dpreatt[t, j] = scale * att[t, j] * (datt[t, j] - sum_j' att[t, j'] datt[t, j']).
    """
    T, hs = q.shape
    scale = 1.0 / math.sqrt(hs)
    _, _, att, _ = head_forward(q, k, v, causal, return_att=True)
    datt = dout_h @ v.T                                # backward pass 4: datt
    dv = att.T @ dout_h                                # backward pass 4: dv
    D = (att * datt).sum(axis=1)                       # kernel7 local_sum
    dpreatt = scale * att * (datt - D[:, None])        # kernel7 identity
    dq = dpreatt @ k                                   # backward pass 1
    dk = dpreatt.T @ q
    if return_parts:
        return dq, dk, dv, {"att": att, "datt": datt, "dpreatt": dpreatt, "D": D}
    return dq, dk, dv


def head_dpreatt_jacobian(att: np.ndarray, datt: np.ndarray, causal: bool) -> np.ndarray:
    """Softmax backward in the Jacobian form of [LLMC attention_backward_cpu, passes 2&3].

    For row t: dpreatt[t, t3] = sum_{t2 in J(t)} scale * att[t, t2] * (delta(t2, t3) - att[t, t3]) * datt[t, t2],
    built as the full (t2, t3) local-derivative matrix per row. O(T^3); small T only.
    `scale` is folded in by the caller.
    """
    T = att.shape[0]
    allowed = _allowed(T, causal)
    out = np.zeros_like(att)
    for t in range(T):
        js = np.nonzero(allowed[t])[0]
        a = att[t, js]
        local = a[:, None] * (np.eye(js.size) - a[None, :])   # [t2, t3]
        out[t, js] = local.T @ datt[t, js]
    return out


def forward(qkv: np.ndarray, B: int, T: int, C: int, NH: int, causal: bool, heads=None):
    """Full forward. Returns out (B, T, C) and lse (B, NH, T), float64.

    `heads`: optional iterable of (b, h) to compute; other entries are NaN.
    """
    q, k, v = split_heads(qkv, C, NH)
    hs = C // NH
    out = np.full((B, T, C), np.nan)
    lse = np.full((B, NH, T), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(NH)]
    for b, h in pairs:
        o, l = head_forward(q[b, h], k[b, h], v[b, h], causal)
        out[b, :, h * hs:(h + 1) * hs] = o
        lse[b, h] = l
    return out, lse


def backward(dout: np.ndarray, qkv: np.ndarray, B: int, T: int, C: int, NH: int,
             causal: bool, heads=None):
    """Full backward. Returns dqkv (B, T, 3C) float64, written with = [ANNO 1.1]."""
    q, k, v = split_heads(qkv, C, NH)
    hs = C // NH
    do = np.asarray(dout, dtype=np.float64).reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    dqkv = np.full((B, T, 3 * C), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(NH)]
    for b, h in pairs:
        dq, dk, dv = head_backward(q[b, h], k[b, h], v[b, h], do[b, h], causal)
        dqkv[b, :, h * hs:(h + 1) * hs] = dq
        dqkv[b, :, C + h * hs:C + (h + 1) * hs] = dk
        dqkv[b, :, 2 * C + h * hs:2 * C + (h + 1) * hs] = dv
    return dqkv


def row_stat_D(dout: np.ndarray, out: np.ndarray, B: int, T: int, C: int, NH: int) -> np.ndarray:
    """D[b, h, t] = sum_i dout[b, t, h*hs+i] * out[b, t, h*hs+i], shape (B, NH, T).

    Equal to the kernel7 local_sum sum_j att[t, j] * datt[t, j], since out_t = sum_j att[t, j] v_j.
    """
    hs = C // NH
    do = np.asarray(dout, dtype=np.float64).reshape(B, T, NH, hs)
    o = np.asarray(out, dtype=np.float64).reshape(B, T, NH, hs)
    return (do * o).sum(axis=3).transpose(0, 2, 1)
