"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: it only draws numbers. Both the CUDA
path and the CPU oracle receive exactly the arrays made here.

Generator (stated so it can be re-implemented anywhere):
  * SplitMix64 stream: state_i = seed + i * 0x9E3779B97F4A7C15 (mod 2^64), i = 1, 2, ...
    followed by the SplitMix64 finaliser (xor-shift 30, *0xBF58476D1CE4E5B9,
    xor-shift 27, *0x94D049BB133111EB, xor-shift 31).
  * Each normal draw consumes two consecutive words w1, w2:
    u = ((w >> 11) + 0.5) / 2^53  in (0, 1),
    z = sqrt(-2 ln u1) * cos(2 pi u2)   (Box-Muller, float64).
  * x = sigma * z, rounded once to float32; for bf16 inputs the float32 value is
    rounded once more to bf16 (round to nearest, ties to even).

Workloads (shapes and distributions of the GPT-2 and ViT-B/16 attention layers):
  qkv has shape (B, T, 3C); dout has shape (B, T, C).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Words start+1 .. start+n of the SplitMix64 stream for `seed`."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def normal_f64(seed: int, n: int) -> np.ndarray:
    """n standard-normal float64 draws (Box-Muller on SplitMix64 words)."""
    out = np.empty(n, dtype=np.float64)
    scale = 1.0 / 9007199254740992.0  # 2^-53
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        w = _splitmix64(seed, 2 * s, 2 * m)
        u = ((w >> np.uint64(11)).astype(np.float64) + 0.5) * scale
        u1, u2 = u[0::2], u[1::2]
        out[s:s + m] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention layer configuration."""
    name: str
    B: int
    T: int
    C: int
    NH: int
    causal: int
    dtype: str          # "f32" or "bf16"
    sigma_qkv: float
    sigma_dout: float
    seed_qkv: int
    seed_dout: int

    @property
    def hs(self) -> int:
        return self.C // self.NH


def _wl(idx, name, B, T, C, NH, causal, dtype, sq, sd):
    return Workload(name, B, T, C, NH, causal, dtype, sq, sd, 1000 + idx, 2000 + idx)


# The six attention-layer shapes: GPT-2 small/XL widths, a long-context GPT-2
# layer, and ViT-B/16 (224x224 image, 16x16 patches -> 196 tokens, no mask).
WORKLOADS = {
    "tiny": _wl(0, "tiny", 2, 64, 128, 4, 1, "f32", 1.0, 1.0),
    "gpt2s_f32": _wl(1, "gpt2s_f32", 4, 1024, 768, 12, 1, "f32", 0.5, 1e-2),
    "gpt2s_bf16": _wl(2, "gpt2s_bf16", 16, 1024, 768, 12, 1, "bf16", 0.5, 1e-2),
    "xl_bf16": _wl(3, "xl_bf16", 8, 1024, 1600, 25, 1, "bf16", 0.5, 1e-2),
    "long_bf16": _wl(4, "long_bf16", 2, 8192, 768, 12, 1, "bf16", 0.5, 1e-2),
    "vit_bf16": _wl(5, "vit_bf16", 256, 196, 768, 12, 0, "bf16", 0.5, 1e-2),
}


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """A decode step: the last Tq tokens of L-token sequences attend to their cache."""
    name: str
    B: int
    L: int
    C: int
    NH: int
    Tq: int
    dtype: str
    sigma_qkv: float
    seed_qkv: int

    @property
    def hs(self) -> int:
        return self.C // self.NH


# Decode stand-ins (the pages name the inference step offset but no decode
# shape): a batch of 64 GPT-2-small sequences with a 4096-token cache, one new
# token each, and the same with four new tokens (a short draft to verify).
DECODE_WORKLOADS = {
    "gpt2s_decode": DecodeWorkload("gpt2s_decode", 64, 4096, 768, 12, 1, "bf16", 0.5, 3000),
    "gpt2s_decode4": DecodeWorkload("gpt2s_decode4", 64, 4096, 768, 12, 4, "bf16", 0.5, 3001),
}


@dataclasses.dataclass
class HostInputs:
    """Host arrays for one workload.

    `qkv` / `dout` hold the exact values the device sees, as float32 (for bf16
    workloads these are bf16-representable). `qkv_dev` / `dout_dev` hold the
    device representation: float32, or uint16 bf16 bit patterns.
    """
    qkv: np.ndarray
    dout: np.ndarray
    qkv_dev: np.ndarray
    dout_dev: np.ndarray


def draw(shape, sigma: float, seed: int, dtype: str):
    """Return (exact values as float32, device representation)."""
    n = int(np.prod(shape))
    x = (normal_f64(seed, n) * sigma).astype(np.float32).reshape(shape)
    if dtype == "f32":
        return x, x
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x)
        return bf16_bits_to_f32(bits).reshape(shape), bits.reshape(shape)
    raise ValueError(f"unknown dtype {dtype!r}")


# ----------------------------------------------------------------------------- e4m3
# OCP FP8 E4M3 (the "fn" variant the tensor core reads): 1 sign bit, 4 exponent
# bits (bias 7), 3 mantissa bits; exponent 0 holds the subnormals m * 2^-9;
# no infinities; 0x7F / 0xFF are NaN, so the largest finite value is 448 (0x7E).

E4M3_MAX = 448.0


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """float -> e4m3 codes (uint8): round to nearest, ties to even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.uint8)
    a = np.minimum(np.abs(x), E4M3_MAX)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range (a rounding up to 8 * 2^-9 lands on the first normal code, 0x08)
    code[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)
    an = a[~sub]
    e = np.floor(np.log2(an)).astype(np.int64)
    m = np.rint((an / np.exp2(e) - 1.0) * 8.0).astype(np.int64)     # 0..8
    e = np.where(m == 8, e + 1, e)
    m = np.where(m == 8, 0, m)
    code[~sub] = np.minimum((e + 7) * 8 + m, 0x7E)
    return (code.astype(np.uint8) | sign)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) -> float64 values (NaN codes are not produced here)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7))
    return np.where(c & 0x80, -mag, mag)


@dataclasses.dataclass
class Fp8Inputs:
    """qkv as e4m3 codes with one descale per 128-row tile of each head's q, k
    and v (value = code * descale of its tile)."""
    codes: np.ndarray        # (B, T, 3C) uint8
    descale: np.ndarray      # (3, B, NH, ceil(T/128)) float32
    qkv: np.ndarray          # (B, T, 3C) float64, the exact values the codes stand for


FP8_TILE = 128


def fp8_tile_view(x: np.ndarray, C: int, NH: int, part: int):
    """Tiles of part (0 q, 1 k, 2 v) of x (B, T, 3C): yields (b, h, tile, slice)
    with slice selecting rows [128*tile, 128*tile+128) of that head's columns."""
    B, T, _ = x.shape
    hs = C // NH
    for b in range(B):
        for h in range(NH):
            c0 = part * C + h * hs
            for k in range((T + FP8_TILE - 1) // FP8_TILE):
                yield b, h, k, (b, slice(k * FP8_TILE, min(T, (k + 1) * FP8_TILE)), slice(c0, c0 + hs))


def make_fp8_inputs(B, T, C, sigma=0.5, seed=1, NH=None, tile_gain=False) -> Fp8Inputs:
    """Draw qkv ~ N(0, sigma^2) (the bf16 recipe's normals), pick each tile's
    descale so its largest magnitude maps to the largest e4m3 code (a tile is
    128 rows of one head's q, k or v), quantise. NH defaults to C / 64. With
    tile_gain, every tile is first multiplied by 2^u, u uniform in [-1, 1]
    (drawn from seed + 1), so the tiles' descales differ by up to 4x."""
    NH = NH if NH is not None else C // 64
    x = normal_f64(seed, B * T * 3 * C).reshape(B, T, 3 * C) * sigma
    nT = (T + FP8_TILE - 1) // FP8_TILE
    if tile_gain:
        w = _splitmix64(seed + 1, 0, 3 * B * NH * nT)
        u = ((w >> np.uint64(11)).astype(np.float64) + 0.5) / 9007199254740992.0
        gain = np.exp2(2.0 * u - 1.0).reshape(3, B, NH, nT)
        for part in range(3):
            for b, h, k, sl in fp8_tile_view(x, C, NH, part):
                x[sl] *= gain[part, b, h, k]
    codes = np.empty(x.shape, dtype=np.uint8)
    vals = np.empty(x.shape, dtype=np.float64)
    descale = np.empty((3, B, NH, nT), dtype=np.float32)
    for part in range(3):
        for b, h, k, sl in fp8_tile_view(x, C, NH, part):
            tile = x[sl]
            d = np.float32(max(float(np.max(np.abs(tile))), 1e-30) / E4M3_MAX)
            descale[part, b, h, k] = d
            codes[sl] = e4m3_encode(tile / float(d))
            vals[sl] = e4m3_decode(codes[sl]) * float(d)
    return Fp8Inputs(codes, descale, vals)


# FP8 forward workload: the GPT-2-small training shape of the bf16 headline.
FP8_WORKLOADS = {
    "gpt2s_fp8": dict(B=16, T=1024, C=768, NH=12, causal=True, sigma=0.5, seed=4000),
}


# ----------------------------------------------------------------------------- attention block
@dataclasses.dataclass
class BlockInputs:
    """x and the c_attn / c_proj parameters, bf16: exact values (float32) and bits."""
    x: np.ndarray
    w_attn: np.ndarray
    b_attn: np.ndarray
    w_proj: np.ndarray
    b_proj: np.ndarray
    bits: dict


def make_block_inputs(B, T, C, seed=5000, sigma_w=0.02) -> BlockInputs:
    """GPT-2 scales: x ~ N(0, 1) (a layer-normed residual), weights and biases
    ~ N(0, sigma_w^2) (GPT-2's initialisation scale), all rounded to bf16."""
    vals, bits = {}, {}
    for i, (name, shape, sig) in enumerate([("x", (B, T, C), 1.0), ("w_attn", (3 * C, C), sigma_w),
                                            ("b_attn", (3 * C,), sigma_w), ("w_proj", (C, C), sigma_w),
                                            ("b_proj", (C,), sigma_w)]):
        vals[name], bits[name] = draw(shape, sig, seed + i, "bf16")
    return BlockInputs(vals["x"], vals["w_attn"], vals["b_attn"], vals["w_proj"], vals["b_proj"], bits)


BLOCK_WORKLOADS = {
    "gpt2s_block": dict(B=16, T=1024, C=768, NH=12, causal=True, seed=5000),
}


def make_inputs(B, T, C, NH, dtype="bf16", sigma_qkv=0.5, sigma_dout=1e-2,
                seed_qkv=1, seed_dout=2) -> HostInputs:
    del NH  # the layout does not depend on the head split
    qkv, qkv_dev = draw((B, T, 3 * C), sigma_qkv, seed_qkv, dtype)
    dout, dout_dev = draw((B, T, C), sigma_dout, seed_dout, dtype)
    return HostInputs(qkv, dout, qkv_dev, dout_dev)


def workload_inputs(w: Workload) -> HostInputs:
    return make_inputs(w.B, w.T, w.C, w.NH, w.dtype, w.sigma_qkv, w.sigma_dout,
                       w.seed_qkv, w.seed_dout)
