"""Dynamic activation quantizers and 4-bit weight packing (oracle; test infrastructure only).

Method.  Per transformer block and denoising step, activations are quantized
online either to NVFP4 (stable blocks: fast, narrow range) or to INT8
(volatile blocks: more precise), after the online block Hadamard rotation
("6Bit-Diffusion" technical summary, section 2.A, "Mecanismo"; popular
summary, section 1).  Weights are 4-bit (the W4A6 / W4A8 configurations,
technical summary section 4 "Calidad"; popular summary section 4).

The pages leave the quantizer arithmetic open.  Readings taken (all FP32,
every operation IEEE round-to-nearest-even, divisions done as divisions):

NVFP4 (two-level):
  amax_t = max |y| over the whole tensor;  s_t = amax_t / 2688 (2688 = 6 * 448),
  or 1.0 when amax_t == 0.  Per 16 consecutive elements of a row:
  sb = (amax_b / 6) / s_t;  e = E4M3(sb);  S = decode(e) * s_t;
  code_i = E2M1(y_i / S), or +0 (code 0) when S == 0.
INT8 (symmetric, per token):
  s_m = amax_row / 127;  q = clamp(rint(y / s_m), -127, 127), q = 0 when s_m == 0.
INT4 weights (symmetric, per output row and group of 128 along K):
  s = amax_group / 7;  q = clamp(rint(w / s), -7, 7), q = 0 when s == 0.
NVFP4 weights: the same two-level quantizer as the activations with a static
  tensor scale taken from the rotated weight.

Packing: two 4-bit codes per byte, the element with the even K index in the
low nibble.
"""
from __future__ import annotations

import numpy as np

from . import formats
from .hadamard import fwht_blocks

NVFP4_GROUP = 16
INT4_GROUP = 128
F32 = np.float32


def tensor_scale(amax) -> np.float32:
    """s_t = amax / (6 * 448) in FP32, or 1 when amax == 0."""
    amax = F32(amax)
    return F32(1.0) if amax == 0 else F32(amax / F32(2688.0))


def nvfp4_quantize(y, s_t=None):
    """Two-level NVFP4 quantization of float32 ``y`` [M, K] (K % 16 == 0).

    Returns dict(codes=uint8 [M, K] unpacked E2M1 codes, scales=uint8 [M, K/16]
    E4M3 codes, s_t=float32, amax=float32).
    """
    y = np.asarray(y, dtype=F32)
    m, k = y.shape
    amax = F32(np.max(np.abs(y))) if y.size else F32(0)
    if s_t is None:
        s_t = tensor_scale(amax)
    s_t = F32(s_t)
    blk = y.reshape(m, k // NVFP4_GROUP, NVFP4_GROUP)
    amax_b = np.max(np.abs(blk), axis=2).astype(F32)
    sb = (amax_b / F32(6.0)).astype(F32) / s_t
    sb = sb.astype(F32)
    e = formats.e4m3_encode(sb)
    S = (formats.e4m3_decode(e).astype(F32) * s_t).astype(F32)
    Sx = np.repeat(S, NVFP4_GROUP, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (y / np.where(Sx == 0, F32(1), Sx)).astype(F32)
    codes = formats.e2m1_encode(q)
    codes = np.where(Sx == 0, np.uint8(0), codes).astype(np.uint8)
    return dict(codes=codes, scales=e, s_t=s_t, amax=amax)


def nvfp4_dequant(codes, scales, s_t) -> np.ndarray:
    """float64 values s_t * decode(scale) * decode(code)  (unpacked codes)."""
    a = formats.e2m1_decode(codes)
    sf = np.repeat(formats.e4m3_decode(scales), NVFP4_GROUP, axis=1)
    return float(s_t) * (a * sf)


def int8_quantize(y):
    """Symmetric per-row INT8 quantization of float32 ``y`` [M, K].

    Returns dict(q=int8 [M, K], s=float32 [M]).
    """
    y = np.asarray(y, dtype=F32)
    amax = np.max(np.abs(y), axis=1).astype(F32) if y.shape[1] else np.zeros(y.shape[0], F32)
    s = (amax / F32(127.0)).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (y / np.where(s == 0, F32(1), s)[:, None]).astype(F32)
    q = np.clip(np.rint(r), -127, 127)
    q = np.where(s[:, None] == 0, 0, q).astype(np.int8)
    return dict(q=q, s=s)


def int4_quantize_weights(w):
    """Symmetric INT4 quantization per row and group of 128 of float32 ``w`` [N, K].

    Returns dict(q=int8 [N, K] with values in [-7, 7], s=float32 [N, K/128]).
    """
    w = np.asarray(w, dtype=F32)
    n, k = w.shape
    g = w.reshape(n, k // INT4_GROUP, INT4_GROUP)
    amax = np.max(np.abs(g), axis=2).astype(F32)
    s = (amax / F32(7.0)).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (g / np.where(s == 0, F32(1), s)[:, :, None]).astype(F32)
    q = np.clip(np.rint(r), -7, 7)
    q = np.where(s[:, :, None] == 0, 0, q).astype(np.int8).reshape(n, k)
    return dict(q=q, s=s)


def pack_nibbles(codes) -> np.ndarray:
    """Pack 4-bit values (uint8 0..15 or int8 -8..7) two per byte, even index low."""
    c = (np.asarray(codes).astype(np.int64) & 0xF).astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed, signed=False) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    if signed:
        return np.where(out >= 8, out.astype(np.int16) - 16, out).astype(np.int8)
    return out


def hadamard_quant(x_bf16, b: int, mode: str, s_t=None):
    """Online rotation + dynamic quantization of bf16-valued ``x`` [M, K].

    mode 'nvfp4' -> nvfp4_quantize(y) fields; 'int8' -> int8_quantize(y) fields.
    Also returns the rotated FP32 tensor under key 'y'.
    """
    y = fwht_blocks(np.asarray(x_bf16, dtype=F32), b)
    if mode == "nvfp4":
        out = nvfp4_quantize(y, s_t)
    elif mode == "int8":
        out = int8_quantize(y)
    else:
        raise ValueError(mode)
    out["y"] = y
    return out


def pack_weights(w, b: int):
    """Offline weight preparation for one linear layer, W float32 [N, K].

    W' = W . blockdiag(H_b/sqrt(b)) (same FP32 butterfly as the activations),
    then NVFP4 (static two-level) and INT4-g128 quantization of W'; bf16(W)
    (unrotated) is kept for the full-precision path.
    """
    w = np.asarray(w, dtype=F32)
    wr = fwht_blocks(w, b)
    nv = nvfp4_quantize(wr)
    i4 = int4_quantize_weights(wr)
    return dict(w_rot=wr, nvfp4=nv, int4=i4, bf16=formats.bf16_round(w))
