"""Small-float formats used by the method (oracle; test infrastructure only).

Sources.  The method quantizes activations to NVFP4, the 4-bit floating-point
format native to NVIDIA Blackwell ("6Bit-Diffusion" technical summary,
section 2.A; popular summary, section 1).  NVFP4 is E2M1 codes with one
unsigned E4M3 scale per 16 elements and an FP32 tensor scale.  The pages do
not define the formats; the definitions below are the public ones:

* E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.
  Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E4M3 ("FN", OCP FP8): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
  no infinities, exponent-15/mantissa-7 is NaN, largest finite 448,
  smallest subnormal 2**-9.
* bfloat16: the top 16 bits of an IEEE binary32.
* MXFP8 (OCP Microscaling Formats v1.0, E4M3 elements): blocks of 32
  consecutive elements share one E8M0 scale 2**X (an 8-bit biased exponent,
  bias 127, code 255 = NaN, no sign and no mantissa).  X is the exponent of
  the block's largest magnitude minus that of E4M3's largest normal (8),
  floor(log2 amax) - 8, clamped to E8M0's range [-127, 127]; an all-zero
  block takes the smallest scale.  Each element is E4M3(v / 2**X) with the
  rounding below.  Magnitudes in [448, 512) * 2**X saturate to 448 * 2**X.
  The method only says that the temporal delta cache can be kept in a low
  precision ("6Bit-Diffusion" popular summary, section 7); MXFP8 is the
  reading taken for it.

Rounding is round-to-nearest, ties-to-even on the mantissa LSB, and
"satfinite": magnitudes beyond the largest finite value become that value.
The sign of the input is kept, so a negative value that rounds to zero
encodes as negative zero.

The encoder is one generic routine for a (exponent bits, mantissa bits,
bias, max) format, written from the definition of round-to-nearest-even on
a floating-point grid: in the binade of the value (clamped below to the
smallest normal binade) the grid spacing is 2**(e - mbits); divide by it,
round half-to-even to an integer, multiply back.  The integer's parity is
the mantissa LSB, so half-to-even on it is ties-to-even on the mantissa.
"""
from __future__ import annotations

import numpy as np

# (exponent bits, mantissa bits, bias, largest finite magnitude)
E2M1 = (2, 1, 1, 6.0)
E4M3 = (4, 3, 7, 448.0)


def _round_to_format(a: np.ndarray, fmt) -> np.ndarray:
    """Round non-negative float64 magnitudes onto the grid of ``fmt`` (RNE, satfinite)."""
    ebits, mbits, bias, fmax = fmt
    emin = 1 - bias                       # exponent of the smallest normal binade
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    big = a >= fmax                       # includes +inf
    out[big] = fmax
    mid = (~big) & (a > 0)
    am = a[mid]
    _, ex = np.frexp(am)                  # am = f * 2**ex, f in [0.5, 1)
    e = np.maximum(ex - 1, emin)          # binade exponent, clamped to normal range
    quantum = np.ldexp(1.0, e - mbits)
    r = np.rint(am / quantum) * quantum   # np.rint: half to even; am/quantum is exact
    out[mid] = np.minimum(r, fmax)
    return out


def _encode_magnitude(r: np.ndarray, fmt) -> np.ndarray:
    """Bit pattern (without sign) of representable magnitudes ``r``."""
    ebits, mbits, bias, _ = fmt
    emin = 1 - bias
    code = np.zeros(r.shape, dtype=np.int64)
    nz = r > 0
    rn = r[nz]
    _, ex = np.frexp(rn)
    e = ex - 1
    sub = e < emin
    expf = np.where(sub, 0, e + bias)
    mant = np.where(sub,
                    rn / np.ldexp(1.0, emin - mbits),
                    rn / np.ldexp(1.0, e - mbits) - (1 << mbits))
    code[nz] = (expf.astype(np.int64) << mbits) | mant.astype(np.int64)
    return code


def encode(v, fmt) -> np.ndarray:
    """Encode float32/float64 values to the small-float ``fmt`` (uint8 codes)."""
    v = np.asarray(v)
    ebits, mbits, _, _ = fmt
    sign = np.signbit(v).astype(np.int64)
    mag = _round_to_format(np.abs(v.astype(np.float64)), fmt)
    code = _encode_magnitude(mag, fmt) | (sign << (ebits + mbits))
    return code.astype(np.uint8)


def decode(code, fmt) -> np.ndarray:
    """Decode small-float codes to float64 (E4M3 NaN pattern decodes to NaN)."""
    ebits, mbits, bias, _ = fmt
    c = np.asarray(code).astype(np.int64)
    sign = (c >> (ebits + mbits)) & 1
    expf = (c >> mbits) & ((1 << ebits) - 1)
    mant = c & ((1 << mbits) - 1)
    emin = 1 - bias
    val = np.where(expf == 0,
                   np.ldexp(mant.astype(np.float64), emin - mbits),
                   np.ldexp((mant + (1 << mbits)).astype(np.float64), expf - bias - mbits))
    if fmt == E4M3:
        val = np.where((expf == 15) & (mant == 7), np.nan, val)
    return np.where(sign == 1, -val, val)


def e2m1_encode(v):
    return encode(v, E2M1)


def e2m1_decode(c):
    return decode(c, E2M1)


def e4m3_encode(v):
    return encode(v, E4M3)


def e4m3_decode(c):
    return decode(c, E4M3)


def bf16_round(x) -> np.ndarray:
    """Round float32 values to bfloat16 (RNE), returned as float32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = (r << 16).astype(np.uint32).view(np.float32)
    nan = np.isnan(x)
    if nan.any():
        out = out.copy()
        out[nan] = np.nan
    return out.reshape(x.shape)


def bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ MXFP8 --

MX_BLOCK = 32
E8M0_BIAS = 127


def e8m0_decode(code) -> np.ndarray:
    """2**(code - 127) as float64; code 255 is NaN."""
    c = np.asarray(code).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - E8M0_BIAS))


def mx_shared_exponent(amax) -> np.ndarray:
    """X = floor(log2 amax) - 8, clamped to [-127, 127]; amax == 0 gives -127."""
    a = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(a)                   # a = f * 2**ex, f in [0.5, 1): floor(log2 a) = ex - 1
    x = np.where(a > 0, ex - 1 - 8, -E8M0_BIAS)
    return np.clip(x, -E8M0_BIAS, E8M0_BIAS).astype(np.int64)


def mxfp8_encode(v, block: int = MX_BLOCK):
    """MXFP8 (E4M3 elements) of a flat array whose length is a multiple of `block`.

    Returns (codes uint8 [n], scales uint8 [n / block]) with scales the E8M0
    codes X + 127.
    """
    v = np.asarray(v, dtype=np.float64).reshape(-1)
    if v.size % block:
        raise ValueError("length must be a multiple of the block")
    blocks = v.reshape(-1, block)
    x = mx_shared_exponent(np.abs(blocks).max(axis=1) if blocks.size else np.zeros(0))
    scaled = blocks / np.ldexp(1.0, x)[:, None]          # exact: a power of two
    codes = encode(scaled, E4M3).reshape(-1)
    return codes, (x + E8M0_BIAS).astype(np.uint8)


def mxfp8_decode(codes, scales, block: int = MX_BLOCK) -> np.ndarray:
    """float64 values of MXFP8 codes (flat) with one E8M0 scale per `block` codes."""
    c = np.asarray(codes).reshape(-1, block)
    return (decode(c, E4M3) * e8m0_decode(scales)[:, None]).reshape(-1)
