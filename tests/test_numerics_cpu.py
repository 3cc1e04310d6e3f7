"""CPU checks of the floating-point identities the GPU kernels rely on.

The kernels compute some steps of the method in a different but equivalent
way; each equivalence is checked here on the host, independently of the GPU:

- INT8 quantization divides the unscaled rotated value v by s * sqrt(b)
  instead of y = v / sqrt(b) by s: RN(y / s) = RN(v / (s sqrt b)) whenever
  both scalings are exact (and q rounds to 0 either way where y would be an
  inexact subnormal);
- rint(d) for |d| <= 127 (1 + 2^-24) is taken as RN(d + 1.5 * 2^23) - 1.5 * 2^23;
- a quotient y / d is taken from a correctly rounded reciprocal and one FMA
  correction (Markstein's theorem) when d and 1/d are normal and y / d does
  not underflow: checked against the exactly rounded quotient with rationals;
- the GEMM epilogue's GELU (erf(x) = x Q(s), Q a degree-15 Chebyshev
  interpolant in s = 2 x^2 / 3.9^2 - 1, x clamped to +-3.9) stays within the
  epilogue's error budget of 4e-7 |GELU| plus the operand bound, here as
  |error| <= 3.5e-7 max(|v|, 1) in an FP32 emulation with FMAs rounded once;
  the kernel's coefficients are the ones its generator script prints.
"""
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import erf

F32 = np.float32


def _rn32(fr: Fraction) -> np.float32:
    """Exactly rounded (nearest, ties to even) float32 of a rational."""
    c = np.float32(float(fr))   # within a float32 ulp or two
    best = None
    for cand in (np.nextafter(np.nextafter(c, F32(-np.inf)), F32(-np.inf)), np.nextafter(c, F32(-np.inf)), c,
                 np.nextafter(c, F32(np.inf)), np.nextafter(np.nextafter(c, F32(np.inf)), F32(np.inf))):
        if not np.isfinite(cand):
            continue
        err = abs(Fraction(float(cand)) - fr)
        if best is None or err < best[0] or (err == best[0] and (int(cand.view(np.uint32)) & 1) == 0):
            best = (err, cand)
    return best[1]


@pytest.mark.parametrize("b", [16, 64, 256])
def test_int8_divisor_folding(b):
    rng = np.random.default_rng(b)
    sq = F32(np.sqrt(b))
    for scale in (1.0, 1e-3, 1e-30, 1e30):
        v = (rng.standard_normal((64, 512)) * scale).astype(F32)
        v[0, :8] = F32(2.0 ** -140)                              # values whose v / sqrt(b) is subnormal
        y = v / sq                                               # exact unless subnormal
        amax_y = np.abs(y).max(axis=1, keepdims=True)
        s = amax_y / F32(127.0)
        ok = (np.abs(s) >= F32(2.0 ** -100)) & (np.abs(s) <= F32(2.0 ** 100))
        q_ref = np.rint(y / s)
        q_fold = np.rint(v / (s * sq))
        assert np.array_equal(np.where(ok, q_ref, 0), np.where(ok, q_fold, 0))


def test_magic_number_rounding_is_rint():
    k = F32(12582912.0)   # 1.5 * 2^23
    d = np.concatenate([np.arange(-127, 128, dtype=np.float64) + off
                        for off in (0.0, 0.5, -0.5, 0.25, 0.75, 0.4999999, 0.5000001)]).astype(F32)
    d = np.concatenate([d, np.nextafter(d, F32(np.inf)), np.nextafter(d, F32(-np.inf)),
                        F32([127.0 * (1 + 2.0 ** -23), -127.0 * (1 + 2.0 ** -23)])])
    d = d[np.abs(d) <= F32(127.0 * (1 + 2.0 ** -23))]
    assert np.array_equal((d + k) - k, np.rint(d))


def test_markstein_division_equals_ieee_quotient():
    rng = np.random.default_rng(11)
    n = 4000
    d = (rng.uniform(1, 2, n) * 2.0 ** rng.integers(-100, 100, n)).astype(F32)
    d = np.where(rng.uniform(size=n) < 0.5, d, -d).astype(F32)
    q_target = rng.uniform(-128, 128, n)
    y = (q_target * d.astype(np.float64)).astype(F32)
    y[::7] = (np.rint(q_target[::7]) + 0.5).astype(F32) * d[::7]   # near rounding ties
    for yi, di in zip(y, d):
        if not np.isfinite(yi) or yi == 0:
            continue
        rd = _rn32(1 / Fraction(float(di)))
        q0 = _rn32(Fraction(float(yi)) * Fraction(float(rd)))
        res = _rn32(Fraction(float(yi)) - Fraction(float(di)) * Fraction(float(q0)))   # fma: one rounding
        q = _rn32(Fraction(float(res)) * Fraction(float(rd)) + Fraction(float(q0)))      # fma: one rounding
        assert q == _rn32(Fraction(float(yi)) / Fraction(float(di))), (yi, di)


def _fma32(a, b, c):
    """FP32 fused multiply-add: the float64 product of two floats is exact, so one rounding."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(F32)


def _kernel_gelu_constants():
    """(scale of s, [c_0 .. c_15]) as written in gemm_common.cuh."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(__file__), "..", "video_dit_mixed_gb300", "csrc", "gemm_common.cuh")).read()
    body = src[src.index("constexpr float gelu_q(int i)"):]
    body = body[:body.index("return c[i];")]
    coef = [float.fromhex(m) for m in re.findall(r"(-?0x[0-9a-f.]+p-?\d+)f,", body)]
    scale = float.fromhex(re.search(r"kGeluS = (0x[0-9a-f.]+p-?\d+)f", src).group(1))
    return F32(scale), np.array(coef, dtype=F32)


def test_epilogue_gelu_coefficients_are_the_generators():
    import sys
    import os
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), "..", "video_dit_mixed_gb300", "csrc"))
    import gelu_coeffs
    scale, coef = _kernel_gelu_constants()
    assert coef.size == gelu_coeffs.DEGREE + 1
    np.testing.assert_array_equal(coef, gelu_coeffs.coefficients())
    assert scale == gelu_coeffs.s_scale()


def test_epilogue_gelu_error_budget():
    v = np.concatenate([np.linspace(-12, 12, 240001), [-60.0, -30.0, 0.0, 1e-30, -1e-30, 30.0, 60.0],
                        np.random.default_rng(7).standard_normal(100000) * 4])
    g = 0.5 * v * (1 + erf(v / np.sqrt(2.0)))
    scale, coef = _kernel_gelu_constants()
    x = v.astype(F32)
    xs = x * F32(0.7071067811865475244)
    xc = (np.sign(xs) * np.minimum(np.abs(xs), F32(3.9))).astype(F32)  # min.xorsign.abs
    s = _fma32(xc * xc, np.full_like(xc, scale), np.full_like(xc, F32(-1)))
    q = np.full_like(s, coef[-1])
    for c in coef[-2::-1]:
        q = _fma32(q, s, np.full_like(s, c))
    h = x * F32(0.5)
    ours = _fma32(h, xc * q, h).astype(np.float64)
    assert np.all(np.abs(ours - g) <= 3.5e-7 * np.maximum(np.abs(v), 1.0))
    # the stated figures, for the FP32 input the kernel sees: erf within
    # 1.9e-7, GELU within 1.3e-7 |v|
    x64 = x.astype(np.float64)
    assert np.max(np.abs((xc * q).astype(np.float64) - erf(xs.astype(np.float64)))) <= 1.9e-7
    g32 = 0.5 * x64 * (1 + erf(x64 / np.sqrt(2.0)))
    nz = x64 != 0
    assert np.max(np.abs(ours - g32)[nz] / np.abs(x64[nz])) <= 1.3e-7
