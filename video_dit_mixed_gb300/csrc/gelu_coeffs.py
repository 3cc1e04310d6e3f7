"""Coefficients of the GEMM epilogues' GELU (``gelu_pair`` in gemm_common.cuh).

GELU(v) = v * Phi(v) = 0.5 v (1 + erf(v / sqrt 2))   ("6Bit-Diffusion" technical
summary section 2: the FFN's activation; the exact-erf form is the definition).

Method: erf is odd and erf(x) / x is an even entire function, so on |x| <= X
it is a smooth function of u = x^2.  It is interpolated at the n + 1 Chebyshev
nodes of the variable s = 2 u / X^2 - 1 in [-1, 1] (Chebyshev interpolation:
for an analytic function the error falls geometrically with n), and the
interpolant is written as monomial coefficients in s for a Horner evaluation
in s, which stays well conditioned on [-1, 1] (the coefficients are below 1
in magnitude).  Beyond |x| = X = 3.9 the kernel clamps x to +-X, where
erf(X) = 1 - 3.5e-8: the clamped value is erf to within that.

Run this script to print the constants; it needs numpy and scipy (erf in
float64 as the definition).  Rounded to FP32 and evaluated with FP32 FMAs,
the result is within ~2e-7 of erf(x) for every x (checked by
``tests/test_numerics_cpu.py``), the same budget as the Abramowitz and
Stegun 7.1.26 rational form it replaces, without its reciprocal and
exponential (two special-function-unit operations an element).
"""
import numpy as np

X_MAX = 3.9
DEGREE = 15


def coefficients(degree: int = DEGREE, x_max: float = X_MAX) -> np.ndarray:
    """Monomial coefficients c_0 .. c_degree (float32) of Q(s) ~ erf(x) / x, s = 2 x^2 / x_max^2 - 1."""
    from numpy.polynomial import chebyshev
    from scipy.special import erf

    k = np.arange(degree + 1)
    nodes = np.cos(np.pi * (k + 0.5) / (degree + 1))  # Chebyshev points of the first kind in s
    x = x_max * np.sqrt((nodes + 1.0) / 2.0)
    cheb = chebyshev.chebfit(nodes, erf(x) / x, degree)  # interpolation: n + 1 points, degree n
    return chebyshev.cheb2poly(cheb).astype(np.float32)


def s_scale(x_max: float = X_MAX) -> np.float32:
    return np.float32(2.0 / (x_max * x_max))


def main() -> None:
    c = coefficients()
    print(f"// Q(s), s = u * {float(s_scale()).hex()} - 1, u = min(|x|, {X_MAX})^2; c_0 .. c_{DEGREE}")
    for i, v in enumerate(c):
        print(f"  {float(v).hex()}f,  // c_{i} = {float(v):.9g}")


if __name__ == "__main__":
    main()
