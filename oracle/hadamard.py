"""Online block Hadamard rotation (oracle; test infrastructure only).

The method rotates activations with a block Hadamard transform before
quantization so that outliers are spread over the block ("6Bit-Diffusion"
technical summary, section 2.A, "Suavizado de valores atipicos"; popular
summary, section 1, last paragraph).  The pages give neither the block
size, the element order nor the normalisation.  Reading taken:

* y = x . blockdiag(H_b / sqrt(b)) along the reduction (K) axis, with H_b the
  Sylvester-ordered Hadamard matrix (H_1 = [1], H_2n = [[H, H], [H, -H]]),
  b in {16, 64, 256};
* computed as the radix-2 fast Walsh-Hadamard butterfly in FP32 with the
  strides taken in ascending order h = 1, 2, 4, ..., b/2, and the
  normalisation 1/sqrt(b) = 2**-(log2(b)/2) applied once at the end (a power
  of two, so exact).

Because every butterfly step is one FP32 add or subtract, this fixed order
makes the rotated values bit-reproducible.
"""
from __future__ import annotations

import numpy as np

BLOCK_SIZES = (16, 64, 256)


def sylvester(b: int) -> np.ndarray:
    """Dense Sylvester Hadamard matrix H_b (entries +-1), float64."""
    if b < 1 or (b & (b - 1)) != 0:
        raise ValueError("b must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < b:
        h = np.block([[h, h], [h, -h]])
    return h


def inv_sqrt_b(b: int) -> np.float32:
    """1/sqrt(b) for b an even power of two (16, 64, 256): itself an exact power of two."""
    lg = int(b).bit_length() - 1
    if lg % 2:
        raise ValueError("b must be an even power of two")
    return np.float32(2.0 ** (-(lg // 2)))


def fwht_blocks(x, b: int) -> np.ndarray:
    """Blockwise FWHT of each row of ``x`` (float32 [M, K], K % b == 0), FP32 butterfly.

    For stride h = 1, 2, ..., b/2 and every index i of a block with (i & h) == 0,
    (v[i], v[i+h]) <- (v[i] + v[i+h], v[i] - v[i+h]); then v <- v / sqrt(b).
    """
    x = np.asarray(x, dtype=np.float32)
    m, k = x.shape
    if k % b:
        raise ValueError("K must be a multiple of the block size")
    v = x.reshape(m, k // b, b).copy()
    h = 1
    while h < b:
        w = v.reshape(m, k // b, b // (2 * h), 2, h)
        lo = w[:, :, :, 0, :]          # indices with (i & h) == 0
        hi = w[:, :, :, 1, :]          # their partners i + h
        s = lo + hi                    # float32 + float32 -> float32 (RNE)
        d = lo - hi
        v = np.stack([s, d], axis=3).reshape(m, k // b, b)
        h *= 2
    return (v * inv_sqrt_b(b)).reshape(m, k).astype(np.float32)


def rotate_dense(x, b: int) -> np.ndarray:
    """The same rotation as a dense float64 product x . blockdiag(H_b)/sqrt(b)."""
    x = np.asarray(x, dtype=np.float64)
    m, k = x.shape
    h = sylvester(b) / np.sqrt(b)
    return (x.reshape(m, k // b, b) @ h).reshape(m, k)
