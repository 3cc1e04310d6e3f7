"""Reference quantized GEMMs and epilogues (oracle; test infrastructure only).

The quantized activations feed a GEMM with 4-bit weights (W4A4 when the
block runs NVFP4, W4A8 when it runs INT8), and PDR forces an FP16/BF16
recompute ("6Bit-Diffusion" technical summary, sections 2.A, 2.C and 4;
popular summary, sections 1, 3 and 4).  The reference values below are the
plain definitions, evaluated in float64:

  NVFP4:  Y[m,n] = s_tx * s_tw * sum_k a[m,k] * b[n,k],
          a = decode(E2M1 code) * decode(E4M3 block scale)   (same for b)
  INT8:   acc_g[m,n] = sum_{k in group g} qx[m,k] * qw[n,k]   (exact integers)
          Y[m,n] = s_m[m] * sum_g s_w[n,g] * acc_g[m,n]
  BF16:   Y[m,n] = sum_k bf16(x[m,k]) * bf16(w[n,k])

followed by an optional epilogue: GELU(v) = 0.5 v (1 + erf(v / sqrt 2))
(exact-erf reading; the pages do not name the activation) or a residual add.

The tolerance bound that accompanies each reference is
  bound[m,n] = sum_k |a_k * b_k|   (the caller scales it, e.g. by 1e-5).
The matrix products use numpy's float64 matmul as a library primitive.
"""
from __future__ import annotations

import numpy as np
from scipy.special import erfc

from . import formats
from .quant import INT4_GROUP, nvfp4_dequant


def nvfp4_gemm_ref(xcodes, xscales, s_tx, wcodes, wscales, s_tw):
    """(ref, bound) float64 [M, N] for unpacked NVFP4 codes/scales of X [M,K] and W [N,K]."""
    a = nvfp4_dequant(xcodes, xscales, 1.0)
    b = nvfp4_dequant(wcodes, wscales, 1.0)
    s = float(np.float32(s_tx)) * float(np.float32(s_tw))
    ref = s * (a @ b.T)
    bound = abs(s) * (np.abs(a) @ np.abs(b).T)
    return ref, bound


def int8_group_acc(qx, qw):
    """Exact per-group integer accumulators acc[g, m, n] (int64), group size 128."""
    qx = np.asarray(qx, dtype=np.int64)
    qw = np.asarray(qw, dtype=np.int64)
    m, k = qx.shape
    n = qw.shape[0]
    g = k // INT4_GROUP
    acc = np.empty((g, m, n), dtype=np.int64)
    for j in range(g):
        sl = slice(j * INT4_GROUP, (j + 1) * INT4_GROUP)
        acc[j] = qx[:, sl] @ qw[:, sl].T
    return acc


def int8_gemm_ref(qx, s_m, qw, s_w):
    """(ref, bound, acc) for INT8 activations x INT4-g128 weights."""
    acc = int8_group_acc(qx, qw)
    sw = np.asarray(s_w, dtype=np.float32).astype(np.float64)          # [N, G]
    sm = np.asarray(s_m, dtype=np.float32).astype(np.float64)          # [M]
    ref = sm[:, None] * np.einsum("gmn,ng->mn", acc.astype(np.float64), sw)
    absacc = int8_group_acc(np.abs(np.asarray(qx, np.int64)), np.abs(np.asarray(qw, np.int64)))
    bound = np.abs(sm)[:, None] * np.einsum("gmn,ng->mn", absacc.astype(np.float64), np.abs(sw))
    return ref, bound, acc


def bf16_gemm_ref(x, w):
    """(ref, bound) for bf16(x) [M,K] times bf16(w) [N,K] transposed, float64."""
    a = formats.bf16_round(np.asarray(x, np.float32)).astype(np.float64)
    b = formats.bf16_round(np.asarray(w, np.float32)).astype(np.float64)
    return a @ b.T, np.abs(a) @ np.abs(b).T


def gelu(v):
    """Exact-erf GELU in float64, 0.5 v (1 + erf(v / sqrt 2)).

    Evaluated as 0.5 v erfc(-v / sqrt 2), the same function: 1 + erf(z) would
    cancel to 0 for z below about -6 and lose the negative tail entirely.
    """
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * erfc(-v / np.sqrt(2.0))


def epilogue(ref, kind: str, residual=None):
    """Apply 'none' | 'gelu' | 'residual' to a float64 GEMM value."""
    if kind == "none":
        return ref
    if kind == "gelu":
        return gelu(ref)
    if kind == "residual":
        return ref + np.asarray(residual, dtype=np.float32).astype(np.float64)
    raise ValueError(kind)
