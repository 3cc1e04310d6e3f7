"""Block statistics that drive the policy (oracle; test infrastructure only).

* Gamma_{t-1}: the "transformation magnitude" of a transformer block, the
  relative difference between its input and output at the previous step
  ("6Bit-Diffusion" technical summary, section 2.A; popular summary,
  section 1).  Reading (the norm is not given): Frobenius,
  Gamma = ||x_out - x_in|| / ||x_in||.
* The residual delta Delta = x_out - x_in that the Temporal Delta Cache keeps
  (technical summary, section 2.B), stored as bf16:
  Delta = bf16(f32(x_out) - f32(x_in)).
* The TDC predictor: similarity of Delta_{t-1} and Delta_{t-2} (technical
  summary, section 2.B; popular summary, section 2).  Reading: cosine
  similarity over the whole block tensor.
* The PDR outlier ratio: max over mean of the block input data (popular
  summary, section 3).  Reading: max|x| / (sum|x| / count) over the whole
  block-input tensor.

Edge cases (readings): sum x_in^2 == 0 -> Gamma = +inf; one Delta norm zero
-> cos = 0, both zero -> cos = 1; sum|x| == 0 -> ratio = 0.
All sums are float64.
"""
from __future__ import annotations

import math

import numpy as np

from .formats import bf16_round


def delta(x_in, x_out) -> np.ndarray:
    """bf16 residual delta, as float32 values."""
    d = np.asarray(x_out, np.float32) - np.asarray(x_in, np.float32)
    return bf16_round(d.astype(np.float32))


def tensor_stats(x):
    """dict(max_abs, sum_abs, sum_sq, count) of a bf16-valued tensor, float64."""
    a = np.abs(np.asarray(x, np.float32).astype(np.float64))
    return dict(max_abs=float(a.max()) if a.size else 0.0, sum_abs=float(a.sum()),
                sum_sq=float((a * a).sum()), count=float(a.size))


def outlier_ratio(ts) -> float:
    if ts["sum_abs"] == 0:
        return 0.0
    return ts["max_abs"] / (ts["sum_abs"] / ts["count"])


def block_stats(x_in, x_out, delta_prev=None):
    """Everything the policy needs from one computed block step.

    Returns dict with delta (bf16 values), the raw sums and the derived
    gamma / cos (cos is None without a previous delta) and the output
    tensor stats (the next block's input stats).
    """
    d = delta(x_in, x_out).astype(np.float64)
    xi = np.asarray(x_in, np.float32).astype(np.float64)
    out = dict(delta=d.astype(np.float32),
               sum_d2=float((d * d).sum()), sum_xin2=float((xi * xi).sum()))
    if delta_prev is not None:
        p = np.asarray(delta_prev, np.float32).astype(np.float64)
        out["sum_ddp"] = float((d * p).sum())
        out["sum_dp2"] = float((p * p).sum())
    out["out"] = tensor_stats(x_out)
    out["gamma"] = gamma(out["sum_d2"], out["sum_xin2"])
    out["cos"] = cosine(out["sum_ddp"], out["sum_d2"], out["sum_dp2"]) if delta_prev is not None else None
    return out


def gamma(sum_d2: float, sum_xin2: float) -> float:
    if sum_xin2 == 0:
        return math.inf
    return math.sqrt(sum_d2) / math.sqrt(sum_xin2)


def cosine(sum_ddp: float, sum_d2: float, sum_dp2: float) -> float:
    if sum_d2 == 0 and sum_dp2 == 0:
        return 1.0
    if sum_d2 == 0 or sum_dp2 == 0:
        return 0.0
    return sum_ddp / math.sqrt(sum_d2 * sum_dp2)


def skip_apply(x_in, delta_cache):
    """TDC skip: the block output is its input plus the cached delta, in bf16."""
    s = np.asarray(x_in, np.float32) + np.asarray(delta_cache, np.float32)
    return bf16_round(s.astype(np.float32))
