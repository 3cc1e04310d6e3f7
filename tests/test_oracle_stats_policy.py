"""Pins for the oracle's block statistics and policy (CPU only)."""
import math
import os

import numpy as np
import pytest

from oracle import policy, stats
from oracle.formats import bf16_round

F32 = np.float32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_gamma_of_scaled_block_is_exact():
    rng = np.random.default_rng(0)
    x = bf16_round(rng.standard_normal((16, 32)).astype(F32))
    s = stats.block_stats(x, (2 * x).astype(F32))
    assert s["gamma"] == 1.0
    np.testing.assert_array_equal(s["delta"], x)
    assert math.isclose(s["sum_xin2"], float(np.linalg.norm(x.astype(np.float64)) ** 2), rel_tol=1e-12)


def test_cosine_special_cases():
    rng = np.random.default_rng(1)
    x = bf16_round(rng.standard_normal((8, 32)).astype(F32))
    d = bf16_round(rng.standard_normal((8, 32)).astype(F32))
    xo = bf16_round(x + d)
    dd = stats.delta(x, xo)
    assert math.isclose(stats.block_stats(x, xo, dd)["cos"], 1.0, rel_tol=1e-15)
    assert math.isclose(stats.block_stats(x, xo, -dd)["cos"], -1.0, rel_tol=1e-15)
    e1 = np.zeros((1, 4), F32); e1[0, 0] = 1
    e2 = np.zeros((1, 4), F32); e2[0, 1] = 1
    assert stats.block_stats(np.zeros((1, 4), F32), e1, e2)["cos"] == 0.0
    assert stats.cosine(0.0, 0.0, 0.0) == 1.0
    assert stats.cosine(0.0, 0.0, 2.0) == 0.0
    assert stats.gamma(1.0, 0.0) == math.inf


def test_delta_is_rounded_to_bf16():
    x_in = np.array([[1.0, 1.0, 256.0]], F32)
    x_out = np.array([[1.0 + 2 ** -7, 258.0, 1.0]], F32)
    # 2^-7 exact; 257 is a tie between 256 and 258 -> 256; -255 exact
    np.testing.assert_array_equal(stats.delta(x_in, x_out), [[2 ** -7, 256.0, -255.0]])


def test_outlier_ratio():
    x = np.ones((4, 8), F32)
    assert stats.outlier_ratio(stats.tensor_stats(x)) == 1.0
    x = np.zeros((4, 8), F32); x[1, 2] = -3
    assert stats.outlier_ratio(stats.tensor_stats(x)) == 32.0
    assert stats.outlier_ratio(stats.tensor_stats(np.zeros((2, 2), F32))) == 0.0


def test_skip_apply_rounds_once():
    x = np.array([[1.0, 256.0]], F32)
    d = np.array([[2 ** -8, 1.0]], F32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> 1; 257 tie -> 256
    np.testing.assert_array_equal(stats.skip_apply(x, d), [[1.0, 256.0]])


def _traces():
    out = {}
    for line in open(os.path.join(GOLDEN, "policy_traces.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        t, cap, rb, step, ratio, g, c, exp, flags = line.split()
        out.setdefault(t, dict(cfg=policy.PolicyConfig(err_cap=float(cap), refresh_bf16=bool(int(rb))), steps=[]))
        st = dict(ratio=float(ratio), expect=exp, flags=set() if flags == "-" else set(flags.split(",")))
        if g != "-":
            st["gamma"] = float(g)
        if c != "-":
            st["cos"] = float(c)
        out[t]["steps"].append(st)
    return out


@pytest.mark.parametrize("name", ["A", "B", "C", "D"])
def test_policy_hand_traces(name):
    tr = _traces()[name]
    got = policy.run_trace(tr["steps"], tr["cfg"])
    assert [d.mode for d in got] == [s["expect"] for s in tr["steps"]]
    for d, s in zip(got, tr["steps"]):
        flags = {f for f in ("refresh", "pdr", "post_skip") if getattr(d, f)}
        assert flags == s["flags"], (name, d, s)


def test_policy_first_two_computes_never_skip():
    steps = [dict(ratio=1, gamma=0.01, cos=1.0)] * 2 + [dict(ratio=1)]
    got = policy.run_trace(steps)
    assert [d.mode for d in got] == ["INT8", "NVFP4", "SKIP"]


def test_policy_near_threshold_flag():
    cfg = policy.PolicyConfig()
    steps = [dict(ratio=30.0 * (1 + 5e-7), gamma=0.2)]
    got = policy.run_trace(steps, cfg)
    assert got[0].mode == "BF16" and got[0].near
    got = policy.run_trace([dict(ratio=29.0, gamma=0.2)], cfg)
    assert not got[0].near


# A statistic that is not a number fails its threshold test toward the safer path.
NAN = float("nan")
NAN_TRACE = [   # (ratio, gamma, cos of the step's own compute), expected mode, pdr
    (12.0, 0.04, None, "INT8", False),   # first step
    (12.0, NAN, NAN, "NVFP4", False),    # decided on Gamma 0.04; this compute's statistics are NaN
    (12.0, 0.04, 0.98, "INT8", False),   # NaN cosine: no skip; NaN Gamma: INT8, not NVFP4
    (NAN, 0.04, 0.995, "BF16", True),    # NaN input ratio: BF16 with the PDR flag
    (12.0, None, None, "SKIP", False),   # cos 0.995, acc 0.005 <= 0.05
    (12.0, None, None, "SKIP", False),   # acc 0.010 <= 0.05
]


def test_policy_nan_statistics_take_the_safer_path():
    steps = [dict(ratio=r, gamma=g, cos=c) for r, g, c, _, _ in NAN_TRACE]
    got = policy.run_trace(steps, policy.PolicyConfig())
    assert [d.mode for d in got] == [m for *_, m, _ in NAN_TRACE]
    assert [d.pdr for d in got] == [p for *_, p in NAN_TRACE]


def test_policy_nan_statistics_single_steps():
    cfg = policy.PolicyConfig()
    st = policy.PolicyState(n_computed=2, have_gamma=True, gamma=NAN, cos=0.5)
    assert policy.decide(st, 12.0, cfg).mode == "INT8"       # volatile without a usable Gamma
    st = policy.PolicyState(n_computed=2, have_gamma=True, gamma=0.01, cos=NAN)
    assert policy.decide(st, 12.0, cfg).mode == "NVFP4"      # no skip on a NaN cosine; Gamma decides
    st = policy.PolicyState(n_computed=2, have_gamma=True, gamma=0.01, cos=0.5)
    d = policy.decide(st, NAN, cfg)
    assert d.mode == "BF16" and d.pdr
    st = policy.PolicyState(n_computed=2, have_gamma=True, gamma=0.01, cos=0.5)
    assert policy.decide(st, 30.0, cfg).mode == "NVFP4"      # finite values: unchanged (ratio 30 is not > 30)
