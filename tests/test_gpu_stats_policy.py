"""Parity: block statistics, delta cache, skip and the device policy step vs the oracle.

Bar: bit-exact delta / skip outputs and maxima.  Sums, against the float64
oracle: the three behind the delta cosine (sum Delta^2, Delta*Delta_prev,
Delta_prev^2) within 1e-9 * sum|terms| (each thread keeps a TwoSum pair;
partials combine as float-float pairs, ~44 bits); the Kahan-compensated sums for Gamma and the outlier ratio
(sum x_in^2, sum |x|, sum x^2) within 2.5e-7 * sum|terms| (Kahan's bound 2u
per thread partial; the policy compares these statistics to thresholds with a
1e-6 relative band, so 2.4e-7 cannot flip a decision outside it).  Policy
decisions identical to the oracle's on the hand traces and random statistics.
"""
import math
import os

import numpy as np
import pytest
import torch

import synthgen
from oracle import policy, stats
from oracle.formats import bf16_round

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def ops():
    from video_dit_mixed_gb300 import ops as o
    return o


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _np_bits(a):
    return (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16).view(np.int16)


def _close(got, ref, absterms, what, rel=1e-9):
    assert abs(got - ref) <= rel * absterms + 1e-300, (what, got, ref, absterms)


KAHAN = 2.5e-7


SIZES = [8, 8 * 1000 + 8, 1920 * 257, 17776 * 1920]


@pytest.mark.parametrize("n", SIZES)
def test_tensor_stats(ops, n):
    x = synthgen.activations(9, 1, n, "laplace", 0.0, 1.0).reshape(-1)
    out = torch.zeros(4, dtype=torch.float64, device="cuda")
    ops.tensor_stats(_dev_bf16(x), out, ops.new_scratch(n))
    r = stats.tensor_stats(x)
    g = out.cpu().numpy()
    assert g[0] == r["max_abs"] and g[2] == n
    _close(g[1], r["sum_abs"], r["sum_abs"], "sum_abs", KAHAN)
    _close(g[3], r["sum_sq"], r["sum_sq"], "sum_sq", KAHAN)


@pytest.mark.parametrize("n", SIZES)
def test_block_stats_and_delta_cache(ops, n):
    xi = synthgen.activations(11, 1, n, "laplace", 0.0, 1.0).reshape(-1)
    xo = bf16_round(xi + synthgen.normal(12, 1, n).astype(np.float32) * 0.3)
    dp = bf16_round(synthgen.normal(13, 1, n).astype(np.float32) * 0.3)
    cache = _dev_bf16(dp)
    st = ops.new_stats()
    scratch = ops.new_scratch(n)
    for _ in range(2):   # the scratch counter must come back to zero after each call
        cache.copy_(_dev_bf16(dp))
        ops.block_stats(_dev_bf16(xi), _dev_bf16(xo), cache, st, scratch)
        torch.cuda.synchronize()
    r = stats.block_stats(xi, xo, dp)
    np.testing.assert_array_equal(_bits(cache), _np_bits(r["delta"]))
    g = st.cpu().numpy()[0]
    d = r["delta"].astype(np.float64)
    p = dp.astype(np.float64)
    _close(g[0], r["sum_d2"], r["sum_d2"], "sum_d2")
    _close(g[1], r["sum_xin2"], r["sum_xin2"], "sum_xin2", KAHAN)
    _close(g[2], r["sum_ddp"], float(np.abs(d * p).sum()), "sum_ddp")
    _close(g[3], r["sum_dp2"], r["sum_dp2"], "sum_dp2")
    assert g[4] == r["out"]["max_abs"] and g[6] == n
    _close(g[5], r["out"]["sum_abs"], r["out"]["sum_abs"], "sum_abs_out", KAHAN)


def test_skip_apply(ops):
    n = 17776 * 1920 // 16
    xi = synthgen.activations(21, 1, n, "laplace", 0.0, 1.0).reshape(-1)
    d = bf16_round(synthgen.normal(22, 1, n).astype(np.float32) * 0.1)
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    st = ops.new_stats()
    st[0, :4] = torch.tensor([1.0, 2.0, 3.0, 4.0], dtype=torch.float64)
    ops.skip_apply(_dev_bf16(xi), _dev_bf16(d), out, st, ops.new_scratch(n))
    torch.cuda.synchronize()
    ref = stats.skip_apply(xi, d)
    np.testing.assert_array_equal(_bits(out), _np_bits(ref))
    g = st.cpu().numpy()[0]
    assert list(g[:4]) == [1.0, 2.0, 3.0, 4.0]          # compute-side fields untouched
    t = stats.tensor_stats(ref)
    assert g[4] == t["max_abs"] and g[6] == n
    _close(g[5], t["sum_abs"], t["sum_abs"], "sum_abs", KAHAN)


def test_mode_word_gates_stats_and_skip(ops):
    n = 4096
    xi = _dev_bf16(synthgen.activations(31, 1, n, "normal", 0.0, 1.0).reshape(-1))
    cache = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    st = ops.new_stats()
    sc = ops.new_scratch(n)
    skip = torch.tensor([4], dtype=torch.int32, device="cuda")
    comp = torch.tensor([2], dtype=torch.int32, device="cuda")
    ops.block_stats(xi, xi, cache, st, sc, mode_dev=skip)      # skipped block: no stats
    ops.skip_apply(xi, cache, out, st, sc, mode_dev=comp)      # computed block: no skip
    torch.cuda.synchronize()
    assert not bool(st.any()) and not bool(out.float().any())


def _stats_row(gamma, cos):
    """A sixbit_stats record whose folded Gamma / cos are the given values.

    Gamma = sqrt(sum_d2) / sqrt(sum_xin2) and cos = sum_ddp / sqrt(sum_d2 * sum_dp2),
    so sum_d2 = gamma^2, sum_xin2 = 1, sum_dp2 = 1 / gamma^2, sum_ddp = cos.
    """
    return [gamma * gamma, 1.0, cos, 1.0 / (gamma * gamma), 0.0, 0.0, 0.0, 0.0]


def _traces():
    out = {}
    for line in open(os.path.join(GOLDEN, "policy_traces.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        t, cap, rb, step, ratio, g, c, exp, flags = line.split()
        out.setdefault(t, dict(cap=float(cap), rb=bool(int(rb)), steps=[]))
        out[t]["steps"].append(dict(ratio=float(ratio), gamma=None if g == "-" else float(g),
                                    cos=None if c == "-" else float(c), expect=exp, flags=flags))
    return out


def _run_device_trace(ops, cfg, steps, state=None):
    state = ops.new_policy_state() if state is None else state
    last = ops.new_stats()
    ins = torch.zeros(3, dtype=torch.float64, device="cuda")
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = []
    for s in steps:
        ins.copy_(torch.tensor([s["ratio"], 1.0, 1.0], dtype=torch.float64))
        ops.policy_step(cfg, state, last, ins, word)
        w = int(word.item())
        got.append(w)
        if (w & 0xFF) != ops.MODE_SKIP:
            g = s["gamma"] if s["gamma"] is not None else 0.5
            c = s["cos"] if s["cos"] is not None else 0.0
            last.copy_(torch.tensor([_stats_row(g, c)], dtype=torch.float64))
    return got


@pytest.mark.parametrize("name", ["A", "B", "C", "D"])
def test_device_policy_hand_traces(ops, name):
    tr = _traces()[name]
    cfg = ops.policy_cfg(err_cap=tr["cap"], refresh_bf16=tr["rb"])
    got = _run_device_trace(ops, cfg, tr["steps"])
    names = {1: "NVFP4", 2: "INT8", 3: "BF16", 4: "SKIP"}
    assert [names[w & 0xFF] for w in got] == [s["expect"] for s in tr["steps"]]
    for w, s in zip(got, tr["steps"]):
        flags = set()
        if w & ops.abi.FLAG_REFRESH:
            flags.add("refresh")
        if w & ops.abi.FLAG_PDR:
            flags.add("pdr")
        if w & ops.abi.FLAG_POSTSKIP:
            flags.add("post_skip")
        assert flags == (set() if s["flags"] == "-" else set(s["flags"].split(",")))


def test_device_policy_matches_oracle_on_random_statistics(ops):
    u = synthgen.uniform(99, 3, 4 * 400).reshape(400, 4)
    steps = []
    for a, b, c, d in u:
        steps.append(dict(ratio=10 + 30 * a, gamma=0.2 * b, cos=0.97 + 0.03 * c))
    cfg = policy.PolicyConfig()
    ref = policy.run_trace([dict(s) for s in steps], cfg)
    # the oracle folds gamma, cos exactly; feed the device the same through sums
    got = _run_device_trace(ops, ops.policy_cfg(), [dict(s) for s in steps])
    names = {1: "NVFP4", 2: "INT8", 3: "BF16", 4: "SKIP"}
    mism = [(i, r.mode, names[g & 0xFF]) for i, (r, g) in enumerate(zip(ref, got)) if r.mode != names[g & 0xFF]
            and not r.near]
    assert not mism, mism[:5]
    assert {r.mode for r in ref} == {"NVFP4", "INT8", "BF16", "SKIP"}


def test_device_policy_nan_statistics(ops):
    """A statistic that is not a number fails its threshold test toward the safer path, as in the oracle: a NaN
    cosine never skips, a NaN Gamma picks INT8 (not NVFP4), a NaN input ratio picks BF16 with the PDR flag; the
    state counts the decisions taken on a NaN statistic (n_nonfinite)."""
    nan = float("nan")
    steps = [dict(ratio=12.0, gamma=0.04, cos=None),    # INT8 (first step)
             dict(ratio=12.0, gamma=nan, cos=nan),      # NVFP4 (Gamma 0.04); its own statistics are NaN
             dict(ratio=12.0, gamma=0.04, cos=0.98),    # NaN cosine and Gamma: INT8, counted
             dict(ratio=nan, gamma=0.04, cos=0.995),    # NaN ratio: BF16 + PDR, counted
             dict(ratio=12.0, gamma=None, cos=None),    # SKIP
             dict(ratio=12.0, gamma=None, cos=None)]    # SKIP
    ref = policy.run_trace([dict(s) for s in steps], policy.PolicyConfig())
    state = ops.new_policy_state()
    got = _run_device_trace(ops, ops.policy_cfg(), [dict(s) for s in steps], state=state)
    names = {1: "NVFP4", 2: "INT8", 3: "BF16", 4: "SKIP"}
    assert [names[w & 0xFF] for w in got] == [r.mode for r in ref] == ["INT8", "NVFP4", "INT8", "BF16", "SKIP",
                                                                       "SKIP"]
    assert [bool(w & ops.abi.FLAG_PDR) for w in got] == [r.pdr for r in ref]
    st = ops.decode_state(state[0])
    assert st.n_nonfinite == 2 and st.n_pdr == 1 and st.n_skip == 2
