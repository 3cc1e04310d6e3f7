"""bench.py's work accounting and roofline arithmetic (CPU only).

A roofline fraction is only as good as its numerator.
- Each call is credited its algorithmic work, not the bytes or FLOPs its
  kernels happen to move:
  - a GEMM: 2·M·N·K FLOP;
  - the INT8 quantizer: 2 B read + 1 B code per element, plus a 4-byte
    row scale;
  - the NVFP4 quantizer: 2 B + 0.5 B codes + 1/16 B scales per element;
  - a block end: x_in and x_out read, Delta_prev read and Delta written
    (8 B per element with a bf16 cache, 6.0625 B with MXFP8);
  - the input statistics: 2 B per element.
- The table and the dominant kernel's roofline divide that work by the
  measured per-call time and by the measured peak of the kernel's own
  dtype (the FP4 one at 6 x bf16).
- The CPU baseline scales the oracle's per-kind block-step time on a token
  sample to the full token count, over the window's actual decisions.

The workload objects are built without a GPU (no __init__): only the
attributes the accounting reads are set.
"""
import os
import sys
from types import SimpleNamespace

import pytest

T, H, F = 17776, 1920, 7680


@pytest.fixture(scope="module")
def bench():
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench as b
    return b


def _dit(bench, delta_bytes=2.0, fused=True):
    wl = object.__new__(bench.DitStep)
    wl.T, wl.H, wl.F = T, H, F
    wl.delta_bytes = delta_bytes
    wl.skip_run_bytes = 123456789
    wl.model = SimpleNamespace(fused_stats=fused)
    wl.name = "dit_2b"
    return wl


def test_dit_gemm_calls_are_credited_2mnk(bench):
    wl = _dit(bench)
    for label in ("qgemm_up", "qgemm_down"):
        for mode, fp4 in (("int8", False), ("bf16", False), ("nvfp4", True)):
            assert wl.work(f"{label}:{mode}") == ("tensor", 2.0 * T * H * F, fp4)


def test_dit_quantizers_are_credited_their_algorithmic_bytes(bench):
    wl = _dit(bench)
    for label, k in (("hq_x", H), ("hq_h", F)):
        n = T * k
        assert wl.work(f"{label}:int8") == ("hbm", 3 * n + 4 * T, False)
        kind, b, fp4 = wl.work(f"{label}:nvfp4")
        assert (kind, fp4) == ("hbm", False) and b == pytest.approx(2.5625 * n, abs=0)
    assert wl.work("hq_h:bf16")[0] is None          # the BF16 path quantizes nothing


def test_dit_block_end_and_statistics_bytes(bench):
    assert _dit(bench).work("block_stats:int8") == ("hbm", 8.0 * T * H, False)
    assert _dit(bench, delta_bytes=1.0 + 1.0 / 32).work("block_stats:int8") == ("hbm", 6.0625 * T * H, False)
    # fused: a BF16 block's statistics come from its down projection's epilogue, so only a fold is left
    assert _dit(bench, fused=True).work("block_stats:bf16")[0] is None
    assert _dit(bench, fused=False).work("block_stats:bf16") == ("hbm", 8.0 * T * H, False)
    assert _dit(bench).work("tensor_stats") == ("hbm", 2 * T * H, False)
    assert _dit(bench).work("skip_run") == ("hbm", 123456789, False)
    assert _dit(bench).work("qgemm_up:skip")[0] is None


def test_roofline_divides_work_by_time_and_the_dtype_peak(bench):
    wl = _dit(bench)
    peaks = {"bf16": 2000.0, "hbm": 8000.0, "src": "measured"}
    per = {  # per-call milliseconds
        "qgemm_up:int8": [0.50, 0.52],          # the largest total: the dominant kernel
        "qgemm_down:nvfp4": [0.20],
        "hq_h:int8": [0.10, 0.10],
        "block_stats:bf16": [0.01],             # no work credited: in the table, no rate
    }
    roof, table = bench._roofline(wl, per, peaks)
    flops = 2.0 * T * H * F
    ach = flops / (0.51 / 1e3) / 1e12
    assert roof["kernel"] == "qgemm_up:int8" and roof["bound"] == "tensor"
    assert roof["achieved"] == pytest.approx(ach, abs=0.05)
    assert roof["frac"] == pytest.approx(ach / 2000.0, abs=1e-4)
    assert roof["work_per_launch"] == flops
    fp4 = table["qgemm_down:nvfp4"]
    assert fp4["frac"] == pytest.approx(flops / 0.2e-3 / 1e12 / (2000.0 * bench.FP4_OVER_BF16), abs=1e-4)
    q = table["hq_h:int8"]
    assert q["gbs"] == pytest.approx((3 * T * F + 4 * T) / 0.1e-3 / 1e9, abs=0.05)
    assert q["frac"] == pytest.approx(q["gbs"] / 8000.0, abs=1e-4)
    assert "frac" not in table["block_stats:bf16"] and table["block_stats:bf16"]["calls"] == 1
    assert bench.FP4_OVER_BF16 == pytest.approx(13.5 / 2.25)


def test_cpu_baseline_extrapolates_over_the_decision_trace(bench):
    """The oracle's rate is its per-kind block-step time on a token sample, scaled to the full token
    count and summed over each step's actual decisions: here steps of 2.5 s and 1 s on 32 rows, run
    on 64 tokens (x 2), give 2 steps / 7 s."""
    costs = {"int8": 2.0, "nvfp4": 1.5, "bf16": 3.0, "skip": 0.5}
    trace = [["int8", "skip"], ["skip", "skip"]]
    assert bench._dit_rate(costs, trace, tokens=64, rows=32) == pytest.approx(2 / 7, rel=1e-15)
    # every block computing in INT8 (the reference arm's extrapolation)
    assert bench._dit_rate(costs, [["int8"] * 30], tokens=17776, rows=32) == pytest.approx(
        1 / (30 * 2.0 * 17776 / 32), rel=1e-15)
    # the bench's mode names are the cost table's keys
    assert {bench.MODE_NAMES[k] for k in (1, 2, 3, 4)} == set(costs)
