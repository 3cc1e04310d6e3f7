"""Parity: a block's statistics produced by its down projection's epilogue vs the oracle.

sixbit_qgemm_blockstats is the GEMM with the residual epilogue that also
writes Delta = bf16(x_out - x_in) over Delta_prev and the block statistics'
partial rows, which sixbit_block_stats_parts folds.  Bar, against the float64
oracle (oracle/stats.block_stats) evaluated on the GPU's own x_out, the
residual x_in and Delta_prev: Delta bit-exact; the maximum exact; the sums
behind the cosine (sum Delta^2, Delta Delta_prev, Delta_prev^2) within
1e-9 sum|terms| and the Kahan-compensated ones (sum x_in^2, sum |x_out|)
within 2.5e-7 sum|terms|, the bars of the separate statistics pass.  Y is
bit-identical to sixbit_qgemm's, and the folded totals are bit-identical
between two runs (the partial rows sit at fixed places and fold in a fixed
order).  Shapes span ragged M and N (N % 32 == 16 ends in half a 32-column
chunk), K of one and several 128-wide groups, each GEMM kind, and the
dit_2b down projection at full size.
"""
import numpy as np
import pytest
import torch

import synthgen
from oracle import stats
from oracle.formats import bf16_round

pytestmark = pytest.mark.gpu
MODES = {"nvfp4": 1, "int8": 2, "bf16": 3}
KAHAN = 2.5e-7


@pytest.fixture(scope="module")
def ops():
    from video_dit_mixed_gb300 import ops as o
    return o


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


def _f32(t):
    return t.float().cpu().numpy()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def _np_bits(a):
    return (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16).view(np.int16)


def _close(got, ref, absterms, what, rel=1e-9):
    assert abs(got - ref) <= rel * absterms + 1e-300, (what, got, ref, absterms)


def _setup(ops, mode, m, n, k, b, seed):
    x = synthgen.activations(seed, m, k, "laplace", 0.005, 50.0)
    w = synthgen.weights(seed + 1, n, k)
    xi = bf16_round(synthgen.activations(seed + 2, m, n, "normal", 0.0, 1.0))
    dp = bf16_round(synthgen.normal(seed + 3, 1, m * n).astype(np.float32).reshape(m, n) * 0.3)
    xd = _dev_bf16(x)
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    qa = ops.hadamard_quant(xd, b, MODES[mode]) if mode != "bf16" else None
    return xd, pw, qa, xi, dp


def _fused(ops, mode, xd, pw, qa, xi_d, dp, m, n, mode_dev=None):
    y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    cache = _dev_bf16(dp).reshape(-1)
    parts = ops.new_blockstats_parts()
    ops.qgemm_blockstats(qa, xd, pw, 0 if mode_dev is not None else MODES[mode], residual=xi_d, out=y,
                         delta_cache=cache, parts=parts, m=m, mode_dev=mode_dev)
    st = ops.new_stats()
    ops.block_stats_parts(parts, m * n, st)
    torch.cuda.synchronize()
    return y, cache, st.cpu().numpy()[0]


def _check_against_oracle(y, cache, g, xi, dp, m, n):
    xo = _f32(y).reshape(-1)
    r = stats.block_stats(xi.reshape(-1), xo, dp.reshape(-1))
    np.testing.assert_array_equal(_bits(cache), _np_bits(r["delta"]))
    d = r["delta"].astype(np.float64)
    p = dp.reshape(-1).astype(np.float64)
    _close(g[0], r["sum_d2"], r["sum_d2"], "sum_d2")
    _close(g[1], r["sum_xin2"], r["sum_xin2"], "sum_xin2", KAHAN)
    _close(g[2], r["sum_ddp"], float(np.abs(d * p).sum()), "sum_ddp")
    _close(g[3], r["sum_dp2"], r["sum_dp2"], "sum_dp2")
    assert g[4] == r["out"]["max_abs"]
    assert g[6] == m * n
    _close(g[5], r["out"]["sum_abs"], r["out"]["sum_abs"], "sum_abs_out", KAHAN)


SHAPES = [(200, 144, 384, 64), (129, 256, 1920, 64), (300, 640, 256, 16), (1, 16, 128, 16), (1000, 1920, 768, 64)]


@pytest.mark.parametrize("mode", ["nvfp4", "int8", "bf16"])
@pytest.mark.parametrize("m,n,k,b", SHAPES)
def test_epilogue_block_stats(ops, mode, m, n, k, b):
    xd, pw, qa, xi, dp = _setup(ops, mode, m, n, k, b, 3000 + m + n)
    xi_d = _dev_bf16(xi)
    y_ref = ops.qgemm(qa, xd, pw, MODES[mode], epilogue=ops.EPI_RESIDUAL, residual=xi_d, m=m)
    y, cache, g = _fused(ops, mode, xd, pw, qa, xi_d, dp, m, n)
    np.testing.assert_array_equal(_bits(y), _bits(y_ref))
    _check_against_oracle(y, cache, g, xi, dp, m, n)
    _, _, g2 = _fused(ops, mode, xd, pw, qa, xi_d, dp, m, n)
    np.testing.assert_array_equal(g, g2)


@pytest.mark.parametrize("mode", ["int8", "bf16", "nvfp4"])
def test_epilogue_block_stats_dit2b_down_projection(ops, mode):
    """The dit_2b down projection: x_in 17776 x 1920, h 17776 x 7680."""
    m, n, k = 17776, 1920, 7680
    xd, pw, qa, xi, dp = _setup(ops, mode, m, n, k, 64, 4100)
    y, cache, g = _fused(ops, mode, xd, pw, qa, _dev_bf16(xi), dp, m, n)
    _check_against_oracle(y, cache, g, xi, dp, m, n)


def test_epilogue_block_stats_mode_gated(ops):
    """With a device mode word, only the matching kind runs (and writes the partial rows);
    a SKIP word leaves the output and the Delta cache untouched."""
    m, n, k = 256, 384, 512
    xd, pw, qa, xi, dp = _setup(ops, "int8", m, n, k, 64, 4200)
    xi_d = _dev_bf16(xi)
    word = torch.tensor([MODES["int8"]], dtype=torch.int32, device="cuda")
    y, cache, g = _fused(ops, "int8", xd, pw, qa, xi_d, dp, m, n, mode_dev=word)
    _check_against_oracle(y, cache, g, xi, dp, m, n)
    word.fill_(4)   # SKIP
    y = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
    cache = _dev_bf16(dp).reshape(-1)
    ops.qgemm_blockstats(qa, xd, pw, 0, residual=xi_d, out=y, delta_cache=cache, parts=ops.new_blockstats_parts(),
                         m=m, mode_dev=word)
    torch.cuda.synchronize()
    assert not y.any()
    np.testing.assert_array_equal(_bits(cache), _np_bits(dp.reshape(-1)))
