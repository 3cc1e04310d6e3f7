"""Parity: the MXFP8 Delta cache (block statistics, skip, the DiT step protocol) vs the oracle.

Bar: the cache's E4M3 codes and E8M0 scales bit-exact against the oracle's
MXFP8 encoding of bf16(x_out - x_in); skip outputs and maxima bit-exact; the
sums as for the bf16 cache (the cosine's three within 1e-9 of the sum of
|terms|, the Kahan-compensated ones within 2.5e-7), with the previous Delta
dequantized by the oracle.  Sizes span one MX block, a ragged grid, several
waves and the 17776 x 1920 activation; the inputs plant all-zero blocks,
blocks below E8M0's range (scale clamped, bf16 subnormals), saturating
blocks and negative values that round to zero.
"""
import numpy as np
import pytest
import torch

import synthgen
from oracle import formats, stats
from oracle.formats import bf16_round

pytestmark = pytest.mark.gpu
KAHAN = 2.5e-7


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


def _planted(seed, n):
    """x_in, x_out (bf16 values) whose Delta has the special blocks planted (when n allows)."""
    xi = synthgen.activations(seed, 1, n, "laplace", 0.0, 1.0).reshape(-1)
    xo = bf16_round(xi + synthgen.normal(seed + 1, 1, n).astype(np.float32) * 0.3)
    nb = n // 32
    if nb >= 8:
        blk = lambda b: slice(32 * b, 32 * b + 32)  # noqa: E731
        xo[blk(1)] = xi[blk(1)]                                      # Delta = 0
        xi[blk(2)] = 0.0
        xo[blk(2)] = np.float32(2.0 ** -130) * np.arange(32)       # bf16 subnormals: scale clamped to 2^-127
        xi[blk(3)] = 0.0
        xo[blk(3)] = 1.0
        xo[32 * 3] = 500.0                                           # saturates: 500 -> 448
        xo[32 * 3 + 1] = -500.0
        xi[blk(4)] = 0.0
        xo[blk(4)] = -(2.0 ** -12)                                   # rounds to -0 beside a large element
        xo[32 * 4] = 256.0
        xo = bf16_round(xo)
    return xi, xo


def _enc(d):
    return formats.mxfp8_encode(np.asarray(d, np.float32).reshape(-1))


SIZES = [32, 32 * 1001, 1920 * 257, 17776 * 1920]


@pytest.mark.parametrize("n", SIZES)
def test_block_stats_mxfp8(ops, n):
    xi, xo = _planted(11, n)
    dprev = bf16_round(synthgen.normal(13, 1, n).astype(np.float32) * 0.3)
    pc, ps = _enc(dprev)
    prev = formats.mxfp8_decode(pc, ps).astype(np.float32)
    codes = torch.from_numpy(pc).cuda()
    scales = torch.from_numpy(ps).cuda()
    st = ops.new_stats()
    scratch = ops.new_scratch(n)
    xid, xod = _dev_bf16(xi), _dev_bf16(xo)
    for _ in range(2):   # the scratch counter must come back to zero after each call
        codes.copy_(torch.from_numpy(pc))
        scales.copy_(torch.from_numpy(ps))
        ops.block_stats_mxfp8(xid, xod, codes, scales, st, scratch)
        torch.cuda.synchronize()
    r = stats.block_stats(xi, xo, prev)
    wc, ws = _enc(r["delta"])
    np.testing.assert_array_equal(scales.cpu().numpy(), ws)
    np.testing.assert_array_equal(codes.cpu().numpy(), wc)
    g = st.cpu().numpy()[0]
    d = r["delta"].astype(np.float64)
    p = prev.astype(np.float64)
    _close(g[0], r["sum_d2"], r["sum_d2"], "sum_d2")
    _close(g[1], r["sum_xin2"], r["sum_xin2"], "sum_xin2", KAHAN)
    _close(g[2], r["sum_ddp"], float(np.abs(d * p).sum()), "sum_ddp")
    _close(g[3], r["sum_dp2"], r["sum_dp2"], "sum_dp2")
    assert g[4] == r["out"]["max_abs"] and g[6] == n
    _close(g[5], r["out"]["sum_abs"], r["out"]["sum_abs"], "sum_abs_out", KAHAN)


@pytest.mark.parametrize("n", [32, 32 * 1001, 17776 * 1920 // 16])
def test_skip_apply_mxfp8(ops, n):
    xi = synthgen.activations(21, 1, n, "laplace", 0.0, 1.0).reshape(-1)
    _, dv = _planted(22, n)
    dc, ds = _enc(bf16_round(dv * np.float32(0.1)))
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    st = ops.new_stats()
    st[0, :4] = torch.tensor([1.0, 2.0, 3.0, 4.0], dtype=torch.float64)
    ops.skip_apply_mxfp8(_dev_bf16(xi), torch.from_numpy(dc).cuda(), torch.from_numpy(ds).cuda(), out, st,
                         ops.new_scratch(n))
    torch.cuda.synchronize()
    ref = stats.skip_apply(xi, formats.mxfp8_decode(dc, ds).astype(np.float32))
    np.testing.assert_array_equal(_bits(out), _np_bits(ref))
    g = st.cpu().numpy()[0]
    assert list(g[:4]) == [1.0, 2.0, 3.0, 4.0]          # compute-side fields untouched
    t = stats.tensor_stats(ref)
    assert g[4] == t["max_abs"] and g[6] == n
    _close(g[5], t["sum_abs"], t["sum_abs"], "sum_abs", KAHAN)


def test_mode_word_gates_the_mxfp8_calls(ops):
    n = 4096
    xi = _dev_bf16(synthgen.activations(31, 1, n, "normal", 0.0, 1.0).reshape(-1))
    codes, scales = ops.mxfp8_cache(n, "cuda")
    out = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    st = ops.new_stats()
    sc = ops.new_scratch(n)
    skip = torch.tensor([4], dtype=torch.int32, device="cuda")
    comp = torch.tensor([2], dtype=torch.int32, device="cuda")
    ops.block_stats_mxfp8(xi, out, codes, scales, st, sc, mode_dev=skip)
    ops.skip_apply_mxfp8(xi, codes, scales, out, st, sc, mode_dev=comp)
    torch.cuda.synchronize()
    assert not bool(st.any()) and not bool(out.float().any()) and not bool(codes.any())


def _states(ops, L, skipping, cos=0.999):
    raw = ops.new_policy_state("cuda", L)
    host = []
    for l in range(L):
        s = ops.PolicyState()
        if l in skipping:
            s.n_computed, s.have_gamma, s.cos, s.gamma = 2, 1, cos, 0.5
        host.append(bytes(s))
    raw.copy_(torch.frombuffer(bytearray(b"".join(host)), dtype=torch.uint8).view(L, 80))
    return raw


@pytest.mark.parametrize("L,skipping", [(6, {1, 2, 3}), (6, set(range(6))), (40, set(range(1, 38))),
                                        (40, set(range(0, 33)) | {35, 36})])
def test_protocol_with_mxfp8_cache_matches_sequential_calls(ops, L, skipping):
    """sixbit_dit_block_end / _skip_run on an MXFP8 cache against one policy step plus
    sixbit_skip_apply_mxfp8 or sixbit_block_stats_mxfp8 per block: bit-identical decisions,
    states, activations, caches and statistics over three steps."""
    n = 8 * 1536
    g = torch.Generator(device="cuda").manual_seed(7)
    x0 = (torch.randn(n, device="cuda", generator=g) * 3).to(torch.bfloat16)
    d0 = bf16_round((np.random.default_rng(8).normal(size=(L, n)) * 0.05).astype(np.float32))
    enc = [_enc(d0[l]) for l in range(L)]
    codes0 = torch.from_numpy(np.stack([e[0] for e in enc])).cuda()
    scales0 = torch.from_numpy(np.stack([e[1] for e in enc])).cuda()
    bumps = [torch.randn(n, device="cuda", generator=g) * 0.2 for _ in range(L)]
    cfg = ops.policy_cfg()
    scratch = ops.new_scratch(n)

    st_a, stats_a = _states(ops, L, skipping), ops.new_stats("cuda", L)
    modes_a = torch.zeros(L, dtype=torch.int32, device="cuda")
    bufs_a = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    codes_a, scales_a = codes0.clone(), scales0.clone()
    tstats_a = torch.zeros(4, dtype=torch.float64, device="cuda")
    st_b, stats_b = _states(ops, L, skipping), ops.new_stats("cuda", L)
    modes_b = torch.zeros(L, dtype=torch.int32, device="cuda")
    bufs_b = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    codes_b, scales_b = codes0.clone(), scales0.clone()
    tstats_b = torch.zeros(4, dtype=torch.float64, device="cuda")
    run_len = torch.zeros(L, dtype=torch.int32, device="cuda")
    rec = ops.dit_blocks(st_b, stats_b, modes_b, run_len, tstats_b, x0, bufs_b[0], bufs_b[1], codes_b,
                         delta_scales=scales_b)
    for step in range(3):
        ops.tensor_stats(x0, tstats_a, scratch)
        x = x0
        for l in range(L):
            ins = tstats_a if l == 0 else stats_a[l - 1, 4:7]
            ops.policy_step(cfg, st_a[l], stats_a[l], ins, modes_a[l:l + 1])
            out = bufs_a[l % 2]
            if int(modes_a[l].item()) & 0xFF == ops.MODE_SKIP:
                ops.skip_apply_mxfp8(x, codes_a[l], scales_a[l], out, stats_a[l], scratch)
            else:
                out.copy_((x.float() + bumps[l]).to(torch.bfloat16))
                ops.block_stats_mxfp8(x, out, codes_a[l], scales_a[l], stats_a[l], scratch)
            x = out
        ops.dit_begin(cfg, rec, scratch)
        xb = x0
        for l in range(L):
            out = bufs_b[l % 2]
            if int(modes_b[l].item()) & 0xFF != ops.MODE_SKIP:
                out.copy_((xb.float() + bumps[l]).to(torch.bfloat16))
            ops.dit_block_end(cfg, rec, l, scratch)
            ops.dit_skip_run(cfg, rec, l, scratch)
            xb = out
        torch.cuda.synchronize()
        np.testing.assert_array_equal(modes_a.cpu().numpy(), modes_b.cpu().numpy())
        np.testing.assert_array_equal(st_a.cpu().numpy(), st_b.cpu().numpy())
        assert torch.equal(x.view(torch.int16), xb.view(torch.int16)), step
        assert torch.equal(codes_a, codes_b) and torch.equal(scales_a, scales_b), step
        assert not run_len.any()
        low = modes_a.cpu().numpy() & 0xFF
        for l in range(L):
            if low[l] != ops.MODE_SKIP:
                np.testing.assert_array_equal(stats_a[l].cpu().numpy(), stats_b[l].cpu().numpy())
            elif l == L - 1 or low[l + 1] != ops.MODE_SKIP:
                np.testing.assert_array_equal(stats_a[l, 4:7].cpu().numpy(), stats_b[l, 4:7].cpu().numpy())
