"""The DiT step protocol (sixbit_dit_begin / _block_end / _skip_run: decisions at the
tails of the kernels that produce their statistics, skips applied in runs) against
one sixbit_policy_step per block followed by sixbit_skip_apply or the block's work
and sixbit_block_stats.

Bar: bit-identical decisions, policy states, activations, Delta caches and the
statistics later blocks read, over several steps of a stack whose skip runs start
at block 0, in the middle and at the end; the run lengths are back to zero
after each step (runs of up to 40 blocks).  A block's compute is stood in for by a seeded
perturbation of its input (the same on both sides).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from video_dit_mixed_gb300 import ops as o
    return o


def _states(ops, L, skipping, cos=0.999):
    """Policy states: blocks in `skipping` will skip (two computes done, cos >= 0.99, small error)."""
    raw = ops.new_policy_state("cuda", L)
    host = []
    for l in range(L):
        s = ops.PolicyState()
        if l in skipping:
            s.n_computed, s.have_gamma, s.cos, s.gamma = 2, 1, cos, 0.5
        host.append(bytes(s))
    raw.copy_(torch.frombuffer(bytearray(b"".join(host)), dtype=torch.uint8).view(L, 80))
    return raw


def _compute(x, out, bump):
    out.copy_((x.float() + bump).to(torch.bfloat16))


# Stacks of 36-40 blocks put a run across the 32-block groups in which a
# run's blocks are decided in parallel (one per lane).
@pytest.mark.parametrize("L,skipping", [(6, {0, 1, 2}), (6, {1, 2, 3}), (6, {4, 5}), (6, {2}), (6, set(range(6))),
                                        (40, set(range(1, 38))), (40, set(range(40))), (40, set(range(10, 36))),
                                        (36, set(range(3, 36))), (40, set(range(0, 33)) | {35, 36})])
def test_protocol_matches_sequential_steps(ops, L, skipping):
    n = 8 * 1536
    g = torch.Generator(device="cuda").manual_seed(7)
    x0 = (torch.randn(n, device="cuda", generator=g) * 3).to(torch.bfloat16)
    deltas0 = (torch.randn((L, n), device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    bumps = [torch.randn(n, device="cuda", generator=g) * 0.2 for _ in range(L)]
    cfg = ops.policy_cfg()
    scratch = ops.new_scratch(n)

    # sequential reference
    st_a, stats_a = _states(ops, L, skipping), ops.new_stats("cuda", L)
    modes_a = torch.zeros(L, dtype=torch.int32, device="cuda")
    bufs_a = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    deltas_a = deltas0.clone()
    tstats_a = torch.zeros(4, dtype=torch.float64, device="cuda")
    # protocol
    st_b, stats_b = _states(ops, L, skipping), ops.new_stats("cuda", L)
    modes_b = torch.zeros(L, dtype=torch.int32, device="cuda")
    bufs_b = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    deltas_b = deltas0.clone()
    tstats_b = torch.zeros(4, dtype=torch.float64, device="cuda")
    run_len = torch.zeros(L, dtype=torch.int32, device="cuda")
    rec = ops.dit_blocks(st_b, stats_b, modes_b, run_len, tstats_b, x0, bufs_b[0], bufs_b[1], deltas_b)

    first_low = None
    for step in range(3):   # by the third step the computing blocks have two computes and may skip too
        ops.tensor_stats(x0, tstats_a, scratch)
        x = x0
        for l in range(L):
            ins = tstats_a if l == 0 else stats_a[l - 1, 4:7]
            ops.policy_step(cfg, st_a[l], stats_a[l], ins, modes_a[l:l + 1])
            out = bufs_a[l % 2]
            if int(modes_a[l].item()) & 0xFF == ops.MODE_SKIP:
                ops.skip_apply(x, deltas_a[l], out, stats_a[l], scratch)
            else:
                _compute(x, out, bumps[l])
                ops.block_stats(x, out, deltas_a[l], stats_a[l], scratch)
            x = out
        ops.dit_begin(cfg, rec, scratch)
        xb = x0
        for l in range(L):
            out = bufs_b[l % 2]
            if int(modes_b[l].item()) & 0xFF != ops.MODE_SKIP:
                _compute(xb, out, bumps[l])
            ops.dit_block_end(cfg, rec, l, scratch)
            ops.dit_skip_run(cfg, rec, l, scratch)
            xb = out
        torch.cuda.synchronize()
        np.testing.assert_array_equal(modes_a.cpu().numpy(), modes_b.cpu().numpy())
        np.testing.assert_array_equal(st_a.cpu().numpy(), st_b.cpu().numpy())
        assert torch.equal(x.view(torch.int16), xb.view(torch.int16)), step
        assert torch.equal(deltas_a.view(torch.int16), deltas_b.view(torch.int16)), step
        np.testing.assert_array_equal(tstats_a.cpu().numpy(), tstats_b.cpu().numpy())
        assert not run_len.any()
        low = modes_a.cpu().numpy() & 0xFF
        first_low = low if first_low is None else first_low
        for l in range(L):
            if low[l] != ops.MODE_SKIP:        # every statistic of a computed block
                np.testing.assert_array_equal(stats_a[l].cpu().numpy(), stats_b[l].cpu().numpy())
            elif l == L - 1 or low[l + 1] != ops.MODE_SKIP:   # what the block after a run reads
                np.testing.assert_array_equal(stats_a[l, 4:7].cpu().numpy(), stats_b[l, 4:7].cpu().numpy())
    assert set(np.flatnonzero(first_low == ops.MODE_SKIP).tolist()) == skipping
