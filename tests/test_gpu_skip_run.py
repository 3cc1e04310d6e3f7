"""sixbit_policy_skip_run (a block's decision fused with the skips of the run it
starts) against one sixbit_policy_step + sixbit_skip_apply per block.

Bar: bit-identical decisions, policy states, activations and run statistics,
over several steps of a stack whose skip runs start at block 0, in the
middle and at the end; the covered marks are back to zero after each step.
Blocks that compute are stood in for by a copy (the same on both sides).
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


@pytest.mark.parametrize("skipping", [{0, 1, 2}, {1, 2, 3}, {4, 5}, {2}, set(range(6))])
def test_fused_runs_match_sequential_skips(ops, skipping):
    L, n = 6, 8 * 1536
    g = torch.Generator(device="cuda").manual_seed(7)
    x0 = (torch.randn(n, device="cuda", generator=g) * 3).to(torch.bfloat16)
    deltas = (torch.randn((L, n), device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    cfg = ops.policy_cfg()
    scratch = ops.new_scratch(n)
    tstats = torch.zeros(4, dtype=torch.float64, device="cuda")
    ops.tensor_stats(x0, tstats, scratch)

    # sequential reference
    st_a, stats_a = _states(ops, L, skipping), ops.new_stats("cuda", L)
    modes_a = torch.zeros(L, dtype=torch.int32, device="cuda")
    bufs_a = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    # fused
    st_b, stats_b = _states(ops, L, skipping), ops.new_stats("cuda", L)
    modes_b = torch.zeros(L, dtype=torch.int32, device="cuda")
    bufs_b = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    marks = torch.zeros((2, L), dtype=torch.int32, device="cuda")
    rec = ops.dit_blocks(st_b, stats_b, modes_b, marks, tstats, x0, bufs_b[0], bufs_b[1], deltas)

    first_low = None
    for step in range(3):   # by the third step the copying blocks have two computes and skip too
        x = x0
        for l in range(L):
            ins = tstats if l == 0 else stats_a[l - 1, 4:7]
            ops.policy_step(cfg, st_a[l], stats_a[l], ins, modes_a[l:l + 1])
            out = bufs_a[l % 2]
            if int(modes_a[l].item()) & 0xFF == ops.MODE_SKIP:
                ops.skip_apply(x, deltas[l], out, stats_a[l], scratch)
            else:
                out.copy_(x)
            x = out
        xb = x0
        for l in range(L):
            ops.policy_skip_run(cfg, rec, l, scratch)
            out = bufs_b[l % 2]
            if int(modes_b[l].item()) & 0xFF != ops.MODE_SKIP:
                out.copy_(xb)
            xb = out
        torch.cuda.synchronize()
        np.testing.assert_array_equal(modes_a.cpu().numpy(), modes_b.cpu().numpy())
        np.testing.assert_array_equal(st_a.cpu().numpy(), st_b.cpu().numpy())
        assert torch.equal(x.view(torch.int16), xb.view(torch.int16)), step
        assert not marks.any()
        # the statistics a later block reads: those of every run's last block
        low = modes_a.cpu().numpy() & 0xFF
        first_low = low if first_low is None else first_low
        for l in range(L):
            if low[l] == ops.MODE_SKIP and (l == L - 1 or low[l + 1] != ops.MODE_SKIP):
                np.testing.assert_array_equal(stats_a[l, 4:7].cpu().numpy(), stats_b[l, 4:7].cpu().numpy())
    assert set(np.flatnonzero(first_low == ops.MODE_SKIP).tolist()) == skipping
