"""DiT runs checked in lockstep against the oracle (C3 dit_2b, its gated variant, C4 dit_5b, and the
small dit_tiny with every step deep-checked).

At these sizes the oracle cannot run the chain itself (a float64 block-step
is ~1 TFLOP), so the comparison is staged: every block-step is checked on the
GPU's own tensors, the way the DiT chains them.
- Every block-step: the oracle's policy, fed the oracle's statistics of the
  GPU's block input, output and previous delta, must take the GPU's decision
  (mode and refresh / PDR / post-skip flags), except where the oracle flags a
  deciding statistic within 1e-6 (relative) of its threshold.  Such cases
  are counted, and the oracle's state is then aligned to the GPU's decision.
  The delta cache the GPU writes must equal bf16(x_out - x_in) bit for bit,
  and every fused run of skips must equal the chain of single skips (on 256
  seeded rows: the chain is elementwise).
- Every 5th step, on the first computed block at or after a seeded index
  (or, when that step computes none there, the next computed block after it):
  the quantizer's codes and scales of the block input in full (bit-exact),
  and seeded rows of the up and down projections element by element
  (|y - ref| <= 1e-5 * sum_k |a_k b_k| + half a bf16 ulp, with GELU's
  slope and the epilogue's 4e-7 |g| on the up projection).
The weights and the trajectory noise are drawn on the device from a seeded
generator (as the benchmark does); the oracle reads exactly the tensors it
checks.  With the MXFP8 delta cache, the codes and scales the GPU writes are
checked bit for bit on seeded rows against the oracle's encoding of
bf16(x_out - x_in), and the oracle's view of the cache is the GPU's cache
decoded through the oracle's own code and scale tables.
"""
import numpy as np
import pytest
import torch

import synthgen
from oracle import formats, gemm, hadamard, policy, quant, stats

pytestmark = pytest.mark.gpu
TOL = 1e-5
MODE = {1: policy.NVFP4, 2: policy.INT8, 3: policy.BF16, 4: policy.SKIP}
CODE = {v: k for k, v in MODE.items()}


def _np(t):
    return t.float().cpu().numpy()


def _half_ulp_bf16(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 8)


class Run:
    """The product DiT on device-seeded weights and trajectory, driven one block at a time."""

    def __init__(self, name, blocks=None, delta_format="bf16"):
        from video_dit_mixed_gb300 import dit, ops
        self.ops = ops
        c = dict(synthgen.DIT_CONFIGS[name])
        L = blocks or c["blocks"]
        self.T, self.H, self.F, self.L, self.b = c["tokens"], c["hidden"], c["ffn"], L, c["had_block"]
        gen = torch.Generator(device="cuda")
        gen.manual_seed(1000 + c["seed"])
        gates = synthgen.dit_gates(name)
        self.w, packed = [], []
        for l in range(L):
            wu = torch.randn((self.F, self.H), generator=gen, device="cuda") * c["w_std"]
            wd = torch.randn((self.H, self.F), generator=gen, device="cuda") * (c["w_std"] * float(gates[l]))
            packed.append((ops.pack_weights(wu, self.b), ops.pack_weights(wd, self.b)))
            self.w.append((wu, wd))
        self.model = dit.DiT(self.T, self.H, self.F, L, self.b, packed, delta_format=delta_format)
        x0 = synthgen.activations(c["seed"], self.T, self.H, "laplace", c.get("outlier_frac", 0.005),
                                  c.get("outlier_scale", 50.0))
        self.x = torch.from_numpy(x0).to(torch.bfloat16).cuda()
        self.sig = synthgen.sigmas(c["steps"])
        self.gen = gen
        self._packs = {}

    def next_input(self, s):
        if s > 0:
            z = torch.randn((self.T, self.H), generator=self.gen, device="cuda")
            self.x = (self.x.float() + float(self.sig[s - 1]) * z).to(torch.bfloat16)
        return self.x

    def oracle_pack(self, l, which):
        key = (l, which)
        if key not in self._packs:
            self._packs[key] = quant.pack_weights(self.w[l][which].cpu().numpy(), self.b)
        return self._packs[key]


def _align(st, gpu_word):
    """Apply the GPU's decision to the oracle state (near-threshold case): the skip-side update only."""
    if (gpu_word & 0xFF) == CODE[policy.SKIP]:
        st.acc = st.acc + (1.0 - st.cos)
        st.skipped_last = True


def _check_codes(run, mode, x_np):
    m = run.model
    q = quant.hadamard_quant(x_np, run.b, "nvfp4" if mode == policy.NVFP4 else "int8")
    if mode == policy.INT8:
        np.testing.assert_array_equal(m.qa_x.i8_codes.cpu().numpy(), q["q"])
        np.testing.assert_array_equal(m.qa_x.row_scale.cpu().numpy().view(np.uint32), q["s"].view(np.uint32))
    else:
        from tests._layouts import untile_scales
        np.testing.assert_array_equal(quant.unpack_nibbles(m.qa_x.fp4_codes.cpu().numpy()), q["codes"])
        mpad = (run.T + 127) // 128 * 128
        np.testing.assert_array_equal(untile_scales(m.qa_x.fp4_scales.cpu().numpy(), mpad, run.H)[:run.T],
                                      q["scales"])
        assert np.float32(m.qa_x.tensor_scale.item()) == q["s_t"]
    return q


def _ref_rows(run, l, which, mode, s_t, a_rows_np):
    """(ref, bound) float64 of the layer's sampled rows a_rows_np (bf16 values); s_t: NVFP4's tensor scale,
    which the oracle takes from the whole input tensor."""
    pk = run.oracle_pack(l, which)
    if mode == policy.NVFP4:
        q = quant.hadamard_quant(a_rows_np, run.b, "nvfp4", s_t=s_t)
        nv = pk["nvfp4"]
        return gemm.nvfp4_gemm_ref(q["codes"], q["scales"], q["s_t"], nv["codes"], nv["scales"], nv["s_t"])
    if mode == policy.INT8:
        q = quant.hadamard_quant(a_rows_np, run.b, "int8")    # per-row scales: rows are independent
        i4 = pk["int4"]
        r, bd, _ = gemm.int8_gemm_ref(q["q"], q["s"], i4["q"], i4["s"])
        return r, bd
    return gemm.bf16_gemm_ref(a_rows_np, run.w[l][which].cpu().numpy())


def _deep_check(run, l, mode, x_np, h_dev, out_np, rows):
    qx = _check_codes(run, mode, x_np) if mode != policy.BF16 else None
    # up projection + GELU
    ref, bound = _ref_rows(run, l, 0, mode, qx["s_t"] if mode == policy.NVFP4 else None, x_np[rows])
    g = gemm.gelu(ref)
    h = _np(h_dev[torch.from_numpy(rows).cuda()])
    tol = 1.13 * TOL * bound + 4e-7 * np.abs(g) + _half_ulp_bf16(g) * 1.0001 + 1e-30
    err = np.abs(h.astype(np.float64) - g)
    assert np.all(err <= tol), f"up rows of block {l}: {int((err > tol).sum())} outside, worst {float((err - tol).max())}"
    # down projection + residual, on the GPU's h (for NVFP4 the tensor scale comes from all of h)
    s_t = None
    if mode == policy.NVFP4:
        s_t = quant.tensor_scale(np.max(np.abs(hadamard.fwht_blocks(_np(h_dev), run.b))))
    ref, bound = _ref_rows(run, l, 1, mode, s_t, h)
    e = ref + x_np[rows].astype(np.float64)
    tol = TOL * bound + 1.2e-7 * np.abs(e) + _half_ulp_bf16(e) * 1.0001 + 1e-30
    err = np.abs(out_np[rows].astype(np.float64) - e)
    assert np.all(err <= tol), f"down rows of block {l}: {int((err > tol).sum())} outside"


_E4M3 = formats.decode(np.arange(256), formats.E4M3)       # value of every code (NaN for 0x7F / 0xFF)
_E8M0 = formats.e8m0_decode(np.arange(256))


def _mx_cache_check(run, l, delta, rng):
    """GPU MXFP8 cache of block l vs the oracle's encoding of `delta` on seeded rows; returns the
    GPU cache decoded (float32 [T, H])."""
    m = run.model
    codes = m.deltas[l].cpu().numpy().reshape(run.T, run.H)
    scales = m.delta_scales[l].cpu().numpy().reshape(run.T, run.H // 32)
    rows = np.unique(np.append(rng.choice(run.T, 255, replace=False), run.T - 1))
    wc, ws = formats.mxfp8_encode(delta[rows].reshape(-1))
    assert np.array_equal(codes[rows].reshape(-1), wc) and np.array_equal(scales[rows].reshape(-1), ws)
    vals = _E4M3[codes].reshape(run.T, run.H // 32, 32) * _E8M0[scales][:, :, None]
    return vals.reshape(run.T, run.H).astype(np.float32)


def _lockstep(name, steps, blocks=None, deep_every=5, nrows=32, delta_format="bf16"):
    run = Run(name, blocks, delta_format)
    o, m = run.ops, run.model
    cfg = policy.PolicyConfig()
    st = [policy.PolicyState() for _ in range(run.L)]
    prev = [np.zeros((run.T, run.H), np.float32) for _ in range(run.L)]   # the oracle's view of the delta cache
    near, seen, checked = 0, set(), 0
    rng = np.random.default_rng(5)
    deep_from = run.L
    for s in range(steps):
        x = run.next_input(s)
        m.x_in.copy_(x)
        o.dit_begin(m.cfg, m.rec, m.scratch)
        x_np = _np(x)
        ratio = stats.outlier_ratio(stats.tensor_stats(x_np))
        if s % deep_every == 0:
            deep_from = int(rng.integers(0, run.L))      # deep-check one block from here on
        elif deep_from < run.L:
            deep_from = 0                                # still pending: the next computed block
        xd = m.x_in
        l = 0
        while l < run.L:
            word = int(m.modes[l].item())
            d = policy.decide(st[l], ratio, cfg)
            gpu = (MODE[word & 0xFF], bool(word & 256), bool(word & 512), bool(word & 1024))
            ora = (d.mode, d.refresh, d.pdr, d.post_skip)
            near += int(d.near)
            if gpu != ora:
                g = o.decode_state(m.state[l])
                assert d.near, (f"step {s} block {l}: GPU {gpu} oracle {d}; oracle (acc, cos, gamma, n) "
                                f"{(st[l].acc, st[l].cos, st[l].gamma, st[l].n_computed)}; GPU state: acc {g.acc!r} "
                                f"cos {g.cos!r} gamma {g.gamma!r} n {g.n_computed}; ratio {ratio!r}")
                _align(st[l], word)          # counted above; the oracle follows the GPU from here
            mode = gpu[0]
            seen.add(mode)
            if mode == policy.SKIP:
                # a run starts here: the GPU applies the skips of blocks l .. l+k-1 in one pass and
                # records k (later blocks' mode words still hold the previous step's decisions)
                k = int(m.run_len[l].item())
                assert 1 <= k <= run.L - l, (s, l, k)
                for j in range(1, k):        # the oracle decides the rest of the run from their own state
                    wj = int(m.modes[l + j].item())
                    before = (st[l + j].acc, st[l + j].cos, st[l + j].n_computed)
                    dj = policy.decide(st[l + j], 0.0, cfg)
                    near += int(dj.near)
                    if dj.mode != policy.SKIP:
                        g = o.decode_state(m.state[l + j])
                        assert dj.near, (f"step {s} block {l + j}: GPU skips, oracle {dj}; oracle (acc, cos, n) "
                                         f"before {before}; GPU state after: acc {g.acc!r} cos {g.cos!r} "
                                         f"n {g.n_computed} gamma {g.gamma!r}")
                        _align(st[l + j], wj)
                o.dit_skip_run(m.cfg, m.rec, l, m.scratch)
                torch.cuda.synchronize()
                out = m.bufs[(l + k - 1) % 2]
                out_np = _np(out)
                rs = np.sort(rng.choice(run.T, 256, replace=False))
                y = x_np[rs]
                for j in range(k):
                    y = stats.skip_apply(y, prev[l + j][rs])
                assert np.array_equal(out_np[rs].view(np.uint32), y.view(np.uint32)), f"skip run at {s}, {l}"
                x_np, xd = out_np, out
                ratio = stats.outlier_ratio(stats.tensor_stats(x_np))
                l += k
                continue
            out = m.bufs[l % 2]
            m._compute_body(xd, out, l, CODE[mode])
            torch.cuda.synchronize()
            out_np = _np(out)
            bs = stats.block_stats(x_np, out_np, prev[l])
            if delta_format == "bf16":
                assert np.array_equal(_np(m.deltas[l]).view(np.uint32), bs["delta"].view(np.uint32)), \
                    f"delta {s}, {l}"
                new_prev = bs["delta"]
            else:
                new_prev = _mx_cache_check(run, l, bs["delta"], rng)
            if l >= deep_from:
                rows = np.sort(rng.choice(run.T, nrows - 1, replace=False))
                rows = np.unique(np.append(rows, run.T - 1))     # the ragged last tile
                _deep_check(run, l, mode, x_np, m.h, out_np, rows)
                checked += 1
                deep_from = run.L
            policy.fold(st[l], bs["gamma"], bs["cos"])
            prev[l] = new_prev
            x_np, xd = out_np, out
            ratio = stats.outlier_ratio(bs["out"])
            l += 1
    return dict(near=near, seen=seen, checked=checked)


def test_dit_tiny_lockstep_every_step():
    """The small DiT (256 tokens, 4 blocks) in lockstep, one block-step deep-checked every step:
    the element-wise counterpart of the independent-chain comparison in test_gpu_dit.py."""
    r = _lockstep("dit_tiny", steps=20, deep_every=1, nrows=32)
    assert r["checked"] >= 15 and {policy.NVFP4, policy.INT8, policy.BF16, policy.SKIP} <= r["seen"], r
    print(f"dit_tiny: {r}")


def test_dit_2b_lockstep():
    r = _lockstep("dit_2b", steps=50)
    assert {policy.INT8, policy.BF16, policy.SKIP} <= r["seen"] and r["checked"] >= 3, r
    print(f"dit_2b: {r}")


def test_dit_2b_gated_lockstep_takes_nvfp4():
    r = _lockstep("dit_2b_gated", steps=9, deep_every=4)
    assert policy.NVFP4 in r["seen"] and r["checked"] >= 3, r
    print(f"dit_2b_gated: {r}")


def test_dit_5b_lockstep_first_steps():
    r = _lockstep("dit_5b", steps=3, deep_every=1, nrows=16)
    assert r["checked"] >= 2, r
    print(f"dit_5b: {r}")


def test_dit_2b_lockstep_mxfp8_cache():
    r = _lockstep("dit_2b", steps=20, deep_every=10, delta_format="mxfp8")
    assert {policy.INT8, policy.BF16, policy.SKIP} <= r["seen"], r
    print(f"dit_2b mxfp8: {r}")
