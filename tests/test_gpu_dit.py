"""A small residual-MLP DiT run end to end on the GPU path vs the oracle's own chain.

Both sides start from the same seeded weights and input trajectory and run
every step independently (the oracle never sees a GPU tensor).  Bar:
- every per-block decision (mode and refresh / PDR / post-skip flags) is
  identical, except where the oracle's deciding statistic is within 1e-3
  (relative) of its threshold: along a chain the two sides' statistics
  differ by the bf16 rounding of intermediate activations, not only by the
  policy's 1e-6 band; comparison stops at such a point;
- each step's output agrees to 1e-2 relative (Frobenius norm): two
  independent chains drift apart by the bf16 rounding of every
  intermediate activation, so element-wise bounds are checked in lockstep
  instead, on the GPU's own tensors (test_gpu_dit_lockstep.py, dit_tiny
  every step, the full-size configurations on sampled steps);
- the run takes every branch: BF16 (PDR), NVFP4, INT8, SKIP and a refresh;
- the CUDA-graph replay of a step, and host-side dispatch on the mode word,
  give bit-identical results to eager launches.
Both Delta-cache formats (bf16 and MXFP8) are run, each against the oracle
keeping its cache in the same format.
"""
import numpy as np
import pytest
import torch

import synthgen
from oracle import policy
from oracle.dit import OracleDiT

pytestmark = pytest.mark.gpu
NAMES = {1: "NVFP4", 2: "INT8", 3: "BF16", 4: "SKIP"}


def _margin(st, ratio, cfg):
    m = [abs(ratio - cfg.pdr_ratio) / cfg.pdr_ratio]
    if st.n_computed >= 2:
        m.append(abs(st.cos - cfg.cos_thr) / cfg.cos_thr)
        if st.cos >= cfg.cos_thr:
            m.append(abs(st.acc + 1 - st.cos - cfg.err_cap) / cfg.err_cap)
    if st.have_gamma:
        m.append(abs(st.gamma - cfg.gamma_thr) / cfg.gamma_thr)
    return min(m)


def _run_gpu(name, graph, switched=True, host_dispatch=False, delta_format="bf16", cfgs=None, fused_stats=True):
    from video_dit_mixed_gb300 import dit, ops
    c = synthgen.DIT_CONFIGS[name]
    packed = dit.pack_block_weights(synthgen.dit_weights(name), c["had_block"])
    gpu_cfg = None if cfgs is None else [ops.policy_cfg(gamma_thr=k.gamma_thr, cos_thr=k.cos_thr, err_cap=k.err_cap,
                                                        pdr_ratio=k.pdr_ratio, refresh_bf16=k.refresh_bf16)
                                         for k in cfgs]
    model = dit.DiT(c["tokens"], c["hidden"], c["ffn"], c["blocks"], c["had_block"], packed, cfg=gpu_cfg,
                    delta_format=delta_format, fused_stats=fused_stats)
    xs = [torch.from_numpy(x).to(torch.bfloat16).cuda() for x in synthgen.dit_trajectory(name)]
    outs, words = [], []
    for s, x in enumerate(xs):
        if graph and s == 1:
            model.capture(switched=switched)
        y = model.step_host_dispatch(x) if host_dispatch else model.step(x)
        torch.cuda.synchronize()
        outs.append(y.float().cpu().numpy())
        words.append(model.modes.cpu().numpy().copy())
    return outs, words, model


# per-depth thresholds: every block its own (the run must still take every branch)
DEPTH_CFGS = [policy.PolicyConfig(), policy.PolicyConfig(cos_thr=0.995, gamma_thr=0.08),
              policy.PolicyConfig(err_cap=0.03, gamma_thr=0.12), policy.PolicyConfig(cos_thr=0.985, pdr_ratio=28.0)]


# fused: BF16 blocks take their statistics from their down projection's epilogue (bf16
# cache), in the host-dispatched (and graph) steps; the eager mode-gated step and the MXFP8
# cache take the separate statistics pass
@pytest.mark.parametrize("delta_format,depth,fused", [("bf16", False, True), ("mxfp8", False, False),
                                                      ("bf16", True, True), ("bf16", False, False)])
def test_tiny_dit_against_oracle_chain(delta_format, depth, fused):
    name = "dit_tiny"
    c = synthgen.DIT_CONFIGS[name]
    cfgs = DEPTH_CFGS if depth else None
    outs, words, _ = _run_gpu(name, graph=False, delta_format=delta_format, cfgs=cfgs, fused_stats=fused,
                              host_dispatch=fused)
    cfg = policy.PolicyConfig()
    ref = OracleDiT(synthgen.dit_weights(name), c["had_block"], cfgs or cfg, delta_format=delta_format)
    # record the oracle's distance to its thresholds at every decision
    margins = []
    orig = policy.decide

    def decide(st, ratio, cf):
        margins.append(_margin(st, ratio, cf))
        return orig(st, ratio, cf)

    import oracle.dit as odit
    odit.policy.decide = decide
    try:
        seen = set()
        for s, x in enumerate(synthgen.dit_trajectory(name)):
            y = ref.step(x)
            stop = False
            for l, d in enumerate(ref.trace[-1]):
                w = int(words[s][l])
                gpu = (NAMES[w & 0xFF], bool(w & 256), bool(w & 512), bool(w & 1024))
                ora = (d.mode, d.refresh, d.pdr, d.post_skip)
                seen.add(d.mode)
                if d.refresh:
                    seen.add("REFRESH")
                if gpu != ora:
                    assert margins[s * c["blocks"] + l] < 1e-3, (s, l, gpu, ora)
                    stop = True
                    break
            if stop:
                break
            err = np.linalg.norm(outs[s].astype(np.float64) - y) / np.linalg.norm(y)
            assert err <= 1e-2, (s, err)
        assert {"BF16", "NVFP4", "INT8", "SKIP", "REFRESH"} <= seen, seen
    finally:
        odit.policy.decide = orig


@pytest.mark.parametrize("switched,delta_format,depth", [(False, "bf16", False), (True, "bf16", False),
                                                          (True, "mxfp8", False), (True, "bf16", True)])
def test_graph_replay_matches_eager(switched, delta_format, depth):
    cfgs = DEPTH_CFGS if depth else None
    o_eager, w_eager, _ = _run_gpu("dit_tiny", graph=False, delta_format=delta_format, cfgs=cfgs)
    o_graph, w_graph, m = _run_gpu("dit_tiny", graph=True, switched=switched, delta_format=delta_format, cfgs=cfgs)
    assert m.graph is not None
    for a, b in zip(w_eager, w_graph):
        np.testing.assert_array_equal(a, b)
    for a, b in zip(o_eager, o_graph):
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_host_dispatch_matches_eager():
    """Host-side dispatch on the mode word runs the same kernels as the switched graph."""
    o_eager, w_eager, _ = _run_gpu("dit_tiny", graph=False)
    o_host, w_host, _ = _run_gpu("dit_tiny", graph=False, host_dispatch=True)
    for a, b in zip(w_eager, w_host):
        np.testing.assert_array_equal(a, b)
    for a, b in zip(o_eager, o_host):
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_pipelined_host_io_matches_eager():
    """step_pipelined (host copies overlapped with the neighbouring steps) gives the eager outputs."""
    from video_dit_mixed_gb300 import dit
    o_eager, w_eager, _ = _run_gpu("dit_tiny", graph=False)
    name = "dit_tiny"
    c = synthgen.DIT_CONFIGS[name]
    packed = dit.pack_block_weights(synthgen.dit_weights(name), c["had_block"])
    model = dit.DiT(c["tokens"], c["hidden"], c["ffn"], c["blocks"], c["had_block"], packed)
    xs = [torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in synthgen.dit_trajectory(name)]
    model.step(xs[0].cuda())
    torch.cuda.synchronize()
    model.capture()
    model.reset()
    outs = [torch.empty((c["tokens"], c["hidden"]), dtype=torch.bfloat16).pin_memory() for _ in xs]
    for x, o in zip(xs, outs):
        model.step_pipelined(x, o)
    torch.cuda.synchronize()
    for a, b in zip(o_eager, outs):
        np.testing.assert_array_equal(a.view(np.uint32), b.float().numpy().view(np.uint32))


@pytest.mark.parametrize("delta_format", ["bf16", "mxfp8"])
def test_checkpoint_resume_is_bit_identical(delta_format):
    """state_dict() half-way through a trajectory, through torch.save, into a fresh model: the rest of the
    trajectory gives the same outputs and mode words, bit for bit, as the uninterrupted run."""
    import io
    from video_dit_mixed_gb300 import dit
    name = "dit_tiny"
    c = synthgen.DIT_CONFIGS[name]
    packed = dit.pack_block_weights(synthgen.dit_weights(name), c["had_block"])
    xs = [torch.from_numpy(x).to(torch.bfloat16).cuda() for x in synthgen.dit_trajectory(name)]
    k = len(xs) // 2

    def model():
        return dit.DiT(c["tokens"], c["hidden"], c["ffn"], c["blocks"], c["had_block"], packed,
                       delta_format=delta_format)

    a = model()
    outs, words, buf = [], [], None
    for s, x in enumerate(xs):
        outs.append(a.step(x).clone())
        words.append(a.modes.clone())
        if s == k - 1:
            buf = io.BytesIO()
            torch.save(a.state_dict(), buf)
    b = model()
    buf.seek(0)
    b.load_state_dict(torch.load(buf))
    for s in range(k, len(xs)):
        y = b.step(xs[s])
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), outs[s].view(torch.int16)), s
        assert torch.equal(b.modes, words[s]), s
    with pytest.raises(ValueError):
        dit.DiT(c["tokens"], c["hidden"], c["ffn"], c["blocks"], c["had_block"], packed,
                delta_format="mxfp8" if delta_format == "bf16" else "bf16").load_state_dict(a.state_dict())
