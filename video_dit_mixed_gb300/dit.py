"""Runs a residual-MLP diffusion transformer through the hot path, one denoising step at a time.

Every block maps x -> x + W_d . GELU(W_u . x).  Every per-block decision is
taken on the device, at the tail of the kernel that produces the statistics
it needs (libsixbit's DiT step protocol), and every later kernel of the block
reads the mode word and does its work only when the mode is its own, so one
step is a fixed sequence of launches with no host synchronisation; it is
captured once into a CUDA graph in which each block is a SWITCH node whose
condition the deciding kernel sets.

Per step:
  dit_begin: statistics of x_0, decision of block 0
Per block l (reads bufs[(l-1) % 2], x_in for l = 0; writes bufs[l % 2]):
  hadamard_quant(x) -> qa_x                              (NVFP4 / INT8)
  qgemm(qa_x | x, W_up[l], GELU) -> h                    (NVFP4 / INT8 / BF16)
  hadamard_quant(h) -> qa_h
  qgemm(qa_h | h, W_down[l], + x) -> out
  dit_block_end(l): block statistics, Delta cache; decision of block l+1
  dit_skip_run(l): when block l starts a run of k skipping blocks, their
                   skips in one pass; decision of block l+k
"""
from __future__ import annotations

import math

import torch

from . import ops


class DiT:
    def __init__(self, tokens: int, hidden: int, ffn: int, blocks: int, had_block: int, packed, cfg=None,
                 device="cuda", delta_format: str = "bf16", fused_stats: bool = True):
        """packed: list of (PackedWeights up [ffn, hidden], PackedWeights down [hidden, ffn]);
        cfg: one policy_cfg for every block, or a list of one per block (per-depth thresholds);
        delta_format: the Delta cache's storage, "bf16" or "mxfp8" (about half the bytes);
        fused_stats (bf16 cache): a block computed in BF16 takes its statistics and Delta from its
        down projection's epilogue (qgemm_blockstats + dit_block_end_parts) instead of a separate
        pass, in the graph and host-dispatched steps (the mode-gated eager step keeps the pass).
        Measured at dit_2b's down projection, the epilogue adds 31 us to the BF16 GEMM against the
        pass's 63 us, but 131 us to the W4A8 and 130 us to the NVFP4 one (their epilogue runs on
        the warps that also feed the tensor core, or holds its single accumulator), so those keep
        the pass."""
        assert len(packed) == blocks
        assert delta_format in ("bf16", "mxfp8")
        dev = torch.device(device)
        self.T, self.H, self.F, self.L, self.b = tokens, hidden, ffn, blocks, had_block
        self.packed = packed
        cfg = cfg or ops.policy_cfg()
        if isinstance(cfg, (list, tuple)):
            assert len(cfg) == blocks
            self.cfg = cfg[0]          # passed to the calls; each block decides with its own entry
            self.block_cfg = ops.policy_cfgs_tensor(cfg, dev)
        else:
            self.cfg = cfg
            self.block_cfg = None
        bf = torch.bfloat16
        self.x_in = torch.zeros((tokens, hidden), dtype=bf, device=dev)
        self.bufs = [torch.zeros((tokens, hidden), dtype=bf, device=dev) for _ in range(2)]
        self.h = torch.zeros((tokens, ffn), dtype=bf, device=dev)
        self.delta_format = delta_format
        if delta_format == "bf16":
            self.deltas = torch.zeros((blocks, tokens, hidden), dtype=bf, device=dev)
            self.delta_scales = None
        else:
            self.deltas, self.delta_scales = ops.mxfp8_cache(tokens * hidden, dev, blocks)
        self.qa_x = ops.QActTensors(tokens, hidden, dev)
        self.qa_h = ops.QActTensors(tokens, ffn, dev)
        # the W4A8 GEMMs expand their INT4 weights into this (one buffer for both projections)
        self.ws = torch.empty(ops.qgemm_workspace_bytes(ffn, hidden), dtype=torch.uint8, device=dev)
        self.tstats = torch.zeros(4, dtype=torch.float64, device=dev)
        self.stats = ops.new_stats(dev, blocks)
        self.state = ops.new_policy_state(dev, blocks)
        self.modes = torch.zeros(blocks, dtype=torch.int32, device=dev)
        self.run_len = torch.zeros(blocks, dtype=torch.int32, device=dev)   # per run start, within a step
        self.scratch = ops.new_scratch(tokens * ffn, dev)
        self.fused_stats = fused_stats and delta_format == "bf16"
        self.fused_modes = (ops.MODE_BF16,) if self.fused_stats else ()
        self.parts = ops.new_blockstats_parts(dev) if self.fused_stats else None
        self.conds = torch.zeros(blocks, dtype=torch.int64, device=dev)  # graph condition handles
        self.rec = self._record(None)
        self.graph = None
        self.out = self.bufs[(blocks - 1) % 2]

    def _record(self, conds):
        return ops.dit_blocks(self.state, self.stats, self.modes, self.run_len, self.tstats, self.x_in,
                              self.bufs[0], self.bufs[1], self.deltas, conds, self.delta_scales, self.block_cfg)

    def reset(self):
        """Back to the state before the first denoising step."""
        self.deltas.zero_()
        if self.delta_scales is not None:
            self.delta_scales.zero_()
        self.stats.zero_()
        self.state.zero_()
        self.modes.zero_()
        self.run_len.zero_()

    # the trajectory state carried from one denoising step to the next (what reset() clears)
    STATE = ("deltas", "delta_scales", "stats", "state", "modes", "run_len")

    def state_dict(self) -> dict:
        """Checkpoint: host copies of the trajectory state between two steps (delta caches, statistics,
        policy states, mode words), after the steps already enqueued on the current stream have run.
        load_state_dict() on a model of the same shape and delta format resumes the trajectory with
        bit-identical outputs and decisions.  The result can be saved with torch.save."""
        torch.cuda.current_stream().synchronize()
        sd = {k: getattr(self, k).to("cpu", copy=True) for k in self.STATE if getattr(self, k) is not None}
        sd["shape"] = (self.T, self.H, self.F, self.L, self.b)
        sd["delta_format"] = self.delta_format
        return sd

    def load_state_dict(self, sd: dict) -> None:
        """Resume from state_dict(): the buffers are overwritten in place, so a captured graph keeps
        working; raises ValueError on a checkpoint of another shape or delta format."""
        if tuple(sd["shape"]) != (self.T, self.H, self.F, self.L, self.b) or sd["delta_format"] != self.delta_format:
            raise ValueError(f"checkpoint of {sd['shape']} / {sd['delta_format']}, model "
                             f"{(self.T, self.H, self.F, self.L, self.b)} / {self.delta_format}")
        for k in self.STATE:
            t = getattr(self, k)
            if t is not None:
                t.copy_(sd[k].to(device=t.device, dtype=t.dtype), non_blocking=False)

    CALLS = ("hq_x", "qgemm_up", "hq_h", "qgemm_down", "block_stats", "skip_run")

    def enqueue_step(self, after_call=None):
        """Enqueue one denoising step on the current stream (input: self.x_in), every
        kernel launched and gated on the device by the block's mode word.

        after_call(label, block) is invoked on the host after each library call
        (e.g. to record a CUDA event for per-call timing); labels are
        "tensor_stats" (block -1, the step's first call) and DiT.CALLS.
        """
        o = ops
        note = after_call or (lambda label, block: None)
        o.dit_begin(self.cfg, self.rec, self.scratch)
        note("tensor_stats", -1)
        x = self.x_in
        for l in range(self.L):
            out = self.bufs[l % 2]
            mode = self.modes[l:l + 1]
            up, down = self.packed[l]
            o.hadamard_quant(x, self.b, 0, out=self.qa_x, mode_dev=mode)
            note("hq_x", l)
            o.qgemm(self.qa_x, x, up, 0, epilogue=o.EPI_GELU, out=self.h, mode_dev=mode, ws=self.ws)
            note("qgemm_up", l)
            o.hadamard_quant(self.h, self.b, 0, out=self.qa_h, mode_dev=mode)
            note("hq_h", l)
            o.qgemm(self.qa_h, self.h, down, 0, epilogue=o.EPI_RESIDUAL, residual=x, out=out, mode_dev=mode,
                    ws=self.ws)
            note("qgemm_down", l)
            o.dit_block_end(self.cfg, self.rec, l, self.scratch)
            note("block_stats", l)
            o.dit_skip_run(self.cfg, self.rec, l, self.scratch)
            note("skip_run", l)
            x = out
        return x

    def _compute_body(self, x, out, l, mode, rec=None, note=None):
        """The kernels of one computed block in a fixed mode (no mode word), ending with
        dit_block_end (or dit_block_end_parts); note(label) is called on the host after each call when given."""
        o = ops
        rec = rec or self.rec
        note = note or (lambda label: None)
        up, down = self.packed[l]
        quant = mode != o.MODE_BF16
        fused = mode == o.MODE_NVFP4 and self.b in (16, 64)   # the up GEMM also takes h's amax pass
        if quant:
            o.hadamard_quant(x, self.b, mode, out=self.qa_x)
            note("hq_x")
        if fused:
            o.qgemm_rotamax(self.qa_x, up, self.b, self.qa_h.tensor_amax, epilogue=o.EPI_GELU, out=self.h, m=self.T)
        else:
            o.qgemm(self.qa_x if quant else None, x, up, mode, epilogue=o.EPI_GELU, out=self.h, m=self.T, ws=self.ws)
        note("qgemm_up")
        if quant:
            o.hadamard_quant(self.h, self.b, mode, out=self.qa_h, tamax=self.qa_h.tensor_amax if fused else None)
            note("hq_h")
        if mode in self.fused_modes:
            o.qgemm_blockstats(self.qa_h if quant else None, self.h, down, mode, residual=x, out=out,
                               delta_cache=self.deltas[l], parts=self.parts, m=self.T, ws=self.ws)
            note("qgemm_down")
            o.dit_block_end_parts(self.cfg, rec, l, self.parts)
        else:
            o.qgemm(self.qa_h if quant else None, self.h, down, mode, epilogue=o.EPI_RESIDUAL, residual=x, out=out,
                    m=self.T, ws=self.ws)
            note("qgemm_down")
            o.dit_block_end(self.cfg, rec, l, self.scratch)
        note("block_stats")

    def enqueue_step_switched(self, body_stream):
        """One step for graph capture: per block a SWITCH over the NVFP4 / INT8 /
        BF16 bodies and the skip run a block starts, whose condition the deciding
        kernel sets, so only the chosen body's kernels run (the other blocks of a
        run run none).  Returns the handles (filled into self.conds by
        capture())."""
        o = ops
        stream = torch.cuda.current_stream()
        handles = [o.graph_cond_create(stream, 4) for _ in range(self.L)]
        rec = self._record(self.conds)
        o.dit_begin(self.cfg, rec, self.scratch)
        x = self.x_in
        for l in range(self.L):
            out = self.bufs[l % 2]
            sw = o.GraphSwitch(stream, body_stream, None, o.MODE_NVFP4, 4, cond=handles[l])
            for i, m in enumerate((o.MODE_NVFP4, o.MODE_INT8, o.MODE_BF16)):
                with sw.branch(i):
                    self._compute_body(x, out, l, m, rec=rec)
            with sw.branch(3):
                o.dit_skip_run(self.cfg, rec, l, self.scratch)
            sw.close()
            x = out
        self._rec_graph = rec   # keeps the record's buffers referenced with the graph
        return handles

    def step_host_dispatch(self, x_s: torch.Tensor | None = None):
        """One step without a graph: the host reads each block's mode word (one
        synchronisation per block) and launches only that mode's kernels.

        The same kernels as a switched-graph step, minus the selectors; meant
        for profilers that cannot look inside graphs with conditional nodes.
        """
        o = ops
        if x_s is not None:
            self.x_in.copy_(x_s, non_blocking=True)
        o.dit_begin(self.cfg, self.rec, self.scratch)
        x = self.x_in
        for l in range(self.L):
            out = self.bufs[l % 2]
            m = int(self.modes[l].item()) & 0xFF
            if m != o.MODE_SKIP:
                self._compute_body(x, out, l, m)
            elif l == 0 or (int(self.modes[l - 1].item()) & 0xFF) != o.MODE_SKIP:
                o.dit_skip_run(self.cfg, self.rec, l, self.scratch)   # a run starts here
            x = out
        return x

    def capture(self, switched: bool = True):
        """Capture one step into a CUDA graph (call after at least one eager step).

        switched=True uses device-selected SWITCH nodes (only the chosen body
        runs); False captures the flat launch sequence whose kernels return at
        once when the mode word is not theirs.
        """
        g = torch.cuda.CUDAGraph()
        body_stream = torch.cuda.Stream()
        handles = None
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            if switched:
                handles = self.enqueue_step_switched(body_stream)
            else:
                self.enqueue_step()
        if handles is not None:   # read by the deciding kernels when the graph runs
            as_i64 = [h - (1 << 64) if h >= (1 << 63) else h for h in handles]
            self.conds.copy_(torch.tensor(as_i64, dtype=torch.int64))
            torch.cuda.synchronize()
        self.graph = g
        self._body_stream = body_stream
        return g

    def step(self, x_s: torch.Tensor | None = None):
        """One denoising step on input x_s (copied into the graph's input buffer)."""
        if x_s is not None:
            self.x_in.copy_(x_s, non_blocking=True)
        if self.graph is not None:
            self.graph.replay()
        else:
            self.enqueue_step()
        return self.out

    def pipeline_init(self):
        """Allocate step_pipelined's side streams, staging buffers and events (once)."""
        if getattr(self, "_pipe", None) is not None:
            return
        cs = torch.cuda.current_stream()
        dev = self.x_in.device
        mk = lambda: [torch.empty_like(self.x_in) for _ in range(2)]  # noqa: E731
        self._pipe = dict(
            s_in=torch.cuda.Stream(device=dev), s_out=torch.cuda.Stream(device=dev), stage_in=mk(),
            stage_out=mk(), k=0,
            in_ready=[torch.cuda.Event() for _ in range(2)], in_free=[torch.cuda.Event() for _ in range(2)],
            out_ready=[torch.cuda.Event() for _ in range(2)], out_free=[torch.cuda.Event() for _ in range(2)])
        for e in self._pipe["in_free"] + self._pipe["out_free"]:
            e.record(cs)

    def step_pipelined(self, x_host: torch.Tensor, out_host: torch.Tensor):
        """One step with its host copies overlapped with the neighbouring steps.

        x_host and out_host are pinned host tensors [T, H] bf16.  The input is
        copied in on one side stream while the previous step computes, and
        the result is copied back on another while the next step computes
        (each through a device staging buffer, so the copies never race the
        step's own buffers).  Returns the event after which out_host holds
        this step's output.  Nothing here synchronises the host.
        """
        cs = torch.cuda.current_stream()
        self.pipeline_init()
        P = self._pipe
        i = P["k"] % 2
        P["s_in"].wait_event(P["in_free"][i])           # stage_in[i] consumed two steps ago
        with torch.cuda.stream(P["s_in"]):
            P["stage_in"][i].copy_(x_host, non_blocking=True)
            P["in_ready"][i].record(P["s_in"])
        cs.wait_event(P["in_ready"][i])
        self.step(P["stage_in"][i])                     # device-to-device into x_in, then the graph
        P["in_free"][i].record(cs)
        cs.wait_event(P["out_free"][i])                 # stage_out[i] read back two steps ago
        P["stage_out"][i].copy_(self.out)
        P["out_ready"][i].record(cs)
        P["s_out"].wait_event(P["out_ready"][i])
        with torch.cuda.stream(P["s_out"]):
            out_host.copy_(P["stage_out"][i], non_blocking=True)
            P["out_free"][i].record(P["s_out"])
        P["k"] += 1
        return P["out_free"][i]

    def decision_records(self) -> list:
        """Per block, the decision of the last step and the policy values it was taken on (one read of
        the mode words and policy states, after the work already enqueued on the current stream):
        see decode_decisions."""
        torch.cuda.current_stream().synchronize()
        return decode_decisions(self.modes.cpu().numpy(), self.state.cpu().numpy())

    def decision_counts(self):
        """Per block: (n_nvfp4, n_int8, n_bf16, n_skip, n_refresh, n_pdr, n_near) from the device state."""
        out = []
        for l in range(self.L):
            s = ops.decode_state(self.state[l])
            out.append((s.n_nvfp4, s.n_int8, s.n_bf16, s.n_skip, s.n_refresh, s.n_pdr, s.n_near))
        return out


def _num(v: float):
    """A float for a JSON record: non-finite values as the strings "nan", "inf", "-inf"."""
    return v if math.isfinite(v) else ("nan" if math.isnan(v) else ("inf" if v > 0 else "-inf"))


def decode_decisions(modes, states) -> list:
    """Decision records of one step from host copies of the mode words [L] and policy states [L, 80]:
    per block its mode, flags (refresh, pdr, post_skip, near), and the Gamma, cosine, accumulated
    skip error and computed-step count the policy state holds after the decision (Gamma and the
    cosine as used for it; acc including a skip's own 1 - cos).  Gamma is absent before the first
    computed step, the cosine before the second."""
    out = []
    for l, w in enumerate(modes):
        w = int(w)
        st = ops.decode_state(torch.as_tensor(states[l]))
        out.append(dict(block=l, mode=ops.abi.MODE_NAMES.get(w & 0xFF, "?"),
                        refresh=bool(w & ops.abi.FLAG_REFRESH), pdr=bool(w & ops.abi.FLAG_PDR),
                        post_skip=bool(w & ops.abi.FLAG_POSTSKIP), near=bool(w & ops.abi.FLAG_NEAR),
                        gamma=_num(st.gamma) if st.have_gamma else None,
                        cos=_num(st.cos) if st.n_computed >= 2 else None,
                        acc=_num(st.acc), n_computed=int(st.n_computed)))
    return out


def pack_block_weights(weights, had_block, device="cuda"):
    """[(W_up fp32 [F, H], W_down fp32 [H, F])] (host or device) -> packed per block."""
    out = []
    for wu, wd in weights:
        wu = torch.as_tensor(wu).to(device=device, dtype=torch.float32).contiguous()
        wd = torch.as_tensor(wd).to(device=device, dtype=torch.float32).contiguous()
        out.append((ops.pack_weights(wu, had_block), ops.pack_weights(wd, had_block)))
    torch.cuda.synchronize()
    return out
