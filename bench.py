"""Throughput of the quantized-linear hot path on one GB300 (N GPUs run as replicas).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Workloads (synthetic inputs shaped like the method's CogVideoX-2B/5B layers;
random weights, no checkpoints or datasets):
  dit_2b        (default) one step = one denoising step of a 30-block
                residual-MLP DiT (hidden 1920, FFN 7680, 17776 tokens) through
                the whole hot path: input statistics, per-block policy, TDC
                skip, fused Hadamard + NVFP4/INT8 quantization, W4A4 / W4A8 /
                BF16 GEMMs with GELU and residual epilogues, block statistics
                and delta cache.  Input trajectory x_s = x_{s-1} + sigma_s N(0,1),
                sigma 0.5 -> 0.01 over 50 steps.  Metric: DiT steps/s.
  dit_2b_gated  the same with a seeded per-block residual gate in [0.02, 0.5]
                so Gamma straddles the 0.1 threshold (exercises NVFP4).
  dit_5b        42 blocks, hidden 3072, FFN 12288.
  qkv_2b        one step = both quantizers and all three GEMM kinds of a
                17776 x 1920 -> 5760 linear layer.  Metric: TFLOP/s.
  ffn_2b        one step = the FFN pair 1920 -> 7680 (GELU) -> 1920 (+ residual)
                in both mode orders (NVFP4 up / INT8 down and the reverse),
                quantizers included.  Metric: TFLOP/s.
  gemm_sweep_5b one step = quantization + W4A4 and W4A8 GEMM at K = N = 3072
                for M = 1024 .. 35552.  Metric: TFLOP/s.

Timing rules: W untimed warm-up steps, then K timed steps (the DiT restarts
its 50-step trajectory at step 0, so the default K = 50 times one whole
video's denoising, fully computed early steps included) on the device with
CUDA events on the launching stream, barrier + synchronize on both sides,
max over ranks.  The DiT working set (weights 4.5 GB, activations, delta
caches) is far larger than the 129 MB L2; the linear workload writes a 256 MB
buffer between steps (outside the events).  The DiT steps are CUDA-graph
replays; a second, eager pass with one event pair per library call gives the
per-kernel durations behind the roofline.  `--impl reference` times the CPU
oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A4/W4A8 qGEMM TFLOPS+%peak; Hadamard-quant GB/s; MLP-DiT step/s"
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense ratio (FP4 13.5 PFLOP/s, BF16 2.25 PFLOP/s)

# DRAM bytes (read + write) per launch from one ncu capture of the same kernels
# on the same shapes (profiles/); an entry must be removed when its kernel
# changes.
MEASURED_TRAFFIC = {
    # the W4A8 up call (weight expansion + GEMM) at 17776 x 7680 x 1920, captured on the FFN pair
    ("dit_2b", "qgemm_up:int8"): 303.2e6,
    ("ffn_2b", "qgemm_up:int8"): 303.2e6,
}
MODE_NAMES = {1: "nvfp4", 2: "int8", 3: "bf16", 4: "skip"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained") or
                    d["bf16_tflops"], src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class Clocks:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        """Starts sampling every 50 ms; returns once the first sample (taken before the timed
        region, and dropped) has been printed, so the sampler is running when timing starts."""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.proc.stdout.readline()
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [[v.strip() for v in r.split(",")] for r in out.strip().splitlines() if r.strip()]
        rows = [r for r in rows if len(r) >= 9]

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                    power_w_max=max(pw) if pw else None, reasons=reasons, samples=len(rows))


# ------------------------------------------------------------------ workloads --

class QkvLinear:
    """The QKV-shaped linear (17776 x 1920 -> 5760), both quantizers and all three GEMM kinds per step."""

    unit = "TFLOP/s"

    def __init__(self, name, torch, ops, device):
        import synthgen
        self.name, self.t, self.ops, self.dev = name, torch, ops, device
        x, w, c = synthgen.linear_inputs("qkv_2b")
        self.b = c["had_block"]
        self.m, self.k = x.shape
        self.n = w.shape[0]
        self.x_host = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.x_host.to(device)
        self.pw = ops.pack_weights(torch.from_numpy(w).to(device), self.b)
        self.qa = ops.QActTensors(self.m, self.k, device)
        self.y = {k: torch.empty((self.m, self.n), dtype=torch.bfloat16, device=device) for k in ("fp4", "i8", "bf")}
        self.y_host = torch.empty((self.m, self.n), dtype=torch.bfloat16).pin_memory()
        self.ins = torch.zeros(4, dtype=torch.float64, device=device)
        self.scratch = ops.new_scratch(self.x.numel(), device)
        self.state = ops.new_policy_state(device)
        self.stats = ops.new_stats(device)
        self.word = torch.zeros(1, dtype=torch.int32, device=device)
        self.cfg = ops.policy_cfg()
        self.gemm_flops = 2.0 * self.m * self.n * self.k
        self.flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=device)
        self.h2d_bytes = self.x.numel() * 2
        self.d2h_bytes = self.m * self.n * 2
        self.config = dict(workload=name, tokens=self.m, k=self.k, n=self.n, had_block=self.b,
                           l2="256 MB buffer written between steps")

    def calls(self):
        o, b = self.ops, self.b
        return [
            ("tensor_stats", lambda: o.tensor_stats(self.x, self.ins, self.scratch)),
            ("policy_step", lambda: o.policy_step(self.cfg, self.state, self.stats, self.ins, self.word)),
            ("hq_nvfp4", lambda: o.hadamard_quant(self.x, b, o.MODE_NVFP4, out=self.qa)),
            ("qgemm_nvfp4", lambda: o.qgemm(self.qa, self.x, self.pw, o.MODE_NVFP4, out=self.y["fp4"])),
            ("hq_int8", lambda: o.hadamard_quant(self.x, b, o.MODE_INT8, out=self.qa)),
            ("qgemm_int8", lambda: o.qgemm(self.qa, self.x, self.pw, o.MODE_INT8, out=self.y["i8"])),
            ("qgemm_bf16", lambda: o.qgemm(None, self.x, self.pw, o.MODE_BF16, out=self.y["bf"])),
        ]

    def warmup(self, w):
        for _ in range(w):
            for _, f in self.calls():
                f()

    def timed(self, k, stream):
        """(per-step ms, {label: [per-call ms]}) -- one event pair per call, L2 flushed between steps."""
        T = self.t
        recs = []
        for _ in range(k):
            self.flush.fill_(1.0)
            evs = [T.cuda.Event(enable_timing=True)]
            evs[0].record(stream)
            for _, f in self.calls():
                f()
                e = T.cuda.Event(enable_timing=True)
                e.record(stream)
                evs.append(e)
            recs.append(evs)
        T.cuda.synchronize()
        labels = [l for l, _ in self.calls()]
        per = {l: [] for l in labels}
        steps = []
        for evs in recs:
            steps.append(evs[0].elapsed_time(evs[-1]))
            for i, l in enumerate(labels):
                per[l].append(evs[i].elapsed_time(evs[i + 1]))
        return steps, per

    def profile(self, k, stream):
        return self.timed(k, stream)[1]

    def e2e(self, k, stream):
        T = self.t
        pairs = []
        for _ in range(k):
            self.flush.fill_(1.0)
            a, b = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
            a.record(stream)
            self.x.copy_(self.x_host, non_blocking=True)
            for _, f in self.calls():
                f()
            self.y_host.copy_(self.y["i8"], non_blocking=True)
            b.record(stream)
            pairs.append((a, b))
        T.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in pairs]

    def value(self, ms):
        return 3 * self.gemm_flops / (ms / 1e3) / 1e12

    def work(self, label):
        mk = self.m * self.k
        if label.startswith("qgemm"):
            return ("tensor", self.gemm_flops, "nvfp4" in label)
        if label == "hq_nvfp4":
            return ("hbm", mk * 2 + mk // 2 + mk // 16, False)
        if label == "hq_int8":   # read X, write the int8 codes and the row scales
            return ("hbm", mk * 3 + self.m * 4, False)
        if label == "tensor_stats":
            return ("hbm", mk * 2, False)
        return (None, 0, False)

    def launches(self):
        return None

    def extra(self):
        return {}


class FfnPair:
    """The FFN pair of a 2B-shaped block (17776 x 1920 -> 7680 -> 1920, GELU between, residual after),
    run in both mode orders per step: NVFP4 up / INT8 down, then INT8 up / NVFP4 down."""

    unit = "TFLOP/s"

    def __init__(self, name, torch, ops, device):
        import synthgen
        self.name, self.t, self.ops, self.dev = name, torch, ops, device
        x, wu, c = synthgen.linear_inputs("ffn_2b")
        wd = synthgen.weights(c["seed"], c["k"], c["n"], stream=3)
        self.b = c["had_block"]
        self.m, self.h_dim = x.shape
        self.f = wu.shape[0]
        self.x_host = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.x_host.to(device)
        self.pu = ops.pack_weights(torch.from_numpy(wu).to(device), self.b)
        self.pd = ops.pack_weights(torch.from_numpy(wd).to(device), self.b)
        self.qx = ops.QActTensors(self.m, self.h_dim, device)
        self.qh = ops.QActTensors(self.m, self.f, device)
        self.hid = torch.empty((self.m, self.f), dtype=torch.bfloat16, device=device)
        self.y = torch.empty((self.m, self.h_dim), dtype=torch.bfloat16, device=device)
        self.y_host = torch.empty((self.m, self.h_dim), dtype=torch.bfloat16).pin_memory()
        self.ws = torch.empty(ops.qgemm_workspace_bytes(self.f, self.h_dim), dtype=torch.uint8, device=device)
        self.flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=device)
        self.gemm_flops = 2.0 * self.m * self.f * self.h_dim
        self.h2d_bytes = self.x.numel() * 2
        self.d2h_bytes = self.y.numel() * 2
        self.config = dict(workload=name, tokens=self.m, hidden=self.h_dim, ffn=self.f, had_block=self.b,
                           orders="nvfp4 up + int8 down, int8 up + nvfp4 down", l2="256 MB buffer written between steps")

    def calls(self):
        o, b = self.ops, self.b
        out = []
        for up, down in ((o.MODE_NVFP4, o.MODE_INT8), (o.MODE_INT8, o.MODE_NVFP4)):
            nu, nd = MODE_NAMES[up], MODE_NAMES[down]
            out += [
                (f"hq_x:{nu}", lambda up=up: o.hadamard_quant(self.x, b, up, out=self.qx)),
                (f"qgemm_up:{nu}", lambda up=up: o.qgemm(self.qx, self.x, self.pu, up, epilogue=o.EPI_GELU,
                                                         out=self.hid, ws=self.ws)),
                (f"hq_h:{nd}", lambda down=down: o.hadamard_quant(self.hid, b, down, out=self.qh)),
                (f"qgemm_down:{nd}", lambda down=down: o.qgemm(self.qh, self.hid, self.pd, down,
                                                               epilogue=o.EPI_RESIDUAL, residual=self.x, out=self.y,
                                                               ws=self.ws)),
            ]
        return out

    warmup = QkvLinear.warmup
    timed = QkvLinear.timed
    profile = QkvLinear.profile

    def e2e(self, k, stream):
        T = self.t
        pairs = []
        for _ in range(k):
            self.flush.fill_(1.0)
            a, b = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
            a.record(stream)
            self.x.copy_(self.x_host, non_blocking=True)
            for _, f in self.calls():
                f()
            self.y_host.copy_(self.y, non_blocking=True)
            b.record(stream)
            pairs.append((a, b))
        T.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in pairs]

    def value(self, ms):
        return 4 * self.gemm_flops / (ms / 1e3) / 1e12

    def work(self, label):
        kind, _, mode = label.partition(":")
        if kind.startswith("qgemm"):
            return ("tensor", self.gemm_flops, mode == "nvfp4")
        n = self.m * (self.h_dim if kind == "hq_x" else self.f)
        if mode == "nvfp4":
            return ("hbm", n * 2 + n // 2 + n // 16, False)
        return ("hbm", n * 3 + self.m * 4, False)

    def launches(self):
        return None

    def extra(self):
        return {}


class DitStep:
    """One denoising step of the synthetic residual-MLP DiT (all hot-path rows)."""

    unit = "step/s"

    def __init__(self, name, torch, ops, device):
        import synthgen
        from video_dit_mixed_gb300 import dit
        self.name, self.t, self.ops, self.dev = name, torch, ops, device
        c = dict(synthgen.DIT_CONFIGS[name])
        if getattr(self, "blocks_override", None):
            c["blocks"] = self.blocks_override
        self.c = c
        T, H, F, L, b = c["tokens"], c["hidden"], c["ffn"], c["blocks"], c["had_block"]
        self.T, self.H, self.F, self.L, self.b = T, H, F, L, b
        gen = torch.Generator(device=device)
        gen.manual_seed(1000 + c["seed"])
        gates = synthgen.dit_gates(name)
        packed = []
        for l in range(L):
            wu = torch.randn((F, H), generator=gen, device=device, dtype=torch.float32) * c["w_std"]
            wd = torch.randn((H, F), generator=gen, device=device, dtype=torch.float32) * (c["w_std"] * gates[l])
            packed.append((ops.pack_weights(wu, b), ops.pack_weights(wd, b)))
            del wu, wd
        self.model = dit.DiT(T, H, F, L, b, packed, device=device, delta_format=self.delta_format,
                             fused_stats=self.fused_stats)
        # bytes per element of one block's Delta cache (MXFP8: one code byte, one scale byte per 32)
        self.delta_bytes = 2.0 if self.delta_format == "bf16" else 1.0 + 1.0 / 32
        # input trajectory, resident in HBM before timing
        x0 = synthgen.activations(c["seed"], T, H, "laplace", c.get("outlier_frac", 0.005),
                                  c.get("outlier_scale", 50.0))
        sig = synthgen.sigmas(c["steps"])
        self.traj = torch.empty((c["steps"], T, H), dtype=torch.bfloat16, device=device)
        self.traj[0].copy_(torch.from_numpy(x0).to(torch.bfloat16))
        for s in range(1, c["steps"]):
            z = torch.randn((T, H), generator=gen, device=device, dtype=torch.float32)
            self.traj[s].copy_((self.traj[s - 1].float() + float(sig[s - 1]) * z).to(torch.bfloat16))
        self.traj_host = None
        self.out_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        self.s = 0
        self.h2d_bytes = T * H * 2
        self.d2h_bytes = T * H * 2
        self.config = dict(workload=name, tokens=T, hidden=H, ffn=F, blocks=L, steps_per_run=c["steps"],
                           had_block=b, gate=c["gate"], policy="gamma 0.1, cos 0.99, err_cap 0.05, pdr 30",
                           l2="working set > 10 GB, no flush needed", cuda_graph=not self.host_dispatch,
                           delta_cache=self.delta_format,
                           block_stats=("BF16 blocks: down-projection epilogue; others: separate pass"
                                        if self.model.fused_stats else "separate pass"))
        self.mode_log = []
        self.timed_steps = []
        self.skip_run_bytes = 0

    def _next_input(self):
        if self.s >= self.c["steps"]:       # trajectory exhausted: start a new video
            self.s = 0
            self.model.reset()
        x = self.traj[self.s]
        self.s += 1
        return x

    host_dispatch = False   # --dispatch host: no graph, the host launches each block's chosen kernels
    delta_format = "bf16"   # --delta-format mxfp8: the Delta cache in MXFP8
    fused_stats = True      # --unfused-stats: the block statistics as a separate pass
    log_decisions = False   # --log-jsonl: keep every block's decision record of the replayed window

    def _step(self, x):
        if self.host_dispatch:
            return self.model.step_host_dispatch(x)
        return self.model.step(x)

    def warmup(self, w):
        self.model.step(self._next_input())          # eager: sets kernel attributes
        self.t.cuda.synchronize()
        if not self.host_dispatch:
            self.model.capture()
        for _ in range(max(0, w - 1)):
            self._step(self._next_input())
        # timed steps start a fresh trajectory at its first (fully computed) step
        self.t.cuda.synchronize()
        self.model.reset()
        self.s = 0

    def timed(self, k, stream):
        T = self.t
        pairs = []
        self.timed_steps = []
        for _ in range(k):
            a, b = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
            a.record(stream)
            self.timed_steps.append(self.s % self.c["steps"])
            self._step(self._next_input())
            b.record(stream)
            pairs.append((a, b))
        T.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in pairs], None

    # kernels one block runs per decision inside the switched graph: NVFP4
    # (amax + quant for x and h, two GEMMs, block end), INT8, BF16, SKIP (one
    # kernel applying the run when the block starts one, none when an earlier
    # run covered it); the decisions run at the tails of these kernels and of
    # the step's first kernel
    BODY_KERNELS = {1: 7, 2: 5, 3: 3, 4: 0}

    def launches(self):
        """Kernels run in the timed steps (from the device decision log of the same steps)."""
        if len(self.mode_log) == 0:
            return None
        import numpy as np
        low = np.asarray(self.mode_log) & 0xFF
        n = 0
        for row in low:
            row = [int(v) for v in row]
            n += 1 + sum(self.BODY_KERNELS.get(v, 0) for v in row)
            n += sum(1 for l, v in enumerate(row) if v == 4 and (l == 0 or row[l - 1] != 4))  # run starts
        return n

    def profile(self, k, stream):
        """Per-call device times over the timed window's own steps, with the kernels a graph step runs.

        The same trajectory steps as the timed region are replayed (from the
        first, with the model reset wherever the timed region started a new
        video), each block dispatched on the host from its mode word (the
        kernels of the switched graph, minus nothing but the branch selection);
        CUDA events on the launching stream bracket every call.  Before each
        group of calls a GPU-side pause lets the host enqueue them ahead of the
        GPU, so the events bracket device work, not launch gaps.  The decision
        log of these steps is what `decisions`, `gpu_launches` and the CPU
        baseline's extrapolation use.
        """
        import numpy as np
        T = self.t
        m = self.model
        o = self.ops
        steps = list(self.timed_steps) if self.timed_steps else list(range(k))
        pause = int(4e5)          # ~0.2 ms of GPU cycles: covers the host's enqueue of a group of calls
        recs = []                 # (key, start event, end event)
        run_bytes = []
        mh = np.zeros((len(steps), self.L), dtype=np.int64)
        dlog = []

        def timed(key, fn):
            a, b = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            recs.append((key, a, b))

        for j, s in enumerate(steps):
            if j == 0 or s == 0:      # the timed region started a new video here
                m.reset()
            m.x_in.copy_(self.traj[s])
            T.cuda.synchronize()
            T.cuda._sleep(pause)
            timed("tensor_stats", lambda: o.dit_begin(m.cfg, m.rec, m.scratch))   # + block 0's decision
            x = m.x_in
            for l in range(self.L):
                out = m.bufs[l % 2]
                word = int(m.modes[l].item())                  # synchronises
                mh[j, l] = word
                mode = word & 0xFF
                if mode == 4:
                    if l == 0 or (mh[j, l - 1] & 0xFF) != 4:    # a run starts here (its length: from the log)
                        T.cuda._sleep(pause)
                        timed("skip_run", lambda l=l: o.dit_skip_run(m.cfg, m.rec, l, m.scratch))
                        run_bytes.append((j, l))
                else:
                    T.cuda._sleep(pause)
                    last = [None]

                    def note(label, last=last, mode=mode):
                        e = T.cuda.Event(enable_timing=True)
                        e.record(stream)
                        recs.append((f"{label}:{MODE_NAMES.get(mode, '?')}", last[0], e))
                        last[0] = e
                    b2 = T.cuda.Event(enable_timing=True)
                    b2.record(stream)
                    last[0] = b2
                    m._compute_body(x, out, l, mode, note=note)
                x = out
            if self.log_decisions:   # one read of the mode words and policy states after the step
                dlog.extend(dict(step=int(s), **r) for r in m.decision_records())
        T.cuda.synchronize()
        self.decision_log = dlog
        low = mh & 0xFF
        per = {}
        for key, a, b in recs:
            per.setdefault(key, []).append(a.elapsed_time(b))
        # bytes of each run start: x read, k deltas read, x written
        sizes = []
        for j, l in run_bytes:
            kk = 1
            while l + kk < self.L and low[j, l + kk] == 4:
                kk += 1
            sizes.append((4 + self.delta_bytes * kk) * self.T * self.H)
        self.skip_run_bytes = (sum(sizes) / len(sizes)) if sizes else 0
        self.mode_log = mh
        m.reset()
        self.s = 0
        return per

    def e2e(self, k, stream):
        """Host trajectory (pinned) -> device, step, output -> host (pinned), from the trajectory's
        first step, through DiT.step_pipelined: each step's input copy overlaps the previous step's
        compute and its output copy the next one's.  Timed from the first copy to the last
        output's arrival on the host; per-step time = total / k."""
        T = self.t
        if self.traj_host is None:
            self.traj_host = self.traj.cpu().pin_memory()
        outs = [T.empty_like(self.out_host).pin_memory() for _ in range(2)]
        if not self.host_dispatch:
            self.model.pipeline_init()   # side streams and staging buffers, outside the timed region
        self.model.reset()
        self.s = 0
        T.cuda.synchronize()
        a, b = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
        a.record(stream)
        last = None
        for j in range(k):
            if self.s >= self.c["steps"]:
                self.s = 0
                self.model.reset()
            if self.host_dispatch:
                self._step(self.traj_host[self.s])
                outs[j % 2].copy_(self.model.out, non_blocking=True)
            else:
                last = self.model.step_pipelined(self.traj_host[self.s], outs[j % 2])
            self.s += 1
        if last is not None:
            stream.wait_event(last)
        b.record(stream)
        T.cuda.synchronize()
        return [a.elapsed_time(b) / k] * k

    def value(self, ms):
        return 1e3 / ms

    def work(self, key):
        label, _, mode = key.partition(":")
        T, H, F = self.T, self.H, self.F
        if label == "skip_run":
            return ("hbm", self.skip_run_bytes, False)
        if mode in ("skip", "covered"):
            return (None, 0, False)
        if label in ("qgemm_up", "qgemm_down"):
            return ("tensor", 2.0 * T * H * F, mode == "nvfp4")
        if label in ("hq_x", "hq_h"):
            n = T * (H if label == "hq_x" else F)
            if mode == "nvfp4":
                return ("hbm", n * 2 + n // 2 + n // 16, False)
            if mode == "int8":   # read, int8 codes, row scales
                return ("hbm", n * 3 + T * 4, False)
            return (None, 0, False)
        if label == "block_stats":   # x_in, x_out read; Delta read and written
            if mode == "bf16" and self.model.fused_stats:   # only the fold of the down projection's partial rows
                return (None, 0, False)
            return ("hbm", (4 + 2 * self.delta_bytes) * T * H, False)
        if label == "tensor_stats":
            return ("hbm", 2 * T * H, False)
        return (None, 0, False)

    def extra(self):
        import numpy as np
        if len(self.mode_log) == 0:
            return {}
        words = np.asarray(self.mode_log)
        low = words & 0xFF
        hist = {MODE_NAMES[k]: int((low == k).sum()) for k in (1, 2, 3, 4)}
        return dict(decisions=hist, refresh=int(((words & 256) != 0).sum()), pdr=int(((words & 512) != 0).sum()),
                    near_threshold=int(((words & 2048) != 0).sum()), block_steps=int(low.size),
                    window=f"trajectory steps {self.timed_steps[0]}..{self.timed_steps[-1]}" if self.timed_steps
                    else None)

    def trace(self):
        """Per timed step, the list of per-block modes ('nvfp4' | 'int8' | 'bf16' | 'skip')."""
        import numpy as np
        if len(self.mode_log) == 0:
            return None
        return [[MODE_NAMES.get(int(v), "?") for v in row] for row in (np.asarray(self.mode_log) & 0xFF)]


class GemmSweep:
    """The 5B-shaped quantized-GEMM sweep: K = N = 3072, M = 1024 .. 35552, W4A4 and W4A8.

    One step = for every M, fused Hadamard + quantization of X then the GEMM,
    in NVFP4 and in INT8.  Metric: aggregate GEMM TFLOP/s over the step.
    """

    unit = "TFLOP/s"

    def __init__(self, name, torch, ops, device):
        import synthgen
        self.name, self.t, self.ops, self.dev = name, torch, ops, device
        c = synthgen.GEMM_SWEEP
        self.b, self.k, self.n, self.ms = c["had_block"], c["k"], c["n"], c["ms"]
        x, w = synthgen.sweep_inputs(max(self.ms))
        self.x_host = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.x_host.to(device)
        self.pw = ops.pack_weights(torch.from_numpy(w).to(device), self.b)
        self.qa = {m: ops.QActTensors(m, self.k, device) for m in self.ms}
        self.y = torch.empty((max(self.ms), self.n), dtype=torch.bfloat16, device=device)
        self.y_host = torch.empty((max(self.ms), self.n), dtype=torch.bfloat16).pin_memory()
        self.flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=device)
        self.flops = {m: 2.0 * m * self.n * self.k for m in self.ms}
        self.h2d_bytes = max(self.ms) * self.k * 2
        self.d2h_bytes = max(self.ms) * self.n * 2
        self.config = dict(workload=name, k=self.k, n=self.n, m=list(self.ms), had_block=self.b,
                           l2="256 MB buffer written between steps")

    def calls(self):
        o = self.ops
        out = []
        for m in self.ms:
            xm = self.x[:m]
            for mode, code in (("nvfp4", o.MODE_NVFP4), ("int8", o.MODE_INT8)):
                out.append((f"hq_{mode}:M{m}", lambda xm=xm, m=m, code=code:
                            o.hadamard_quant(xm, self.b, code, out=self.qa[m])))
                out.append((f"qgemm_{mode}:M{m}", lambda xm=xm, m=m, code=code:
                            o.qgemm(self.qa[m], xm, self.pw, code, out=self.y[:m], m=m)))
        return out

    warmup = QkvLinear.warmup
    timed = QkvLinear.timed
    profile = QkvLinear.profile

    def e2e(self, k, stream):
        T = self.t
        pairs = []
        for _ in range(k):
            self.flush.fill_(1.0)
            a, b = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
            a.record(stream)
            self.x.copy_(self.x_host, non_blocking=True)
            for _, f in self.calls():
                f()
            self.y_host.copy_(self.y, non_blocking=True)
            b.record(stream)
            pairs.append((a, b))
        T.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in pairs]

    def value(self, ms):
        return 2 * sum(self.flops.values()) / (ms / 1e3) / 1e12

    def work(self, label):
        kind, _, mm = label.partition(":M")
        m = int(mm)
        if kind.startswith("qgemm"):
            return ("tensor", self.flops[m], "nvfp4" in kind)
        n = m * self.k
        if kind == "hq_nvfp4":
            return ("hbm", n * 2 + n // 2 + n // 16, False)
        return ("hbm", n * 3 + m * 4, False)     # INT8: read X, write the codes and the row scales

    def launches(self):
        return None

    def extra(self):
        return {}


WORKLOADS = {"qkv_2b": QkvLinear, "ffn_2b": FfnPair, "dit_2b": DitStep, "dit_2b_gated": DitStep, "dit_5b": DitStep, "gemm_sweep_5b": GemmSweep}


# --------------------------------------------------------------------- timing --

def _roofline(wl, per, peaks):
    """Per-kernel table and the dominant kernel's roofline from per-call durations (ms)."""
    table = {}
    for key, v in per.items():
        kind, work, fp4 = wl.work(key)
        avg = sum(v) / len(v)
        ent = dict(calls=len(v), avg_us=round(avg * 1e3, 2), total_ms=round(sum(v), 3))
        if kind == "tensor":
            pk = peaks["bf16"] * (FP4_OVER_BF16 if fp4 else 1.0)
            ach = work / (avg / 1e3) / 1e12
            ent.update(tflops=round(ach, 1), frac=round(ach / pk, 4))
        elif kind == "hbm":
            ach = work / (avg / 1e3) / 1e9
            ent.update(gbs=round(ach, 1), frac=round(ach / peaks["hbm"], 4))
        table[key] = ent
    cands = {k: sum(v) for k, v in per.items() if wl.work(k)[0] is not None}
    dom = max(cands, key=cands.get)
    kind, work, fp4 = wl.work(dom)
    avg = sum(per[dom]) / len(per[dom]) / 1e3
    if kind == "tensor":
        pk = peaks["bf16"] * (FP4_OVER_BF16 if fp4 else 1.0)
        ach = work / avg / 1e12
        roof = dict(bound="tensor", kernel=dom, achieved=round(ach, 1), peak=round(pk, 1), unit="TFLOP/s",
                    frac=round(ach / pk, 4), traffic=MEASURED_TRAFFIC.get((wl.name, dom)), work_per_launch=work,
                    peak_source=f"{peaks['src']} bf16 burst" + (" x6 nominal fp4/bf16" if fp4 else ""))
    else:
        ach = work / avg / 1e9
        roof = dict(bound="hbm", kernel=dom, achieved=round(ach, 1), peak=peaks["hbm"], unit="GB/s",
                    frac=round(ach / peaks["hbm"], 4), traffic=MEASURED_TRAFFIC.get((wl.name, dom)),
                    work_per_launch=work,
                    peak_source=f"{peaks['src']} copy")
    return roof, table


def metric_parts(torch, ops, dev, peaks):
    """The metric's kernel parts, timed with CUDA events on the current stream (median of 7, after 3 warm-up
    launches; every input is larger than L2, and a 256 MB buffer is written between launches):
      qgemm: W4A4 (NVFP4) and W4A8 (INT8, including its per-call INT4 -> fp16 weight expansion) at
             M x N x K = 35552 x 3072 x 3072, TFLOP/s and the fraction of the dtype's peak;
      hadamard_quant: the fused rotation + quantization of a 17776 x 7680 bf16 tensor (the FFN hidden
             activation), GB/s over its algorithmic bytes (read 2 B, write 0.5625 B (NVFP4) or 1 B (INT8) per
             element), with the NVFP4 amax pass separate or supplied by the producer.
    Synthetic inputs: Laplace(0, 1) activations with 0.5% of channels x50, N(0, 0.02^2) weights, drawn on
    the device from a seeded generator."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def laplace(m, k):
        # u strictly inside (-1/2, 1/2): rand can return 0, and u = -1/2 would give log1p(-1) = -inf
        u = (torch.rand((m, k), generator=gen, device=dev) - 0.5).clamp(-0.5 + 2.0 ** -24, 0.5 - 2.0 ** -24)
        x = -torch.sign(u) * torch.log1p(-2 * u.abs())
        idx = torch.randperm(k, generator=gen, device=dev)[: max(1, round(0.005 * k))]
        x[:, idx] *= 50.0
        return x.to(torch.bfloat16)

    def med_us(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(7):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return sorted(ts)[len(ts) // 2]

    out = {}
    m, n, k, b = 35552, 3072, 3072, 64
    x = laplace(m, k)
    w = torch.randn((n, k), generator=gen, device=dev) * 0.02
    pw = ops.pack_weights(w, b)
    qa = ops.QActTensors(m, k, dev)
    ops.hadamard_quant(x, b, ops.MODE_NVFP4, out=qa)
    ops.hadamard_quant(x, b, ops.MODE_INT8, out=qa)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(ops.qgemm_workspace_bytes(n, k), dtype=torch.uint8, device=dev)
    flops = 2.0 * m * n * k
    g = {}
    for name, code, pk, pk_src in (("w4a4_nvfp4", ops.MODE_NVFP4, peaks["bf16"] * FP4_OVER_BF16,
                                    "bf16 burst x6 nominal fp4/bf16"),
                                   ("w4a8_int8", ops.MODE_INT8, peaks["bf16"], "bf16 burst (fp16 MMAs)")):
        us = med_us(lambda: ops.qgemm(qa, x, pw, code, out=y, ws=ws))
        tf = flops / us / 1e6
        g[name] = dict(us=round(us, 1), tflops=round(tf, 1), peak=round(pk, 1), frac=round(tf / pk, 4),
                       peak_source=f"{peaks['src']} {pk_src}")
    out["qgemm"] = dict(shape=[m, n, k], **g)
    del x, qa, y, w, pw, ws
    m, k = 17776, 7680
    x = laplace(m, k)
    qa = ops.QActTensors(m, k, dev)
    nel = m * k
    hq = {}
    us2 = med_us(lambda: ops.hadamard_quant(x, b, ops.MODE_NVFP4, out=qa))
    amax = qa.tensor_amax.clone()
    us1 = med_us(lambda: ops.hadamard_quant(x, b, ops.MODE_NVFP4, out=qa, tamax=amax))
    us8 = med_us(lambda: ops.hadamard_quant(x, b, ops.MODE_INT8, out=qa))
    for name, us, byt in (("nvfp4_two_pass", us2, nel * 2 + nel // 2 + nel // 16),
                          ("nvfp4_amax_supplied", us1, nel * 2 + nel // 2 + nel // 16),
                          ("int8", us8, nel * 3 + m * 4)):
        gbs = byt / us / 1e3
        hq[name] = dict(us=round(us, 1), gbs=round(gbs, 1), frac=round(gbs / peaks["hbm"], 4),
                        algorithmic_bytes=byt)
    out["hadamard_quant"] = dict(shape=[m, k], had_block=b, peak_gbs=peaks["hbm"],
                                 peak_source=f"{peaks['src']} copy", **hq)
    return out


def reduce_max(v: float, world: int, device) -> float:
    """The largest of every rank's value (the slowest rank's time); a no-op on one rank."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(per_rank_value_at_max_time: float, world: int) -> float:
    """Replicas do the same work each, so the job's throughput is N x one rank's at the slowest time."""
    return per_rank_value_at_max_time * world


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from video_dit_mixed_gb300 import ops

    cls = WORKLOADS[args.workload]
    if args.blocks:
        cls = type(cls.__name__, (cls,), dict(blocks_override=args.blocks))
    if args.dispatch == "host":
        cls = type(cls.__name__, (cls,), dict(host_dispatch=True))
    if args.delta_format != "bf16":
        cls = type(cls.__name__, (cls,), dict(delta_format=args.delta_format))
    if args.unfused_stats:
        cls = type(cls.__name__, (cls,), dict(fused_stats=False))
    if args.log_jsonl:
        cls = type(cls.__name__, (cls,), dict(log_decisions=True))
    wl = cls(args.workload, torch, ops, dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
            torch.cuda.synchronize()

    def max_over_ranks(v):
        return reduce_max(v, world, dev)

    wl.warmup(args.warmup)
    barrier()
    clocks = Clocks(local)
    clocks.start()
    launches0 = ops.launch_count()
    t0 = time.perf_counter()
    torch.cuda.nvtx.range_push("timed")   # lets a profiler select the timed region (ncu --nvtx-include timed/)
    steps_ms, per = wl.timed(args.steps, stream)
    barrier()
    torch.cuda.nvtx.range_pop()
    wall = time.perf_counter() - t0
    launches = ops.launch_count() - launches0
    clk = clocks.stop()
    ms = max_over_ranks(sum(steps_ms) / len(steps_ms))

    if per is None:
        per = wl.profile(args.steps, stream)
    if args.log_jsonl and rank == 0:
        with open(args.log_jsonl, "w") as f:
            for r in getattr(wl, "decision_log", []):
                f.write(json.dumps(r) + "\n")
    barrier()
    e2e_ms = max_over_ranks(statistics.fmean(wl.e2e(args.steps, stream)))
    if wl.launches() is not None:
        launches = wl.launches()
    parts = None
    if args.workload.startswith("dit") and not args.no_metric_parts:
        barrier()
        parts = metric_parts(torch, ops, dev, _peaks())

    if rank == 0:
        peaks = _peaks()
        roof, table = _roofline(wl, per, peaks)
        line = dict(metric=METRIC, value=round(whole_job_value(wl.value(ms), world), 4), unit=wl.unit, n_gpus=world,
                    steps=args.steps, warmup=args.warmup, ms_per_step=round(ms, 4), higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="nvfp4/int8/bf16 operands, fp32 accumulate",
                    data="synthetic", config=dict(wl.config, parallelism=f"replicas x{world}"),
                    e2e=dict(value=round(whole_job_value(wl.value(e2e_ms), world), 4), unit=wl.unit,
                             h2d_bytes_per_step=wl.h2d_bytes, d2h_bytes_per_step=wl.d2h_bytes),
                    gpu_launches=launches, roofline=roof, kernels=table, clocks=clk, wall_s=round(wall, 3))
        line.update(wl.extra())
        if parts is not None:
            line["metric_parts"] = parts
        if not args.no_cpu_baseline:
            trace = wl.trace() if hasattr(wl, "trace") else None
            line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget, trace=trace)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------ CPU oracle leg --

def _oracle_linear_sample(workload, budget_s):
    import synthgen
    from oracle import gemm, quant
    c = synthgen.CONFIGS[workload]
    rows = 128
    x, w, _ = synthgen.linear_inputs(workload, m=rows)
    b = c["had_block"]
    pw = quant.pack_weights(w, b)
    t0 = time.perf_counter()
    done = 0
    while True:
        qx = quant.hadamard_quant(x, b, "nvfp4")
        gemm.nvfp4_gemm_ref(qx["codes"], qx["scales"], qx["s_t"], pw["nvfp4"]["codes"], pw["nvfp4"]["scales"],
                            pw["nvfp4"]["s_t"])
        q8 = quant.hadamard_quant(x, b, "int8")
        gemm.int8_gemm_ref(q8["q"], q8["s"], pw["int4"]["q"], pw["int4"]["s"])
        gemm.bf16_gemm_ref(x, w)
        done += rows
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    flops = 3 * 2.0 * done * c["n"] * c["k"]
    return dict(value=round(flops / dt / 1e12, 6), unit="TFLOP/s", cores=os.cpu_count(), kind="oracle",
                sample=f"{done} of {c['m']} token rows of {workload}: oracle quantizers and float64 reference "
                       f"GEMMs of all three kinds (weights packed once, untimed), {dt:.1f} s")


def cpu_model() -> str:
    """The host CPU's model name (x86 'model name', else lscpu's 'Model name', else the platform)."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_block_costs(workload, rows, budget_s):
    """Seconds the oracle takes for one block-step of each kind on `rows` token rows.

    compute kinds (nvfp4, int8, bf16): both quantized linears (or bf16 GEMMs)
    with GELU and residual, then the block statistics; skip: the TDC skip and
    its output statistics.  Weights are packed once, untimed.  Each kind is
    repeated until budget_s / 4 has passed; the mean is returned.
    """
    import numpy as np

    import synthgen
    from oracle import dit as odit
    from oracle import policy, quant, stats
    c = synthgen.DIT_CONFIGS[workload]
    x = synthgen.activations(c["seed"], rows, c["hidden"], "laplace", 0.005, 50.0)
    wu = synthgen.weights(c["seed"], c["ffn"], c["hidden"], c["w_std"], stream=100)
    wd = synthgen.weights(c["seed"], c["hidden"], c["ffn"], c["w_std"], stream=101)
    pu, pd = quant.pack_weights(wu, c["had_block"]), quant.pack_weights(wd, c["had_block"])
    prev = np.zeros_like(x)

    def compute(mode):
        h = odit.linear(x, pu, mode, c["had_block"], "gelu")
        out = odit.linear(h, pd, mode, c["had_block"], "residual", x)
        stats.block_stats(x, out, prev)

    def skip():
        stats.tensor_stats(stats.skip_apply(x, prev))

    kinds = {"nvfp4": lambda: compute(policy.NVFP4), "int8": lambda: compute(policy.INT8),
             "bf16": lambda: compute(policy.BF16), "skip": skip}
    out = {}
    for name, fn in kinds.items():
        t0 = time.perf_counter()
        n = 0
        while True:
            fn()
            n += 1
            if time.perf_counter() - t0 > budget_s / 4:
                break
        out[name] = (time.perf_counter() - t0) / n
    return out


def _costs_one_core(workload, rows, budget_s):
    """oracle_block_costs in a fresh process whose numerical libraries use one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-costs", "--workload", workload,
                        "--rows", str(rows), "--cpu-budget", str(budget_s)],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def _dit_rate(costs, trace, tokens, rows):
    """DiT steps/s of the oracle extrapolated over a decision trace (list of per-block mode lists)."""
    per_step = [sum(costs[mode] for mode in step) * tokens / rows for step in trace]
    return len(per_step) / sum(per_step)


def cpu_baseline(workload: str, budget_s: float = 15.0, trace=None):
    """The oracle, as it stands, on a bounded sample of the workload (host cores).

    DiT workloads: per-kind block-step times on a token sample, extrapolated
    over `trace` (the timed window's decisions; every block computing in INT8
    when no trace is given), on all cores and, in a child process, on one.
    """
    if not workload.startswith("dit"):
        return _oracle_linear_sample(workload, budget_s)
    import synthgen
    c = synthgen.DIT_CONFIGS[workload]
    rows = 32
    costs = oracle_block_costs(workload, rows, budget_s / 2)
    costs1 = _costs_one_core(workload, rows, budget_s / 2)
    if trace is None:
        trace = [["int8"] * c["blocks"]]
        how = "every block computing in INT8 (no decision trace)"
    else:
        how = f"the decisions of the timed window ({len(trace)} steps x {c['blocks']} blocks)"
    v = _dit_rate(costs, trace, c["tokens"], rows)
    out = dict(value=round(v, 10), unit="step/s", cores=os.cpu_count(), kind="oracle",
               sample=f"oracle block-steps of each kind (NVFP4, INT8, BF16: both linears, GELU, residual, "
                      f"quantizers, block statistics; SKIP: skip and statistics) on {rows} of {c['tokens']} token "
                      f"rows, extrapolated to full size over {how}: extrapolated",
               cpu_model=cpu_model(),
               block_step_s_per_row={k: round(t / rows, 6) for k, t in costs.items()})
    if costs1 is not None:
        out["value_1core"] = round(_dit_rate(costs1, trace, c["tokens"], rows), 10)
        out["block_step_s_per_row_1core"] = {k: round(t / rows, 6) for k, t in costs1.items()}
    return out


def _reference_dit_step(workload, budget_s):
    """One reference-arm step: oracle block-steps on a token sample, every block computing in INT8."""
    import synthgen
    c = synthgen.DIT_CONFIGS[workload]
    rows = 32
    costs = oracle_block_costs(workload, rows, budget_s)
    v = _dit_rate(costs, [["int8"] * c["blocks"]], c["tokens"], rows)
    return dict(value=round(v, 10), unit="step/s", cores=os.cpu_count(), kind="oracle", cpu_model=cpu_model(),
                sample=f"oracle block-steps on {rows} of {c['tokens']} token rows, extrapolated to full size with "
                       f"every block computing in INT8: extrapolated")


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = max(1.0, args.cpu_budget / max(1, args.steps))
    vals, times = [], []
    cb = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        if args.workload.startswith("dit"):
            cb = _reference_dit_step(args.workload, per_step if i >= args.warmup else 0.5)
        else:
            cb = cpu_baseline(args.workload, budget_s=per_step if i >= args.warmup else 0.5)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
            vals.append(cb["value"])
    v = statistics.fmean(vals)
    cb = dict(cb, value=v)
    line = dict(impl="reference", metric=METRIC, value=v, unit=cb["unit"], n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(1e3 * statistics.fmean(times), 3), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64 reference GEMMs, f32 quantizers", data="synthetic",
                config=dict(workload=args.workload), cpu_baseline=cb,
                e2e=dict(value=v, unit=cb["unit"], h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="dit_2b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-metric-parts", action="store_true",
                    help="DiT workloads: skip the qGEMM / Hadamard-quant kernel figures added to the line")
    ap.add_argument("--dispatch", default="graph", choices=["graph", "host"],
                    help="DiT workloads: 'host' replaces the CUDA graph by host-side dispatch on each block's mode "
                         "word (one sync per block; for profilers that cannot profile conditional graph nodes)")
    ap.add_argument("--delta-format", default="bf16", choices=["bf16", "mxfp8"],
                    help="storage of the DiT's Delta cache (MXFP8: E4M3 codes, one E8M0 scale per 32)")
    ap.add_argument("--unfused-stats", action="store_true",
                    help="DiT workloads: a computed block's statistics and Delta update as a separate pass "
                         "instead of in its down projection's epilogue")
    ap.add_argument("--blocks", type=int, default=0,
                    help="DiT workloads: use only this many blocks (profiling runs on a smaller device footprint)")
    ap.add_argument("--log-jsonl", default=None, metavar="PATH",
                    help="DiT workloads: write one JSON record per timed step and block (mode, flags, Gamma, cosine, "
                         "accumulated skip error) to PATH, read in the replay pass after the timed region")
    ap.add_argument("--oracle-costs", action="store_true", help=argparse.SUPPRESS)  # the 1-core CPU leg's child
    ap.add_argument("--rows", type=int, default=32, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.log_jsonl and not args.workload.startswith("dit"):
        ap.error("--log-jsonl records DiT decisions: use a dit_* workload")
    if args.oracle_costs:
        print(json.dumps(oracle_block_costs(args.workload, args.rows, args.cpu_budget)), flush=True)
        return
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        # one process per GPU: relaunch this command under torch.distributed.run
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", os.environ.get("MASTER_PORT", "29511"),
               os.path.abspath(__file__), *sys.argv[1:]]
        os.execv(sys.executable, cmd)
    if world is not None and int(world) != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one process per GPU")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
