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
# on the same shapes (profiles/dram_traffic_dit_2b.md); an entry must be
# removed when its kernel changes.
MEASURED_TRAFFIC = {
    ("dit_2b", "qgemm_up:int8"): 335972608,
    ("dit_2b", "qgemm_down:int8"): 632774656,
    ("dit_2b", "qgemm_up:bf16"): 333682841,
    ("dit_2b", "qgemm_down:bf16"): 543600844,
    ("dit_2b", "hq_x:int8"): 86360960,
    ("dit_2b", "hq_h:int8"): 495195520,
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
        self.qa = ops.QActTensors(self.m, self.k, device, i8_codes=False)   # the GEMM reads the bf16 operand
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
        if label == "hq_int8":   # read X, write the bf16 integer operand and the row scales
            return ("hbm", mk * 4 + self.m * 4, False)
        if label == "tensor_stats":
            return ("hbm", mk * 2, False)
        return (None, 0, False)

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
        self.model = dit.DiT(T, H, F, L, b, packed, device=device)
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
                           l2="working set > 10 GB, no flush needed", cuda_graph=not self.host_dispatch)
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
        """Kernels run in the timed steps (from the device decision log of the same trajectory)."""
        if len(self.mode_log) == 0:
            return None
        import numpy as np
        low = np.asarray(self.mode_log) & 0xFF
        n = 0
        for s in self.timed_steps:
            row = [int(v) for v in low[s]]
            n += 1 + sum(self.BODY_KERNELS.get(v, 0) for v in row)
            n += sum(1 for l, v in enumerate(row) if v == 4 and (l == 0 or row[l - 1] != 4))  # run starts
        return n

    def profile(self, k, stream):
        """Per-call device times over a full trajectory, with the kernels a graph step runs.

        Each block is dispatched on the host from its mode word (the kernels of
        the switched graph, minus nothing but the branch selection); CUDA
        events on the launching stream bracket every call.  Before each group
        of calls a GPU-side pause lets the host enqueue them ahead of the GPU,
        so the events bracket device work, not launch gaps.
        """
        import numpy as np
        T = self.t
        m = self.model
        o = self.ops
        m.reset()
        self.s = 0
        pause = int(4e5)          # ~0.2 ms of GPU cycles: covers the host's enqueue of a group of calls
        recs = []                 # (key, start event, end event)
        run_bytes = []
        mh = np.zeros((self.c["steps"], self.L), dtype=np.int64)

        def timed(key, fn):
            a, b = T.cuda.Event(enable_timing=True), T.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            recs.append((key, a, b))

        for s in range(self.c["steps"]):
            m.x_in.copy_(self.traj[s])
            T.cuda.synchronize()
            T.cuda._sleep(pause)
            timed("tensor_stats", lambda: o.dit_begin(m.cfg, m.rec, m.scratch))   # + block 0's decision
            x = m.x_in
            for l in range(self.L):
                out = m.bufs[l % 2]
                word = int(m.modes[l].item())                  # synchronises
                mh[s, l] = word
                mode = word & 0xFF
                if mode == 4:
                    if l == 0 or (mh[s, l - 1] & 0xFF) != 4:    # a run starts here (its length: from the log)
                        T.cuda._sleep(pause)
                        timed("skip_run", lambda l=l: o.dit_skip_run(m.cfg, m.rec, l, m.scratch))
                        run_bytes.append((s, l))
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
        T.cuda.synchronize()
        low = mh & 0xFF
        per = {}
        for key, a, b in recs:
            per.setdefault(key, []).append(a.elapsed_time(b))
        # bytes of each run start: x read, k deltas read, x written
        sizes = []
        for s, l in run_bytes:
            k = 1
            while l + k < self.L and low[s, l + k] == 4:
                k += 1
            sizes.append((4 + 2 * k) * self.T * self.H)
        run_bytes = sizes
        self.skip_run_bytes = (sum(run_bytes) / len(run_bytes)) if run_bytes else 0
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
            if mode == "int8":   # read, bf16 integer operand, row scales
                return ("hbm", n * 4 + T * 4, False)
            return (None, 0, False)
        if label == "block_stats":
            return ("hbm", 8 * T * H, False)
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
                    near_threshold=int(((words & 2048) != 0).sum()), block_steps=int(low.size))


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
        self.qa = {m: ops.QActTensors(m, self.k, device, i8_codes=False) for m in self.ms}
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
        return ("hbm", n * 4 + m * 4, False)

    def launches(self):
        return None

    def extra(self):
        return {}


WORKLOADS = {"qkv_2b": QkvLinear, "dit_2b": DitStep, "dit_2b_gated": DitStep, "dit_5b": DitStep, "gemm_sweep_5b": GemmSweep}


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
    barrier()
    e2e_ms = max_over_ranks(statistics.fmean(wl.e2e(args.steps, stream)))
    if wl.launches() is not None:
        launches = wl.launches()

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
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
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


def _oracle_dit_sample(workload, budget_s):
    """One INT8 block (both linears, quantizers, statistics) on a token sample, extrapolated to a DiT step."""
    import numpy as np

    import synthgen
    from oracle import dit as odit
    from oracle import policy, quant, stats
    c = synthgen.DIT_CONFIGS[workload]
    rows = 64
    x = synthgen.activations(c["seed"], rows, c["hidden"], "laplace", 0.005, 50.0)
    wu = synthgen.weights(c["seed"], c["ffn"], c["hidden"], c["w_std"], stream=100)
    wd = synthgen.weights(c["seed"], c["hidden"], c["ffn"], c["w_std"], stream=101)
    pu, pd = quant.pack_weights(wu, c["had_block"]), quant.pack_weights(wd, c["had_block"])
    t0 = time.perf_counter()
    done = 0
    while True:
        h = odit.linear(x, pu, policy.INT8, c["had_block"], "gelu")
        out = odit.linear(h, pd, policy.INT8, c["had_block"], "residual", x)
        stats.block_stats(x, out, np.zeros_like(x))
        done += rows
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    sec_per_step = dt / done * c["tokens"] * c["blocks"]
    return dict(value=round(1.0 / sec_per_step, 8), unit="step/s", cores=os.cpu_count(), kind="oracle",
                sample=f"{done} token rows of one INT8 block (up GEMM + GELU, down GEMM + residual, both "
                       f"quantizers, block statistics; weights packed once, untimed) in {dt:.1f} s, "
                       f"extrapolated to {c['tokens']} tokens x {c['blocks']} blocks per step (all computed)")


def cpu_baseline(workload: str, budget_s: float = 15.0):
    """The oracle, as it stands, on a bounded sample of the workload (host cores)."""
    if workload.startswith("dit"):
        return _oracle_dit_sample(workload, budget_s)
    return _oracle_linear_sample(workload, budget_s)


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
    ap.add_argument("--dispatch", default="graph", choices=["graph", "host"],
                    help="DiT workloads: 'host' replaces the CUDA graph by host-side dispatch on each block's mode "
                         "word (one sync per block; for profilers that cannot profile conditional graph nodes)")
    ap.add_argument("--blocks", type=int, default=0,
                    help="DiT workloads: use only this many blocks (profiling runs on a smaller device footprint)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
