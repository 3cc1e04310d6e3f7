"""Throughput of the quantized-linear hot path on one GB300 (or N, as replicas).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Workloads (synthetic inputs of the shapes and distributions of the method's
CogVideoX-shaped layers; no model weights or datasets are used):
  qkv_2b  one step = input statistics, policy step, fused Hadamard + NVFP4
          quantization, W4A4 GEMM, fused Hadamard + INT8 quantization, W4A8
          GEMM and the BF16 (PDR) GEMM of a 17776 x 1920 -> 5760 linear layer.

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events on
the launching stream; between steps a 256 MB buffer is written to flush the
129 MB L2 (outside the events).  Barrier + synchronize around the timed
region; the max over ranks is reported.  N > 1 runs independent replicas
(weak scaling; the path needs no collective for independent inputs).
`--impl reference` times the CPU oracle on a bounded sample of the same
workload instead.
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

import numpy as np  # noqa: E402

METRIC = "W4A4/W4A8 qGEMM TFLOPS+%peak; Hadamard-quant GB/s; MLP-DiT step/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# nominal dense ratios to bf16 (2.25 PFLOP/s): fp8 x2, fp4 x6
FP4_OVER_BF16 = 13.5 / 2.25


class Clocks:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) >= 9 for i in range(4) if r[5 + i].strip() == "Active"})
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=reasons, samples=len(rows))


# ------------------------------------------------------------------ workloads --

class QkvLinear:
    """The QKV-shaped linear (17776 x 1920 -> 5760), all three GEMM kinds per step."""

    name = "qkv_2b"

    def __init__(self, torch, ops, device):
        import synthgen
        self.t, self.ops = torch, ops
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
        self.flops_per_step = 3 * self.gemm_flops
        self.unit = "TFLOP/s"
        self.h2d_bytes = self.x.numel() * 2
        self.d2h_bytes = self.m * self.n * 2

    def kernels(self):
        """(label, callable) of the step, in order."""
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

    def step(self):
        for _, f in self.kernels():
            f()

    def step_e2e(self, stream):
        self.x.copy_(self.x_host, non_blocking=True)
        self.step()
        self.y_host.copy_(self.y["i8"], non_blocking=True)

    def value(self, seconds_per_step):
        return self.flops_per_step / seconds_per_step / 1e12

    # algorithmic work of each kernel per launch, for the roofline
    def algorithmic(self, label):
        mk = self.m * self.k
        if label.startswith("qgemm"):
            return ("tensor", self.gemm_flops)
        if label == "hq_nvfp4":
            # read X once (bf16), write E2M1 codes and E4M3 scales
            return ("hbm", mk * 2 + mk // 2 + mk // 16)
        if label == "hq_int8":
            # read X once, write int8 codes and row scales
            return ("hbm", mk * 2 + mk + self.m * 4)
        if label == "tensor_stats":
            return ("hbm", mk * 2)
        return (None, 0)


WORKLOADS = {"qkv_2b": QkvLinear}


# --------------------------------------------------------------------- timing --

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

    wl = WORKLOADS[args.workload](torch, ops, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
            torch.cuda.synchronize()

    for _ in range(args.warmup):
        wl.step()
    barrier()

    # ---- device-resident timed region: one event pair per step, L2 flushed between steps
    labels = [l for l, _ in wl.kernels()]
    per_kernel = {l: 0.0 for l in labels}
    clocks = Clocks(local)
    clocks.start()
    launches0 = ops.launch_count()
    step_ms = []
    barrier()
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.fill_(1.0)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(labels) + 1)]
        evs[0].record(stream)
        for i, (_, f) in enumerate(wl.kernels()):
            f()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        step_ms.append(evs[0].elapsed_time(evs[-1]))
        for i, l in enumerate(labels):
            per_kernel[l] += evs[i].elapsed_time(evs[i + 1])
    barrier()
    wall = time.perf_counter() - t_wall0
    launches = ops.launch_count() - launches0
    clk = clocks.stop()
    ms = sum(step_ms) / len(step_ms)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # ---- end to end: pinned host input -> device -> hot path -> host output, per step
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for _ in range(max(1, args.steps)):
        flush.fill_(1.0)
        e0.record(stream)
        wl.step_e2e(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e = sum(e2e_ms) / len(e2e_ms)
    if world > 1:
        t = torch.tensor([e2e], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e = float(t.item())

    if rank == 0:
        peaks = _peaks()
        kavg = {l: per_kernel[l] / args.steps for l in labels}
        dom = max(kavg, key=kavg.get)
        kind, work = wl.algorithmic(dom)
        dur = kavg[dom] / 1e3
        if kind == "tensor":
            peak = peaks["bf16"] * (FP4_OVER_BF16 if "nvfp4" in dom else 1.0)
            achieved = work / dur / 1e12
            roof = dict(bound="tensor", kernel=dom, achieved=round(achieved, 1), peak=round(peak, 1),
                        unit="TFLOP/s", frac=round(achieved / peak, 4), traffic=None,
                        peak_source=f"{peaks['src']} bf16 burst" + (" x6 nominal fp4/bf16" if "nvfp4" in dom else ""))
        else:
            achieved = work / dur / 1e9
            roof = dict(bound="hbm", kernel=dom, achieved=round(achieved, 1), peak=peaks["hbm"], unit="GB/s",
                        frac=round(achieved / peaks["hbm"], 4), traffic=None, peak_source=peaks["src"])
        kernels = {}
        for l in labels:
            kd, wk = wl.algorithmic(l)
            d = kavg[l] / 1e3
            ent = dict(us=round(kavg[l] * 1e3, 2))
            if kd == "tensor":
                pk = peaks["bf16"] * (FP4_OVER_BF16 if "nvfp4" in l else 1.0)
                ent.update(tflops=round(wk / d / 1e12, 1), frac=round(wk / d / 1e12 / pk, 4))
            elif kd == "hbm":
                ent.update(gbs=round(wk / d / 1e9, 1), frac=round(wk / d / 1e9 / peaks["hbm"], 4))
            kernels[l] = ent
        value = wl.value(ms / 1e3) * world
        line = dict(metric=METRIC, value=round(value, 3), unit=wl.unit, n_gpus=world, steps=args.steps,
                    warmup=args.warmup, ms_per_step=round(ms, 4), higher_is_better=True, scaling="weak",
                    vs_baseline=None, dtype="nvfp4/int8/bf16 operands, fp32 accumulate", data="synthetic",
                    config=dict(workload=wl.name, tokens=wl.m, k=wl.k, n=wl.n, had_block=wl.b,
                                l2="flushed between steps (256 MB write)", parallelism=f"replicas x{world}"),
                    e2e=dict(value=round(wl.value(e2e / 1e3) * world, 3), unit=wl.unit,
                             h2d_bytes_per_step=wl.h2d_bytes, d2h_bytes_per_step=wl.d2h_bytes),
                    gpu_launches=launches, roofline=roof, kernels=kernels, clocks=clk,
                    wall_s=round(wall, 3))
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------ CPU oracle leg --

def cpu_baseline(workload: str, budget_s: float = 15.0):
    """The oracle, as it stands, on a bounded sample of the workload (host cores)."""
    import synthgen
    from oracle import gemm, quant
    cores = os.cpu_count()
    c = synthgen.CONFIGS[workload]
    rows = 128
    x, w, _ = synthgen.linear_inputs(workload, m=rows)
    b = c["had_block"]
    t0 = time.perf_counter()
    done_rows = 0
    while True:
        qx = quant.hadamard_quant(x, b, "nvfp4")
        pw = quant.pack_weights(w, b)
        gemm.nvfp4_gemm_ref(qx["codes"], qx["scales"], qx["s_t"], pw["nvfp4"]["codes"], pw["nvfp4"]["scales"],
                            pw["nvfp4"]["s_t"])
        q8 = quant.hadamard_quant(x, b, "int8")
        gemm.int8_gemm_ref(q8["q"], q8["s"], pw["int4"]["q"], pw["int4"]["s"])
        gemm.bf16_gemm_ref(x, w)
        done_rows += rows
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    flops = 3 * 2.0 * done_rows * c["n"] * c["k"]
    return dict(value=round(flops / dt / 1e12, 6), unit="TFLOP/s", cores=cores, kind="oracle",
                sample=f"{done_rows} of {c['m']} token rows of {workload} (oracle quantizers, weight packing "
                       f"and float64 reference GEMMs of all three kinds), {dt:.1f} s")


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    t_steps = []
    cb = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        cb = cpu_baseline(args.workload, budget_s=args.cpu_budget / max(1, args.steps))
        if i >= args.warmup:
            t_steps.append(time.perf_counter() - t0)
    v = cb["value"]
    line = dict(impl="reference", metric=METRIC, value=v, unit=cb["unit"], n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(1e3 * sum(t_steps) / len(t_steps), 3),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64 reference, f32 quantizers",
                data="synthetic", config=dict(workload=args.workload), cpu_baseline=cb,
                e2e=dict(value=v, unit=cb["unit"], h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="qkv_2b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
