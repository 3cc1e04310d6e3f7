"""Torch-facing binding of libsixbit: argument marshalling only.

Every function here allocates its output tensors with torch (device memory),
passes raw pointers and the current CUDA stream to the C ABI, and raises
``SixbitError`` on a non-zero status.  All arithmetic runs in the library's
CUDA kernels; there is no CPU path.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import abi
from .abi import (EPI_GELU, EPI_NONE, EPI_RESIDUAL, MODE_BF16, MODE_INT8, MODE_NVFP4, MODE_SKIP,  # noqa: F401
                  DitBlocks, PolicyCfg, PolicyState, QAct, Stats, Weights, check, lib)

_lib = lib()


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def fp4_scale_bytes(rows: int, k: int) -> int:
    return int(_lib.sixbit_fp4_scale_bytes(rows, k))


def stats_scratch_bytes(n: int) -> int:
    return int(_lib.sixbit_stats_scratch_bytes(n))


def launch_count() -> int:
    return int(_lib.sixbit_launch_count())


def qgemm_workspace_bytes(n: int, k: int) -> int:
    return int(_lib.sixbit_qgemm_workspace_bytes(n, k))


_workspaces = {}


def workspace(n: int, k: int, device) -> torch.Tensor:
    """A device buffer of at least qgemm_workspace_bytes(n, k) bytes, shared by every call on `device`
    that passes none of its own (calls that share it must be ordered, e.g. on one stream)."""
    dev = torch.device(device)
    need = qgemm_workspace_bytes(n, k)
    buf = _workspaces.get(dev)
    if buf is None or buf.numel() < need:
        buf = torch.empty(need, dtype=torch.uint8, device=dev)
        _workspaces[dev] = buf
    return buf


class QActTensors:
    """Device buffers of one quantized activation tensor [M, K]."""

    def __init__(self, m: int, k: int, device="cuda", nvfp4=True, int8=True, rotated=False):
        self.m, self.k = m, k
        dev = torch.device(device)
        u8, f32 = torch.uint8, torch.float32
        self.fp4_codes = torch.empty((m, k // 2), dtype=u8, device=dev) if nvfp4 else None
        self.fp4_scales = torch.zeros(fp4_scale_bytes(m, k), dtype=u8, device=dev) if nvfp4 else None
        self.tensor_amax = torch.zeros(1, dtype=f32, device=dev) if nvfp4 else None
        self.tensor_scale = torch.zeros(1, dtype=f32, device=dev) if nvfp4 else None
        self.i8_codes = torch.empty((m, k), dtype=torch.int8, device=dev) if int8 else None
        self.row_scale = torch.empty(m, dtype=f32, device=dev) if int8 else None
        self.rotated = torch.empty((m, k), dtype=f32, device=dev) if rotated else None

    def c(self) -> QAct:
        return QAct(*[_p(getattr(self, f)) for f, _ in QAct._fields_])


class PackedWeights:
    """Device buffers of one packed linear layer W [N, K]."""

    def __init__(self, n: int, k: int, device="cuda"):
        self.n, self.k = n, k
        dev = torch.device(device)
        self.fp4_codes = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
        self.fp4_scales = torch.zeros(fp4_scale_bytes(n, k), dtype=torch.uint8, device=dev)
        self.fp4_amax = torch.zeros(1, dtype=torch.float32, device=dev)
        self.fp4_tensor_scale = torch.zeros(1, dtype=torch.float32, device=dev)
        self.i4_codes = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
        self.i4_scales = torch.empty((k // 128, n), dtype=torch.float32, device=dev)
        self.bf16_w = torch.empty((n, k), dtype=torch.bfloat16, device=dev)

    def c(self) -> Weights:
        return Weights(*[_p(getattr(self, f)) for f, _ in Weights._fields_])


def pack_weights(w: torch.Tensor, had_block: int, out: PackedWeights | None = None, stream=None) -> PackedWeights:
    assert w.dtype == torch.float32 and w.is_contiguous()
    n, k = w.shape
    out = out or PackedWeights(n, k, w.device)
    cw = out.c()
    check(_lib.sixbit_pack_weights(_p(w), n, k, had_block, C.byref(cw), None, _stream(stream)), "pack_weights")
    return out


def hadamard_quant(x: torch.Tensor, had_block: int, mode: int, out: QActTensors | None = None, mode_dev=None,
                   tamax=None, stream=None) -> QActTensors:
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    m, k = x.shape
    out = out or QActTensors(m, k, x.device)
    ca = out.c()
    check(_lib.sixbit_hadamard_quant(_p(x), m, k, had_block, mode, _p(mode_dev), _p(tamax), C.byref(ca), None,
                                     _stream(stream)), "hadamard_quant")
    return out


def qgemm(a: QActTensors | None, x_bf16, w: PackedWeights, mode: int, epilogue: int = EPI_NONE, residual=None,
          out=None, out_f32: bool = False, acc_dbg=None, mode_dev=None, err=None, stream=None, m: int | None = None,
          ws=None):
    """ws: the INT8 kind's workspace (qgemm_workspace_bytes); by default the device's shared one."""
    n, k = w.n, w.k
    if ws is None and (mode == MODE_INT8 or mode_dev is not None):
        ws = workspace(n, k, w.bf16_w.device)
    m = m if m is not None else (a.m if a is not None else x_bf16.shape[0])
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32 if out_f32 else torch.bfloat16, device=w.bf16_w.device)
    ca = a.c() if a is not None else None
    cw = w.c()
    y = out if out.dtype == torch.bfloat16 else None
    yf = out if out.dtype == torch.float32 else None
    check(_lib.sixbit_qgemm(C.byref(ca) if ca is not None else None, _p(x_bf16), C.byref(cw), m, n, k, mode,
                            _p(mode_dev), epilogue, _p(residual), _p(y), _p(yf), _p(acc_dbg), _p(ws), _p(err),
                            _stream(stream)), "qgemm")
    return out


def qgemm_rotamax(a: QActTensors, w: PackedWeights, had_block: int, amax_out: torch.Tensor, epilogue: int = EPI_NONE,
                  residual=None, out=None, mode_dev=None, err=None, stream=None, m: int | None = None):
    """NVFP4 qgemm whose epilogue also writes the rotated amax of its bf16 output to amax_out."""
    n, k = w.n, w.k
    m = m if m is not None else a.m
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=w.bf16_w.device)
    ca, cw = a.c(), w.c()
    check(_lib.sixbit_qgemm_rotamax(C.byref(ca), C.byref(cw), m, n, k, _p(mode_dev), epilogue, _p(residual), _p(out),
                                    had_block, _p(amax_out), _p(err), _stream(stream)), "qgemm_rotamax")
    return out


def qgemm_blockstats(a: QActTensors | None, x_bf16, w: PackedWeights, mode: int, residual, out, delta_cache,
                     parts, mode_dev=None, err=None, stream=None, m: int | None = None, ws=None):
    """qgemm with the RESIDUAL epilogue that also updates delta_cache (Delta_prev -> Delta) and writes
    the block statistics' partial rows to parts (blockstats_parts_bytes(); fold with block_stats_parts
    or dit_block_end_parts)."""
    n, k = w.n, w.k
    if ws is None and (mode == MODE_INT8 or mode_dev is not None):
        ws = workspace(n, k, w.bf16_w.device)
    m = m if m is not None else (a.m if a is not None else x_bf16.shape[0])
    ca = a.c() if a is not None else None
    cw = w.c()
    check(_lib.sixbit_qgemm_blockstats(C.byref(ca) if ca is not None else None, _p(x_bf16), C.byref(cw), m, n, k,
                                       mode, _p(mode_dev), _p(residual), _p(out), _p(delta_cache), _p(parts), _p(ws),
                                       _p(err), _stream(stream)), "qgemm_blockstats")
    return out


def blockstats_parts_bytes() -> int:
    return int(_lib.sixbit_blockstats_parts_bytes())


def new_blockstats_parts(device="cuda") -> torch.Tensor:
    return torch.zeros(blockstats_parts_bytes(), dtype=torch.uint8, device=device)


def block_stats_parts(parts: torch.Tensor, n: int, stats: torch.Tensor, stream=None):
    check(_lib.sixbit_block_stats_parts(_p(parts), n, _p(stats), None, _stream(stream)), "block_stats_parts")
    return stats


def tensor_stats(x: torch.Tensor, out: torch.Tensor, scratch: torch.Tensor, stream=None) -> torch.Tensor:
    check(_lib.sixbit_tensor_stats(_p(x), x.numel(), _p(out), _p(scratch), None, _stream(stream)), "tensor_stats")
    return out


def block_stats(x_in, x_out, delta_cache, stats: torch.Tensor, scratch: torch.Tensor, mode_dev=None, stream=None):
    check(_lib.sixbit_block_stats(_p(x_in), _p(x_out), _p(delta_cache), x_in.numel(), _p(mode_dev), _p(stats),
                                  _p(scratch), None, _stream(stream)), "block_stats")
    return stats


def block_stats_noalloc(x_in, x_out, delta_cache, stats: torch.Tensor, mode_dev=None, stream=None):
    """sixbit_block_stats without caller scratch (the library's fixed array is used).

    For callers that cannot allocate device memory for scratch; calls must not
    overlap on the GPU, since they share that array.
    """
    check(_lib.sixbit_block_stats_noalloc(_p(x_in), _p(x_out), _p(delta_cache), x_in.numel(), _p(mode_dev),
                                          _p(stats), None, _stream(stream)), "block_stats_noalloc")
    return stats


def skip_apply(x_in, delta_cache, x_out, stats: torch.Tensor, scratch: torch.Tensor, mode_dev=None, stream=None):
    check(_lib.sixbit_skip_apply(_p(x_in), _p(delta_cache), _p(x_out), x_in.numel(), _p(mode_dev), _p(stats),
                                 _p(scratch), None, _stream(stream)), "skip_apply")
    return x_out


DELTA_BF16, DELTA_MXFP8 = 0, 1
MX_BLOCK = 32


def mxfp8_cache(n: int, device, blocks: int | None = None):
    """A zeroed MXFP8 Delta cache of n elements (per block when `blocks` is given): (codes, scales) uint8."""
    assert n % MX_BLOCK == 0
    lead = () if blocks is None else (blocks,)
    return (torch.zeros(lead + (n,), dtype=torch.uint8, device=device),
            torch.zeros(lead + (n // MX_BLOCK,), dtype=torch.uint8, device=device))


def block_stats_mxfp8(x_in, x_out, codes, scales, stats: torch.Tensor, scratch: torch.Tensor, mode_dev=None,
                      stream=None):
    """sixbit_block_stats_mxfp8: the Delta cache in MXFP8 (codes [n] uint8, scales [n / 32] uint8)."""
    n = x_in.numel()
    assert codes.dtype == torch.uint8 and codes.numel() == n and scales.numel() == n // MX_BLOCK
    check(_lib.sixbit_block_stats_mxfp8(_p(x_in), _p(x_out), _p(codes), _p(scales), n, _p(mode_dev), _p(stats),
                                        _p(scratch), None, _stream(stream)), "block_stats_mxfp8")
    return stats


def skip_apply_mxfp8(x_in, codes, scales, x_out, stats: torch.Tensor, scratch: torch.Tensor, mode_dev=None,
                     stream=None):
    n = x_in.numel()
    assert codes.dtype == torch.uint8 and codes.numel() == n and scales.numel() == n // MX_BLOCK
    check(_lib.sixbit_skip_apply_mxfp8(_p(x_in), _p(codes), _p(scales), _p(x_out), n, _p(mode_dev), _p(stats),
                                       _p(scratch), None, _stream(stream)), "skip_apply_mxfp8")
    return x_out


def policy_cfg(gamma_thr=0.1, cos_thr=0.99, err_cap=0.05, pdr_ratio=30.0, near_rel=1e-6, refresh_bf16=False):
    return PolicyCfg(gamma_thr, cos_thr, err_cap, pdr_ratio, near_rel, int(refresh_bf16), 0)


def policy_step(cfg: PolicyCfg, state: torch.Tensor, last_stats: torch.Tensor, in_stats: torch.Tensor,
                mode_word: torch.Tensor, stream=None):
    check(_lib.sixbit_policy_step(C.byref(cfg), _p(state), _p(last_stats), _p(in_stats), _p(mode_word), None,
                                  _stream(stream)), "policy_step")
    return mode_word


def policy_cfgs_tensor(cfgs, device="cuda") -> torch.Tensor:
    """Per-block thresholds as the device array sixbit_dit_blocks.block_cfg points to."""
    raw = b"".join(bytes(c) for c in cfgs)
    return torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(device)


def dit_blocks(states, stats, modes, run_len, in_stats0, x0, buf0, buf1, deltas, conds=None,
               delta_scales=None, block_cfg=None) -> DitBlocks:
    """The sixbit_dit_blocks record of a stack of residual blocks (device tensors; deltas [L, ...];
    run_len: int32 [L], zeroed; conds: int64 [L] graph condition handles, or None).  The Delta
    cache is bf16 (deltas bf16 [L, n]) or, with delta_scales, MXFP8 (deltas uint8 [L, n] E4M3
    codes, delta_scales uint8 [L, n / 32] E8M0 codes).  block_cfg: the policy_cfgs_tensor of L
    per-block thresholds, or None."""
    L = states.shape[0]
    n = x0.numel()
    assert stats.shape[0] == L and modes.numel() == L and run_len.numel() == L and deltas.shape[0] == L
    assert run_len.dtype == torch.int32 and run_len.is_contiguous() and deltas.numel() == L * n
    assert in_stats0.dtype == torch.float64 and in_stats0.numel() >= 4
    assert conds is None or (conds.dtype == torch.int64 and conds.numel() == L)
    if delta_scales is None:
        assert deltas.dtype == torch.bfloat16
        fmt = DELTA_BF16
    else:
        assert deltas.dtype == torch.uint8 and delta_scales.dtype == torch.uint8
        assert delta_scales.is_contiguous() and delta_scales.numel() == L * (n // MX_BLOCK)
        fmt = DELTA_MXFP8
    assert block_cfg is None or (block_cfg.dtype == torch.uint8 and block_cfg.numel() == L * C.sizeof(PolicyCfg))
    return DitBlocks(_p(states), _p(stats), _p(modes), _p(in_stats0), _p(x0),
                     (C.c_void_p * 2)(buf0.data_ptr(), buf1.data_ptr()), _p(deltas), _p(delta_scales), _p(run_len),
                     _p(conds), _p(block_cfg), n, L, fmt)


def dit_begin(cfg: PolicyCfg, blocks: DitBlocks, scratch: torch.Tensor, err=None, stream=None):
    """sixbit_dit_begin: statistics of the step input, then block 0's decision."""
    check(_lib.sixbit_dit_begin(C.byref(cfg), C.byref(blocks), _p(scratch), _p(err), _stream(stream)), "dit_begin")


def dit_block_end_parts(cfg: PolicyCfg, blocks: DitBlocks, l: int, parts: torch.Tensor, err=None, stream=None):
    """sixbit_dit_block_end_parts: fold the statistics block l's down projection wrote to parts, then
    block l+1's decision (nothing when block l skipped)."""
    check(_lib.sixbit_dit_block_end_parts(C.byref(cfg), C.byref(blocks), l, _p(parts), _p(err), _stream(stream)),
          "dit_block_end_parts")


def dit_block_end(cfg: PolicyCfg, blocks: DitBlocks, l: int, scratch: torch.Tensor, err=None, stream=None):
    """sixbit_dit_block_end: block l's statistics and Delta update (if it computed), then block l+1's decision."""
    check(_lib.sixbit_dit_block_end(C.byref(cfg), C.byref(blocks), l, _p(scratch), _p(err), _stream(stream)),
          "dit_block_end")


def dit_skip_run(cfg: PolicyCfg, blocks: DitBlocks, l: int, scratch: torch.Tensor, err=None, stream=None):
    """sixbit_dit_skip_run: the run of skips block l starts (if any), then the decisions up to its end + 1."""
    check(_lib.sixbit_dit_skip_run(C.byref(cfg), C.byref(blocks), l, _p(scratch), _p(err), _stream(stream)),
          "dit_skip_run")


def graph_cond_create(stream, nbranches: int) -> int:
    """A conditional handle in the graph `stream` is capturing (default value: no body)."""
    h = C.c_uint64()
    check(_lib.sixbit_graph_cond_create(C.c_void_p(stream.cuda_stream), nbranches, C.byref(h)), "graph_cond_create")
    return int(h.value)


class GraphSwitch:
    """A device-selected branch in the CUDA graph being captured on `stream` (sixbit_graph_switch_*).

    Body i runs when the low byte of mode_word equals first_mode + i.  Use
    ``with sw.branch(i):`` to capture body i: inside it the current torch
    stream is `body_stream`, which is capturing into that body.
    """

    def __init__(self, stream, body_stream, mode_word: torch.Tensor | None, first_mode: int, nbranches: int,
                 cond: int | None = None):
        """With cond (a handle from graph_cond_create, set by a kernel already captured) no selector is added."""
        self.h = C.c_void_p()
        self.body_stream = body_stream
        if cond is not None:
            check(_lib.sixbit_graph_switch_begin_cond(C.c_void_p(stream.cuda_stream),
                                                      C.c_void_p(body_stream.cuda_stream), cond, nbranches,
                                                      C.byref(self.h)), "graph_switch_begin_cond")
        else:
            check(_lib.sixbit_graph_switch_begin(C.c_void_p(stream.cuda_stream),
                                                 C.c_void_p(body_stream.cuda_stream), _p(mode_word), first_mode,
                                                 nbranches, C.byref(self.h)), "graph_switch_begin")

    def branch(self, i: int):
        sw = self

        class _Branch:
            def __enter__(self):
                s = C.c_void_p()
                check(_lib.sixbit_graph_branch_begin(sw.h, i, C.byref(s)), "graph_branch_begin")
                self.ctx = torch.cuda.stream(sw.body_stream)
                self.ctx.__enter__()
                return sw.body_stream

            def __exit__(self, *exc):
                self.ctx.__exit__(*exc)
                check(_lib.sixbit_graph_branch_end(sw.h), "graph_branch_end")
                return False

        return _Branch()

    def close(self):
        check(_lib.sixbit_graph_switch_end(self.h), "graph_switch_end")


def new_stats(device="cuda", count: int = 1) -> torch.Tensor:
    """Zeroed device storage for `count` sixbit_stats records (float64 x 8 each)."""
    return torch.zeros((count, 8), dtype=torch.float64, device=device)


def new_policy_state(device="cuda", count: int = 1) -> torch.Tensor:
    """Zeroed device storage for `count` sixbit_policy_state records (80 bytes each)."""
    assert C.sizeof(PolicyState) == 80
    return torch.zeros((count, 80), dtype=torch.uint8, device=device)


def decode_state(raw: torch.Tensor) -> PolicyState:
    b = bytes(raw.cpu().numpy().tobytes())
    return PolicyState.from_buffer_copy(b)


def new_scratch(n: int, device="cuda") -> torch.Tensor:
    """Zeroed scratch for the statistics kernels (its counter must start at zero)."""
    return torch.zeros(stats_scratch_bytes(n), dtype=torch.uint8, device=device)
