"""ctypes declarations of libsixbit's C ABI (include/sixbit.h), one to one."""
from __future__ import annotations

import ctypes as C
import os

from . import _build

c_p = C.c_void_p

MODE_NVFP4, MODE_INT8, MODE_BF16, MODE_SKIP = 1, 2, 3, 4
FLAG_REFRESH, FLAG_PDR, FLAG_POSTSKIP, FLAG_NEAR = 1 << 8, 1 << 9, 1 << 10, 1 << 11
EPI_NONE, EPI_GELU, EPI_RESIDUAL = 0, 1, 2
MODE_NAMES = {MODE_NVFP4: "NVFP4", MODE_INT8: "INT8", MODE_BF16: "BF16", MODE_SKIP: "SKIP"}


class QAct(C.Structure):
    _fields_ = [("fp4_codes", c_p), ("fp4_scales", c_p), ("tensor_amax", c_p), ("tensor_scale", c_p),
                ("i8_codes", c_p), ("row_scale", c_p), ("rotated", c_p)]


class Weights(C.Structure):
    _fields_ = [("fp4_codes", c_p), ("fp4_scales", c_p), ("fp4_amax", c_p), ("fp4_tensor_scale", c_p),
                ("i4_codes", c_p), ("i4_scales", c_p), ("bf16_w", c_p)]


class Stats(C.Structure):
    _fields_ = [(n, C.c_double) for n in ("sum_d2", "sum_xin2", "sum_ddp", "sum_dp2", "max_abs_out",
                                          "sum_abs_out", "count", "reserved")]


class PolicyCfg(C.Structure):
    _fields_ = [("gamma_thr", C.c_double), ("cos_thr", C.c_double), ("err_cap", C.c_double),
                ("pdr_ratio", C.c_double), ("near_rel", C.c_double), ("refresh_bf16", C.c_int32),
                ("reserved", C.c_int32)]


class PolicyState(C.Structure):
    _fields_ = [("n_computed", C.c_int32), ("skipped_last", C.c_int32), ("have_gamma", C.c_int32),
                ("pending", C.c_int32), ("gamma", C.c_double), ("cos", C.c_double), ("acc", C.c_double),
                ("last_word", C.c_int32), ("steps", C.c_int32)] + \
               [(n, C.c_int32) for n in ("n_skip", "n_refresh", "n_pdr", "n_near", "n_nvfp4", "n_int8",
                                         "n_bf16", "n_nonfinite")]


class DitBlocks(C.Structure):
    _fields_ = [("states", c_p), ("stats", c_p), ("modes", c_p), ("in_stats0", c_p),
                ("x0", c_p), ("buf", c_p * 2), ("deltas", c_p), ("delta_scales", c_p), ("run_len", c_p),
                ("conds", c_p), ("block_cfg", c_p), ("n", C.c_int64), ("L", C.c_int32), ("delta_format", C.c_int32)]


EXPORTS = {
    "sixbit_fp4_scale_bytes": (C.c_size_t, [C.c_int, C.c_int]),
    "sixbit_fp4_scale_offset": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "sixbit_stats_scratch_bytes": (C.c_size_t, [C.c_int64]),
    "sixbit_pack_weights": (C.c_int, [c_p, C.c_int, C.c_int, C.c_int, C.POINTER(Weights), c_p, c_p]),
    "sixbit_hadamard_quant": (C.c_int, [c_p, C.c_int, C.c_int, C.c_int, C.c_int, c_p, c_p,
                                        C.POINTER(QAct), c_p, c_p]),
    "sixbit_qgemm": (C.c_int, [C.POINTER(QAct), c_p, C.POINTER(Weights), C.c_int, C.c_int, C.c_int, C.c_int,
                               c_p, C.c_int, c_p, c_p, c_p, c_p, c_p, c_p, c_p]),
    "sixbit_qgemm_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int]),
    "sixbit_qgemm_rotamax": (C.c_int, [C.POINTER(QAct), C.POINTER(Weights), C.c_int, C.c_int, C.c_int, c_p, C.c_int,
                                       c_p, c_p, C.c_int, c_p, c_p, c_p]),
    "sixbit_block_stats": (C.c_int, [c_p, c_p, c_p, C.c_int64, c_p, c_p, c_p, c_p, c_p]),
    "sixbit_qgemm_blockstats": (C.c_int, [C.POINTER(QAct), c_p, C.POINTER(Weights), C.c_int, C.c_int, C.c_int,
                                          C.c_int, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p]),
    "sixbit_blockstats_parts_bytes": (C.c_size_t, []),
    "sixbit_block_stats_parts": (C.c_int, [c_p, C.c_int64, c_p, c_p, c_p]),
    "sixbit_policy_step": (C.c_int, [C.POINTER(PolicyCfg), c_p, c_p, c_p, c_p, c_p, c_p]),
    "sixbit_tensor_stats": (C.c_int, [c_p, C.c_int64, c_p, c_p, c_p, c_p]),
    "sixbit_skip_apply": (C.c_int, [c_p, c_p, c_p, C.c_int64, c_p, c_p, c_p, c_p, c_p]),
    "sixbit_block_stats_mxfp8": (C.c_int, [c_p, c_p, c_p, c_p, C.c_int64, c_p, c_p, c_p, c_p, c_p]),
    "sixbit_skip_apply_mxfp8": (C.c_int, [c_p, c_p, c_p, c_p, C.c_int64, c_p, c_p, c_p, c_p, c_p]),
    "sixbit_block_stats_noalloc": (C.c_int, [c_p, c_p, c_p, C.c_int64, c_p, c_p, c_p, c_p]),
    "sixbit_block_stats_noalloc_max_elems": (C.c_int64, []),
    "sixbit_dit_begin": (C.c_int, [C.POINTER(PolicyCfg), C.POINTER(DitBlocks), c_p, c_p, c_p]),
    "sixbit_dit_block_end": (C.c_int, [C.POINTER(PolicyCfg), C.POINTER(DitBlocks), C.c_int, c_p, c_p, c_p]),
    "sixbit_dit_block_end_parts": (C.c_int, [C.POINTER(PolicyCfg), C.POINTER(DitBlocks), C.c_int, c_p, c_p, c_p]),
    "sixbit_dit_skip_run": (C.c_int, [C.POINTER(PolicyCfg), C.POINTER(DitBlocks), C.c_int, c_p, c_p, c_p]),
    "sixbit_graph_switch_begin": (C.c_int, [c_p, c_p, c_p, C.c_int, C.c_int, C.POINTER(c_p)]),
    "sixbit_graph_cond_create": (C.c_int, [c_p, C.c_int, C.POINTER(C.c_uint64)]),
    "sixbit_graph_switch_begin_cond": (C.c_int, [c_p, c_p, C.c_uint64, C.c_int, C.POINTER(c_p)]),
    "sixbit_graph_branch_begin": (C.c_int, [c_p, C.c_int, C.POINTER(c_p)]),
    "sixbit_graph_branch_end": (C.c_int, [c_p]),
    "sixbit_graph_switch_end": (C.c_int, [c_p]),
    "sixbit_debug_gemm_timeout": (C.c_int, [C.c_uint64, C.c_int32]),
    "sixbit_check": (C.c_int, [c_p, c_p]),
    "sixbit_status_str": (C.c_char_p, [C.c_int]),
    "sixbit_launch_count": (C.c_uint64, []),
}

_lib = None


def lib(build_if_missing: bool = False):
    """The loaded libsixbit (raises if it is not built)."""
    global _lib
    if _lib is None:
        if build_if_missing:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libsixbit.so is not built ({_build.LIB}); run __graft_entry__.build()")
        h = C.CDLL(_build.LIB)
        for name, (res, args) in EXPORTS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


class SixbitError(RuntimeError):
    pass


def check(status: int, what: str) -> None:
    if status != 0:
        msg = lib().sixbit_status_str(status).decode()
        raise SixbitError(f"{what}: {msg} (status {status})")
