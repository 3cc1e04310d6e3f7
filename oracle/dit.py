"""A synthetic residual-MLP diffusion transformer run end to end (oracle; test infrastructure only).

Each block maps x -> x + W_d . GELU(W_u . x); per denoising step and block
the policy ("6Bit-Diffusion" technical summary sections 2.A-2.C; popular
summary sections 1-3) picks NVFP4 / INT8 / BF16 compute or a TDC skip, both
linear layers of a computed block use the chosen precision, and the block's
statistics (Gamma, delta cosine, the next block's input outlier ratio) feed
the next decision.  The GEMM outputs are the float64 references rounded to
FP32 and then to bf16, as a bf16 activation tensor is stored.

Per-depth thresholds: `cfg` may be one PolicyConfig for every block or a
list with one per block (the finding that blocks at different depths differ
in temporal stability, popular summary section 5, read as: each block may
carry its own thresholds under the same rules).

The delta cache is kept in bf16, or (delta_format="mxfp8") in MXFP8: the
fresh bf16 delta is used as it is by the block statistics and then encoded;
the previous delta enters the statistics, and a skip, dequantized.

This chains every other oracle module; it is compared with the GPU path on
small sizes only.
"""
from __future__ import annotations

import numpy as np

from . import gemm, policy, quant, stats
from .formats import bf16_round, mxfp8_decode, mxfp8_encode


def _round_bf16(v64):
    return bf16_round(np.asarray(v64, dtype=np.float64).astype(np.float32))


def linear(x, pk, mode, b, epilogue, residual=None):
    """One quantized linear layer in the given mode; returns bf16-valued float32."""
    if mode == policy.NVFP4:
        q = quant.hadamard_quant(x, b, "nvfp4")
        nv = pk["nvfp4"]
        ref, _ = gemm.nvfp4_gemm_ref(q["codes"], q["scales"], q["s_t"], nv["codes"], nv["scales"], nv["s_t"])
    elif mode == policy.INT8:
        q = quant.hadamard_quant(x, b, "int8")
        i4 = pk["int4"]
        ref, _, _ = gemm.int8_gemm_ref(q["q"], q["s"], i4["q"], i4["s"])
    elif mode == policy.BF16:
        ref = np.asarray(x, np.float64) @ pk["bf16"].astype(np.float64).T
    else:
        raise ValueError(mode)
    return _round_bf16(gemm.epilogue(ref, epilogue, residual))


class OracleDiT:
    def __init__(self, weights, had_block, cfg: policy.PolicyConfig | None = None, delta_format: str = "bf16"):
        """weights: list of (W_up [F, H], W_down [H, F]) float32 per block."""
        if delta_format not in ("bf16", "mxfp8"):
            raise ValueError(delta_format)
        self.b = had_block
        self.delta_format = delta_format
        self.L = len(weights)
        cfg = cfg or policy.PolicyConfig()
        self.cfgs = list(cfg) if isinstance(cfg, (list, tuple)) else [cfg] * self.L
        if len(self.cfgs) != self.L:
            raise ValueError("one policy configuration per block")
        self.cfg = self.cfgs[0]
        self.packs = [(quant.pack_weights(wu, had_block), quant.pack_weights(wd, had_block)) for wu, wd in weights]
        self.states = [policy.PolicyState() for _ in range(self.L)]
        self.deltas = [None] * self.L
        self.trace = []          # per step: list of Decision per block

    def step(self, x0):
        x = np.asarray(x0, np.float32)
        ratio = stats.outlier_ratio(stats.tensor_stats(x))
        decisions = []
        for l in range(self.L):
            st = self.states[l]
            d = policy.decide(st, ratio, self.cfgs[l])
            decisions.append(d)
            if self.deltas[l] is None:
                self.store_delta(l, np.zeros_like(x))
            if d.mode == policy.SKIP:
                out = stats.skip_apply(x, self.cached_delta(l))
                out_stats = stats.tensor_stats(out)
            else:
                pu, pd = self.packs[l]
                h = linear(x, pu, d.mode, self.b, "gelu")
                out = linear(h, pd, d.mode, self.b, "residual", x)
                bs = stats.block_stats(x, out, self.cached_delta(l))
                self.store_delta(l, bs["delta"])
                policy.fold(st, bs["gamma"], bs["cos"])
                out_stats = bs["out"]
            ratio = stats.outlier_ratio(out_stats)
            x = out
        self.trace.append(decisions)
        return x

    def store_delta(self, l, d):
        """Keeps block l's bf16 delta in the cache's format."""
        d = np.asarray(d, np.float32)
        self.deltas[l] = (d.copy(), None) if self.delta_format == "bf16" else (d.shape, mxfp8_encode(d))

    def cached_delta(self, l):
        """Block l's cached delta as float32 values (dequantized for MXFP8; exact in float32)."""
        a, enc = self.deltas[l]
        if enc is None:
            return a
        return mxfp8_decode(*enc).astype(np.float32).reshape(a)
