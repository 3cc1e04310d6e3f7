"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the method: it only draws numbers.  Every
draw is a pure function of (seed, stream, index), so any slice can be
regenerated independently, on any machine:

* splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) in counter form: r_i = mix(key + (i + 1) * gamma),
  gamma = 0x9E3779B97F4A7C15, key = mix(seed * 2**32 + stream);
* uniform  u = ((r >> 11) + 0.5) * 2**-53, in the open interval (0, 1);
* normal   Box-Muller on consecutive pairs (u1, u2):
           z0 = sqrt(-2 ln u1) cos(2 pi u2), z1 = sqrt(-2 ln u1) sin(2 pi u2);
* Laplace(0, 1)  -sign(u - 1/2) ln(1 - 2 |u - 1/2|)   (inverse CDF);
* outlier channels: the first round(p * K) channels of the permutation that
  sorts K uniforms, multiplied by a factor.

Activations are rounded to bf16 (round-to-nearest-even) because the layer's
input is a bf16 tensor; weights stay float32.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    v = np.array([((int(seed) & 0xFFFFFFFF) << 32) | (int(stream) & 0xFFFFFFFF)], dtype=np.uint64)
    return _mix(v + _GAMMA)[0]


def raw64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(_key(seed, stream) + i * _GAMMA)


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    r = raw64(seed, stream, n, start)
    return ((r >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


def laplace(seed: int, stream: int, n: int) -> np.ndarray:
    u = uniform(seed, stream, n) - 0.5
    return -np.sign(u) * np.log1p(-2.0 * np.abs(u))


def bf16_rne(x) -> np.ndarray:
    """Round finite float32 values to bf16 (RNE); returns float32 values (input preparation only)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # finite values stay below 0xFF800000, so the 32-bit sum cannot wrap
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32).reshape(x.shape)


def outlier_channels(seed: int, stream: int, k: int, frac: float) -> np.ndarray:
    n_out = int(round(frac * k))
    perm = np.argsort(uniform(seed, stream, k), kind="stable")
    return np.sort(perm[:n_out])


def activations(seed: int, m: int, k: int, dist: str = "laplace", outlier_frac: float = 0.0,
                outlier_scale: float = 1.0, stream: int = 1) -> np.ndarray:
    """bf16-valued float32 activations [m, k] with scaled outlier channels."""
    n = m * k
    v = laplace(seed, stream, n) if dist == "laplace" else normal(seed, stream, n)
    v = v.reshape(m, k)
    if outlier_frac > 0:
        ch = outlier_channels(seed, stream + 1000, k, outlier_frac)
        v[:, ch] *= outlier_scale
    return bf16_rne(v.astype(np.float32))


def weights(seed: int, n: int, k: int, std: float = 0.02, stream: int = 2) -> np.ndarray:
    """float32 weights [n, k] ~ N(0, std^2)."""
    return (normal(seed, stream, n * k) * std).astype(np.float32).reshape(n, k)


# Named workloads (shapes and distributions of the configurations in the
# design notes).  tokens = 13*30*45 video latents + 226 text tokens.
TOKENS = 13 * 30 * 45 + 226

CONFIGS = {
    # tiny single linear: X ~ N(0,1), 1% channels x20, W 512x512, block 16
    "tiny_linear": dict(seed=0, m=256, k=512, n=512, dist="normal", outlier_frac=0.01,
                        outlier_scale=20.0, had_block=16),
    # QKV-shaped linear of a 2B-parameter video DiT: Laplace X, 0.5% channels x50
    "qkv_2b": dict(seed=1, m=TOKENS, k=1920, n=5760, dist="laplace", outlier_frac=0.005,
                   outlier_scale=50.0, had_block=64),
    # FFN pair of the same model: 1920 -> 7680 -> 1920
    "ffn_2b": dict(seed=2, m=TOKENS, k=1920, n=7680, dist="laplace", outlier_frac=0.005,
                   outlier_scale=50.0, had_block=64),
}


def linear_inputs(name: str, m: int | None = None):
    """(x, w, cfg) for a named single-linear workload; ``m`` truncates the token count."""
    c = dict(CONFIGS[name])
    mm = c["m"] if m is None else m
    x = activations(c["seed"], mm, c["k"], c["dist"], c["outlier_frac"], c["outlier_scale"])
    w = weights(c["seed"], c["n"], c["k"])
    return x, w, c


# Synthetic residual-MLP DiTs: block l maps x -> x + g_l W_d GELU(W_u x).
# tokens x hidden, ffn, blocks, denoising steps; x_0 like the QKV input
# (Laplace, 0.5% channels x50); x_s = bf16(x_{s-1} + sigma_s z_s) with sigma
# falling linearly from 0.5 (s = 1) to 0.01 (last step).  gate: None (all 1)
# or (lo, hi) for a seeded log-uniform per-block gate folded into W_d.
DIT_CONFIGS = {
    # small enough for the oracle to run end to end; its 20 steps x 4 blocks
    # take every branch: PDR -> BF16, NVFP4, INT8, SKIP, refresh after skips
    "dit_tiny": dict(seed=12, tokens=256, hidden=256, ffn=1024, blocks=4, steps=20, had_block=64,
                     w_std=0.05, gate=(0.02, 0.5), outlier_frac=0.01, outlier_scale=4.0),
    "dit_2b": dict(seed=3, tokens=TOKENS, hidden=1920, ffn=7680, blocks=30, steps=50, had_block=64,
                   w_std=0.02, gate=None),
    # a deviation that exercises the NVFP4 branch: per-block residual gates
    # put Gamma around 0.1, and milder outlier channels (x2) keep the PDR
    # ratio below 30
    "dit_2b_gated": dict(seed=3, tokens=TOKENS, hidden=1920, ffn=7680, blocks=30, steps=50, had_block=64,
                         w_std=0.02, gate=(0.02, 0.5), outlier_frac=0.005, outlier_scale=2.0),
    "dit_5b": dict(seed=4, tokens=TOKENS, hidden=3072, ffn=12288, blocks=42, steps=50, had_block=64,
                   w_std=0.02, gate=None),
}


def sigmas(steps: int) -> np.ndarray:
    """sigma_s for s = 1 .. steps-1, linear from 0.5 to 0.01."""
    if steps <= 1:
        return np.zeros(0)
    return np.linspace(0.5, 0.01, steps - 1)


def dit_gates(name: str) -> np.ndarray:
    c = DIT_CONFIGS[name]
    if c["gate"] is None:
        return np.ones(c["blocks"])
    lo, hi = c["gate"]
    u = uniform(c["seed"], 40, c["blocks"])
    return np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))


def dit_weights(name: str):
    """[(W_up [ffn, hidden], W_down [hidden, ffn])] float32, the gate folded into W_down."""
    c = DIT_CONFIGS[name]
    g = dit_gates(name)
    out = []
    for l in range(c["blocks"]):
        wu = (normal(c["seed"], 100 + 2 * l, c["ffn"] * c["hidden"]) * c["w_std"]).astype(np.float32)
        wd = (normal(c["seed"], 101 + 2 * l, c["hidden"] * c["ffn"]) * c["w_std"] * g[l]).astype(np.float32)
        out.append((wu.reshape(c["ffn"], c["hidden"]), wd.reshape(c["hidden"], c["ffn"])))
    return out


def dit_trajectory(name: str):
    """List of bf16-valued float32 inputs x_0 .. x_{steps-1} [tokens, hidden]."""
    c = DIT_CONFIGS[name]
    x = activations(c["seed"], c["tokens"], c["hidden"], "laplace", c.get("outlier_frac", 0.005),
                    c.get("outlier_scale", 50.0))
    xs = [x]
    n = c["tokens"] * c["hidden"]
    for s, sg in enumerate(sigmas(c["steps"]), start=1):
        z = normal(c["seed"], 1000 + s, n).reshape(c["tokens"], c["hidden"])
        x = bf16_rne((x + sg * z).astype(np.float32))
        xs.append(x)
    return xs


# The 5B-shaped GEMM sweep: X [M, 3072] like the QKV input, W [3072, 3072].
GEMM_SWEEP = dict(seed=5, ms=(1024, 2048, 4096, 8192, TOKENS, 2 * TOKENS), k=3072, n=3072, had_block=64)


def sweep_inputs(m: int):
    c = GEMM_SWEEP
    x = activations(c["seed"], m, c["k"], "laplace", 0.005, 50.0)
    w = weights(c["seed"], c["n"], c["k"])
    return x, w


def ffn_hidden(seed: int, m: int, f: int, tile: int = 8):
    """A bf16 stand-in for GELU(W_up x) [m, f]: GELU of N(0, 0.9^2) samples (tanh form, input prep only).

    f/tile columns are drawn and repeated `tile` times along the row (cheap to
    generate at 17776 x 7680; the repetition does not matter to a GEMM test).
    """
    fc = f // tile
    z = normal(seed, 7, m * fc).reshape(m, fc) * 0.9
    g = 0.5 * z * (1.0 + np.tanh(0.7978845608028654 * (z + 0.044715 * z ** 3)))
    return np.tile(bf16_rne(g.astype(np.float32)), (1, tile))
