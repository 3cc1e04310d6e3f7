"""Parity at the full sizes of the FFN-pair and 5B-shaped GEMM-sweep workloads (sampled rows).

FFN pair (17776 tokens, 1920 -> 7680 -> 1920): the up projection with its
GELU epilogue and the down projection with its residual epilogue, in both
per-layer mode orders (NVFP4 up / INT8 down and the reverse).  The down
projection reads a seeded stand-in for the hidden activations, so the oracle
never sees a GPU tensor.  GEMM sweep: K = N = 3072, M from 1024 to 35552,
NVFP4 and INT8.  The GPU runs every full-size kernel; the oracle checks 32
seeded rows (the last row included) against the float64 references.  For
NVFP4 the oracle takes the tensor amax over all rows (rotated in chunks) and
quantizes the sampled rows with that tensor scale.
"""
import numpy as np
import pytest
import torch

import synthgen
from oracle import gemm, quant
from oracle.hadamard import fwht_blocks

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def ops():
    from video_dit_mixed_gb300 import ops as o
    return o


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


def _rows(m, seed):
    r = np.unique((synthgen.uniform(seed, 9, 32) * m).astype(np.int64))
    r[-1] = m - 1
    return np.unique(r)


def _rotated_amax(x, b, chunk=2048):
    a = 0.0
    for i in range(0, x.shape[0], chunk):
        a = max(a, float(np.abs(fwht_blocks(x[i:i + chunk], b)).max()))
    return np.float32(a)


def _ref_rows(mode, x, w, b, rows, epi, residual=None):
    if mode == "nvfp4":
        s_t = quant.tensor_scale(_rotated_amax(x, b))
        qx = quant.hadamard_quant(x[rows], b, "nvfp4", s_t=s_t)
        pw = quant.pack_weights(w, b)["nvfp4"]
        ref, bound = gemm.nvfp4_gemm_ref(qx["codes"], qx["scales"], qx["s_t"], pw["codes"], pw["scales"], pw["s_t"])
    else:
        qx = quant.hadamard_quant(x[rows], b, "int8")
        i4 = quant.pack_weights(w, b)["int4"]
        ref, bound, _ = gemm.int8_gemm_ref(qx["q"], qx["s"], i4["q"], i4["s"])
    out = gemm.epilogue(ref, epi, None if residual is None else residual[rows])
    return out, bound


def _half_ulp_bf16(v):
    a = np.abs(v).astype(np.float64)
    return 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 8)


def _gpu(ops, mode, x, w, b, epi, residual=None):
    m = x.shape[0]
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    xd = _dev_bf16(x)
    code = ops.MODE_NVFP4 if mode == "nvfp4" else ops.MODE_INT8
    qa = ops.hadamard_quant(xd, b, code)
    res = _dev_bf16(residual) if residual is not None else None
    e = {"none": ops.EPI_NONE, "gelu": ops.EPI_GELU, "residual": ops.EPI_RESIDUAL}[epi]
    y = ops.qgemm(qa, xd, pw, code, epilogue=e, residual=res, m=m)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("up_mode,down_mode", [("nvfp4", "int8"), ("int8", "nvfp4")])
def test_ffn_pair_full_size(ops, up_mode, down_mode):
    c = synthgen.CONFIGS["ffn_2b"]
    b = c["had_block"]
    x, w_up, _ = synthgen.linear_inputs("ffn_2b")
    w_down = synthgen.weights(c["seed"], c["k"], c["n"], stream=3)
    rows = _rows(x.shape[0], 21)
    # up projection + GELU, bf16 out
    y = _gpu(ops, up_mode, x, w_up, b, "gelu")[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    ref, bound = _ref_rows(up_mode, x, w_up, b, rows, "gelu")
    err = np.abs(y - ref)
    assert np.all(err <= 1.13 * TOL * bound + 4e-7 * np.abs(ref) + _half_ulp_bf16(ref) * 1.0001 + 1e-30), err.max()
    del y
    # down projection + residual, bf16 out, from a seeded hidden tensor
    h = synthgen.ffn_hidden(c["seed"], x.shape[0], c["n"])
    y = _gpu(ops, down_mode, h, w_down, b, "residual", residual=x)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    ref, bound = _ref_rows(down_mode, h, w_down, b, rows, "residual", residual=x)
    err = np.abs(y - ref)
    assert np.all(err <= TOL * bound + 1.2e-7 * np.abs(ref) + _half_ulp_bf16(ref) * 1.0001 + 1e-30), err.max()


@pytest.mark.parametrize("mode", ["nvfp4", "int8"])
@pytest.mark.parametrize("m", [1024, 8192, 2 * synthgen.TOKENS])
def test_gemm_sweep_5b_shapes(ops, mode, m):
    b = synthgen.GEMM_SWEEP["had_block"]
    x, w = synthgen.sweep_inputs(m)
    rows = _rows(m, 31)
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    xd = _dev_bf16(x)
    code = ops.MODE_NVFP4 if mode == "nvfp4" else ops.MODE_INT8
    qa = ops.hadamard_quant(xd, b, code)
    y = ops.qgemm(qa, xd, pw, code, out_f32=True, m=m)
    torch.cuda.synchronize()
    got = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref, bound = _ref_rows(mode, x, w, b, rows, "none")
    assert np.all(np.abs(got - ref) <= TOL * bound + 1e-30)
