"""Parity: tcgen05 quantized GEMMs (NVFP4 W4A4, INT8 W4A8, BF16) vs the float64 oracle.

Bar: FP32 output within 1e-5 * sum_k |a_k b_k| of the exact value (before
bf16 rounding); bf16 output within that bound plus half a bf16 ulp; INT8
group accumulators bit-exact.  Both sides quantize the same seeded inputs
independently (the quantizers are checked bit-exact elsewhere).
"""
import numpy as np
import pytest
import torch

import synthgen
from oracle import formats, gemm, quant
from tests._layouts import bf16_bits_to_f32

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def ops():
    from video_dit_mixed_gb300 import ops as o
    return o


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


def _ref(mode, x, w, b):
    """(ref, bound, extra) from the oracle on the same seeded inputs."""
    if mode == "nvfp4":
        qx = quant.hadamard_quant(x, b, "nvfp4")
        pw = quant.pack_weights(w, b)["nvfp4"]
        r, bd = gemm.nvfp4_gemm_ref(qx["codes"], qx["scales"], qx["s_t"], pw["codes"], pw["scales"], pw["s_t"])
        return r, bd, None
    if mode == "int8":
        qx = quant.hadamard_quant(x, b, "int8")
        i4 = quant.pack_weights(w, b)["int4"]
        r, bd, acc = gemm.int8_gemm_ref(qx["q"], qx["s"], i4["q"], i4["s"])
        return r, bd, acc
    r, bd = gemm.bf16_gemm_ref(x, w)
    return r, bd, None


def _half_ulp_bf16(v):
    a = np.abs(v).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def _assert_close(y, ref, tol_abs, what):
    err = np.abs(y.astype(np.float64) - ref)
    bad = err > tol_abs
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {tuple(i)}: "
                             f"got {y[tuple(i)]!r} ref {ref[tuple(i)]!r} tol {tol_abs[tuple(i)]!r}")


MODES = {"nvfp4": 1, "int8": 2, "bf16": 3}
SHAPES = [(256, 512, 512, 16), (200, 144, 384, 64), (129, 256, 1920, 64), (64, 128, 7680, 64),
          (300, 640, 256, 256), (1, 16, 128, 16)]


def _run(ops, mode, x, w, b, epi=0, residual=None, out_f32=True, acc=False):
    m, k = x.shape
    n = w.shape[0]
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    xd = _dev_bf16(x)
    qa = None
    if mode != "bf16":
        qa = ops.hadamard_quant(xd, b, MODES[mode])
    acc_dbg = torch.zeros((k // 128, m, n), dtype=torch.int32, device="cuda") if acc else None
    res = _dev_bf16(residual) if residual is not None else None
    y = ops.qgemm(qa, xd, pw, MODES[mode], epilogue=epi, residual=res, out_f32=out_f32, acc_dbg=acc_dbg, m=m)
    torch.cuda.synchronize()
    y = y.float().cpu().numpy() if not out_f32 else y.cpu().numpy()
    return y, (acc_dbg.cpu().numpy() if acc else None)


@pytest.mark.parametrize("mode", ["nvfp4", "int8", "bf16"])
@pytest.mark.parametrize("m,n,k,b", SHAPES)
def test_gemm_fp32_within_bound(ops, mode, m, n, k, b):
    x = synthgen.activations(400 + m, m, k, "laplace", 0.005, 50.0)
    w = synthgen.weights(500 + n, n, k)
    y, acc = _run(ops, mode, x, w, b, acc=(mode == "int8"))
    ref, bound, acc_ref = _ref(mode, x, w, b)
    _assert_close(y, ref, TOL * bound + 1e-30, f"{mode} {m}x{n}x{k}")
    if mode == "int8":
        np.testing.assert_array_equal(acc, acc_ref.astype(np.int64))


@pytest.mark.parametrize("mode", ["nvfp4", "int8", "bf16"])
@pytest.mark.parametrize("m,n,k,b", SHAPES)
def test_gemm_bf16_output_ragged(ops, mode, m, n, k, b):
    """bf16 Y at ragged M and N (N = 144 and 16 end in half of a 32-column
    output box; the BF16 kind stores through TMA, which must clip at N and M
    rather than spill into the next row or past the last)."""
    x = synthgen.activations(600 + m, m, k, "laplace", 0.005, 50.0)
    w = synthgen.weights(700 + n, n, k)
    ref, bound, _ = _ref(mode, x, w, b)
    y, _ = _run(ops, mode, x, w, b, out_f32=False)
    _assert_close(y, ref, TOL * bound + _half_ulp_bf16(ref) * 1.0001 + 1e-30, f"{mode} bf16 {m}x{n}x{k}")
    r = synthgen.activations(800 + m, m, n, "normal", 0.0, 1.0)
    y, _ = _run(ops, mode, x, w, b, epi=2, residual=r, out_f32=False)
    e = gemm.epilogue(ref, "residual", r)
    _assert_close(y, e, TOL * bound + 1.2e-7 * np.abs(e) + _half_ulp_bf16(e) * 1.0001 + 1e-30, "residual")


@pytest.mark.parametrize("mode", ["nvfp4", "int8", "bf16"])
def test_gemm_epilogues_bf16_output(ops, mode):
    m, n, k, b = 200, 256, 512, 64
    x = synthgen.activations(41, m, k, "laplace", 0.005, 50.0)
    w = synthgen.weights(42, n, k)
    ref, bound, _ = _ref(mode, x, w, b)
    # GELU: |GELU'| <= 1.13; plus a few FP32 ulps for erff and the products
    y, _ = _run(ops, mode, x, w, b, epi=1, out_f32=False)
    g = gemm.gelu(ref)
    _assert_close(y, g, 1.13 * TOL * bound + 4e-7 * np.abs(g) + _half_ulp_bf16(g) * 1.0001 + 1e-30, "gelu")
    r = synthgen.activations(43, m, n, "normal", 0.0, 1.0)
    y, _ = _run(ops, mode, x, w, b, epi=2, residual=r, out_f32=False)
    e = gemm.epilogue(ref, "residual", r)
    _assert_close(y, e, TOL * bound + 1.2e-7 * np.abs(e) + _half_ulp_bf16(e) * 1.0001 + 1e-30, "residual")


def test_int8_group_sums_at_the_extremes(ops):
    """All activation codes +-127 and weight codes +-7: the largest group sums."""
    m, n, k, b = 128, 128, 512, 16
    from oracle.hadamard import fwht_blocks
    sgn = np.where(synthgen.uniform(5, 1, m * k).reshape(m, k) < 0.5, -1.0, 1.0)
    y = (sgn * 4.0).astype(np.float32)          # every rotated value has |y| = row amax -> code +-127
    x = fwht_blocks(y, b)
    assert np.array_equal(formats.bf16_round(x), x)
    flip = np.where(synthgen.uniform(6, 1, n) < 0.5, -1.0, 1.0)
    wsg = (sgn * flip[:, None]).astype(np.float32)   # row j of W matches row j of X up to sign
    w = fwht_blocks(wsg * 0.25, b)              # rotated weight = +-0.25 -> INT4 codes +-7
    y_gpu, acc = _run(ops, "int8", x, w, b, acc=True)
    ref, bound, acc_ref = _ref("int8", x, w, b)
    assert np.abs(acc_ref).max() > 100000
    np.testing.assert_array_equal(acc, acc_ref.astype(np.int64))
    _assert_close(y_gpu, ref, TOL * bound + 1e-30, "int8 extremes")


@pytest.mark.parametrize("mode", ["nvfp4", "int8", "bf16"])
def test_qkv_full_size_sampled_rows(ops, mode):
    """Full QKV-shaped problem (17776 x 5760 x 1920); 64 seeded rows checked against the oracle."""
    x, w, c = synthgen.linear_inputs("qkv_2b")
    b = c["had_block"]
    y, _ = _run(ops, mode, x, w, b, out_f32=True)
    rows = np.sort((synthgen.uniform(77, 9, 64) * x.shape[0]).astype(np.int64))
    rows[-1] = x.shape[0] - 1                     # the ragged last tile
    if mode == "nvfp4":
        qx = quant.hadamard_quant(x, b, "nvfp4")
        pw = quant.pack_weights(w, b)["nvfp4"]
        ref, bound = gemm.nvfp4_gemm_ref(qx["codes"][rows], qx["scales"][rows], qx["s_t"],
                                         pw["codes"], pw["scales"], pw["s_t"])
    elif mode == "int8":
        qx = quant.hadamard_quant(x[rows], b, "int8")   # per-row scales: rows are independent
        i4 = quant.pack_weights(w, b)["int4"]
        ref, bound, _ = gemm.int8_gemm_ref(qx["q"], qx["s"], i4["q"], i4["s"])
    else:
        ref, bound = gemm.bf16_gemm_ref(x[rows], w)
    _assert_close(y[rows], ref, TOL * bound + 1e-30, f"qkv {mode}")


def test_device_mode_word_selects_the_kernel(ops):
    m, n, k, b = 128, 128, 256, 16
    x = synthgen.activations(61, m, k, "laplace", 0.0, 1.0)
    w = synthgen.weights(62, n, k)
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    xd = _dev_bf16(x)
    for mode in ("nvfp4", "int8", "bf16"):
        word = torch.tensor([MODES[mode]], dtype=torch.int32, device="cuda")
        qa = ops.QActTensors(m, k)
        ops.hadamard_quant(xd, b, 0, out=qa, mode_dev=word)
        y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        ops.qgemm(qa, xd, pw, 0, out=y, mode_dev=word)
        torch.cuda.synchronize()
        ref, bound, _ = _ref(mode, x, w, b)
        _assert_close(y.cpu().numpy(), ref, TOL * bound + 1e-30, f"device mode {mode}")
    word = torch.tensor([4], dtype=torch.int32, device="cuda")          # SKIP: nothing written
    y = torch.full((m, n), 7.0, dtype=torch.float32, device="cuda")
    ops.qgemm(qa, xd, pw, 0, out=y, mode_dev=word)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


@pytest.mark.parametrize("m,n,k,b,epi", [(300, 256, 384, 64, "gelu"), (17, 512, 256, 16, "none"),
                                         (1000, 7680, 1920, 64, "gelu")])
def test_rotamax_epilogue_equals_quantizer_amax_pass(m, n, k, b, epi):
    """qgemm_rotamax: the same Y as the NVFP4 qgemm, and an amax equal to the quantizer's own
    amax pass over that Y (bit for bit)."""
    from video_dit_mixed_gb300 import ops
    x = synthgen.activations(77 + m, m, k, "laplace", 0.005, 20.0)
    w = synthgen.weights(78, n, k)
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    xd = torch.from_numpy(x).to(torch.bfloat16).cuda()
    qa = ops.hadamard_quant(xd, b, ops.MODE_NVFP4)
    e = ops.EPI_GELU if epi == "gelu" else ops.EPI_NONE
    y_ref = ops.qgemm(qa, xd, pw, ops.MODE_NVFP4, epilogue=e)
    amax = torch.full((1,), 123.0, device="cuda")
    y = ops.qgemm_rotamax(qa, pw, b, amax, epilogue=e)
    qh = ops.hadamard_quant(y_ref, b, ops.MODE_NVFP4)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert amax.item() == qh.tensor_amax.item() and amax.item() > 0
