"""Parity: fused block-Hadamard + NVFP4/INT8 quantization and weight packing, GPU vs oracle.

Bar: bit-exact rotated values, tensor amax, tensor scale, E4M3 scales, E2M1
codes, INT8 codes and row scales, packed INT4 weights and scales.
"""
import numpy as np
import pytest
import torch

import synthgen
from oracle import formats, quant
from tests._layouts import untile_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from video_dit_mixed_gb300 import ops as o
    return o


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


def _u32(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


CASES = [(256, 512, 16), (200, 384, 64), (17, 1920, 64), (130, 768, 256), (1, 128, 16), (129, 256, 16),
         (64, 7680, 64)]


def _check_nvfp4(ops, x, b):
    m, k = x.shape
    q = ops.QActTensors(m, k, rotated=True, int8=False)
    ops.hadamard_quant(_dev_bf16(x), b, ops.MODE_NVFP4, out=q)
    torch.cuda.synchronize()
    ref = quant.hadamard_quant(x, b, "nvfp4")
    assert np.array_equal(_u32(q.rotated.cpu().numpy()), _u32(ref["y"]))
    assert q.tensor_amax.item() == float(ref["amax"])
    assert np.float32(q.tensor_scale.item()) == ref["s_t"]
    codes = quant.unpack_nibbles(q.fp4_codes.cpu().numpy())
    np.testing.assert_array_equal(codes, ref["codes"])
    mpad = (m + 127) // 128 * 128
    sc = untile_scales(q.fp4_scales.cpu().numpy(), mpad, k)
    np.testing.assert_array_equal(sc[:m], ref["scales"])
    assert not sc[m:].any()


def _check_int8(ops, x, b):
    m, k = x.shape
    q = ops.QActTensors(m, k, rotated=True, nvfp4=False)
    ops.hadamard_quant(_dev_bf16(x), b, ops.MODE_INT8, out=q)
    torch.cuda.synchronize()
    ref = quant.hadamard_quant(x, b, "int8")
    assert np.array_equal(_u32(q.rotated.cpu().numpy()), _u32(ref["y"]))
    np.testing.assert_array_equal(q.i8_codes.cpu().numpy(), ref["q"])
    np.testing.assert_array_equal(_u32(q.row_scale.cpu().numpy()), _u32(ref["s"]))


@pytest.mark.parametrize("m,k,b", CASES)
def test_nvfp4_quant_bit_exact(ops, m, k, b):
    _check_nvfp4(ops, synthgen.activations(100 + m, m, k, "laplace", 0.005, 50.0), b)


@pytest.mark.parametrize("m,k,b", CASES)
def test_int8_quant_bit_exact(ops, m, k, b):
    _check_int8(ops, synthgen.activations(200 + m, m, k, "normal", 0.01, 20.0), b)


# Row lengths that exercise every team size of the one-pass INT8 kernel
# (1, 2, 4, 8 and 16 warps per row, ragged last chunk) and, past 16384
# elements, the two-pass kernel.
INT8_WIDE = [(40, 1152, 64), (9, 2048, 256), (5, 3968, 16), (3, 8064, 64), (2, 16384, 256), (3, 12288, 64),
             (2, 16640, 64)]


@pytest.mark.parametrize("m,k,b", INT8_WIDE)
def test_int8_quant_row_teams_bit_exact(ops, m, k, b):
    _check_int8(ops, synthgen.activations(300 + k, m, k, "laplace", 0.01, 30.0), b)


@pytest.mark.parametrize("k", [1920, 16640])
def test_int8_extreme_row_magnitudes(ops, k):
    """Rows whose scale s = amax/127 is below 2^-100 or above 2^100 take the
    IEEE-division path; a row with amax ~1e-26 keeps the reciprocal path while
    some of its rotated values are subnormal.  Bit-exact against the oracle in
    both INT8 kernels (one-pass rows kernel, two-pass kernel past 16384)."""
    x = synthgen.activations(77, 6, k, "normal", 0.0, 1.0)
    x[0] *= 1e-30                      # s ~ 1e-32 < 2^-100
    x[1] *= 1e35                       # s ~ 1e33 > 2^100
    x[2] *= 1e-26
    x[2, 64:128] = np.where(np.arange(64) % 3 == 0, 1.0, -1.0) * 2.0 ** -130  # a block of subnormals
    x[3] = 0.0
    x[3, 5] = 2.0 ** -120              # a lone tiny value: s subnormal
    _check_int8(ops, synthgen.bf16_rne(x), 64)


def test_int8_needs_codes(ops):
    q = ops.QActTensors(16, 256, nvfp4=False)
    q.i8_codes = None
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.abi.SixbitError):
        ops.hadamard_quant(x, 64, ops.MODE_INT8, out=q)


def test_tiny_linear_config(ops):
    c = synthgen.CONFIGS["tiny_linear"]
    x = synthgen.activations(c["seed"], c["m"], c["k"], c["dist"], c["outlier_frac"], c["outlier_scale"])
    _check_nvfp4(ops, x, c["had_block"])
    _check_int8(ops, x, c["had_block"])


def test_zero_and_one_hot_inputs(ops):
    z = np.zeros((3, 256), np.float32)
    _check_nvfp4(ops, z, 64)
    _check_int8(ops, z, 64)
    o = np.zeros((5, 256), np.float32)
    o[2, 7] = 96.0
    o[4, 200] = -3.0
    _check_nvfp4(ops, o, 16)
    _check_int8(ops, o, 256)


def test_qkv_full_size_bit_exact(ops):
    x, _, c = synthgen.linear_inputs("qkv_2b")
    _check_nvfp4(ops, x, c["had_block"])
    _check_int8(ops, x, c["had_block"])


def test_supplied_tensor_amax_is_used(ops):
    x = synthgen.activations(7, 64, 256, "laplace", 0.0, 1.0)
    q = ops.QActTensors(64, 256, int8=False)
    amax = torch.tensor([100.0], device="cuda")
    ops.hadamard_quant(_dev_bf16(x), 16, ops.MODE_NVFP4, out=q, tamax=amax)
    torch.cuda.synchronize()
    ref = quant.hadamard_quant(x, 16, "nvfp4", s_t=quant.tensor_scale(100.0))
    np.testing.assert_array_equal(quant.unpack_nibbles(q.fp4_codes.cpu().numpy()), ref["codes"])
    assert np.float32(q.tensor_scale.item()) == quant.tensor_scale(100.0)


@pytest.mark.parametrize("n,k,b", [(512, 512, 16), (200, 384, 64), (144, 256, 256), (5760, 1920, 64)])
def test_pack_weights_bit_exact(ops, n, k, b):
    w = synthgen.weights(300 + n, n, k)
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    torch.cuda.synchronize()
    ref = quant.pack_weights(w, b)
    nv, i4 = ref["nvfp4"], ref["int4"]
    assert pw.fp4_amax.item() == float(nv["amax"])
    assert np.float32(pw.fp4_tensor_scale.item()) == nv["s_t"]
    np.testing.assert_array_equal(quant.unpack_nibbles(pw.fp4_codes.cpu().numpy()), nv["codes"])
    npad = (n + 127) // 128 * 128
    sc = untile_scales(pw.fp4_scales.cpu().numpy(), npad, k)
    np.testing.assert_array_equal(sc[:n], nv["scales"])
    assert not sc[n:].any()
    np.testing.assert_array_equal(quant.unpack_nibbles(pw.i4_codes.cpu().numpy(), signed=True), i4["q"])
    np.testing.assert_array_equal(_u32(pw.i4_scales.cpu().numpy().T), _u32(i4["s"]))
    np.testing.assert_array_equal(_u32(pw.bf16_w.float().cpu().numpy()), _u32(formats.bf16_round(w)))


def test_e2m1_ties_and_signed_zero_through_the_kernel(ops):
    """Rows built so that y / S lands exactly on E2M1 rounding ties.

    Block 0 of row 0 holds 2688 so s_t = 1; every other 16-block holds 6 (its
    scale is exactly 1, S = 1) and one probe value t, so code = E2M1(t).  x is
    the inverse rotation of y (the rotation is an involution), exact in bf16
    because each x entry is (+-6 +- t) / 4.
    """
    from oracle.hadamard import fwht_blocks
    probes = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5, -5.0, -0.0625, 0.0625, 7.0, -6.5]
    y = np.zeros((2, 16 * (len(probes) + 1)), np.float32)
    y[0, 0] = 2688.0
    for j, t in enumerate(probes):
        y[1, 16 * (j + 1)] = 6.0
        y[1, 16 * (j + 1) + 5] = t
    y = np.concatenate([y, np.zeros((2, (-y.shape[1]) % 128), np.float32)], axis=1)
    x = fwht_blocks(y, 16)
    assert np.array_equal(formats.bf16_round(x), x)
    _check_nvfp4(ops, x, 16)
    ref = quant.hadamard_quant(x, 16, "nvfp4")
    got = [int(ref["codes"][1, 16 * (j + 1) + 5]) for j in range(len(probes))]
    assert got == [0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x8, 0xC, 0xE, 0x8, 0x0, 0x7, 0xF]
