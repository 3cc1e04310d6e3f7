"""Pins for the oracle's quantizers (CPU only): hand-worked blocks, invariants."""
import numpy as np

from oracle import formats, quant

F32 = np.float32


def test_nvfp4_hand_worked_blocks():
    # amax_t = 2688 makes s_t exactly 1, so every step can be checked by hand
    y = np.zeros((1, 64), F32)
    y[0, :8] = [2688, 1344, -672, 224, 112, 336, -1, 0]        # block 0: amax 2688
    y[0, 16:22] = [12, -3, 5, 1, 0.5, -12]                      # block 1: amax 12
    # block 2 all zero
    y[0, 48:51] = [102, -51, 20]                                # block 3: amax 102
    out = quant.nvfp4_quantize(y)
    assert out["s_t"] == F32(1.0) and out["amax"] == F32(2688)
    # block scales: 448 -> 0x7E, 2 -> 0x40, 0 -> 0x00, 17 -> 16 -> 0x58 (tie to even)
    assert list(out["scales"][0]) == [0x7E, 0x40, 0x00, 0x58]
    c = out["codes"][0]
    # block 0, S = 448: 6, 3, -1.5, 0.5, 0.25 (tie -> 0), 0.75 (tie -> 1), -1/448 -> -0, 0
    assert list(c[:8]) == [0x7, 0x5, 0xB, 0x1, 0x0, 0x2, 0x8, 0x0]
    # block 1, S = 2: 6, -1.5, 2.5 (tie -> 2), 0.5, 0.25 (tie -> 0), -6
    assert list(c[16:22]) == [0x7, 0xB, 0x4, 0x1, 0x0, 0xF]
    assert not c[32:48].any()
    # block 3, S = 16: 102/16 = 6.375 saturates to 6; -51/16 = -3.1875 -> -3; 1.25 (tie -> 1)
    assert list(c[48:51]) == [0x7, 0xD, 0x2]


def test_nvfp4_zero_tensor():
    out = quant.nvfp4_quantize(np.zeros((2, 32), F32))
    assert out["s_t"] == F32(1.0) and not out["codes"].any() and not out["scales"].any()


def test_nvfp4_rounding_error_bound_random():
    rng = np.random.default_rng(11)
    y = (rng.laplace(size=(64, 256)) * 3).astype(F32)
    y[:, 5] *= 50
    out = quant.nvfp4_quantize(y)
    S = np.repeat(formats.e4m3_decode(out["scales"]) * float(out["s_t"]), 16, axis=1)
    q = formats.e2m1_decode(out["codes"])
    r = y.astype(np.float64) / np.where(S == 0, 1, S)
    # RNE on the E2M1 grid: error at most half the local spacing, or saturation
    half = np.where(np.abs(r) <= 2, 0.25, np.where(np.abs(r) <= 4, 0.5, 1.0))
    sat = np.abs(r) > 6
    assert np.all((np.abs(q - r) <= half + 1e-12) | (sat & (np.abs(q) == 6)))
    # the tensor maximum lands on the top of the grid (scale chosen from it)
    i = np.unravel_index(np.argmax(np.abs(y)), y.shape)
    assert abs(q[i]) >= 4


def test_int8_hand_worked_rows():
    y = np.array([[127, -63.5, 0.5, 1.5, 2.5, -127, 0, 3.49],
                  [0, 0, 0, 0, 0, 0, 0, 0]], F32)
    out = quant.int8_quantize(y)
    assert list(out["s"]) == [F32(1.0), F32(0.0)]
    assert list(out["q"][0]) == [127, -64, 0, 2, 2, -127, 0, 3]
    assert not out["q"][1].any()


def test_int8_row_max_maps_to_127():
    rng = np.random.default_rng(5)
    y = rng.standard_normal((32, 128)).astype(F32)
    out = quant.int8_quantize(y)
    am = np.argmax(np.abs(y), axis=1)
    assert np.all(np.abs(out["q"][np.arange(32), am]) == 127)
    err = np.abs(out["q"] * out["s"][:, None].astype(np.float64) - y)
    assert np.all(err <= 0.5 * out["s"][:, None] * (1 + 1e-6))


def test_int4_weight_groups():
    w = np.zeros((2, 256), F32)
    w[0, :6] = [7, 3.5, 2.5, -0.5, -7, 1]        # group 0: amax 7 -> s = 1
    w[0, 128:130] = [0.7, -0.35]                   # group 1: amax 0.7 -> s = 0.1
    out = quant.int4_quantize_weights(w)
    assert out["s"][0, 0] == F32(1.0) and out["s"][0, 1] == F32(F32(0.7) / F32(7))
    assert list(out["q"][0, :6]) == [7, 4, 2, 0, -7, 1]
    assert out["q"][0, 128] == 7 and out["q"][0, 129] in (-3, -4)
    assert not out["q"][1].any() and not out["s"][1].any()


def test_nibble_packing_order():
    c = np.array([[1, 2, 0xF, 0x7]], np.uint8)
    assert list(quant.pack_nibbles(c)[0]) == [0x21, 0x7F]
    s = np.array([[-1, 7, -7, 0]], np.int8)
    p = quant.pack_nibbles(s)
    assert list(p[0]) == [0x7F, 0x09]
    np.testing.assert_array_equal(quant.unpack_nibbles(p, signed=True), s)
    np.testing.assert_array_equal(quant.unpack_nibbles(quant.pack_nibbles(c)), c)


def test_pack_weights_rotates_before_quantizing():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((4, 128)) * 0.02).astype(F32)
    p = quant.pack_weights(w, 16)
    from oracle.hadamard import fwht_blocks
    np.testing.assert_array_equal(p["w_rot"], fwht_blocks(w, 16))
    np.testing.assert_array_equal(p["bf16"], formats.bf16_round(w))
    deq = p["int4"]["q"].reshape(4, 1, 128) * p["int4"]["s"][:, :, None]
    assert np.max(np.abs(deq.reshape(4, 128) - p["w_rot"])) <= 0.5 * p["int4"]["s"].max() * (1 + 1e-6)
