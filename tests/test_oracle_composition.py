"""Pins for the oracle's composed steps (CPU only): rotate-then-quantize,
the packed weights, and the quantized branches of the DiT's linear layer.

Each expected value below comes from the mathematics, not from the oracle:

* One-hot rows.  A row holding a at channel j rotates to a * H[j % b, i] / sqrt(b)
  on the b channels of j's block (Sylvester H, signs from scipy) and to 0
  elsewhere.  With b = 64, a = 96 gives +-12, a = 48 gives +-6.  Then by the
  format definitions:
    NVFP4: tensor amax 12, so each 16-element block of magnitude 12 gets the
    E4M3 scale 448 (0x7E) and of magnitude 6 the scale 224 (0x76); the block
    scale times s_t is 2 (resp. 1), so every code is E2M1 6 (0x7, or 0xF when
    negative); all-zero blocks get scale 0 and code 0.
    INT8: each row's nonzero block maps to +-127, the rest to 0, and s_m * 127
    recovers the row's magnitude.
* The block-Hadamard matrix as a weight.  W = blockdiag(H_b / sqrt b) rotates
  to W' = W H / sqrt b = I exactly (H H = b I), so its INT4 form is 7 on the
  diagonal with group scale 1/7 and its NVFP4 form is code 6 with scale 448 on
  the diagonal; a linear layer with this W maps x to x W^T, which for the
  one-hot rows above is again +-12 / +-6 -- through the NVFP4, the INT8 and
  the BF16 branch alike, then GELU (Python's math.erfc) or a residual add.
* Random data.  (XH)(WH)^T = XW^T, so each quantized branch must land within
  the quantizers' own rounding bounds of the float64 product X W^T: INT8
  |e| <= s/2 per element on both sides, NVFP4 |e| <= the block's scale S, which
  is at most (block amax / 6) * (1 + 1/16) (E4M3 rounds to within 1/16), BF16
  2^-9 relative on W; plus half a bf16 ulp of the stored output.
"""
import math

import numpy as np
import pytest
import scipy.linalg

from oracle import dit, policy, quant
from oracle.formats import bf16_round, e2m1_decode, e4m3_decode

F32 = np.float32
B = 64
H64 = scipy.linalg.hadamard(B).astype(np.float64)


def _one_hot_rows():
    """x [3, 256]: 96 at channel 0, 96 at channel 65, 48 at channel 130; and its exact rotation."""
    x = np.zeros((3, 256), F32)
    x[0, 0], x[1, 65], x[2, 130] = 96.0, 96.0, 48.0
    y = np.zeros((3, 256), np.float64)
    y[0, 0:64] = 12.0 * H64[0]
    y[1, 64:128] = 12.0 * H64[1]
    y[2, 128:192] = 6.0 * H64[2]
    return x, y


def test_hadamard_quant_nvfp4_one_hot_rows():
    x, y = _one_hot_rows()
    out = quant.hadamard_quant(x, B, "nvfp4")
    np.testing.assert_array_equal(out["y"].astype(np.float64), y)
    assert out["amax"] == F32(12.0)
    sc = out["scales"]
    assert list(sc[0]) == [0x7E] * 4 + [0] * 12
    assert list(sc[1]) == [0] * 4 + [0x7E] * 4 + [0] * 8
    assert list(sc[2]) == [0] * 8 + [0x76] * 4 + [0] * 4
    expect = np.where(y > 0, 0x7, np.where(y < 0, 0xF, 0)).astype(np.uint8)
    np.testing.assert_array_equal(out["codes"], expect)
    # the two levels reproduce the inputs: 6 * 448 * s_t = 12, 6 * 224 * s_t = 6
    assert abs(6 * 448 * float(out["s_t"]) - 12.0) <= 12.0 * 2.0 ** -22
    assert abs(6 * 224 * float(out["s_t"]) - 6.0) <= 6.0 * 2.0 ** -22


def test_hadamard_quant_int8_one_hot_rows():
    x, y = _one_hot_rows()
    out = quant.hadamard_quant(x, B, "int8")
    np.testing.assert_array_equal(out["q"], (127 * np.sign(y)).astype(np.int8))
    for r, mag in enumerate((12.0, 12.0, 6.0)):
        assert abs(127 * float(out["s"][r]) - mag) <= mag * 2.0 ** -22


def _hadamard_weight(k):
    """blockdiag(H_64 / 8) as an fp32 [k, k] weight (entries +-1/8, exact)."""
    w = np.zeros((k, k), F32)
    for j in range(k // B):
        w[j * B:(j + 1) * B, j * B:(j + 1) * B] = H64 / 8.0
    return w


def test_pack_weights_of_the_hadamard_matrix_is_the_identity():
    k = 256
    pk = quant.pack_weights(_hadamard_weight(k), B)
    np.testing.assert_array_equal(pk["w_rot"], np.eye(k, dtype=F32))
    np.testing.assert_array_equal(pk["int4"]["q"], 7 * np.eye(k, dtype=np.int8))
    s = pk["int4"]["s"]                      # [N, K/128]: only the diagonal's group is nonzero
    for n in range(k):
        g = n // 128
        assert abs(7 * float(s[n, g]) - 1.0) <= 2.0 ** -22 and not np.any(np.delete(s[n], g))
    nv = pk["nvfp4"]
    np.testing.assert_array_equal(nv["codes"], 7 * np.eye(k, dtype=np.uint8))
    sc = nv["scales"]
    for n in range(k):
        assert sc[n, n // 16] == 0x7E and not np.any(np.delete(sc[n], n // 16))
    deq = e2m1_decode(nv["codes"]) * np.repeat(e4m3_decode(sc), 16, axis=1) * float(nv["s_t"])
    np.testing.assert_allclose(deq, np.eye(k), rtol=2.0 ** -21, atol=0)
    np.testing.assert_array_equal(pk["bf16"], _hadamard_weight(k))


def _gelu(v):
    return 0.5 * v * math.erfc(-v / math.sqrt(2.0))


@pytest.mark.parametrize("mode", [policy.NVFP4, policy.INT8, policy.BF16])
def test_linear_with_the_hadamard_weight_closed_form(mode):
    x, _ = _one_hot_rows()
    w = _hadamard_weight(256)
    exact = x.astype(np.float64) @ w.astype(np.float64).T      # +-12 / +-6 by hand: a * H[n % 64, j % 64] / 8
    assert set(np.unique(np.abs(exact))) == {0.0, 6.0, 12.0}
    pk = quant.pack_weights(w, B)
    y = dit.linear(x, pk, mode, B, "none")
    np.testing.assert_array_equal(y.astype(np.float64), exact)
    g = dit.linear(x, pk, mode, B, "gelu")
    ge = np.vectorize(_gelu)(exact)
    np.testing.assert_array_equal(g, bf16_round(ge.astype(F32)))
    r = np.full_like(x, 0.5)
    z = dit.linear(x, pk, mode, B, "residual", r)
    np.testing.assert_array_equal(z.astype(np.float64), exact + 0.5)


def _rot(a):
    m, k = a.shape
    return (a.astype(np.float64).reshape(m, k // B, B) @ (H64 / 8.0)).reshape(m, k)


def _half_ulp_bf16(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 8)


@pytest.mark.parametrize("mode", [policy.NVFP4, policy.INT8, policy.BF16])
def test_linear_random_within_quantizer_bounds(mode):
    rng = np.random.default_rng(21)
    m, k, n = 16, 256, 48
    x = bf16_round((rng.laplace(size=(m, k)) * 2).astype(F32))
    x[:, 7] *= 20
    w = (rng.standard_normal((n, k)) * 0.05).astype(F32)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    y, wr = _rot(x), _rot(w)                 # exact rotations (float64 dense product)
    ay, aw = np.abs(y), np.abs(wr)
    if mode == policy.INT8:
        ex = (np.max(ay, axis=1, keepdims=True) / 127.0) * (0.5 + 1e-5) * np.ones_like(y)
        ew = np.repeat(np.max(aw.reshape(n, k // 128, 128), axis=2) / 7.0, 128, axis=1) * (0.5 + 1e-5)
    elif mode == policy.NVFP4:
        ex = np.repeat(np.max(ay.reshape(m, k // 16, 16), axis=2) / 6.0, 16, axis=1) * (1 + 1 / 16) * (1 + 1e-5)
        ew = np.repeat(np.max(aw.reshape(n, k // 16, 16), axis=2) / 6.0, 16, axis=1) * (1 + 1 / 16) * (1 + 1e-5)
    else:
        y, ay = x.astype(np.float64), np.abs(x.astype(np.float64))
        wr, aw = w.astype(np.float64), np.abs(w.astype(np.float64))
        ex = np.zeros_like(y)
        ew = aw * 2.0 ** -9
    bound = ex @ aw.T + ay @ ew.T + ex @ ew.T + 1e-5 * (ay @ aw.T)
    got = dit.linear(x, quant.pack_weights(w, B), mode, B, "none").astype(np.float64)
    err = np.abs(got - exact)
    assert np.all(err <= bound + _half_ulp_bf16(exact)), float(np.max(err - bound))
    # (worst-case bounds add |terms| while the result cancels, so they are loose on random signs;
    # the grid test below pins the quantized branches exactly)


E2M1_GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _on_nvfp4_grid(rng, rows, k, s_t_exp):
    """Rotated values that NVFP4 represents exactly: per 16-block a scale S = E4M3 value * 2^s_t_exp
    (448 or 224), entries S * (E2M1 grid value, random sign), one entry per block at +-6 S; the
    first block uses 448 so the tensor amax is 6 * 448 * 2^s_t_exp = 2688 * s_t, making s_t exact."""
    g = rng.choice(E2M1_GRID, size=(rows, k)) * rng.choice([-1.0, 1.0], size=(rows, k))
    g.reshape(rows, k // 16, 16)[:, :, 0] = rng.choice([-6.0, 6.0], size=(rows, k // 16))
    sc = rng.choice([448.0, 224.0], size=(rows, k // 16))
    sc[0, 0] = 448.0
    return g * np.repeat(sc, 16, axis=1) * 2.0 ** s_t_exp


def _on_int8_grid(rng, rows, k, group, qmax):
    """Rotated values that the symmetric quantizer represents exactly: integers times a power of two
    per row (INT8, group = k) or per 128-group (INT4), with one entry of each group at +-qmax."""
    q = rng.integers(-qmax, qmax + 1, size=(rows, k)).astype(np.float64)
    q.reshape(rows, k // group, group)[:, :, 3] = rng.choice([-qmax, qmax], size=(rows, k // group))
    e = rng.integers(-9, -3, size=(rows, k // group)).astype(np.float64)
    return q * np.repeat(2.0 ** e, group, axis=1)


@pytest.mark.parametrize("mode", [policy.NVFP4, policy.INT8])
def test_linear_exact_on_the_quantizer_grids(mode):
    """With rotated activations and weights on the quantizers' grids, quantization loses nothing, so a
    quantized branch must return x W^T itself -- the inputs are built in the rotated basis and rotated
    back (H / sqrt b is its own inverse), and (XH)(WH)^T = X W^T."""
    rng = np.random.default_rng(7)
    m, k, n = 8, 256, 40
    if mode == policy.NVFP4:
        y, wr = _on_nvfp4_grid(rng, m, k, -8), _on_nvfp4_grid(rng, n, k, -11)
    else:
        y, wr = _on_int8_grid(rng, m, k, k, 127), _on_int8_grid(rng, n, k, 128, 7)
    x, w = _rot(y), _rot(wr)
    assert np.array_equal(x.astype(F32).astype(np.float64), x) and np.array_equal(w.astype(F32).astype(np.float64), w)
    exact = y @ wr.T                                        # = x w^T
    np.testing.assert_allclose(exact, x @ w.T, rtol=1e-12, atol=1e-12)
    got = dit.linear(x.astype(F32), quant.pack_weights(w.astype(F32), B), mode, B, "none")
    np.testing.assert_array_equal(got, bf16_round(exact.astype(F32)))
