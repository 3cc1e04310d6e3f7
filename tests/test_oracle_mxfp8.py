"""Pins for the oracle's MXFP8 delta-cache format (oracle/formats.py) and its
use in the DiT chain (oracle/dit.py), CPU only.

MXFP8 is the OCP Microscaling format with E4M3 elements: 32 consecutive
values share an E8M0 scale 2**X, X = floor(log2 amax) - 8 clamped to
[-127, 127], and each element is E4M3(v / 2**X), round-to-nearest-even,
saturating at 448.  The method itself only says the delta cache may be held
in a low precision ("6Bit-Diffusion" popular summary, section 7).

Pins, none of which re-runs the encoder's own arithmetic:
- hand-worked blocks (scale codes and element codes written out by hand);
- brute force: each element against the nearest point of an E4M3 grid that
  the test enumerates from the bit layout, with the scale from an integer
  search for floor(log2 amax);
- the special cases: all-zero block, a block below E8M0's range (clamped
  scale), a block above it, saturation in [448, 512) * 2**X;
- the DiT chain with the MXFP8 cache: with the same delta every step the
  cosine is the closed form of a delta against its own dequantized copy, and
  a skip adds the dequantized delta, not the fresh one.
"""
import math

import numpy as np
import pytest

from oracle import formats, policy, stats
from oracle.dit import OracleDiT


def _block(vals):
    v = np.zeros(32)
    v[: len(vals)] = vals
    return v


# (block values, expected E8M0 code, {index: expected element code}), worked by hand:
#   amax 448 = 1.75 * 2**8 -> X = 0, code 127; 448 -> 0x7E (E=15, M=6); 1 -> 0x38 (E=7, M=0)
#   amax 3 -> X = 1 - 8 = -7, code 120; 3 * 2**7 = 384 = 1.5 * 2**8 -> 0x7C; -3 -> 0xFC;
#     0.01 * 2**7 = 1.28, between 1.25 (M=2) and 1.375 (M=3), nearer 1.25 -> 0x3A
#   amax 500 -> X = 0 (2**8 <= 500 < 2**9): 500 saturates to 448 -> 0x7E
#   amax 2**-130 -> X = -138, clamped to -127, code 0; 2**-130 * 2**127 = 0.125 = 2**-3 -> 0x20
#   amax 2**-3 * 1.5 -> X = -11, code 116; 0.1875 * 2**11 = 384 -> 0x7C;
#     2**-12 * 2**11 = 0.5 -> 0x30; 2**-20 * 2**11 = 2**-9, the smallest subnormal -> 0x01
HAND = [
    ([448.0, 1.0], 127, {0: 0x7E, 1: 0x38, 2: 0x00}),
    ([3.0, 0.01, -3.0], 120, {0: 0x7C, 1: 0x3A, 2: 0xFC}),
    ([500.0, -500.0], 127, {0: 0x7E, 1: 0xFE}),
    ([2.0 ** -130], 0, {0: 0x20}),
    ([0.1875, 2.0 ** -12, 2.0 ** -20], 116, {0: 0x7C, 1: 0x30, 2: 0x01}),
    ([], 0, {0: 0x00, 31: 0x00}),
]


@pytest.mark.parametrize("vals,scale,elems", HAND)
def test_hand_worked_blocks(vals, scale, elems):
    codes, scales = formats.mxfp8_encode(_block(vals))
    assert scales.tolist() == [scale]
    for i, c in elems.items():
        assert int(codes[i]) == c, (i, hex(int(codes[i])))


def test_scale_above_the_e8m0_range_is_clamped():
    codes, scales = formats.mxfp8_encode(_block([2.0 ** 140, 1.0]))
    assert scales.tolist() == [254]                     # X = 132 - 8 = 132 -> clamped to 127
    assert int(codes[0]) == 0x7E                        # 2**13 saturates to 448


def _e4m3_grid():
    """Non-negative finite E4M3 magnitudes indexed by code (0x00 .. 0x7E), from the bit layout."""
    out = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        out.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(out)


def _floor_log2(a):
    e = 0
    while 2.0 ** (e + 1) <= a:
        e += 1
    while 2.0 ** e > a:
        e -= 1
    return e


def test_brute_force_nearest_on_random_blocks():
    rng = np.random.default_rng(11)
    grid = _e4m3_grid()
    n_blocks = 60
    # bf16-valued inputs over a wide range of block magnitudes, some blocks with zeros
    mags = 2.0 ** rng.integers(-40, 40, size=n_blocks)
    v = (rng.laplace(size=(n_blocks, 32)) * mags[:, None]).astype(np.float32)
    v = formats.bf16_round(v).astype(np.float64)
    v[::7, ::3] = 0.0
    codes, scales = formats.mxfp8_encode(v.reshape(-1))
    codes = codes.reshape(n_blocks, 32)
    for b in range(n_blocks):
        amax = np.abs(v[b]).max()
        x = max(_floor_log2(amax) - 8, -127) if amax > 0 else -127
        assert int(scales[b]) == x + 127
        for i in range(32):
            t = abs(v[b, i]) / 2.0 ** x
            dist = np.abs(grid - t)
            best = np.flatnonzero(dist == dist.min())
            want = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]   # ties to even mantissa
            if t >= 448.0:
                want = 0x7E
            got = int(codes[b, i])
            assert got & 0x7F == want, (b, i, v[b, i], hex(got))
            assert (got >> 7) == (1 if np.signbit(v[b, i]) else 0)


def test_decode_is_code_value_times_scale():
    grid = _e4m3_grid()
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F].reshape(-1, 2)[:, 0][:96]   # 96 finite codes, 3 blocks
    scales = np.array([0, 127, 250], np.uint8)
    got = formats.mxfp8_decode(codes, scales)
    for j, c in enumerate(codes):
        mag = grid[c & 0x7F] * 2.0 ** (int(scales[j // 32]) - 127)
        assert got[j] == (-mag if c & 0x80 else mag)


def test_roundtrip_error_bound():
    rng = np.random.default_rng(5)
    v = formats.bf16_round(rng.normal(size=4096).astype(np.float32) * 0.03).astype(np.float64)
    codes, scales = formats.mxfp8_encode(v)
    d = formats.mxfp8_decode(codes, scales)
    x = np.repeat(scales.astype(np.int64) - 127, 32)
    # half a unit in the last place of E4M3 at the element's binade (never below the subnormal spacing),
    # or the saturation gap
    binade = np.floor(np.log2(np.maximum(np.abs(v) / np.ldexp(1.0, x), 2.0 ** -9))).astype(np.int64)
    step = np.ldexp(1.0, np.maximum(binade, -6) - 3 + x)
    sat = np.abs(v) >= 448 * np.ldexp(1.0, x)
    err = np.abs(d - v)
    assert np.all(err[~sat] <= step[~sat] / 2)
    assert np.all(np.abs(d[sat]) == 448 * np.ldexp(1.0, x[sat]))


def test_length_must_be_a_multiple_of_the_block():
    with pytest.raises(ValueError):
        formats.mxfp8_encode(np.zeros(33))


def _x(m, k, seed):
    rng = np.random.default_rng(seed)
    return formats.bf16_round(rng.normal(size=(m, k)).astype(np.float32))


def _identity_blocks(h, a=4.0, b=0.5):
    eye = np.eye(h, dtype=np.float32)
    return [(a * eye, b * eye)]


def test_dit_mxfp8_cache_cosine_and_skip_closed_forms():
    m, h = 4, 128
    cfg = policy.PolicyConfig(pdr_ratio=0.0, cos_thr=0.9, err_cap=0.5)   # BF16 compute; skips allowed
    x = _x(m, h, 7)
    dit = OracleDiT(_identity_blocks(h), 64, cfg, delta_format="mxfp8")
    ref = OracleDiT(_identity_blocks(h), 64, cfg)                       # bf16 cache
    y1 = dit.step(x)
    np.testing.assert_array_equal(y1, ref.step(x))                      # the first step reads a zero cache
    d = stats.delta(x, y1).astype(np.float64)                           # the same delta every step
    q = formats.mxfp8_decode(*formats.mxfp8_encode(d.reshape(-1))).reshape(d.shape)
    assert not np.array_equal(q, d)                                     # the format loses something here
    y2 = dit.step(x)
    np.testing.assert_array_equal(y2, y1)
    cos = float((d * q).sum() / math.sqrt((d * d).sum() * (q * q).sum()))
    assert dit.states[0].cos == pytest.approx(cos, rel=1e-12, abs=0)
    assert cos < 1.0
    ref.step(x)
    assert ref.states[0].cos == 1.0
    y3 = dit.step(x)                                                    # cos >= 0.9: the block skips
    assert dit.trace[-1][0].mode == policy.SKIP
    want = formats.bf16_round((x.astype(np.float64) + q).astype(np.float32))
    np.testing.assert_array_equal(y3, want)                             # x + dequantized delta
    assert not np.array_equal(y3, formats.bf16_round((x + d).astype(np.float32)))


def test_dit_mxfp8_cache_zero_weights_unchanged():
    m, h, f, L = 8, 128, 256, 2
    w = [(np.zeros((f, h), np.float32), np.zeros((h, f), np.float32)) for _ in range(L)]
    dit = OracleDiT(w, 64, delta_format="mxfp8")
    x = _x(m, h, 3)
    for _ in range(4):
        np.testing.assert_array_equal(dit.step(x), x)
    assert [d.mode for d in dit.trace[-1]] == [policy.SKIP] * L
    for l in range(L):
        assert not np.any(dit.cached_delta(l))
