"""Pins for the oracle's small-float formats (CPU only).

The oracle encoders are checked against hand-worked encodings, against an
independent library conversion (torch's float8_e4m3fn cast, which rounds to
nearest-even inside the finite range), and against a brute-force nearest-
value search over the whole E2M1 grid.
"""
import os

import numpy as np
import pytest
import torch

from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pins(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if not line:
            continue
        v, code, dec = line.split()[:3]
        rows.append((float(v), int(code, 16), float(dec)))
    return rows


@pytest.mark.parametrize("name,enc,dec", [
    ("e2m1_pins.txt", formats.e2m1_encode, formats.e2m1_decode),
    ("e4m3_pins.txt", formats.e4m3_encode, formats.e4m3_decode),
])
def test_hand_worked_encodings(name, enc, dec):
    for v, code, d in _read_pins(name):
        got = int(enc(np.array([v], np.float32))[0])
        assert got == code, (name, v, hex(got), hex(code))
        back = float(dec(np.array([code]))[0])
        assert back == d or (back == 0 and d == 0), (name, code, back, d)


def test_e2m1_decode_table():
    # the format's eight magnitudes, then the same negated
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    got = formats.e2m1_decode(np.arange(16))
    assert list(got[:8]) == mags
    assert list(-got[8:]) == mags


def _brute_e2m1(v):
    """Nearest E2M1 magnitude by exhaustive search; ties -> even mantissa."""
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    a = min(abs(float(v)), 6.0)
    best = None
    for idx, g in enumerate(grid):
        d = abs(a - g)
        key = (d, idx & 1)          # prefer mantissa bit 0 on ties
        if best is None or key < best[0]:
            best = (key, idx)
    return best[1] | (8 if np.signbit(v) else 0)


def test_e2m1_brute_force():
    vals = np.concatenate([
        np.linspace(-8, 8, 4097, dtype=np.float32),
        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5], np.float32),
        np.nextafter(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32), np.float32(10)),
        np.nextafter(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32), np.float32(-10)),
    ])
    got = formats.e2m1_encode(vals)
    exp = np.array([_brute_e2m1(v) for v in vals], np.uint8)
    np.testing.assert_array_equal(got, exp)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = formats.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_in_range():
    # every representable value, every midpoint between neighbours, and one
    # float32 ulp either side of each midpoint (where RNE decisions happen)
    reps = np.unique(np.abs(formats.e4m3_decode(np.arange(127))))
    mids = ((reps[:-1] + reps[1:]) / 2).astype(np.float32)
    probe = np.concatenate([reps.astype(np.float32), mids,
                            np.nextafter(mids, np.float32(1e9)), np.nextafter(mids, np.float32(-1))])
    probe = np.concatenate([probe, -probe])
    rng = np.random.default_rng(123)
    rnd = (rng.standard_normal(200000) * np.exp2(rng.integers(-12, 9, 200000))).astype(np.float32)
    rnd = rnd[np.abs(rnd) < 448]
    probe = np.concatenate([probe, rnd])
    np.testing.assert_array_equal(formats.e4m3_encode(probe), _torch_e4m3(probe))


def test_e4m3_saturates_where_torch_gives_nan():
    big = np.array([465.0, 480.0, 1e6, np.inf], np.float32)
    assert list(formats.e4m3_encode(big)) == [0x7E] * 4
    assert list(formats.e4m3_encode(-big)) == [0xFE] * 4


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 1000,
        np.frombuffer(rng.integers(0, 2**32, 100000, dtype=np.uint64).astype(np.uint32).tobytes(), np.float32),
    ])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = formats.bf16_round(x)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
