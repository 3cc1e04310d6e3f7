"""Seeded input generator: determinism, slicing and distribution sanity (CPU only)."""
import numpy as np

import synthgen


def test_splitmix64_known_values():
    # first outputs of the reference splitmix64 stream seeded with 0
    # (state += golden gamma, then the two multiply-xorshift rounds)
    gamma = 0x9E3779B97F4A7C15
    def ref(state):
        z = (state + gamma) & (2**64 - 1)
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & (2**64 - 1)
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & (2**64 - 1)
        return z ^ (z >> 31)
    assert ref(0) == 0xE220A8397B1DCDAF     # published first value of splitmix64(0)
    key = ref((3 << 32) | 5)
    got = synthgen.raw64(3, 5, 4)
    exp = [ref((key + i * gamma - gamma) & (2**64 - 1)) for i in range(1, 5)]
    assert [int(v) for v in got] == exp


def test_deterministic_and_sliceable():
    a = synthgen.uniform(1, 2, 1000)
    b = synthgen.uniform(1, 2, 500, start=500)
    np.testing.assert_array_equal(a[500:], b)
    assert np.all((a > 0) & (a < 1))


def test_distributions():
    z = synthgen.normal(0, 1, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1) < 0.02
    l = synthgen.laplace(0, 1, 200000)
    assert abs(l.mean()) < 0.02 and abs(l.var() - 2) < 0.05


def test_activation_outliers_and_bf16():
    x = synthgen.activations(0, 64, 512, "normal", 0.01, 20.0)
    ch = synthgen.outlier_channels(0, 1001, 512, 0.01)
    assert len(ch) == 5
    assert np.all((x.view(np.uint32) & 0xFFFF) == 0)        # bf16-valued
    big = np.abs(x[:, ch]).mean()
    rest = np.abs(np.delete(x, ch, axis=1)).mean()
    assert 10 < big / rest < 30
