"""Pins for the oracle's DiT chain (oracle/dit.py), from what the block
structure x -> x + W_d . GELU(W_u . x) and the policy rules fix by hand:

- zero weights: every block is the identity, so every step returns its input
  bit for bit, every Delta is zero (Gamma 0, cosine of two zero deltas 1) and
  the decisions follow from the rules alone: INT8 on the first compute (no
  Gamma yet), NVFP4 on the second (Gamma 0 < 0.1), then skips for ever (cos 1,
  predicted error 0);
- W_u = 4 I, W_d = I / 2 with the BF16 path forced by the outlier rule: on
  inputs +-2 the block gives x + GELU(4x) / 2, which is 6 for x = 2 and -2 for
  x = -2 after bf16 rounding (GELU(8) = 8 (1 - 6e-16), GELU(-8) = -5e-15), and
  a second such block maps 6 to 6 + 12 = 18; with W_d = -I / 2 both inputs
  map to -2 (GELU applied after the down projection would give 2 + GELU(-4)
  = 2 and -2 + GELU(4) = 2 instead).

A dropped residual, a swapped layer order, GELU applied after the down
projection, or a wrong decision sequence fails one of these.
"""
import numpy as np

from oracle import policy
from oracle.dit import OracleDiT


def _x(m, k, seed=3):
    rng = np.random.default_rng(seed)
    x = rng.choice(np.array([-1.5, -0.5, 0.25, 0.75, 1.0], np.float32), size=(m, k))
    return x.astype(np.float32)     # small dyadic values: exact in bf16, outlier ratio < 30


def test_zero_weights_identity_and_decision_sequence():
    m, h, f, L = 8, 128, 256, 3
    w = [(np.zeros((f, h), np.float32), np.zeros((h, f), np.float32)) for _ in range(L)]
    dit = OracleDiT(w, 64)
    x = _x(m, h)
    for _ in range(5):
        y = dit.step(x)
        assert np.array_equal(y.view(np.uint32), x.view(np.uint32))
    modes = [[d.mode for d in step] for step in dit.trace]
    assert modes[0] == [policy.INT8] * L
    assert modes[1] == [policy.NVFP4] * L
    for s in modes[2:]:
        assert s == [policy.SKIP] * L
    for l in range(L):
        assert not np.any(dit.cached_delta(l))
    for st in dit.states:
        assert st.gamma == 0.0 and st.cos == 1.0 and st.acc == 0.0


def test_scaled_identity_blocks_closed_form():
    m, h = 4, 128
    eye = np.eye(h, dtype=np.float32)
    w = [(4.0 * eye, 0.5 * eye), (4.0 * eye, 0.5 * eye)]
    cfg = policy.PolicyConfig(pdr_ratio=0.0)          # any nonzero input: BF16 (PDR)
    x = np.where((np.arange(m * h).reshape(m, h) % 3) == 0, -2.0, 2.0).astype(np.float32)
    one = OracleDiT(w[:1], 64, cfg).step(x)
    np.testing.assert_array_equal(one, np.where(x > 0, 6.0, -2.0).astype(np.float32))
    dit = OracleDiT(w, 64, cfg)
    two = dit.step(x)
    np.testing.assert_array_equal(two, np.where(x > 0, 18.0, -2.0).astype(np.float32))
    assert [d.mode for d in dit.trace[0]] == [policy.BF16, policy.BF16]
    assert all(d.pdr for d in dit.trace[0])


def test_gelu_sits_between_the_projections():
    m, h = 4, 128
    eye = np.eye(h, dtype=np.float32)
    cfg = policy.PolicyConfig(pdr_ratio=0.0)
    x = np.where((np.arange(m * h).reshape(m, h) % 3) == 0, -2.0, 2.0).astype(np.float32)
    y = OracleDiT([(4.0 * eye, -0.5 * eye)], 64, cfg).step(x)
    np.testing.assert_array_equal(y, np.full_like(x, -2.0))


def test_per_depth_thresholds_closed_form():
    """Per-block thresholds (one PolicyConfig per block).  Zero weights keep
    every Delta zero, so Gamma = 0 and cos = 1 at every block: a block whose
    gamma_thr is 0 computes INT8 (Gamma >= 0) where the others take NVFP4,
    and a block whose cos_thr is above 1 never skips."""
    m, h, f, L = 8, 128, 256, 3
    w = [(np.zeros((f, h), np.float32), np.zeros((h, f), np.float32)) for _ in range(L)]
    base = policy.PolicyConfig()
    cfgs = [base, policy.PolicyConfig(cos_thr=1.5), policy.PolicyConfig(gamma_thr=0.0)]
    dit = OracleDiT(w, 64, cfgs)
    x = _x(m, h)
    for _ in range(5):
        y = dit.step(x)
        assert np.array_equal(y.view(np.uint32), x.view(np.uint32))
    modes = [[d.mode for d in step] for step in dit.trace]
    assert modes[0] == [policy.INT8] * L
    assert modes[1] == [policy.NVFP4, policy.NVFP4, policy.INT8]
    for s in modes[2:]:
        assert s == [policy.SKIP, policy.NVFP4, policy.SKIP]


def test_per_depth_list_of_equal_configs_equals_one_config():
    rng = np.random.default_rng(4)
    m, h, f, L = 4, 128, 256, 3
    w = [((rng.normal(size=(f, h)) * 0.02).astype(np.float32), (rng.normal(size=(h, f)) * 0.02).astype(np.float32))
         for _ in range(L)]
    cfg = policy.PolicyConfig(pdr_ratio=1e9)
    a, b = OracleDiT(w, 64, cfg), OracleDiT(w, 64, [cfg] * L)
    x = _x(m, h, seed=9)
    for _ in range(4):
        np.testing.assert_array_equal(a.step(x), b.step(x))
    assert [[d.mode for d in s] for s in a.trace] == [[d.mode for d in s] for s in b.trace]
