"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case patches one plausible error into an oracle function (a dropped
term, a wrong sign, a wrong constant, a wrong tie rule, a dropped rule) and
checks that at least one pin test then fails.
"""
import numpy as np
import pytest

from oracle import dit, formats, gemm, hadamard, policy, quant, stats

import tests.test_oracle_composition as tc
import tests.test_oracle_dit as td
import tests.test_oracle_formats as tf
import tests.test_oracle_hadamard as th
import tests.test_oracle_quant as tq
import tests.test_oracle_stats_policy as ts


def _fails(fn, *args):
    """True when the pin rejects the mutant: a failed assertion, or an error the mutant raises."""
    try:
        fn(*args)
    except Exception:  # noqa: BLE001 -- AssertionError included
        return True
    return False


def _bad_fwht_sign(x, b):
    x = np.asarray(x, np.float32)
    m, k = x.shape
    v = x.reshape(m, k // b, b).copy()
    h = 1
    while h < b:
        w = v.reshape(m, k // b, b // (2 * h), 2, h)
        v = np.stack([w[:, :, :, 0] + w[:, :, :, 1], w[:, :, :, 1] - w[:, :, :, 0]], axis=3).reshape(m, k // b, b)
        h *= 2
    return (v * hadamard.inv_sqrt_b(b)).reshape(m, k)


def _bad_fwht_no_norm(x, b):
    return hadamard.fwht_blocks(x, b) / hadamard.inv_sqrt_b(b)


def test_fwht_mutations_are_caught(monkeypatch):
    monkeypatch.setattr(hadamard, "fwht_blocks", _bad_fwht_sign)
    assert _fails(th.test_fwht_of_unit_vectors_is_normalised_hadamard, 16)
    monkeypatch.undo()
    orig = hadamard.fwht_blocks
    monkeypatch.setattr(hadamard, "fwht_blocks", lambda x, b: orig(x, b) / hadamard.inv_sqrt_b(b))
    assert _fails(th.test_fwht_is_an_involution_on_small_integers, 64)


def test_format_tie_rule_mutation_is_caught(monkeypatch):
    def away(a, fmt):   # ties away from zero instead of to even
        ebits, mbits, bias, fmax = fmt
        a = np.asarray(a, np.float64)
        out = np.zeros_like(a)
        nz = a > 0
        _, ex = np.frexp(a[nz])
        q = np.ldexp(1.0, np.maximum(ex - 1, 1 - bias) - mbits)
        out[nz] = np.minimum(np.floor(a[nz] / q + 0.5) * q, fmax)
        return out
    monkeypatch.setattr(formats, "_round_to_format", away)
    assert _fails(tf.test_hand_worked_encodings, "e2m1_pins.txt", formats.e2m1_encode, formats.e2m1_decode)
    assert _fails(tf.test_e4m3_encode_matches_torch_in_range)


def test_quantizer_constant_mutations_are_caught(monkeypatch):
    monkeypatch.setattr(quant, "tensor_scale", lambda amax: np.float32(amax) / np.float32(448.0))
    assert _fails(tq.test_nvfp4_hand_worked_blocks)
    monkeypatch.undo()
    orig = quant.int8_quantize
    def int8_128(y):
        y = np.asarray(y, np.float32)
        s = (np.max(np.abs(y), axis=1) / np.float32(128.0)).astype(np.float32)
        q = np.clip(np.rint(y / np.where(s == 0, 1, s)[:, None]), -127, 127).astype(np.int8)
        return dict(q=q, s=s)
    monkeypatch.setattr(quant, "int8_quantize", int8_128)
    assert _fails(tq.test_int8_hand_worked_rows)


def test_policy_rule_mutation_is_caught(monkeypatch):
    orig = policy.decide
    def no_post_skip(st, ratio, cfg):
        st.skipped_last = False
        return orig(st, ratio, cfg)
    monkeypatch.setattr(policy, "decide", no_post_skip)
    assert _fails(ts.test_policy_hand_traces, "B")


def test_cosine_mutation_is_caught(monkeypatch):
    monkeypatch.setattr(stats, "cosine", lambda a, b, c: a / b if b else 0.0)
    assert _fails(ts.test_cosine_special_cases)


def test_dit_block_mutations_are_caught(monkeypatch):
    orig = dit.linear

    def no_residual(x, pk, mode, b, epilogue, residual=None):   # x -> W_d . GELU(W_u . x)
        return orig(x, pk, mode, b, "none" if epilogue == "residual" else epilogue)

    def gelu_after_down(x, pk, mode, b, epilogue, residual=None):   # x -> x + GELU(W_d . W_u . x)
        y = orig(x, pk, mode, b, "none")
        if epilogue == "residual":
            return dit._round_bf16(gemm.gelu(y.astype(np.float64)) + np.asarray(residual, np.float64))
        return y

    monkeypatch.setattr(dit, "linear", no_residual)
    assert _fails(td.test_zero_weights_identity_and_decision_sequence)
    monkeypatch.setattr(dit, "linear", gelu_after_down)
    assert _fails(td.test_gelu_sits_between_the_projections)


def test_rotate_then_quantize_mutations_are_caught(monkeypatch):
    orig_hq = quant.hadamard_quant

    def unrotated(x, b, mode, s_t=None):      # quantizes x instead of its rotation
        out = quant.nvfp4_quantize(np.asarray(x, np.float32), s_t) if mode == "nvfp4" else \
            quant.int8_quantize(np.asarray(x, np.float32))
        out["y"] = np.asarray(x, np.float32)
        return out
    monkeypatch.setattr(quant, "hadamard_quant", unrotated)
    assert _fails(tc.test_hadamard_quant_nvfp4_one_hot_rows)
    assert _fails(tc.test_hadamard_quant_int8_one_hot_rows)
    assert _fails(tc.test_linear_exact_on_the_quantizer_grids, policy.NVFP4)
    assert _fails(tc.test_linear_exact_on_the_quantizer_grids, policy.INT8)
    monkeypatch.setattr(quant, "hadamard_quant", lambda x, b, mode, s_t=None: orig_hq(x, b, mode, np.float32(1.0)))
    assert _fails(tc.test_hadamard_quant_nvfp4_one_hot_rows)            # s_t forced to 1


def test_weight_packing_mutations_are_caught(monkeypatch):
    orig = quant.pack_weights

    def unrotated_weights(w, b):              # quantizes W instead of W . blockdiag(H / sqrt b)
        out = orig(w, b)
        w = np.asarray(w, np.float32)
        return dict(out, w_rot=w, nvfp4=quant.nvfp4_quantize(w), int4=quant.int4_quantize_weights(w))
    monkeypatch.setattr(quant, "pack_weights", unrotated_weights)
    assert _fails(tc.test_pack_weights_of_the_hadamard_matrix_is_the_identity)
    assert _fails(tc.test_linear_exact_on_the_quantizer_grids, policy.NVFP4)
    assert _fails(tc.test_linear_exact_on_the_quantizer_grids, policy.INT8)


def test_quantized_linear_mutations_are_caught(monkeypatch):
    orig_lin = dit.linear
    swapped = lambda x, pk, mode, b, epi, residual=None: orig_lin(  # noqa: E731 -- the packings swapped
        x, dict(pk, nvfp4=pk["int4"], int4=pk["nvfp4"]), mode, b, epi, residual)
    monkeypatch.setattr(dit, "linear", swapped)
    for mode in (policy.NVFP4, policy.INT8):
        assert _fails(tc.test_linear_with_the_hadamard_weight_closed_form, mode)
    monkeypatch.undo()
    orig_nv = gemm.nvfp4_gemm_ref
    monkeypatch.setattr(gemm, "nvfp4_gemm_ref", lambda xc, xs, stx, wc, ws, stw: orig_nv(xc, xs, 1.0, wc, ws, stw))
    assert _fails(tc.test_linear_with_the_hadamard_weight_closed_form, policy.NVFP4)   # activation s_t dropped
    assert _fails(tc.test_linear_exact_on_the_quantizer_grids, policy.NVFP4)
    monkeypatch.undo()
    orig_i8 = gemm.int8_gemm_ref
    monkeypatch.setattr(gemm, "int8_gemm_ref", lambda qx, sm, qw, sw: orig_i8(qx, np.ones_like(sm), qw, sw))
    assert _fails(tc.test_linear_with_the_hadamard_weight_closed_form, policy.INT8)    # row scale dropped
    assert _fails(tc.test_linear_exact_on_the_quantizer_grids, policy.INT8)
    monkeypatch.undo()
    monkeypatch.setattr(gemm, "int8_gemm_ref", lambda qx, sm, qw, sw: orig_i8(qx, sm, qw, sw[:, ::-1]))
    assert _fails(tc.test_linear_exact_on_the_quantizer_grids, policy.INT8)            # group scales misindexed
    monkeypatch.undo()
    monkeypatch.setattr(gemm, "gelu", lambda v: 0.5 * np.asarray(v, np.float64) * (1 + np.tanh(np.asarray(v))))
    assert _fails(tc.test_linear_with_the_hadamard_weight_closed_form, policy.BF16)    # a different activation


def test_mxfp8_mutations_are_caught(monkeypatch):
    import tests.test_oracle_mxfp8 as tm
    orig_x = formats.mx_shared_exponent
    monkeypatch.setattr(formats, "mx_shared_exponent", lambda a: orig_x(a) + 1)        # exponent one too high
    assert _fails(tm.test_hand_worked_blocks, *tm.HAND[1])
    assert _fails(tm.test_brute_force_nearest_on_random_blocks)
    monkeypatch.setattr(formats, "mx_shared_exponent", lambda a: orig_x(a) - 1)        # one too low: saturates
    assert _fails(tm.test_hand_worked_blocks, *tm.HAND[0])

    def unclamped(a):
        a = np.asarray(a, np.float64)
        _, ex = np.frexp(a)
        return np.where(a > 0, ex - 9, -127).astype(np.int64)
    monkeypatch.setattr(formats, "mx_shared_exponent", unclamped)                      # no E8M0 range clamp
    assert _fails(tm.test_hand_worked_blocks, *tm.HAND[3])
    monkeypatch.undo()
    orig_dec = formats.mxfp8_decode
    monkeypatch.setattr(formats, "mxfp8_decode",
                        lambda c, s, block=32: formats.decode(np.asarray(c), formats.E4M3))  # scale dropped
    assert _fails(tm.test_decode_is_code_value_times_scale)
    monkeypatch.undo()
    monkeypatch.setattr(dit.OracleDiT, "store_delta",
                        lambda self, l, d: self.deltas.__setitem__(l, (np.asarray(d, np.float32).copy(), None)))
    assert _fails(tm.test_dit_mxfp8_cache_cosine_and_skip_closed_forms)                # cache kept in bf16
    monkeypatch.undo()
    assert orig_dec is formats.mxfp8_decode


def test_per_depth_threshold_mutation_is_caught(monkeypatch):
    orig = dit.OracleDiT.__init__

    def first_config_everywhere(self, weights, had_block, cfg=None, delta_format="bf16"):
        orig(self, weights, had_block, cfg, delta_format)
        self.cfgs = [self.cfgs[0]] * self.L      # per-block thresholds ignored
    monkeypatch.setattr(dit.OracleDiT, "__init__", first_config_everywhere)
    assert _fails(td.test_per_depth_thresholds_closed_form)


def test_nan_statistic_reading_mutations_are_caught(monkeypatch):
    """Reading a NaN Gamma as stable (NVFP4), or a NaN input ratio as no outlier (no PDR), fails the
    NaN pins."""
    import math
    orig = policy.decide

    def nan_gamma_stable(st, ratio, cfg):
        if math.isnan(st.gamma):
            st.gamma = 0.0
        return orig(st, ratio, cfg)

    def nan_ratio_no_pdr(st, ratio, cfg):
        return orig(st, 0.0 if math.isnan(ratio) else ratio, cfg)

    for mutant in (nan_gamma_stable, nan_ratio_no_pdr):
        monkeypatch.setattr(policy, "decide", mutant)
        assert _fails(ts.test_policy_nan_statistics_take_the_safer_path), mutant.__name__
        assert _fails(ts.test_policy_nan_statistics_single_steps), mutant.__name__
    monkeypatch.setattr(policy, "decide", orig)
    ts.test_policy_nan_statistics_take_the_safer_path()
