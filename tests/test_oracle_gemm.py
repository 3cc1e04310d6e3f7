"""Pins for the oracle's reference GEMMs (CPU only): brute force on tiny shapes."""
import math

import numpy as np
import torch

from oracle import formats, gemm, quant

F32 = np.float32


def _tiny(seed, m=3, n=2, k=128):
    rng = np.random.default_rng(seed)
    x = formats.bf16_round((rng.laplace(size=(m, k)) * 2).astype(F32))
    w = (rng.standard_normal((n, k)) * 0.05).astype(F32)
    return x, w


def test_nvfp4_gemm_brute_force():
    x, w = _tiny(1)
    qx = quant.nvfp4_quantize(x)
    qw = quant.nvfp4_quantize(w)
    ref, bound = gemm.nvfp4_gemm_ref(qx["codes"], qx["scales"], qx["s_t"], qw["codes"], qw["scales"], qw["s_t"])
    m, k = x.shape
    n = w.shape[0]
    e2 = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    def val(code, sc):   # decode by the format tables, not by formats.decode
        mag = e2[code & 7] * (-1 if code & 8 else 1)
        e, mnt = (sc >> 3) & 15, sc & 7
        s = (mnt / 8) * 2.0 ** -6 if e == 0 else (1 + mnt / 8) * 2.0 ** (e - 7)
        return mag * s
    for i in range(m):
        for j in range(n):
            acc, acc_abs = 0.0, 0.0
            for t in range(k):
                a = val(int(qx["codes"][i, t]), int(qx["scales"][i, t // 16]))
                b = val(int(qw["codes"][j, t]), int(qw["scales"][j, t // 16]))
                acc += a * b
                acc_abs += abs(a * b)
            s = float(qx["s_t"]) * float(qw["s_t"])
            assert math.isclose(ref[i, j], s * acc, rel_tol=1e-12, abs_tol=1e-300)
            assert math.isclose(bound[i, j], s * acc_abs, rel_tol=1e-12, abs_tol=1e-300)


def test_int8_gemm_brute_force():
    x, w = _tiny(2, k=256)
    qx = quant.int8_quantize(x)
    qw = quant.int4_quantize_weights(w)
    ref, bound, acc = gemm.int8_gemm_ref(qx["q"], qx["s"], qw["q"], qw["s"])
    m, k = x.shape
    n = w.shape[0]
    for i in range(m):
        for j in range(n):
            tot = 0.0
            for g in range(k // 128):
                a = 0
                for t in range(g * 128, (g + 1) * 128):
                    a += int(qx["q"][i, t]) * int(qw["q"][j, t])
                assert acc[g, i, j] == a
                tot += float(qw["s"][j, g]) * a
            assert math.isclose(ref[i, j], float(qx["s"][i]) * tot, rel_tol=1e-12)
    # the group form equals the plain dequantized product
    deq_x = qx["q"].astype(np.float64) * qx["s"][:, None].astype(np.float64)
    deq_w = qw["q"].astype(np.float64) * np.repeat(qw["s"].astype(np.float64), 128, axis=1)
    np.testing.assert_allclose(ref, deq_x @ deq_w.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bound, np.abs(deq_x) @ np.abs(deq_w).T, rtol=1e-12)


def test_bf16_gemm_brute_force():
    x, w = _tiny(3, k=64)
    ref, bound = gemm.bf16_gemm_ref(x, w)
    wb = formats.bf16_round(w)
    for i in range(x.shape[0]):
        for j in range(w.shape[0]):
            s = sum(float(x[i, t]) * float(wb[j, t]) for t in range(x.shape[1]))
            assert math.isclose(ref[i, j], s, rel_tol=1e-12, abs_tol=1e-15)


def test_gelu_matches_torch_exact_erf():
    v = np.linspace(-8, 8, 1001)
    ref = torch.nn.functional.gelu(torch.from_numpy(v), approximate="none").numpy()
    np.testing.assert_allclose(gemm.gelu(v), ref, rtol=1e-14, atol=1e-15)
    assert gemm.gelu(0.0) == 0.0
    # GELU(1) = Phi(1), the standard normal CDF at 1
    assert math.isclose(float(gemm.gelu(1.0)), 0.8413447460685429, rel_tol=1e-14)


def test_residual_epilogue():
    ref = np.array([[1.0, -2.0]])
    res = np.array([[0.5, 0.25]], F32)
    np.testing.assert_array_equal(gemm.epilogue(ref, "residual", res), [[1.5, -1.75]])
    np.testing.assert_array_equal(gemm.epilogue(ref, "none"), ref)
