"""The GEMMs' bounded-wait failure path, exercised without faulting anything.

With sixbit_debug_gemm_timeout, every CTA's producer skips the copies of its
first pipeline stage and the wait limit is 20 ms, so the tensor-core thread's
wait for that stage runs out: the kernel must record SIXBIT_ETIMEOUT in the
caller's error word, stop its other roles, drain, free its tensor memory and
return.  The next launch on the same context must then run normally and give
the oracle's result (it could not even allocate tensor memory had the failed
launch kept it).
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synthgen
from oracle import gemm, quant

pytestmark = pytest.mark.gpu
MODES = {"nvfp4": 1, "int8": 2, "bf16": 3}
ETIMEOUT = 6


def _ref(mode, x, w, b):
    if mode == "nvfp4":
        qx = quant.hadamard_quant(x, b, "nvfp4")
        pw = quant.pack_weights(w, b)["nvfp4"]
        return gemm.nvfp4_gemm_ref(qx["codes"], qx["scales"], qx["s_t"], pw["codes"], pw["scales"], pw["s_t"])
    if mode == "int8":
        qx = quant.hadamard_quant(x, b, "int8")
        i4 = quant.pack_weights(w, b)["int4"]
        r, bd, _ = gemm.int8_gemm_ref(qx["q"], qx["s"], i4["q"], i4["s"])
        return r, bd
    return gemm.bf16_gemm_ref(x, w)


@pytest.mark.parametrize("mode", ["bf16", "nvfp4", "int8"])
def test_gemm_wait_timeout_is_reported_and_the_context_recovers(mode):
    from video_dit_mixed_gb300 import abi, ops
    lib = abi.lib()
    m, n, k, b = 384, 512, 640, 64
    x = synthgen.activations(91, m, k, "normal", 0.0, 1.0)
    w = synthgen.weights(92, n, k)
    xd = torch.from_numpy(x).to(torch.bfloat16).cuda()
    pw = ops.pack_weights(torch.from_numpy(w).cuda(), b)
    code = MODES[mode]
    qa = ops.hadamard_quant(xd, b, code) if mode != "bf16" else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    y = torch.full((m, n), 7.0, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert lib.sixbit_debug_gemm_timeout(20_000_000, 1) == 0
    try:
        ops.qgemm(qa, xd, pw, code, out=y, err=err, m=m)
        status = lib.sixbit_check(C.c_void_p(err.data_ptr()), stream)
    finally:
        assert lib.sixbit_debug_gemm_timeout(0, 0) == 0
    assert status == ETIMEOUT, lib.sixbit_status_str(status)
    assert int(err.item()) == 0                       # sixbit_check cleared the word
    # same context, next launch: normal result
    y2 = ops.qgemm(qa, xd, pw, code, out_f32=True, err=err, m=m)
    assert lib.sixbit_check(C.c_void_p(err.data_ptr()), stream) == 0
    ref, bound = _ref(mode, x, w, b)
    got = y2.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-5 * bound + 1e-30)


def test_debug_setting_rejects_bad_arguments():
    from video_dit_mixed_gb300 import abi
    lib = abi.lib()
    assert lib.sixbit_debug_gemm_timeout(0, 2) == 1
    assert lib.sixbit_debug_gemm_timeout(0, 0) == 0
