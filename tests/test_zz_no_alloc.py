"""The allocation-free block-statistics entry point agrees with the regular one.

sixbit_block_stats_noalloc serves callers that cannot call cudaMalloc (and so
cannot hand the library a scratch buffer): it reduces through a fixed array
inside the library instead.  This file is named to be collected last, so a
run that stops at the first failure has already run every other test; it
passes on its own in a fresh process as well.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synthgen
from oracle.formats import bf16_round

pytestmark = pytest.mark.gpu


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


def _inputs(seed, n):
    xi = synthgen.activations(seed, 1, n, "laplace", 0.0, 1.0).reshape(-1)
    xo = bf16_round(xi + synthgen.normal(seed + 1, 1, n).astype(np.float32) * 0.3)
    dp = bf16_round(synthgen.normal(seed + 2, 1, n).astype(np.float32) * 0.3)
    return _dev_bf16(xi), _dev_bf16(xo), _dev_bf16(dp)


def test_noalloc_matches_regular_entry_point_twice_in_a_row():
    from video_dit_mixed_gb300 import abi, ops
    lib = abi.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (seed, n) in enumerate([(5, 17776 * 1920), (8, 1920 * 257 + 8)]):
        xi, xo, dp = _inputs(seed, n)
        # the existing entry point, with caller scratch
        cache_ref = dp.clone()
        st_ref = ops.new_stats()
        ops.block_stats(xi, xo, cache_ref, st_ref, ops.new_scratch(n))
        # the allocation-free entry point, straight through the C ABI
        cache = dp.clone()
        st = ops.new_stats()
        status = lib.sixbit_block_stats_noalloc(C.c_void_p(xi.data_ptr()), C.c_void_p(xo.data_ptr()),
                                                C.c_void_p(cache.data_ptr()), n, None,
                                                C.c_void_p(st.data_ptr()), None, stream)
        assert status == 0, lib.sixbit_status_str(status)
        torch.cuda.synchronize()
        assert torch.equal(cache.view(torch.int16), cache_ref.view(torch.int16)), f"delta differs (call {call})"
        a = st.cpu().numpy()[0]
        b = st_ref.cpu().numpy()[0]
        assert a[4] == b[4] and a[6] == b[6] == n
        # sums of non-negative terms: TwoSum-accumulated (0, 3) agree to 1e-9;
        # Kahan-accumulated (1, 5) to twice Kahan's 2u bound, since the two
        # entry points use different grids and so different summation orders
        for i, rel in ((0, 1e-9), (1, 5e-7), (3, 1e-9), (5, 5e-7)):
            assert abs(a[i] - b[i]) <= rel * abs(b[i]), (call, i, a[i], b[i])
        d = cache_ref.float().double()
        p = dp.float().double()
        assert abs(a[2] - b[2]) <= 1e-9 * float((d * p).abs().sum()), (call, a[2], b[2])


def test_noalloc_rejects_oversized_input_without_launching():
    from video_dit_mixed_gb300 import abi
    lib = abi.lib()
    big = lib.sixbit_block_stats_noalloc_max_elems() + 8
    before = lib.sixbit_launch_count()
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(8, dtype=torch.float64, device="cuda")
    p = C.c_void_p(x.data_ptr())
    status = lib.sixbit_block_stats_noalloc(p, p, p, big, None, C.c_void_p(st.data_ptr()), None, None)
    assert status == 2 and lib.sixbit_status_str(status) == b"unsupported shape"
    assert lib.sixbit_launch_count() == before


def test_noalloc_skip_mode_touches_nothing_then_still_matches():
    """With the mode word at SKIP the kernel returns at once: the delta cache and the statistics keep
    their contents.  The next computing call, which finds the shared array as the skipped call left
    it, still matches the regular entry point."""
    from video_dit_mixed_gb300 import abi, ops
    lib = abi.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    n = 1920 * 520
    xi, xo, dp = _inputs(13, n)
    mode = torch.tensor([ops.MODE_SKIP], dtype=torch.int32, device="cuda")
    cache = dp.clone()
    st = torch.full((1, 8), -1.0, dtype=torch.float64, device="cuda")

    def call():
        return lib.sixbit_block_stats_noalloc(C.c_void_p(xi.data_ptr()), C.c_void_p(xo.data_ptr()),
                                              C.c_void_p(cache.data_ptr()), n, C.c_void_p(mode.data_ptr()),
                                              C.c_void_p(st.data_ptr()), None, stream)
    assert call() == 0
    torch.cuda.synchronize()
    assert torch.equal(cache.view(torch.int16), dp.view(torch.int16))
    assert bool((st == -1.0).all())
    mode.fill_(ops.MODE_INT8)
    assert call() == 0
    cache_ref = dp.clone()
    st_ref = ops.new_stats()
    ops.block_stats(xi, xo, cache_ref, st_ref, ops.new_scratch(n), mode_dev=mode)
    torch.cuda.synchronize()
    assert torch.equal(cache.view(torch.int16), cache_ref.view(torch.int16))
    a, b = st.cpu().numpy()[0], st_ref.cpu().numpy()[0]
    assert a[4] == b[4] and a[6] == b[6] == n
    for i, rel in ((0, 1e-9), (1, 5e-7), (3, 1e-9), (5, 5e-7)):
        assert abs(a[i] - b[i]) <= rel * abs(b[i]), (i, a[i], b[i])
