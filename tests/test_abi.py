"""The C-ABI library loads and exports every call include/sixbit.h declares (CPU only).

No compute is launched here: only host-side functions and argument checks
that fail before any kernel would be enqueued.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

from tests._layouts import scale_offsets

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from video_dit_mixed_gb300 import abi
    return abi.lib(build_if_missing=True)


def _declared():
    src = open(os.path.join(ROOT, "include", "sixbit.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sixbit_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    from video_dit_mixed_gb300 import abi
    assert set(names) == set(abi.EXPORTS)


def test_scale_layout_host_functions(lib):
    rows, k = 300, 384
    off = scale_offsets(rows, k)
    for r in (0, 1, 31, 32, 127, 128, 255, 299):
        for kb in (0, 1, 3, 4, 7, 23):
            assert lib.sixbit_fp4_scale_offset(r, kb, k) == off[r, kb]
    assert lib.sixbit_fp4_scale_bytes(rows, k) == 384 * (k // 16)
    # a bijection onto the buffer for full tiles
    full = scale_offsets(256, k)
    assert np.array_equal(np.sort(full.ravel()), np.arange(256 * k // 16))


def test_argument_errors_return_status_without_launching(lib):
    from video_dit_mixed_gb300 import abi
    before = lib.sixbit_launch_count()
    qa = abi.QAct()
    w = abi.Weights()
    # NULL input
    assert lib.sixbit_hadamard_quant(None, 16, 128, 16, abi.MODE_NVFP4, None, None, C.byref(qa), None, None) == 1
    # K not a multiple of 128
    buf = C.create_string_buffer(64)
    p = C.cast(buf, C.c_void_p)
    assert lib.sixbit_hadamard_quant(p, 16, 96, 16, abi.MODE_INT8, None, None, C.byref(qa), None, None) == 2
    # unsupported Hadamard block
    assert lib.sixbit_hadamard_quant(p, 16, 128, 32, abi.MODE_INT8, None, None, C.byref(qa), None, None) == 2
    # GEMM: missing output, bad epilogue, bad N
    assert lib.sixbit_qgemm(C.byref(qa), None, C.byref(w), 16, 128, 128, 1, None, 0, None, None, None, None,
                            None, None, None) == 1
    assert lib.sixbit_qgemm(C.byref(qa), None, C.byref(w), 16, 120, 128, 1, None, 0, None, p, None, None,
                            None, None, None) == 2
    assert lib.sixbit_qgemm(C.byref(qa), None, C.byref(w), 16, 128, 128, 1, None, 7, None, p, None, None,
                            None, None, None) == 1
    # INT8 without the weight-expansion workspace
    assert lib.sixbit_qgemm(C.byref(qa), None, C.byref(w), 16, 128, 128, abi.MODE_INT8, None, 0, None, p, None,
                            None, None, None, None) == 1
    assert lib.sixbit_qgemm_workspace_bytes(5760, 1920) == 5760 * 1920 * 2
    # stats: n not a multiple of 8
    assert lib.sixbit_block_stats(p, p, p, 12, None, p, p, None, None) == 2
    # MXFP8 Delta cache: n a multiple of 32, both cache arrays given
    assert lib.sixbit_block_stats_mxfp8(p, p, p, p, 48, None, p, p, None, None) == 2
    assert lib.sixbit_block_stats_mxfp8(p, p, p, None, 64, None, p, p, None, None) == 1
    assert lib.sixbit_skip_apply_mxfp8(p, p, p, p, 40, None, p, p, None, None) == 2
    assert lib.sixbit_skip_apply_mxfp8(p, None, p, p, 64, None, p, p, None, None) == 1
    blocks = abi.DitBlocks()
    for f in ("states", "stats", "modes", "in_stats0", "x0", "deltas", "run_len"):
        setattr(blocks, f, p.value)
    blocks.buf[0] = blocks.buf[1] = p.value
    blocks.n, blocks.L = 64, 2
    cfg = abi.PolicyCfg()
    blocks.delta_format = 2                                    # no such format
    assert lib.sixbit_dit_block_end(C.byref(cfg), C.byref(blocks), 0, p, None, None) == 1
    blocks.delta_format = 1                                    # MXFP8 without its scales
    assert lib.sixbit_dit_block_end(C.byref(cfg), C.byref(blocks), 0, p, None, None) == 1
    blocks.delta_scales = p.value
    blocks.n = 40                                              # MXFP8 needs n % 32 == 0
    assert lib.sixbit_dit_skip_run(C.byref(cfg), C.byref(blocks), 0, p, None, None) == 2
    # the down projection with the block statistics: residual, Y, Delta cache and parts required;
    # their fold: parts given, n > 0; the DiT's fold: a bf16 Delta cache only
    assert lib.sixbit_qgemm_blockstats(C.byref(qa), None, C.byref(w), 16, 128, 128, 1, None, None, p, p, p, None,
                                       None, None) == 1
    assert lib.sixbit_qgemm_blockstats(C.byref(qa), None, C.byref(w), 16, 128, 128, 1, None, p, p, p, None, None,
                                       None, None) == 1
    assert lib.sixbit_block_stats_parts(None, 64, p, None, None) == 1
    assert lib.sixbit_block_stats_parts(p, 0, p, None, None) == 2
    blocks.n, blocks.delta_format = 64, 1
    assert lib.sixbit_dit_block_end_parts(C.byref(cfg), C.byref(blocks), 0, p, None, None) == 1
    assert lib.sixbit_policy_step(None, p, p, p, p, None, None) == 1
    assert lib.sixbit_launch_count() == before
    assert lib.sixbit_status_str(6) == b"device-side wait timed out"


def test_struct_sizes_match_header():
    from video_dit_mixed_gb300 import abi
    assert C.sizeof(abi.QAct) == 56 and C.sizeof(abi.Weights) == 56
    assert C.sizeof(abi.Stats) == 64 and C.sizeof(abi.PolicyCfg) == 48
    assert C.sizeof(abi.PolicyState) == 80 and C.sizeof(abi.DitBlocks) == 112


def test_struct_layouts_match_the_c_compiler(tmp_path):
    """Every field offset of the ctypes mirrors equals the C compiler's offsetof on include/sixbit.h."""
    import shutil
    import subprocess
    from video_dit_mixed_gb300 import abi
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"sixbit_qact": abi.QAct, "sixbit_weights": abi.Weights, "sixbit_stats": abi.Stats,
               "sixbit_policy_cfg": abi.PolicyCfg, "sixbit_policy_state": abi.PolicyState,
               "sixbit_dit_blocks": abi.DitBlocks}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "sixbit.h"', 'int main(void) {']
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in structs.items():
        assert got[(cname, "sizeof")] == C.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)
