"""Host-side helpers for the tests: the tiled E4M3 scale layout the GEMM reads.

The layout is a property of the CUDA path's data layout, not of the method:
scales of 128 rows x 4 consecutive 16-element blocks form one 512-byte chunk,
byte (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4; chunks run along K
within a 128-row tile, tiles along rows.
"""
import numpy as np


def scale_offsets(rows: int, k: int) -> np.ndarray:
    r = np.arange(rows)[:, None]
    kb = np.arange(k // 16)[None, :]
    return (r // 128) * (128 * (k // 16)) + (kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4


def untile_scales(buf: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Canonical [rows, K/16] scale codes from the tiled byte buffer."""
    return np.asarray(buf)[scale_offsets(rows, k)]


def bf16_bits_to_f32(t) -> np.ndarray:
    a = np.asarray(t).view(np.uint16).astype(np.uint32) << 16
    return a.view(np.float32)
