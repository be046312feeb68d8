"""Test-side readers of the quantized-view layout documented in
include/fp4lin.h (written from that description; shares no code with the
library or the oracle)."""
import numpy as np


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[rows, cols/2] bytes -> [rows, cols] 4-bit codes (value k in byte k/2,
    low nibble for even k)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), np.uint8)
    out[:, 0::2] = p & 0x0F
    out[:, 1::2] = p >> 4
    return out


def scale_index(rows: int, nblk: int) -> np.ndarray:
    """Byte offset of (r, j) in the 128x4 atom layout, as an int64 [rows, nblk] array."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    j = np.arange(nblk, dtype=np.int64)[None, :]
    atom = (r // 128) * (nblk // 4) + j // 4
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (j % 4)


def unswizzle_scales(flat: np.ndarray, rows: int, cols: int, bs: int) -> np.ndarray:
    flat = np.asarray(flat, dtype=np.uint8).reshape(-1)
    return flat[scale_index(rows, cols // bs)]


def swizzle_scales(logical: np.ndarray) -> np.ndarray:
    rows, nblk = logical.shape
    out = np.zeros(rows * nblk, np.uint8)
    out[scale_index(rows, nblk)] = logical
    return out


def expand_outer(outer: np.ndarray, count: int, rows: int) -> np.ndarray:
    """Per-stored-row S_enc from the view's outer array."""
    o = np.asarray(outer, dtype=np.float32)[:count]
    if count == 1:
        return np.full(rows, o[0], np.float32)
    return np.repeat(o, 128)[:rows]
