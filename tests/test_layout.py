"""The test-side layout readers invert each other (no GPU needed)."""
import numpy as np

from layout import scale_index, swizzle_scales, unswizzle_scales, unpack_codes


def test_scale_index_is_a_permutation():
    for rows, nblk in ((128, 4), (256, 16), (384, 8)):
        idx = scale_index(rows, nblk).reshape(-1)
        assert np.array_equal(np.sort(idx), np.arange(rows * nblk))


def test_swizzle_roundtrip_and_atom_shape():
    rng = np.random.default_rng(0)
    s = rng.integers(0, 255, (256, 8)).astype(np.uint8)
    flat = swizzle_scales(s)
    assert np.array_equal(unswizzle_scales(flat, 256, 8 * 32, 32), s)
    # one atom = 128 rows x 4 blocks in 512 bytes, rows r, r+32, r+64, r+96 share a 16-byte line
    assert flat[16 * 3 + 4 * 2 + 1] == s[2 * 32 + 3, 1]


def test_unpack_codes_nibble_order():
    p = np.array([[0x21, 0xF0]], np.uint8)
    assert unpack_codes(p).tolist() == [[1, 2, 0, 15]]
