"""Host checks of the producer kernel's shared-memory layout arithmetic,
restated here in Python from the kernel's comments (the GPU parity tests
then check the kernel's outputs against the oracle):

* tiles are unpadded 128 x 128 bf16 with the 16-byte chunks of row r XOR-ed
  by r & 7; the map must be a bijection onto the tile's 16,384 elements, and
  every access pattern the kernel issues must touch each of the 32 banks
  once per phase (8 lanes for 16-byte accesses, 32 lanes for 2- and 4-byte
  ones): the cp.async copies, the row-segment loads and the column loads;
* the row segments are numbered so that each warp holds 32 consecutive rows
  at one block index: a bijection onto the 128 x 4 (row, block) pairs, with
  every 32 x 32 block (2D weights) inside one warp.
"""

TILE = 128


def tile_off(r: int, c: int) -> int:
    ch = c >> 3
    return r * TILE + ((((ch ^ r) & 7) | (ch & ~7)) * 8) + (c & 7)


def banks(byte_addr: int, nbytes: int) -> set:
    return {((byte_addr // 4) + i) % 32 for i in range(max(nbytes // 4, 1))}


def seg_row(idx: int) -> int:
    return (idx & 31) + 32 * (idx >> 7)


def seg_j(idx: int) -> int:
    return (idx >> 5) & 3


def test_swizzle_is_a_bijection_within_rows():
    seen = set()
    for r in range(TILE):
        row = {tile_off(r, c) for c in range(TILE)}
        assert row == set(range(r * TILE, (r + 1) * TILE))  # stays in its own row
        seen |= row
    assert len(seen) == TILE * TILE


def test_cp_async_copies_are_conflict_free():
    # thread t copies chunk q & 15 of row q >> 4, q = t + 256 i; 8 lanes per phase
    for i in range(8):
        for t0 in range(0, 256, 8):
            used = set()
            for lane in range(8):
                q = t0 + lane + 256 * i
                b = banks(2 * tile_off(q >> 4, (q & 15) * 8), 16)
                assert not (used & b)
                used |= b


def test_row_segment_loads_are_conflict_free():
    # each lane loads chunk q of its segment (16 bytes); phases of 8 lanes
    for k in range(2):
        for w in range(8):
            for q in range(4):
                for p0 in range(0, 32, 8):
                    used = set()
                    for lane in range(p0, p0 + 8):
                        idx = 32 * w + lane + 256 * k
                        b = banks(2 * tile_off(seg_row(idx), 32 * seg_j(idx) + 8 * q), 16)
                        assert not (used & b)
                        used |= b


def test_column_loads_are_conflict_free():
    # lane = column pair cp (32 consecutive per warp), one 16-bit load per row
    for j in range(4):
        for cp0 in (0, 32):
            for h in range(2):
                for i in range(32):
                    words = {tile_off(j * 32 + i, 2 * (cp0 + lane) + h) // 2 for lane in range(32)}
                    assert len({w % 32 for w in words}) == 32


def test_segment_numbering_covers_every_block_once_per_warp():
    pairs = {(seg_row(i), seg_j(i)) for i in range(512)}
    assert pairs == {(r, j) for r in range(TILE) for j in range(4)}
    for w in range(16):  # 16 warps of segments (two passes of 8 warps)
        rows = {seg_row(32 * w + lane) for lane in range(32)}
        js = {seg_j(32 * w + lane) for lane in range(32)}
        assert len(js) == 1 and rows == set(range(min(rows), min(rows) + 32)) and min(rows) % 32 == 0
