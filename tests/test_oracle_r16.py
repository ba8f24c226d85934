"""Pins of the oracle's 16-row tile order of Q2_K (q2k_to_r16 / q2k_from_r16 /
r16_dequant).

The tile order is this library's own storage order (the pages give none):
the bytes of the Q2_K block of "【#2】ds4.c 해독하기" (layout table and qs
packing) permuted inside every 16-row x 256-column tile-block.  It is pinned
against the plain Q2_K decode, itself pinned by hand-derived golden blocks
(tests/test_oracle_formats.py): a byte permutation that keeps every value,
with hand-derived positions for single codes and scale bytes.
"""
import numpy as np
import pytest

import oracle


def _random_q2k(rng, rows, cols):
    """Random Q2_K bytes with finite, normal fp16 d / dmin."""
    nb = rows * cols // 256
    b = rng.integers(0, 256, size=(nb, 84), dtype=np.uint8)
    for off in (80, 82):
        h = (rng.integers(5, 20, size=nb) << 10) | rng.integers(0, 1024, size=nb)
        b[:, off] = h & 0xFF
        b[:, off + 1] = h >> 8
    return b.reshape(-1)


def test_round_trip_random_bytes():
    rng = np.random.default_rng(11)
    for rows, cols in ((16, 256), (32, 512), (48, 1024)):
        b = rng.integers(0, 256, size=rows * cols // 256 * 84, dtype=np.uint8)
        r = oracle.q2k_to_r16(b, rows, cols)
        assert r.size == b.size
        assert np.array_equal(oracle.q2k_from_r16(r, rows, cols), b)


def test_bit_permutation():
    """Every source bit lands on exactly one destination bit, all distinct:
    the tile order is a bijection on the 1344 * 8 bits of a tile-block pair."""
    rows, cols = 16, 512
    n = rows * cols // 256 * 84
    zero = np.zeros(n, dtype=np.uint8)
    assert not oracle.q2k_to_r16(zero, rows, cols).any()
    seen = np.zeros(n * 8, dtype=bool)
    for byte in range(n):
        for bit in range(8):
            src = zero.copy()
            src[byte] = 1 << bit
            out = np.unpackbits(oracle.q2k_to_r16(src, rows, cols), bitorder="little")
            hits = np.flatnonzero(out)
            assert hits.size == 1, (byte, bit, hits)
            assert not seen[hits[0]], (byte, bit)
            seen[hits[0]] = True
    assert seen.all()


def test_values_equal_plain_q2k_decode():
    rng = np.random.default_rng(5)
    rows, cols = 48, 768
    b = _random_q2k(rng, rows, cols)
    ref = oracle.dequant(oracle.Q2_K, b, rows * cols).reshape(rows, cols)
    got = oracle.r16_dequant(oracle.q2k_to_r16(b, rows, cols), rows, cols)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# Hand-derived from the layout rule: (row, value) of a single code 1 in an
# otherwise zero 16 x 256 matrix -> (byte offset in the tile-block, byte value).
#  row 0, value 0:    sub-block 0, half 0, lane 0, word 0, bit 0   -> byte 0,    0x01
#  row 9, value 37:   sub-block 2 (v 5), lane 4*1+2 = 6, word 1, bit 16+4 = 20
#                     -> word at 96 + 4 = 100, byte 102, bit 4        -> 0x10
#  row 15, value 255: sub-block 15 (v 15), half 1, lane 4*7+3 = 31, word 3,
#                     bit 16+14 = 30 -> word at 512+496+12 = 1020, byte 1023, bit 6 -> 0x40
#  row 4, value 130:  sub-block 8 (v 2), half 1, lane 16, word 0, bit 2
#                     -> word at 512+256 = 768, byte 768, bit 2        -> 0x04
SINGLE_CODES = [((0, 0), (0, 0x01)), ((9, 37), (102, 0x10)), ((15, 255), (1023, 0x40)), ((4, 130), (768, 0x04))]


@pytest.mark.parametrize("pos,expect", SINGLE_CODES)
def test_single_code_positions(pos, expect):
    row, val = pos
    blocks = np.zeros((16, 84), dtype=np.uint8)
    # plain Q2_K: value i -> qs[32 (i / 128) + i % 32] at bit 2 ((i % 128) / 32)
    blocks[row, 16 + 32 * (val // 128) + val % 32] |= 1 << (2 * ((val % 128) // 32))
    out = oracle.q2k_to_r16(blocks.reshape(-1), 16, 256)
    nz = np.flatnonzero(out)
    assert nz.tolist() == [expect[0]]
    assert out[expect[0]] == expect[1]


# Scale bytes: (row, sub-block) -> byte offset, hand-derived:
#  row 10, sub-block 13: lane 4*2 + 5//2 = 10, row word 1, byte 1 + 2 = 3 -> 1024 + 80 + 4 + 3 = 1111
#  row 3, sub-block 0:   lane 12, word 0, byte 0                        -> 1024 + 96 = 1120
#  row 8, sub-block 9:   lane 0, word 1, byte 1 + 2 = 3                 -> 1024 + 4 + 3 = 1031
SCALES = [((10, 13), 1111), ((3, 0), 1120), ((8, 9), 1031)]


@pytest.mark.parametrize("pos,off", SCALES)
def test_scale_byte_positions(pos, off):
    row, sb = pos
    blocks = np.zeros((16, 84), dtype=np.uint8)
    blocks[row, sb] = 0xA5
    out = oracle.q2k_to_r16(blocks.reshape(-1), 16, 256)
    assert np.flatnonzero(out).tolist() == [off]
    assert out[off] == 0xA5


def test_d_dmin_positions():
    blocks = np.zeros((16, 84), dtype=np.uint8)
    blocks[7, 80:84] = [1, 2, 3, 4]
    out = oracle.q2k_to_r16(blocks.reshape(-1), 16, 256)
    assert np.flatnonzero(out).tolist() == [1308, 1309, 1310, 1311]
    assert out[1308:1312].tolist() == [1, 2, 3, 4]


def test_tiles_stay_in_place():
    """Each 16-row tile-block keeps the byte range the plain layout gives it."""
    rng = np.random.default_rng(3)
    rows, cols = 32, 512
    b = rng.integers(0, 256, size=rows * cols // 256 * 84, dtype=np.uint8)
    r = oracle.q2k_to_r16(b, rows, cols)
    rowb = cols // 256 * 84
    for t in range(rows // 16):
        for blk in range(cols // 256):
            src = np.concatenate([b[(16 * t + i) * rowb + 84 * blk:(16 * t + i) * rowb + 84 * blk + 84]
                                  for i in range(16)])
            dst = r[16 * t * rowb + 1344 * blk:16 * t * rowb + 1344 * blk + 1344]
            assert sorted(np.unpackbits(src).tolist()) == sorted(np.unpackbits(dst).tolist())


@pytest.mark.parametrize("rows,cols", [(8, 256), (16, 128), (24, 256)])
def test_rejects_partial_tiles(rows, cols):
    with pytest.raises(ValueError):
        oracle.q2k_to_r16(np.zeros(max(rows * cols // 256, 1) * 84, dtype=np.uint8), rows, cols)
