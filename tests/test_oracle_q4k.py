"""Pins of the oracle's Q4_K block (the ds4.c page's type-trait table fixes
256 values in 144 bytes; the layout is the standard k-quant reading:
fp16 d @0, fp16 dmin @2, scales[12] @4 with eight 6-bit (scale, min) pairs,
qs[128] @16, value 64c + l in the low nibble of qs[32c + l], 64c + 32 + l in
its high nibble).

Pinned by: the byte count; hand-derived single-code positions; every one of
the 96 scale / min bits lands on its own bit of scales[12] (a bijection, so
pack(unpack(b)) == b for random bytes); closed forms of constant blocks;
one fp32 rounding of d * sc * q - dmin * mn.
"""
import numpy as np

import oracle

RNG = np.random.default_rng(144)
Q4K = oracle.Q4_K


def test_block_size_from_the_type_table():
    assert oracle.block_values(Q4K) == 256 and oracle.block_bytes(Q4K) == 144


def _blank(nb=1):
    return (np.zeros(nb * 256, np.uint8), np.zeros(nb * 8, np.uint8), np.zeros(nb * 8, np.uint8),
            np.full(nb, 0x3C00, np.uint16), np.zeros(nb, np.uint16))


def test_single_code_positions_hand_derived():
    # (value index, byte offset, high nibble?)
    cases = [(0, 16, False), (31, 47, False), (32, 16, True), (63, 47, True), (64, 48, False),
             (100, 52, True), (128, 80, False), (200, 120, False), (255, 143, True)]
    for i, byte, high in cases:
        codes, sc, mn, d, dmin = _blank()
        codes[i] = 0xA
        blk = oracle.q4k_pack(codes, sc, mn, d, dmin)
        nz = np.nonzero(blk[16:])[0] + 16
        assert list(nz) == [byte], (i, nz)
        assert blk[byte] == (0xA0 if high else 0x0A)


def test_scale_and_min_bits_are_a_bijection_onto_scales12():
    seen = {}
    for j in range(8):
        for field in ("sc", "mn"):
            for bit in range(6):
                codes, sc, mn, d, dmin = _blank()
                (sc if field == "sc" else mn)[j] = 1 << bit
                blk = oracle.q4k_pack(codes, sc, mn, d, dmin)
                bits = np.unpackbits(blk[4:16])
                pos = tuple(np.nonzero(bits)[0])
                assert len(pos) == 1, (j, field, bit)
                assert pos[0] not in seen, (j, field, bit, seen.get(pos[0]))
                seen[pos[0]] = (j, field, bit)
    assert len(seen) == 96  # all 12 bytes of scales used


def test_random_bytes_round_trip():
    raw = RNG.integers(0, 256, size=144 * 50, dtype=np.uint8)
    assert np.array_equal(oracle.q4k_pack(*oracle.q4k_unpack(raw)), raw)


def test_constant_block_closed_forms():
    # d = 0.5, dmin = 0.25; sub-block j: sc = j + 1 (j + 60 for j >= 4: both 6-bit
    # halves used), mn = 2 j; all codes 7: value = 0.5 * sc * 7 - 0.25 * mn
    codes, sc, mn, d, dmin = _blank()
    codes[:] = 7
    sc[:] = [1, 2, 3, 4, 61, 62, 63, 33]
    mn[:] = [0, 2, 4, 6, 48, 50, 52, 63]
    d[:] = np.float16(0.5).view(np.uint16)
    dmin[:] = np.float16(0.25).view(np.uint16)
    y = oracle.dequant(Q4K, oracle.q4k_pack(codes, sc, mn, d, dmin), 256)
    ref = np.repeat(0.5 * sc.astype(np.float64) * 7 - 0.25 * mn.astype(np.float64), 32)
    assert np.array_equal(y, ref.astype(np.float32))


def test_dequant_is_one_rounding_of_the_exact_value():
    nb = 20
    codes = RNG.integers(0, 16, nb * 256).astype(np.uint8)
    sc = RNG.integers(0, 64, nb * 8).astype(np.uint8)
    mn = RNG.integers(0, 64, nb * 8).astype(np.uint8)
    d = (np.abs(RNG.standard_normal(nb)) * 0.003).astype(np.float16).view(np.uint16)
    dmin = (np.abs(RNG.standard_normal(nb)) * 0.003).astype(np.float16).view(np.uint16)
    y = oracle.dequant(Q4K, oracle.q4k_pack(codes, sc, mn, d, dmin), nb * 256)
    D = np.repeat(d.view(np.float16).astype(np.float64), 256)
    M = np.repeat(dmin.view(np.float16).astype(np.float64), 256)
    S = np.repeat(sc.astype(np.float64), 32)
    Mn = np.repeat(mn.astype(np.float64), 32)
    assert np.array_equal(y, (D * S * codes - M * Mn).astype(np.float32))
