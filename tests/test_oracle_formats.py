"""Pins of the oracle's block formats against what the pages fix.

Sources: molayo1419.me "【#2】ds4.c 해독하기" (Q2_K type trait 256 values /
84 bytes, layout table, qs_out packing expression) and thakicloud.com
"자체 저비트 포맷을 llama.cpp로 옮기기: 복원값이 비트까지 같은 GGUF Q4_1 재부호화"
(Q4_1 block and nibble order; the two lossless conditions; explicit bits and
group; read-back verification, max abs error 0.0).
"""
import numpy as np
import pytest

import oracle
from tests import golden_io as G

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f16(h):
    return np.array([h], dtype=np.uint16).view(np.float16)[0].astype(np.float64)


# -------------------------------------------------------------- block sizes
def test_block_sizes_match_pages():
    # Q2_K: 256 values in 84 bytes (type-trait table); Q4_1: 32 values in 20 bytes.
    assert oracle.block_values(oracle.Q2_K) == 256
    assert oracle.block_bytes(oracle.Q2_K) == 84
    assert oracle.block_values(oracle.Q4_1) == 32
    assert oracle.block_bytes(oracle.Q4_1) == 20
    # Q2_K vs raw f16: 512 / 84 ~ 6.1x smaller (the page's own ratio).
    assert round(512 / 84, 1) == 6.1
    # gguf byte shape of a Q4_1 row: cols / 32 * 20 (Q4_1 re-encode page).
    assert 4096 // 32 * 20 == 2560


# ------------------------------------------------------------ fp16 decoding
def test_f16_decode_all_patterns_match_numpy():
    hs = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = hs.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16(int(h)) for h in hs])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros
    assert np.signbit(oracle.f16(0x8000)) and not np.signbit(oracle.f16(0x0000))


def _ref_round_bf16(x: float) -> float:
    """Exact reference: round |x| to 8 significand bits (quantum floor 2^-133)
    with Python's rational round-half-even."""
    import math
    from fractions import Fraction
    if x == 0 or not math.isfinite(x):
        return x
    m, e = math.frexp(abs(x))                  # |x| = m * 2^e, m in [0.5, 1)
    q_exp = max(e - 8, -133)
    n = round(Fraction(abs(x)) / Fraction(2) ** q_exp)
    v = float(n * Fraction(2) ** q_exp)
    if v >= 2.0 ** 128:
        v = math.inf
    return math.copysign(v, x)


def test_round_bf16_matches_exact_rounding():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-45, 39, 4000),
                        [0.0, -0.0, np.inf, -np.inf, 1.0, 3.0e38, 3.4e38, 1e-40, 9.2e-41, 5.877e-39,
                         1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8 + 2.0 ** -40)]])
    got = oracle.round_bf16(v)
    for x, g in zip(v.tolist(), got.tolist()):
        r = _ref_round_bf16(x)
        gv = oracle.bf16(int(g))
        assert gv == r and np.signbit(gv) == np.signbit(r), (x, hex(g), r)
    assert np.isnan(oracle.bf16(int(oracle.round_bf16([np.nan])[0])))


# ----------------------------------------------------------- Q4_1 (pinned)
def test_q4_1_golden_block():
    g = G.load("q4_1_block.txt")
    codes = np.array(G.ints(g["codes"]), np.uint8)
    d, m = int(g["d_f16"], 16), int(g["m_f16"], 16)
    blk = oracle.q41_pack(codes, [d], [m])
    assert blk.tolist() == G.hex_bytes(g["bytes"])
    vals = oracle.dequant(oracle.Q4_1, blk, 32)
    assert vals.tolist() == G.floats(g["values"])


@pytest.mark.parametrize("j", range(32))
def test_q4_1_single_code_bit_position(j):
    # value j -> low nibble of qs[j] (j < 16), high nibble of qs[j-16] (j >= 16);
    # qs starts after the two fp16 fields, at byte 4.
    base = oracle.q41_pack(np.zeros(32, np.uint8), [0x3C00], [0])
    for v in range(1, 16):
        c = np.zeros(32, np.uint8)
        c[j] = v
        blk = oracle.q41_pack(c, [0x3C00], [0])
        diff = np.nonzero(blk != base)[0].tolist()
        byte = 4 + (j % 16)
        assert diff == [byte]
        assert blk[byte] == (v if j < 16 else v << 4)
        vals = oracle.dequant(oracle.Q4_1, blk, 32)
        expect = np.zeros(32, np.float32)
        expect[j] = v
        assert np.array_equal(vals, expect)


def test_q4_1_roundtrip_random_bytes_is_bijection():
    rng = np.random.default_rng(1)
    blocks = rng.integers(0, 256, 20 * 500, dtype=np.uint8)
    codes, d, m = oracle.q41_unpack(blocks)
    assert codes.max() <= 15
    assert np.array_equal(oracle.q41_pack(codes, d, m), blocks)


def test_q4_1_dequant_is_single_rounding_of_exact_value():
    rng = np.random.default_rng(2)
    nb = 4000
    codes = rng.integers(0, 16, nb * 32).astype(np.uint8)
    # finite fp16 patterns of either sign, incl. subnormals
    d = rng.integers(0, 0x7C00, nb).astype(np.uint16) | (rng.integers(0, 2, nb) << 15).astype(np.uint16)
    m = rng.integers(0, 0x7C00, nb).astype(np.uint16) | (rng.integers(0, 2, nb) << 15).astype(np.uint16)
    blk = oracle.q41_pack(codes, d, m)
    got = oracle.dequant(oracle.Q4_1, blk, nb * 32)
    dd = np.repeat(d.view(np.float16).astype(np.float64), 32)
    mm = np.repeat(m.view(np.float16).astype(np.float64), 32)
    # d*q is exact in float64 and d*q + m too: one rounding to float32
    ref = (dd * codes.astype(np.float64) + mm).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ----------------------------------------------------------- Q2_K (pinned)
def test_q2_k_golden_block_a():
    g = G.load("q2_k_block_a.txt")
    i = np.arange(256)
    codes = ((i % 128) // 32).astype(np.uint8)
    sc = np.array(G.ints(g["sc"]), np.uint8)
    mn = np.array(G.ints(g["mn"]), np.uint8)
    d, dmin = int(g["d_f16"], 16), int(g["dmin_f16"], 16)
    blk = oracle.q2k_pack(codes, sc, mn, [d], [dmin])
    assert blk.tolist() == G.hex_bytes(g["bytes"])
    vals = oracle.dequant(oracle.Q2_K, blk, 256)
    expect = sc[i // 16].astype(np.float64) * codes - 0.25 * mn[i // 16]
    assert vals.tolist() == expect.tolist()


def test_q2_k_golden_block_b():
    g = G.load("q2_k_block_b.txt")
    codes = np.zeros(256, np.uint8)
    codes[int(g["code_index"])] = int(g["code_value"])
    sc = np.full(16, int(g["sc_all"]), np.uint8)
    mn = np.full(16, int(g["mn_all"]), np.uint8)
    blk = oracle.q2k_pack(codes, sc, mn, [int(g["d_f16"], 16)], [int(g["dmin_f16"], 16)])
    assert blk[int(g["byte_index"])] == int(g["byte_value"], 16)
    vals = oracle.dequant(oracle.Q2_K, blk, 256)
    assert vals[int(g["code_index"])] == float(g["value_at_index"])
    assert np.count_nonzero(vals) == 1


@pytest.mark.parametrize("i", range(0, 256, 1))
def test_q2_k_single_code_bit_position(i):
    # qs byte j/4 + l, shift 2 * term, with j = 128 * (i // 128),
    # term = (i - j) // 32 and l = (i - j) % 32; qs starts at block byte 16.
    zero = np.zeros(256, np.uint8)
    sc = np.ones(16, np.uint8)
    mn = np.zeros(16, np.uint8)
    base = oracle.q2k_pack(zero, sc, mn, [0x3C00], [0])
    j = 128 * (i // 128)
    term, l = (i - j) // 32, (i - j) % 32
    for v in (1, 2, 3):
        c = zero.copy()
        c[i] = v
        blk = oracle.q2k_pack(c, sc, mn, [0x3C00], [0])
        diff = np.nonzero(blk != base)[0].tolist()
        assert diff == [16 + j // 4 + l]
        assert blk[16 + j // 4 + l] == v << (2 * term)
        vals = oracle.dequant(oracle.Q2_K, blk, 256)
        assert vals[i] == v and np.count_nonzero(vals) == 1


def test_q2_k_scale_nibbles_and_field_offsets():
    # sub-block n's byte is scales[n] at offset n; d at 80, dmin at 82 (little endian)
    codes = np.zeros(256, np.uint8)
    for n in range(16):
        sc = np.zeros(16, np.uint8)
        mn = np.zeros(16, np.uint8)
        sc[n], mn[n] = 5, 9
        blk = oracle.q2k_pack(codes, sc, mn, [0x1234], [0xABCD])
        assert blk[n] == 5 | (9 << 4)
        assert np.count_nonzero(blk[:16]) == 1
        assert blk[80:84].tolist() == [0x34, 0x12, 0xCD, 0xAB]
        vals = oracle.dequant(oracle.Q2_K, blk, 256)
        dmin = f16(0xABCD)
        # codes are 0, so only the min term: -dmin * 9 on sub-block n
        expect = np.zeros(256)
        expect[16 * n:16 * n + 16] = -dmin * 9
        assert np.array_equal(vals, expect.astype(np.float32))


def test_q2_k_roundtrip_random_bytes_is_bijection():
    rng = np.random.default_rng(3)
    blocks = rng.integers(0, 256, 84 * 300, dtype=np.uint8)
    fields = oracle.q2k_unpack(blocks)
    assert np.array_equal(oracle.q2k_pack(*fields), blocks)


def test_q2_k_dequant_is_single_rounding_of_exact_value():
    rng = np.random.default_rng(4)
    nb = 2000
    codes = rng.integers(0, 4, nb * 256).astype(np.uint8)
    sc = rng.integers(0, 16, nb * 16).astype(np.uint8)
    mn = rng.integers(0, 16, nb * 16).astype(np.uint8)
    d = rng.integers(0, 0x7C00, nb).astype(np.uint16)
    dmin = rng.integers(0, 0x7C00, nb).astype(np.uint16) | np.uint16(0x8000) * (rng.integers(0, 2, nb)).astype(np.uint16)
    blk = oracle.q2k_pack(codes, sc, mn, d, dmin)
    got = oracle.dequant(oracle.Q2_K, blk, nb * 256)
    dd = np.repeat(d.view(np.float16).astype(np.float64), 256)
    dm = np.repeat(dmin.view(np.float16).astype(np.float64), 256)
    s = np.repeat(sc, 16).astype(np.float64)
    m = np.repeat(mn, 16).astype(np.float64)
    ref = (dd * s * codes - dm * m).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_pack_rejects_out_of_range_fields():
    with pytest.raises(oracle.OracleError):
        oracle.q2k_pack(np.full(256, 4, np.uint8), np.zeros(16, np.uint8), np.zeros(16, np.uint8), [0], [0])
    with pytest.raises(oracle.OracleError):
        oracle.q2k_pack(np.zeros(256, np.uint8), np.full(16, 16, np.uint8), np.zeros(16, np.uint8), [0], [0])
    with pytest.raises(oracle.OracleError):
        oracle.q41_pack(np.full(32, 16, np.uint8), [0], [0])


# ------------------------------------------------ lossless re-encode to Q4_1
def _asym_source(rng, n, bits, group):
    codes = rng.integers(0, 1 << bits, n).astype(np.uint8)
    scale = (np.abs(rng.standard_normal(n // group)) * 0.01).astype(np.float16).view(np.uint16)
    mins = (rng.standard_normal(n // group) * 0.05).astype(np.float16).view(np.uint16)
    return codes, scale, mins


@pytest.mark.parametrize("bits,group,n", [(3, 32, 32 * 64), (4, 64, 64 * 64), (3, 64, 64 * 64),
                                          (3, 32, 1024 * 3072)])
def test_reencode_is_bit_identical_to_code_times_scale_plus_min(bits, group, n):
    # The page's local unit tests: (3-bit, 32), (4-bit, 64), (3-bit, 64) and a
    # large matrix, read back and compared bit for bit with code*scale + min.
    rng = np.random.default_rng(bits * 1000 + group)
    codes, scale, mins = _asym_source(rng, n, bits, group)
    st, blk = oracle.q41_reencode(bits, group, codes, scale, mins)
    assert st == oracle.OK
    assert blk.size == n // 32 * 20
    got = oracle.dequant(oracle.Q4_1, blk, n)
    s = np.repeat(scale.view(np.float16).astype(np.float64), group)
    m = np.repeat(mins.view(np.float16).astype(np.float64), group)
    ref = (codes * s + m).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.max(np.abs(got.astype(np.float64) - ref.astype(np.float64))) == 0.0
    # nothing recomputed: each block carries its group's fp16 pair verbatim
    c2, d2, m2 = oracle.q41_unpack(blk)
    assert np.array_equal(c2, codes)
    assert np.array_equal(d2, np.repeat(scale, group // 32))
    assert np.array_equal(m2, np.repeat(mins, group // 32))


@pytest.mark.parametrize("bits,group,bad_code,why", [
    (4, 48, None, "group not a multiple of 32"),
    (5, 32, None, "bit width above 4"),
    (4, 32, 16, "code does not fit a nibble"),
    (3, 32, 8, "code outside the declared 3-bit range"),
])
def test_reencode_blockers(bits, group, bad_code, why):
    rng = np.random.default_rng(5)
    n = 96 * 32
    codes = rng.integers(0, min(1 << bits, 16), n).astype(np.uint8)
    if bad_code is not None:
        codes[17] = bad_code
    scale = np.full(n // group, 0x2000, np.uint16)
    mins = np.zeros(n // group, np.uint16)
    st, _ = oracle.q41_reencode(bits, group, codes, scale, mins)
    assert st == oracle.EBLOCKER, why


def test_bits_and_group_are_not_inferred_from_byte_counts():
    # n_groups * group * bits == packed_bytes * 8 fixes only the product
    # group * bits: with 8 groups, (bits 4, group 64) and (bits 2, group 128)
    # both fill 256 packed bytes.  Reading the same bytes under each
    # declaration gives different tensors; only the explicit (bits, group)
    # arguments say which one the bytes hold.
    n_groups, packed_bytes = 8, 256
    assert n_groups * 64 * 4 == n_groups * 128 * 2 == packed_bytes * 8
    rng = np.random.default_rng(6)
    packed = rng.integers(0, 256, packed_bytes, dtype=np.uint8)
    bitsarr = np.unpackbits(packed, bitorder="little")

    def read(bits):
        return (bitsarr.reshape(-1, bits) * (1 << np.arange(bits))).sum(1).astype(np.uint8)

    scale = np.arange(0x2000, 0x2000 + n_groups, dtype=np.uint16)
    mins = np.zeros(n_groups, np.uint16)
    st_a, a = oracle.q41_reencode(4, 64, read(4), scale, mins)
    st_b, b = oracle.q41_reencode(2, 128, read(2), scale, mins)
    assert st_a == st_b == oracle.OK
    assert a.size == 512 // 32 * 20 and b.size == 1024 // 32 * 20
    da = oracle.dequant(oracle.Q4_1, a, 512)
    db = oracle.dequant(oracle.Q4_1, b, 1024)
    assert da.size != db.size and not np.array_equal(da, db[:512])
    # a declared width is enforced: a 4-bit code under a 2-bit declaration is a BLOCKER
    assert oracle.q41_reencode(2, 128, read(4)[:1024] if read(4).size >= 1024 else
                               np.concatenate([read(4), read(4)]), scale, mins)[0] == oracle.EBLOCKER
