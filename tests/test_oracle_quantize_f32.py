"""Pins of the oracle's float-input quantizer ("【#2】ds4.c 해독하기", Q2_K
block writer: per-16-value scale / min, codes rounded to 0..3, importance
used as the weight of the quantisation error).

The pages give no search, so the pins are properties any reading must have
and that a slip in this one would break:
  * its binary16 encoder agrees with numpy's round-to-nearest-even cast;
  * every code is the nearest one for the block's own stored parameters;
  * values inside a sub-block's representable range are within half a step;
  * blocks that are already representable come back byte for byte;
  * with an importance vector the weighted error never exceeds the plain
    choice's weighted error;
  * degenerate blocks (all zero, constant) and argument errors.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(20261202)


def test_f16_encoder_matches_numpy_round_to_nearest_even():
    v = np.concatenate([
        (RNG.standard_normal(20000) * 10.0 ** RNG.integers(-9, 5, 20000)).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.99, 1e-8, 2.9802322e-08, 2.9802326e-08, 6.1035156e-05,
                  6.097555e-05, 1.00048828125, 1.000732421875, -3.0517578e-05], np.float32)])
    assert np.array_equal(oracle.f32_to_f16(v), v.astype(np.float16).view(np.uint16))


def _q2k_fields(blk):
    codes, sc, mn, d, dmin = oracle.q2k_unpack(blk)
    return codes.astype(np.int64), sc.astype(np.int64), mn.astype(np.int64), d, dmin


def _q2k_values(codes, sc, mn, d, dmin):
    """A, B per value (value = A q - B), float32 like the format's dequant."""
    sub = np.arange(codes.size) // 16
    blk = np.arange(codes.size) // 256
    D = np.array([oracle.f16(int(h)) for h in d], np.float32)[blk]
    M = np.array([oracle.f16(int(h)) for h in dmin], np.float32)[blk]
    A = (D * sc[sub].astype(np.float32)).astype(np.float32)
    B = (M * mn[sub].astype(np.float32)).astype(np.float32)
    return A, B


@pytest.mark.parametrize("scale", [1.0, 1e-3, 250.0])
def test_q2k_codes_are_nearest_for_the_stored_parameters(scale):
    x = (RNG.standard_normal(256 * 6) * scale).astype(np.float32)
    blk = oracle.quantize_f32(oracle.Q2_K, x)
    codes, sc, mn, d, dmin = _q2k_fields(blk)
    A, B = _q2k_values(codes, sc, mn, d, dmin)
    cand = (A[:, None] * np.arange(4, dtype=np.float32)[None, :] - B[:, None]).astype(np.float64)
    err = np.abs(x[:, None].astype(np.float64) - cand)
    chosen = err[np.arange(x.size), codes]
    assert np.all(chosen <= err.min(axis=1) + 1e-6 * np.maximum(A, 1e-30))
    # inside [-B, 3A - B] the error is at most half a step
    inside = (x >= -B) & (x <= 3 * A - B)
    assert np.all(chosen[inside] <= 0.5 * A[inside] * (1 + 1e-5) + 1e-30)
    assert inside.mean() > 0.9


def test_q41_codes_are_nearest_and_block_parameters_cover_the_range():
    x = (RNG.standard_normal(32 * 20) * 3.0 + 1.0).astype(np.float32)
    blk = oracle.quantize_f32(oracle.Q4_1, x)
    codes, d, m = oracle.q41_unpack(blk)
    D = np.repeat(np.array([oracle.f16(int(h)) for h in d], np.float32), 32)
    Mv = np.repeat(np.array([oracle.f16(int(h)) for h in m], np.float32), 32)
    q = codes.astype(np.int64)
    cand = (D[:, None] * np.arange(16, dtype=np.float32)[None, :] + Mv[:, None]).astype(np.float64)
    err = np.abs(x[:, None].astype(np.float64) - cand)
    assert np.all(err[np.arange(x.size), q] <= err.min(axis=1) + 1e-6 * D)
    # the step is the block's range over 15 (to binary16 precision)
    xb = x.reshape(-1, 32)
    rng = (xb.max(1) - xb.min(1)) / 15
    Db = D.reshape(-1, 32)[:, 0]
    assert np.allclose(Db, rng, rtol=2 ** -10)


def _representable_q2k(nb):
    """Blocks whose values the plain reading must reproduce exactly: every
    sub-block holds codes 0 and 3, one sub-block has sc = 15 and one mn = 15,
    scales >= 1 (so no sub-block is degenerate)."""
    codes = RNG.integers(0, 4, size=(nb, 16, 16)).astype(np.uint8)
    codes[:, :, 0] = 0
    codes[:, :, 1] = 3
    sc = RNG.integers(1, 16, size=(nb, 16)).astype(np.uint8)
    mn = RNG.integers(0, 16, size=(nb, 16)).astype(np.uint8)
    sc[:, 3] = 15
    mn[:, 7] = 15
    d = (np.abs(RNG.standard_normal(nb)) * 0.01 + 1e-3).astype(np.float16).view(np.uint16)
    dmin = (np.abs(RNG.standard_normal(nb)) * 0.01 + 1e-3).astype(np.float16).view(np.uint16)
    return oracle.q2k_pack(codes.reshape(-1), sc.reshape(-1), mn.reshape(-1), d, dmin)


def test_q2k_representable_blocks_round_trip_byte_for_byte():
    blk = _representable_q2k(12)
    x = oracle.dequant(oracle.Q2_K, blk, 12 * 256).astype(np.float32)
    assert np.array_equal(oracle.quantize_f32(oracle.Q2_K, x), blk)


def test_q41_representable_blocks_round_trip_byte_for_byte():
    nb = 16
    codes = RNG.integers(0, 16, size=(nb, 32)).astype(np.uint8)
    codes[:, 0] = 0
    codes[:, 1] = 15
    d = (np.abs(RNG.standard_normal(nb)) * 0.01 + 1e-3).astype(np.float16).view(np.uint16)
    m = (RNG.standard_normal(nb) * 0.02).astype(np.float16).view(np.uint16)
    blk = oracle.q41_pack(codes.reshape(-1), d, m)
    x = oracle.dequant(oracle.Q4_1, blk, nb * 32).astype(np.float32)
    assert np.array_equal(oracle.quantize_f32(oracle.Q4_1, x), blk)


@pytest.mark.parametrize("qtype", [oracle.Q2_K, oracle.Q4_1])
def test_importance_never_increases_the_weighted_error(qtype):
    cols = 512
    x = (RNG.standard_normal(cols * 8) * np.linspace(0.2, 3.0, cols)[None, :].repeat(8, 0).ravel()).astype(np.float32)
    imp = (RNG.exponential(1.0, cols) ** 2).astype(np.float32)
    plain = oracle.quantize_f32(qtype, x)
    weighted = oracle.quantize_f32(qtype, x, imp, cols)
    ep = oracle.weighted_sq_error(qtype, x, imp, cols, plain)
    ew = oracle.weighted_sq_error(qtype, x, imp, cols, weighted)
    assert ew <= ep * (1 + 1e-6)
    assert ew < ep  # and on this data the search does find something better
    # uniform importance changes the choice only towards a smaller plain error
    ones = np.ones(cols, np.float32)
    e1 = oracle.weighted_sq_error(qtype, x, None, cols, oracle.quantize_f32(qtype, x, ones, cols))
    assert e1 <= oracle.weighted_sq_error(qtype, x, None, cols, plain) * (1 + 1e-6)


def test_degenerate_blocks():
    z = np.zeros(512, np.float32)
    assert not oracle.quantize_f32(oracle.Q2_K, z).any()
    assert not oracle.quantize_f32(oracle.Q4_1, z).any()
    # a constant positive Q2_K block: zero mins, the value at code 3
    c = np.full(256, 0.75, np.float32)
    blk = oracle.quantize_f32(oracle.Q2_K, c)
    y = oracle.dequant(oracle.Q2_K, blk, 256)
    assert np.abs(y - 0.75).max() <= 0.75 * 2 ** -10
    # a constant Q4_1 block: step 0, min = the value in binary16
    c4 = np.full(32, -1.2345, np.float32)
    y4 = oracle.dequant(oracle.Q4_1, oracle.quantize_f32(oracle.Q4_1, c4), 32)
    assert np.all(y4 == np.float32(np.float16(-1.2345)))


def test_argument_errors():
    with pytest.raises(oracle.OracleError):
        oracle.quantize_f32(oracle.Q2_K, np.zeros(100, np.float32))
    with pytest.raises(oracle.OracleError):  # columns not whole blocks
        oracle.quantize_f32(oracle.Q4_1, np.zeros(96, np.float32), np.ones(48, np.float32), 48)
    bad = np.zeros(32, np.float32)
    bad[5] = np.inf
    with pytest.raises(oracle.OracleError):
        oracle.quantize_f32(oracle.Q4_1, bad)
