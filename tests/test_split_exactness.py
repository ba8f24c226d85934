"""The exact gate/up operands of the tensor-core prefill, checked on the host
in numpy's IEEE fp16: for every code q and scale sc of a block format, the
integer sc * q is exact in fp16, and hi = RN16(d * (sc * q)) plus the FMA
residual lo = RN16(d * (sc * q) - hi) recovers d * sc * q exactly whenever the
residual stays out of fp16's subnormal range -- at the formats' d ranges it
does, with one ulp of the residual's spacing at most otherwise.  The same
holds for the minimum -dmin * mn split into mh + ml, and for Q4_1's d * q
(the block minimum m is an fp16 value itself)."""
import numpy as np
import pytest

F16_MIN_NORMAL = 2.0 ** -14


def _split(v):
    """hi = RN16(v), lo = RN16(v - hi): the fp16 pair the kernels build (an
    FMA computes v - hi exactly before its one rounding)."""
    hi = np.float16(v)
    lo = np.float16(v - np.float64(hi))
    return np.float64(hi), np.float64(lo)


def _random_d(rng, n, sigma):
    # fp16 scales as the synthetic recipes draw them: |N(0, sigma)| rounded to fp16, nonzero
    d = np.abs(rng.normal(0.0, sigma, n)).astype(np.float16).astype(np.float64)
    return d[d > 0]


@pytest.mark.parametrize("qmax,scmax,sigma", [(3, 15, 0.002), (15, 63, 0.0002)])  # Q2_K, Q4_K
def test_scaled_codes_split_exactly(qmax, scmax, sigma):
    rng = np.random.default_rng(qmax)
    sc = np.arange(scmax + 1, dtype=np.float64)
    q = np.arange(qmax + 1, dtype=np.float64)
    scq = (sc[:, None] * q[None, :]).ravel()
    assert np.all(scq <= 2048) and np.array_equal(np.float16(scq).astype(np.float64), scq)  # sc q exact in fp16
    for d in _random_d(rng, 400, sigma):
        v = d * scq                                    # exact in float64 (11 + 10 bits)
        hi, lo = _split(v)
        exact = hi + lo == v
        # misses only where the residual falls below fp16's normal range
        tiny = (np.abs(v - hi) < F16_MIN_NORMAL) & ~exact
        assert np.all(exact | tiny)
        # and then by at most half the subnormal spacing
        assert np.all(np.abs(hi + lo - v) <= 2.0 ** -25)


@pytest.mark.parametrize("mnmax,sigma", [(15, 0.002), (63, 0.0002)])
def test_minima_split_exactly(mnmax, sigma):
    rng = np.random.default_rng(mnmax)
    mn = np.arange(mnmax + 1, dtype=np.float64)
    for dmin in _random_d(rng, 400, sigma):
        v = -dmin * mn
        mh, ml = _split(v)
        assert np.all(np.abs(mh + ml - v) <= 2.0 ** -25)


def test_q4_1_codes_split_exactly():
    rng = np.random.default_rng(41)
    q = np.arange(16, dtype=np.float64)
    for d in _random_d(rng, 400, 0.01):
        v = d * q
        hi, lo = _split(v)
        assert np.all(np.abs(hi + lo - v) <= 2.0 ** -25)
        # at the Q4_1 recipe's scales the residual is always representable: exact
        assert np.all((hi + lo == v) | (np.abs(v - hi) < F16_MIN_NORMAL))


def test_one_rounding_is_not_exact():
    """Why the split: RN16(d * sc * q) alone misses by up to half an fp16 ulp
    (2^-12 relative), which flips the bf16 rounding of some h."""
    d = np.float64(np.float16(0.0013))
    v = d * 45.0
    assert np.float64(np.float16(v)) != v
