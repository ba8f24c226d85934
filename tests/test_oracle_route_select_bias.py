"""Pins of the oracle's routing variant with the bias used for selection
only (the survey's "next" routing row; DeepSeek-style): ranking by
logit + bias, weights = softmax of the selected experts' unbiased logits.

Pinned by: a zero bias reduces it to the plain route (a separate code
path); brute force over all subsets on tiny inputs (the chosen set is the
k largest biased logits, ties to lower ids); weights depend on the
unbiased logits only (a huge bias on one expert forces it in without
changing the other experts' relative weights); weights sum to one and are
ordered like the unbiased logits.
"""
import itertools

import numpy as np

import oracle

RNG = np.random.default_rng(77)


def _layer(T, D, E):
    x = (RNG.standard_normal((T, D)).astype(np.float32)).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation: some bf16 pattern
    Wr = (RNG.standard_normal((E, D)) * 0.05).astype(np.float32)
    return xb, Wr


def test_zero_bias_is_the_plain_route():
    xb, Wr = _layer(9, 64, 12)
    idx, w, _, _ = oracle.route_select_bias(xb, Wr, np.zeros(12, np.float32), 4)
    ridx, rw, _ = oracle.route(xb, Wr, None, 4)
    assert np.array_equal(idx, ridx)
    assert np.array_equal(w.view(np.uint32), rw.view(np.uint32))


def test_selection_is_the_k_largest_biased_logits_by_brute_force():
    xb, Wr = _layer(6, 32, 7)
    bias = RNG.standard_normal(7).astype(np.float32)
    idx, w, lu, lb = oracle.route_select_bias(xb, Wr, bias, 3)
    for t in range(6):
        best = max(itertools.combinations(range(7), 3),
                   key=lambda c: (sorted((lb[t, e] for e in c), reverse=True), [-e for e in c]))
        assert set(idx[t]) == set(best)
        # rank order: biased logit descending
        assert all(lb[t, idx[t, i]] >= lb[t, idx[t, i + 1]] for i in range(2))


def test_weights_follow_the_unbiased_logits_only():
    xb, Wr = _layer(5, 48, 10)
    bias = np.zeros(10, np.float32)
    bias[8] = 1e6  # expert 8 is always selected
    idx, w, lu, _ = oracle.route_select_bias(xb, Wr, bias, 3)
    assert np.all(idx[:, 0] == 8)
    for t in range(5):
        u = lu[t, idx[t]].astype(np.float64)
        ref = np.exp(u - u.max())
        ref /= ref.sum()
        assert np.allclose(w[t], ref, rtol=1e-6)
        assert abs(w[t].astype(np.float64).sum() - 1.0) < 1e-6
        order = np.argsort(-u, kind="stable")
        assert np.all(np.diff(w[t][order]) <= 0)
