"""Pins of the oracle's routing and expert FFN.

The pages give the model shape (molayo1419.me "ds4.c 해독하기 1/8": 256 routed
experts, 6 used per token; "【#2】ds4.c 해독하기": w1 = gate, w2 = down,
w3 = up) but no worked numeric example, so these pins are exact brute force,
closed forms, hand-derived layers (tests/golden/tiny_ffn.txt) and
invariants.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests import golden_io as G
from tests.layers import build_layer, oracle_forward


def _round_f32(fr: Fraction) -> float:
    """Correct rounding of an exact rational to binary32 (ties to even)."""
    if fr == 0:
        return 0.0
    a = abs(fr)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 23, -149)
    n = round(a / Fraction(2) ** q)
    v = float(n * Fraction(2) ** q)
    return math.copysign(v, fr)


def _bf16_vals(b):
    return oracle.bf16_to_f32(b).astype(np.float64)


# ------------------------------------------------------------------ routing
def test_router_logits_equal_correctly_rounded_exact_dot():
    rng = np.random.default_rng(11)
    T, E, D = 5, 9, 96
    x = oracle.round_bf16(rng.standard_normal((T, D)))
    Wr = (rng.standard_normal((E, D)) * 0.02).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32)
    for b in (None, bias):
        got = oracle.router_logits(x, Wr, b)
        xv = _bf16_vals(x)
        for t in range(T):
            for e in range(E):
                exact = sum(Fraction(float(xv[t, j])) * Fraction(float(Wr[e, j])) for j in range(D))
                if b is not None:
                    exact += Fraction(float(b[e]))
                assert got[t, e] == np.float32(_round_f32(exact)), (t, e)


def test_topk_matches_full_sort_brute_force_with_ties_and_nan():
    rng = np.random.default_rng(12)
    T, E = 200, 17
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[::3, 5] = logits[::3, 2]             # exact ties -> lower id first
    logits[::7, 4] = np.nan                       # NaN ranks below -inf
    logits[::11, 8] = -np.inf
    logits[::13, :] = 0.5                         # all equal
    for k in (1, 2, 6, E):
        idx, _ = oracle.topk_softmax(logits, k)
        for t in range(T):
            def key(e):
                v = float(logits[t, e])
                return (1, 0.0, e) if math.isnan(v) else (0, -v, e)
            ref = sorted(range(E), key=key)[:k]
            assert idx[t].tolist() == ref, (t, k)


def test_softmax_over_selected_closed_forms():
    # equal logits -> uniform weights; k = E -> weights sum to 1;
    # w_i / w_j = exp(l_i - l_j)
    lg = np.zeros((1, 8), np.float32)
    for k in (1, 2, 4, 8):
        _, w = oracle.topk_softmax(lg, k)
        assert np.all(w == np.float32(1.0 / k))
    _, w6 = oracle.topk_softmax(np.zeros((1, 8), np.float32), 6)
    assert np.all(w6 == np.float32(1.0 / 6.0))
    rng = np.random.default_rng(13)
    lg = (rng.standard_normal((50, 256)) * 1.3).astype(np.float32)
    idx, w = oracle.topk_softmax(lg, 256)
    assert np.allclose(w.astype(np.float64).sum(1), 1.0, rtol=0, atol=256 * 2 ** -24)
    idx, w = oracle.topk_softmax(lg, 6)
    for t in range(50):
        sel = lg[t, idx[t]].astype(np.float64)
        assert np.all(np.diff(sel) <= 0)
        ratio = w[t, 1:].astype(np.float64) / w[t, 0]
        assert np.allclose(ratio, np.exp(sel[1:] - sel[0]), rtol=4e-7, atol=0)
        # two experts: the logistic function
    _, w2 = oracle.topk_softmax(np.array([[2.0, -2.0]], np.float32), 2)
    assert w2[0, 0] == np.float32(1.0 / (1.0 + math.exp(-4.0)))
    assert w2[0, 1] == np.float32(math.exp(-4.0) / (1.0 + math.exp(-4.0)))


def test_bias_enters_selection_and_weights():
    # A bias that flips the ranking: logits without bias favour expert 0,
    # with bias expert 1 -- and the weights follow the biased logits.
    D = 32
    x = oracle.round_bf16(np.ones((1, D)))
    Wr = np.zeros((2, D), np.float32)
    Wr[0, :] = 2 ** -5                      # logit 1.0
    bias = np.array([0.0, 3.0], np.float32)  # expert 1: 0 + 3
    idx, w, lg = oracle.route(x, Wr, bias, 2)
    assert lg.tolist() == [[1.0, 3.0]]
    assert idx.tolist() == [[1, 0]]
    assert w[0, 0] == np.float32(1.0 / (1.0 + math.exp(-2.0)))


# ---------------------------------------------------------------------- FFN
def _tiny_layer_from_golden():
    g = G.load("tiny_ffn.txt")
    D, F = int(g["d_model"]), int(g["d_ff"])
    w = synth.Workload("golden", D, F, 2, 1, 2, 0, synth.Q41_4BIT, synth.Q41_4BIT, synth.Q2K)

    def q41(spec, rows, cols):
        s = G.kv(spec)
        n = rows * cols
        return oracle.q41_pack(np.full(n, int(s["code"]), np.uint8), np.full(n // 32, int(s["d"], 16), np.uint16),
                               np.full(n // 32, int(s["m"], 16), np.uint16))

    def q2k(spec, rows, cols):
        s = G.kv(spec)
        n = rows * cols
        return oracle.q2k_pack(np.full(n, int(s["code"]), np.uint8), np.full(n // 16, int(s["sc"]), np.uint8),
                               np.full(n // 16, int(s["mn"]), np.uint8), np.full(n // 256, int(s["d"], 16), np.uint16),
                               np.full(n // 256, int(s["dmin"], 16), np.uint16))

    gate = np.concatenate([q41(g["e0_gate"], F, D), q41(g["e1_gate"], F, D)])
    up = np.concatenate([q41(g["e0_up"], F, D), q41(g["e1_up"], F, D)])
    down = np.concatenate([q2k(g["e0_down"], D, F), q2k(g["e1_down"], D, F)])
    Wr = np.stack([np.full(D, float(g["router_row0"]), np.float32), np.full(D, float(g["router_row1"]), np.float32)])
    x = np.stack([np.full(D, int(g["x_token0_bf16"], 16), np.uint16), np.full(D, int(g["x_token1_bf16"], 16), np.uint16)])
    return g, w, gate, up, down, Wr, x


def test_hand_computed_tiny_layer():
    g, w, gate, up, down, Wr, x = _tiny_layer_from_golden()
    D, F = w.d_model, w.d_ff
    idx, wt, lg = oracle.route(x, Wr, None, 1)
    assert lg[0].tolist() == G.floats(g["logits_token0"])
    assert lg[1].tolist() == G.floats(g["logits_token1"])
    assert idx[:, 0].tolist() == G.ints(g["idx"])
    assert wt.tolist() == [[1.0], [1.0]]
    for t in range(2):
        y, h, gg, uu = oracle.expert_ffn(D, F, oracle.Q4_1, gate, oracle.Q4_1, up, oracle.Q2_K, down,
                                         int(idx[t, 0]), x[t])
        assert np.all(h == int(g[f"h_token{t}_bf16"], 16))
    out = oracle.moe_ffn(D, F, 2, oracle.Q4_1, gate, oracle.Q4_1, up, oracle.Q2_K, down, x, idx, wt)
    assert np.all(out[0] == float(g["out_token0"]))
    assert np.all(out[1] == float(g["out_token1"]))


def test_constant_q4_1_rows_give_closed_form_projection():
    # every code c, constant d and m: each gate row is (d*c + m) * sum(x)
    D, F = 512, 256
    rng = np.random.default_rng(21)
    x = oracle.round_bf16(rng.standard_normal(D))
    for c, dh, mh in ((7, 0x2118, 0xA0C0), (15, 0x1C00, 0x0000), (0, 0x2400, 0x3555)):
        n = F * D
        gate = oracle.q41_pack(np.full(n, c, np.uint8), np.full(n // 32, dh, np.uint16), np.full(n // 32, mh, np.uint16))
        down = oracle.q2k_pack(np.zeros(n, np.uint8), np.zeros(n // 16, np.uint8), np.zeros(n // 16, np.uint8),
                               np.zeros(n // 256, np.uint16), np.zeros(n // 256, np.uint16))
        y, h, g, u = oracle.expert_ffn(D, F, oracle.Q4_1, gate, oracle.Q4_1, gate, oracle.Q2_K, down, 0, x)
        entry = Fraction(oracle.f16(dh)) * c + Fraction(oracle.f16(mh))
        sx = sum(Fraction(float(v)) for v in _bf16_vals(x))
        exact = float(entry * sx)
        assert np.allclose(g, exact, rtol=1e-13, atol=0) and np.allclose(u, exact, rtol=1e-13, atol=0)
        # h = bf16(silu(g) * u) of that closed form
        hv = exact / (1.0 + math.exp(-exact)) * exact
        assert np.all(h == oracle.round_bf16([hv])[0])
        # Q2_K down with codes 0 and mins 0 is the zero matrix
        assert np.all(y == 0.0)
    # a Q2_K down matrix needs d_ff to be a whole number of 256-value blocks
    with pytest.raises(oracle.OracleError):
        oracle.expert_ffn(D, 64, oracle.Q4_1, gate, oracle.Q4_1, gate, oracle.Q2_K, down, 0, x)


@pytest.fixture(scope="module")
def small_layer():
    # 4 experts of a reduced layer: d_model 512, d_ff 256 (several Q2_K/Q4_1 blocks per row)
    w = synth.WORKLOADS[0].replace(d_model=512, d_ff=256, n_expert=4, k=2, T=6, seed=5)
    return build_layer(w)


def test_identical_experts_with_k_equal_E_reduce_to_one_expert(small_layer):
    L = small_layer
    w = L.w
    E = w.n_expert
    gate = np.tile(L.gate[: L.gate.size // E], E)
    up = np.tile(L.up[: L.up.size // E], E)
    down = np.tile(L.down[: L.down.size // E], E)
    x = synth.activations(w, T=3)
    idx, wt, _ = oracle.route(x, L.Wr, None, E)
    out = oracle.moe_ffn(w.d_model, w.d_ff, E, L.qg, gate, L.qu, up, L.qd, down, x, idx, wt)
    for t in range(3):
        y, *_ = oracle.expert_ffn(w.d_model, w.d_ff, L.qg, gate, L.qu, up, L.qd, down, 0, x[t])
        # out = sum_i w_i * y with sum_i w_i = 1 up to fp32 rounding of each w_i
        assert np.allclose(out[t], y, rtol=0, atol=E * 2 ** -24 * np.abs(y).max() + 1e-30)


def test_expert_permutation_invariance(small_layer):
    L = small_layer
    w = L.w
    E = w.n_expert
    perm = np.array([2, 0, 3, 1])
    x = synth.activations(w, T=6)
    out, idx, wt, _ = oracle_forward(L, x)
    per_g, per_u, per_d = L.gate.size // E, L.up.size // E, L.down.size // E

    def permute(buf, per):
        return np.concatenate([buf[p * per:(p + 1) * per] for p in perm])

    idx2, wt2, _ = oracle.route(x, L.Wr[perm], None, w.k)
    assert np.array_equal(perm[idx2], idx) and np.array_equal(wt2, wt)
    out2 = oracle.moe_ffn(w.d_model, w.d_ff, E, L.qg, permute(L.gate, per_g), L.qu, permute(L.up, per_u),
                          L.qd, permute(L.down, per_d), x, idx2, wt2)
    assert np.array_equal(out.view(np.uint32), out2.view(np.uint32))


def test_token_permutation_and_linearity_in_routing_weights(small_layer):
    L = small_layer
    w = L.w
    x = synth.activations(w, T=6)
    out, idx, wt, _ = oracle_forward(L, x)
    p = np.array([5, 3, 1, 0, 2, 4])
    out_p = oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down,
                           x[p], idx[p], wt[p])
    assert np.array_equal(out_p, out[p])
    # the combine is linear in the routing weights: doubling them doubles out
    # (exact: the accumulation is in double and doubling is exact)
    out2 = oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down,
                          x, idx, wt * 2)
    assert np.array_equal(out2, out * 2)


def test_rejects_out_of_range_expert_ids(small_layer):
    L = small_layer
    w = L.w
    x = synth.activations(w, T=1)
    with pytest.raises(oracle.OracleError):
        oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down,
                       x, np.array([[0, w.n_expert]], np.int32), np.ones((1, 2), np.float32))


# ----------------------------------------------------------- layer stack
def test_rmsnorm_layer_input_closed_forms():
    """bf16(x / sqrt(mean(x^2) + eps)): a constant row maps to +-1 (eps = 0);
    scaling a row by a power of two leaves it unchanged (eps = 0, exact);
    the result's mean square is 1 within bf16 rounding; eps damps tiny rows
    by exactly sqrt(ms / (ms + eps))."""
    import oracle
    D = 256
    x = np.full((2, D), 3.0, dtype=np.float32)
    x[1] = -0.125
    y = oracle.bf16_to_f32(oracle.rmsnorm_bf16(x, 0.0))
    assert (y[0] == 1.0).all() and (y[1] == -1.0).all()
    rng = np.random.default_rng(3)
    r = rng.standard_normal((5, D)).astype(np.float32)
    a = oracle.rmsnorm_bf16(r, 0.0)
    assert np.array_equal(a, oracle.rmsnorm_bf16(r * np.float32(64.0), 0.0))
    assert np.array_equal(a, oracle.rmsnorm_bf16(r * np.float32(2.0 ** -20), 0.0))
    ms = (oracle.bf16_to_f32(a).astype(np.float64) ** 2).mean(axis=1)
    assert np.abs(ms - 1.0).max() < 2 ** -7
    # constant row c with eps: value = c / sqrt(c^2 + eps), rounded to bf16
    c, eps = np.float32(0.001), 3e-6
    got = oracle.bf16_to_f32(oracle.rmsnorm_bf16(np.full((1, D), c, np.float32), eps))[0, 0]
    want = float(c) / np.sqrt(float(c) ** 2 + eps)
    assert abs(got - want) <= abs(want) * 2 ** -8
    assert got < 1.0
