"""GPU parity of the tensor-core prefill path (tcgen05 grouped GEMMs) against
the CPU oracle, through ds4moe_ffn_prefill.

Covers: the kernels really run (profiling names them) for eligible layers
(gate and up in one of Q4_1 / Q4_K / Q2_K, d_model a multiple of 1024) and
not for others; Q2_K, Q4_1 and Q4_K down; the exact gate/up tiles of every
gate/up format (Q2_K: a minima step per 8 main steps, 16-value sub-block
sums); token chunks that split an expert (more than 128 / 256 pairs on one
expert); experts with no tokens; a single token; ragged chunk tails (n not a
multiple of 16 or 32); run-to-run bit equality (static schedule, fixed
accumulation order).  Bar as for every FFN test: max |err| <= 2e-3 * max |ref|.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err
from tests.layers import build_layer, to_device
from tests.test_gpu_ffn import gpu_forward, oracle_out

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


TC_SHAPES = [
    # Q4_1 gate/up, Q2_K down (the prefill workload's formats)
    synth.WORKLOADS[3].replace(d_model=1024, d_ff=1024, n_expert=8, k=2, T=150, seed=301),
    # Q4_1 down, d_ff a multiple of 128 but not of 256
    synth.WORKLOADS[3].replace(d_model=1024, d_ff=384, n_expert=5, k=3, T=77, seed=302, down=synth.Q41_4BIT),
    # 3-bit codes re-encoded as Q4_1, router bias
    synth.WORKLOADS[2].replace(d_model=2048, d_ff=1024, n_expert=12, k=4, T=45, seed=303, bias_sigma=1.0),
    # all Q2_K (the decode workload's formats at prefill): two 512-value
    # minima groups per 1024 values, four per row here
    synth.WORKLOADS[1].replace(d_model=2048, d_ff=1024, n_expert=8, k=3, T=140, seed=304),
    # all Q4_K, d_ff a multiple of 256 but not of 1024
    synth.WORKLOADS[5].replace(d_model=1024, d_ff=768, n_expert=6, k=2, T=130, seed=305),
    # Q4_K gate/up, Q2_K down (the mixed recipe's Q4 layers next to 2-bit ones)
    synth.WORKLOADS[5].replace(d_model=2048, d_ff=1024, n_expert=7, k=2, T=90, seed=306, down=synth.Q2K),
    # Q2_K gate/up, Q4_1 down, one token per expert at most on some experts
    synth.WORKLOADS[1].replace(d_model=1024, d_ff=512, n_expert=16, k=2, T=9, seed=307, down=synth.Q41_4BIT),
]


def _profiled_names(M, fn):
    M.ds4moe_profile_enable(True)
    try:
        fn()
        return set(M.ds4moe_profile_read())
    finally:
        M.ds4moe_profile_enable(False)


def test_tensor_core_kernels_run_only_for_eligible_layers(M):
    w = TC_SHAPES[0].replace(T=20)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    names = _profiled_names(M, lambda: gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill=True))
    assert {"gate_up_tc", "down_tc"} <= names
    # gate and up in different formats: the prefill call takes the warp-MMA
    # kernels instead
    w2 = w.replace(gate=synth.Q2K)
    L2 = build_layer(w2)
    dev2 = to_device(L2)
    names2 = _profiled_names(M, lambda: gpu_forward(M, dev2, x, L2.Wr, L2.bias, w2.k, prefill=True))
    assert not ({"gate_up_tc", "down_tc"} & names2)
    # d_model not a multiple of 1024: likewise
    w3 = w.replace(d_model=512, d_ff=1024)
    L3 = build_layer(w3)
    dev3 = to_device(L3)
    x3 = synth.activations(w3)
    names3 = _profiled_names(M, lambda: gpu_forward(M, dev3, x3, L3.Wr, L3.bias, w3.k, prefill=True))
    assert not ({"gate_up_tc", "down_tc"} & names3)


@pytest.mark.parametrize("wi", [3, 4, 5, 6])
def test_every_gate_up_format_takes_the_tensor_cores(M, wi):
    w = TC_SHAPES[wi]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    names = _profiled_names(M, lambda: gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill=True))
    assert {"gate_up_tc", "down_tc"} <= names
    assert not ({"gate_up_simt", "down_simt"} & names)


@pytest.mark.parametrize("wi", range(len(TC_SHAPES)))
def test_prefill_tc_matches_oracle_all_tokens(M, wi):
    w = TC_SHAPES[wi]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    out, idx, wt, st = gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill=True)
    assert st == M.DS4MOE_OK
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx, ridx)
    assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL
    # same inputs, same bits
    out2, _, _, _ = gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill=True)
    assert np.array_equal(out2.view(np.uint32), out.view(np.uint32))


@pytest.mark.parametrize("T,k,wi", [(300, 1, 0), (301, 2, 0), (1, 6, 0), (260, 2, 3), (270, 2, 4)])
def test_prefill_tc_heavy_expert_and_single_token(M, T, k, wi):
    """Slot 0 of every token goes to expert 3: 300 pairs on one expert span
    three 128-pair gate/up chunks and two 256-pair down chunks; the other
    slots spread over the remaining experts, several of which stay empty."""
    w = TC_SHAPES[wi].replace(T=T, k=k, n_expert=8, seed=310 + k + wi)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    rng = np.random.default_rng(T * 10 + k)
    idx = np.empty((T, k), dtype=np.int32)
    idx[:, 0] = 3
    pool = [0, 1, 5] if k <= 4 else [e for e in range(8) if e != 3]
    for t in range(T):
        idx[t, 1:] = rng.choice(pool, size=k - 1, replace=False) if k > 1 else []
    wt = rng.random((T, k)).astype(np.float32)
    wt /= wt.sum(axis=1, keepdims=True)
    out, _, _, st = gpu_forward(M, dev, x, L.Wr, None, k, True, idx, wt)
    assert st == M.DS4MOE_OK
    assert rel_err(out, oracle_out(L, x, idx, wt)) <= TOL


@pytest.mark.parametrize("wi", [0, 3, 5])
def test_prefill_split_small_experts_stream(M, wi):
    """Experts with at most ds4moe_prefill_small_pairs() pairs take the
    weight-streaming kernels, the rest the grouped GEMMs, in one call: 150
    pairs on expert 3, 17 on expert 5 (just above), 16, 9, 5, 2 and 1 on
    others (at or below), none on expert 7."""
    w = TC_SHAPES[wi].replace(T=200, k=1, n_expert=8, seed=330 + wi)
    L = build_layer(w)
    dev = to_device(L)
    n_small = M.ds4moe_prefill_small_pairs(dev.abi)
    assert n_small == 16
    x = synth.activations(w)
    sizes = [(3, 150), (5, 17), (4, 16), (2, 9), (1, 5), (0, 2), (6, 1)]
    idx = np.concatenate([np.full(n, e, np.int32) for e, n in sizes]).reshape(200, 1)
    idx = idx[np.random.default_rng(wi).permutation(200)]
    wt = np.ones((200, 1), np.float32)
    names = _profiled_names(M, lambda: gpu_forward(M, dev, x, L.Wr, None, 1, True, idx, wt))
    assert {"gate_up_tc", "down_tc", "gate_up", "down"} <= names
    out, _, _, st = gpu_forward(M, dev, x, L.Wr, None, 1, True, idx, wt)
    assert st == M.DS4MOE_OK
    assert rel_err(out, oracle_out(L, x, idx, wt)) <= TOL


def test_prefill_tc_out_of_range_expert_is_flagged_and_skipped(M):
    w = TC_SHAPES[0].replace(T=40, k=2, seed=320)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    idx = ridx.copy()
    idx[7, 1] = 99  # out of range: reported, contributes nothing
    out, _, _, st = gpu_forward(M, dev, x, L.Wr, None, w.k, True, idx, rw)
    assert st == M.DS4MOE_EDEVICE
    keep = np.ones(w.T, dtype=bool)
    keep[7] = False
    ref = oracle_out(L, x[keep], ridx[keep], rw[keep])
    assert rel_err(out[keep], ref) <= TOL
