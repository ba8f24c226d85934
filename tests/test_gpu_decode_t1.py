"""GPU parity of the single-token decode kernels (T = 1: Q2_K or Q4_K
gate/up with d_model a multiple of 1024 up to 4096, Q2_K or Q4_K down with
d_ff 1024 or 2048), against the CPU oracle, through both decode entry points.

Covers: every (d_model, d_ff) the kernels take, including layers where only
one of the two single-token kernels applies and the other side runs the
multi-token kernel; k = 1, 2, 6; a router bias; an expert id out of range
(the valid experts are still combined); run-to-run bit equality; the
profiling names of the launched kernels.  Bar as for every FFN test:
max |err| <= 2e-3 * max |ref|, routing bit-exact.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err, ulp_diff_f32
from tests.layers import build_layer, to_device
from tests.test_gpu_ffn import gpu_forward, gpu_moe_decode, oracle_out

pytestmark = pytest.mark.gpu
TOL = 2e-3

Q2 = synth.WORKLOADS[1]
Q4 = synth.WORKLOADS[5]
SHAPES = [
    # both single-token kernels
    Q2.replace(d_model=1024, d_ff=1024, n_expert=8, k=6, seed=401),
    Q2.replace(d_model=2048, d_ff=2048, n_expert=16, k=2, seed=402, bias_sigma=1.0),
    Q2.replace(d_model=4096, d_ff=1024, n_expert=4, k=1, seed=403),
    Q2.replace(d_model=3072, d_ff=2048, n_expert=6, k=3, seed=404),
    # all Q2_K with d_model = 2 d_ff: the merged gate/up + down grid
    Q2.replace(d_model=4096, d_ff=2048, n_expert=12, k=6, seed=408),
    Q2.replace(d_model=2048, d_ff=1024, n_expert=7, k=3, seed=409, bias_sigma=1.0),
    Q2.replace(d_model=2048, d_ff=1024, n_expert=3, k=1, seed=410),
    # gate/up single-token, down multi-token (d_ff not a multiple of 1024)
    Q2.replace(d_model=1024, d_ff=768, n_expert=5, k=2, seed=405),
    # gate/up multi-token (d_model not a multiple of 1024), down single-token
    Q2.replace(d_model=768, d_ff=1024, n_expert=5, k=2, seed=406),
    # Q4_1 gate/up (multi-token kernel), Q2_K down single-token
    synth.WORKLOADS[0].replace(d_model=1024, d_ff=2048, n_expert=6, k=2, T=1, seed=407),
    # Q4_K: both single-token kernels
    Q4.replace(d_model=1024, d_ff=1024, n_expert=8, k=6, seed=411),
    Q4.replace(d_model=4096, d_ff=2048, n_expert=6, k=2, seed=412, bias_sigma=1.0),
    Q4.replace(d_model=3072, d_ff=1024, n_expert=4, k=1, seed=413),
    # Q4_K gate/up with Q2_K down, and Q2_K gate/up with Q4_K down
    Q4.replace(d_model=2048, d_ff=1024, n_expert=5, k=3, seed=414, down=synth.Q2K),
    Q2.replace(d_model=1024, d_ff=2048, n_expert=5, k=2, seed=415, down=synth.Q4K),
]


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


@pytest.mark.parametrize("wi", range(len(SHAPES)))
def test_single_token_matches_oracle(M, wi):
    w = SHAPES[wi]
    L = build_layer(w)
    dev = to_device(L)
    for batch in (0, 1):
        x = synth.activations(w, T=1, batch=batch)
        ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
        ref = oracle_out(L, x, ridx, rw)
        out, idx, wt, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        assert st == M.DS4MOE_OK
        assert np.array_equal(idx, ridx)
        assert ulp_diff_f32(wt, rw).max() <= 2
        assert rel_err(out, ref) <= TOL
        out2, idx2, wt2, st2 = gpu_forward(M, dev, x, L.Wr, L.bias, w.k)
        assert st2 == M.DS4MOE_OK and np.array_equal(idx2, ridx)
        assert rel_err(out2, ref) <= TOL
        # the fused entry (merged grid where the layer allows it) and the
        # separate kernels do the same arithmetic in the same order
        if np.array_equal(wt.view(np.uint32), wt2.view(np.uint32)):
            assert np.array_equal(out.view(np.uint32), out2.view(np.uint32))
        # same inputs, same bits
        out3, _, _, _ = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        assert np.array_equal(out3.view(np.uint32), out.view(np.uint32))


MERGED = [4, 5, 6]


@pytest.mark.parametrize("wi", [0, 4, 5, 10])
def test_single_token_kernels_are_the_ones_launched(M, wi):
    w = SHAPES[wi]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w, T=1)
    M.ds4moe_profile_enable(True)
    try:
        gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        names = set(M.ds4moe_profile_read())
    finally:
        M.ds4moe_profile_enable(False)
    # the all-Q2_K layers with d_model = 2 d_ff run the merged grid
    if wi in MERGED:
        assert "ffn_t1" in names and not {"gate_up", "down"} & names
    else:
        assert {"gate_up", "down"} <= names
    assert not {"gate_up_simt", "down_simt"} & names


def test_single_token_out_of_range_expert(M):
    w = SHAPES[0].replace(k=3)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w, T=1)
    idx = np.array([[2, 99, 5]], np.int32)
    wt = np.array([[0.5, 0.3, 0.2]], np.float32)
    out, _, _, st = gpu_forward(M, dev, x, L.Wr, None, 3, False, idx, wt)
    assert st == M.DS4MOE_EDEVICE
    ref = oracle_out(L, x, np.array([[2, 5, 5]], np.int32), np.array([[0.5, 0.2, 0.0]], np.float32))
    assert rel_err(out, ref) <= TOL


def test_single_token_agrees_with_the_batched_kernels(M):
    """The same token alone (single-token kernels) and inside a batch of
    three (multi-token kernels) gives the same output within the bar."""
    w = SHAPES[1]
    L = build_layer(w)
    dev = to_device(L)
    x3 = synth.activations(w, T=3)
    o3, i3, w3, st3 = gpu_forward(M, dev, x3, L.Wr, L.bias, w.k)
    o1, i1, w1, st1 = gpu_forward(M, dev, x3[1:2], L.Wr, L.bias, w.k)
    assert st1 == st3 == M.DS4MOE_OK
    assert np.array_equal(i1, i3[1:2])
    assert rel_err(o1, o3[1:2]) <= TOL
