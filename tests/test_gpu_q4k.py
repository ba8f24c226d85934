"""GPU parity of the Q4_K expert path (dequant and the FFN entry points;
Q4_K layers run the single-token, persistent multi-token and, at prefill
with d_model a multiple of 1024, the tcgen05 kernels) against the oracle: dequant bit for bit
(incl. arbitrary bytes with inf / NaN / subnormal scales), the layer output
within 2e-3 * max |ref| with routing bit-exact, for all-Q4_K layers and
Q4_K mixed with Q2_K / Q4_1 matrices."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err
from tests.layers import build_layer, expert_matrix, to_device
from tests.test_gpu_ffn import gpu_forward, gpu_moe_decode, oracle_out

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _gpu_dequant(M, blocks, n):
    import torch
    b = torch.from_numpy(np.ascontiguousarray(blocks)).cuda()
    out = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    M.ds4moe_dequant(M.DS4MOE_Q4_K, b, n, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _same_bits(a, b):
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


@pytest.mark.parametrize("nb", [1, 9, 4097])
def test_dequant_q4k_bit_exact(M, nb):
    rng = np.random.default_rng(nb)
    blk = oracle.q4k_pack(rng.integers(0, 16, nb * 256).astype(np.uint8), rng.integers(0, 64, nb * 8).astype(np.uint8),
                          rng.integers(0, 64, nb * 8).astype(np.uint8), rng.integers(0, 0x7C00, nb).astype(np.uint16),
                          rng.integers(0, 0x7C00, nb).astype(np.uint16))
    assert _same_bits(_gpu_dequant(M, blk, nb * 256), oracle.dequant(oracle.Q4_K, blk, nb * 256))


def test_dequant_q4k_arbitrary_bytes(M):
    nb = 3000
    blk = np.random.default_rng(5).integers(0, 256, nb * 144, dtype=np.uint8)
    assert _same_bits(_gpu_dequant(M, blk, nb * 256), oracle.dequant(oracle.Q4_K, blk, nb * 256))


def test_dequant_q4k_full_expert_matrix(M):
    w = synth.WORKLOADS[5]
    blk = expert_matrix(w, 0, synth.T_DOWN, 17)
    n = w.d_model * w.d_ff
    assert _same_bits(_gpu_dequant(M, blk, n), oracle.dequant(oracle.Q4_K, blk, n))


Q4 = synth.WORKLOADS[5]
SHAPES = [
    Q4.replace(d_model=1024, d_ff=512, n_expert=8, k=6, T=1, seed=601),
    Q4.replace(d_model=512, d_ff=1024, n_expert=12, k=2, T=19, seed=602, bias_sigma=1.0),
    Q4.replace(d_model=768, d_ff=256, n_expert=5, k=3, T=33, seed=603, down=synth.Q2K),
    Q4.replace(d_model=1024, d_ff=768, n_expert=6, k=2, T=7, seed=604, gate=synth.Q41_4BIT, up=synth.Q41_4BIT),
    # the persistent multi-token kernels: all Q4_K at the Flash shape, and
    # Q4_K gate/up with Q2_K down (the mixed recipe's neighbour layers)
    Q4.replace(d_model=4096, d_ff=2048, n_expert=6, k=3, T=21, seed=605),
    Q4.replace(d_model=2048, d_ff=1024, n_expert=9, k=2, T=40, seed=606, down=synth.Q2K),
    synth.WORKLOADS[1].replace(d_model=2048, d_ff=1024, n_expert=9, k=2, T=12, seed=607, down=synth.Q4K),
]


@pytest.mark.parametrize("wi", range(len(SHAPES)))
@pytest.mark.parametrize("prefill", [False, True])
def test_q4k_layers_match_oracle(M, wi, prefill):
    w = SHAPES[wi]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    out, idx, wt, st = gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill)
    assert st == M.DS4MOE_OK
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx, ridx)
    assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL


def test_q4k_fused_decode_entry_point(M):
    w = SHAPES[0]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    out, idx, wt, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
    assert st == M.DS4MOE_OK
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx, ridx)
    assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL


@pytest.mark.parametrize("wi", [1, 4, 5, 6])
def test_q4k_multi_token_layers_take_the_tensor_core_kernels(M, wi):
    """More than one token on layers with Q4_K gate/up or down (every shape
    here fits the persistent kernels): no SIMT kernel runs."""
    w = SHAPES[wi]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    M.ds4moe_profile_enable(True)
    try:
        gpu_forward(M, dev, x, L.Wr, L.bias, w.k)
        names = set(M.ds4moe_profile_read())
    finally:
        M.ds4moe_profile_enable(False)
    assert {"gate_up", "down"} <= names
    assert not ({"gate_up_simt", "down_simt"} & names)
