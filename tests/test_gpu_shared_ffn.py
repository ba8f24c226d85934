"""GPU parity of the shared expert (ds4moe_shared_ffn) against the oracle:
the GEMV path (up to 8 tokens) and the tcgen05 path (more tokens), with and
without accumulation, ragged token counts, a shape the tensor-core path does
not take, width zero, run-to-run bit equality, and the routed layer plus the
shared expert against the oracle's composition.  Bar as for every FFN test:
max |err| <= 2e-3 * max |ref|."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err
from tests.layers import build_layer, to_device
from tests.test_gpu_ffn import gpu_moe_decode

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _bf16_bits(a):
    """Seeded inputs as bf16 bit patterns (the top half of each fp32)."""
    return (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _inputs(D, Fs, T, seed, wscale=0.02):
    rng = np.random.default_rng(seed)
    w1 = _bf16_bits(rng.standard_normal((Fs, D)) * wscale)
    w3 = _bf16_bits(rng.standard_normal((Fs, D)) * wscale)
    w2 = _bf16_bits(rng.standard_normal((D, Fs)) * wscale)
    x = _bf16_bits(rng.standard_normal((T, D)))
    return w1, w3, w2, x


def _gpu(M, w1, w3, w2, x, base=None, spans=False):
    import torch
    T, D = x.shape
    Fs = w1.shape[0]
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    out = torch.from_numpy(base.copy()).cuda() if base is not None else torch.full((T, D), float("nan"), device="cuda")
    ws = torch.empty(M.ds4moe_shared_workspace_bytes(D, Fs, T), dtype=torch.uint8, device="cuda")
    M.ds4moe_workspace_init(ws)
    if spans:
        M.ds4moe_profile_span(1)
    try:
        M.ds4moe_shared_ffn(d(w1), d(w3), d(w2), d(x), out, ws, accumulate=base is not None)
        torch.cuda.synchronize()
        ran = M.ds4moe_profile_span(0) if spans else None
    finally:
        if spans:
            M.ds4moe_profile_span(0)
    st = M.ds4moe_stream_status(ws)
    return out.cpu().numpy(), st, ran


# (d_model, d_shared, tokens): GEMV path up to 8 tokens, or a shape without tensor-core tiles
SIMT = [(256, 64, 1), (1024, 512, 5), (4096, 2048, 8), (512, 200, 64), (640, 96, 13)]
# tensor-core path: d_model % 256 == 0, d_shared % 128 == 0, more than 8 tokens
TC = [(1024, 512, 9), (1024, 512, 65), (2048, 1024, 300), (4096, 2048, 130), (1536, 384, 256)]


@pytest.mark.parametrize("D,Fs,T", SIMT)
@pytest.mark.parametrize("acc", [False, True])
def test_gemv_path_matches_oracle(M, D, Fs, T, acc):
    w1, w3, w2, x = _inputs(D, Fs, T, seed=D + Fs + T)
    base = np.random.default_rng(7).standard_normal((T, D)).astype(np.float32) if acc else None
    got, st, ran = _gpu(M, w1, w3, w2, x, base, spans=True)
    assert st == M.DS4MOE_OK
    assert not ({"shared_gate_up_tc", "shared_down_tc"} & set(ran))
    ref = oracle.shared_ffn(w1, w3, w2, x, base)
    assert rel_err(got, ref) <= TOL


@pytest.mark.parametrize("D,Fs,T", TC)
@pytest.mark.parametrize("acc", [False, True])
def test_tensor_core_path_matches_oracle(M, D, Fs, T, acc):
    w1, w3, w2, x = _inputs(D, Fs, T, seed=3 * D + Fs + T)
    base = np.random.default_rng(8).standard_normal((T, D)).astype(np.float32) if acc else None
    got, st, ran = _gpu(M, w1, w3, w2, x, base, spans=True)
    assert st == M.DS4MOE_OK
    assert {"shared_gate_up_tc", "shared_down_tc"} <= set(ran)
    ref = oracle.shared_ffn(w1, w3, w2, x, base)
    assert rel_err(got, ref) <= TOL


def test_many_tokens_on_a_shape_without_tensor_core_tiles(M):
    D, Fs, T = 640, 200, 100  # d_model not a multiple of 256: the GEMV path for every token
    w1, w3, w2, x = _inputs(D, Fs, T, seed=11)
    got, st, ran = _gpu(M, w1, w3, w2, x, spans=True)
    assert st == M.DS4MOE_OK and not ({"shared_gate_up_tc", "shared_down_tc"} & set(ran))
    assert rel_err(got, oracle.shared_ffn(w1, w3, w2, x)) <= TOL


@pytest.mark.parametrize("T", [3, 200])
def test_runs_are_bit_identical(M, T):
    w1, w3, w2, x = _inputs(1024, 512, T, seed=12)
    a, _, _ = _gpu(M, w1, w3, w2, x)
    b, _, _ = _gpu(M, w1, w3, w2, x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_width_zero(M):
    import torch
    D, T = 256, 3
    z = np.zeros((0, D), np.uint16)
    x = _bf16_bits(np.ones((T, D)))
    base = np.arange(T * D, dtype=np.float32).reshape(T, D)
    got, st, _ = _gpu(M, z, z, np.zeros((D, 0), np.uint16), x, base)
    assert st == M.DS4MOE_OK and np.array_equal(got, base)
    got, st, _ = _gpu(M, z, z, np.zeros((D, 0), np.uint16), x)
    assert st == M.DS4MOE_OK and np.array_equal(got, np.zeros((T, D), np.float32))


@pytest.mark.parametrize("T", [1, 96])
def test_routed_layer_plus_shared_expert(M, T):
    """ds4moe_moe_decode (routed combine) then ds4moe_shared_ffn accumulating:
    the oracle's shared expert added to its routed layer."""
    import torch
    w = synth.WORKLOADS[1].replace(d_model=2048, d_ff=1024, n_expert=8, k=2, T=T, seed=950)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w, T=T)
    routed, idx, _, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
    assert st == M.DS4MOE_OK
    w1, w3, w2, _ = _inputs(2048, 512, T, seed=951)
    got, st, _ = _gpu(M, w1, w3, w2, x, base=routed)
    assert st == M.DS4MOE_OK
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx, ridx)
    ref_routed = oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, x, ridx, rw)
    ref = oracle.shared_ffn(w1, w3, w2, x, ref_routed)
    assert rel_err(got, ref) <= TOL
