"""GPU parity: the routed expert FFN (decode and prefill paths, through the
C ABI) against the CPU oracle.  Bar: max |err| <= 2e-3 * max |ref| (fp32
accumulation over bf16-rounded activations vs a double-precision oracle);
routing indices bit-exact."""
import numpy as np
import pytest

import oracle
import synth
from tests import golden_io as G
from tests.gpu_util import rel_err, torch_bf16_bits
from tests.layers import build_layer, cached_layer, to_device

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def gpu_forward(M, dev, x, Wr, bias, k, prefill=False, idx_override=None, w_override=None):
    """Route + FFN on the GPU.  Returns (out, idx, w, status)."""
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    T = x.shape[0]
    xd = torch_bf16_bits(x)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = torch.full((T, dev.d_model), float("nan"), dtype=torch.float32, device="cuda")
    ws = workspace(dev, T, k, prefill)
    if idx_override is None:
        M.ds4moe_route_topk(xd, torch.from_numpy(Wr).cuda(), None if bias is None else torch.from_numpy(bias).cuda(),
                            k, idx, w, None, ws)
    else:
        idx.copy_(torch.from_numpy(idx_override))
        w.copy_(torch.from_numpy(w_override))
    fn = M.ds4moe_ffn_prefill if prefill else M.ds4moe_ffn_decode
    fn(dev.abi, xd, idx, w, out, ws)
    st = M.ds4moe_stream_status(ws)
    return out.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), st


def gpu_moe_decode(M, dev, x, Wr, bias, k):
    """The fused decode entry point: (out, idx, w, status)."""
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    T = x.shape[0]
    idx = torch.full((T, k), -5, dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = torch.full((T, dev.d_model), float("nan"), dtype=torch.float32, device="cuda")
    ws = workspace(dev, T, k)
    M.ds4moe_moe_decode(dev.abi, torch_bf16_bits(x), torch.from_numpy(Wr).cuda(),
                        None if bias is None else torch.from_numpy(bias).cuda(), k, out, idx, w, ws)
    st = M.ds4moe_stream_status(ws)
    return out.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), st


def oracle_out(L, x, idx, w):
    ww = L.w
    return oracle.moe_ffn(ww.d_model, ww.d_ff, ww.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, x, idx, w)


# ------------------------------------------------------------ hand-computed
@pytest.mark.parametrize("prefill", [False, True])
def test_hand_computed_tiny_layer(M, prefill):
    from tests.test_oracle_route_ffn import _tiny_layer_from_golden
    from bit_quantized_moe_q2_gb300.device import DeviceLayer
    g, w, gate, up, down, Wr, x = _tiny_layer_from_golden()
    dev = DeviceLayer.from_host(w.d_model, w.d_ff, 2, M.DS4MOE_Q4_1, M.DS4MOE_Q4_1, M.DS4MOE_Q2_K, gate, up, down)
    out, idx, wt, st = gpu_forward(M, dev, x, Wr, None, 1, prefill)
    assert st == M.DS4MOE_OK
    assert idx[:, 0].tolist() == G.ints(g["idx"])
    assert np.all(out[0] == float(g["out_token0"]))
    assert np.all(out[1] == float(g["out_token1"]))


# --------------------------------------------------------- reduced layers
REDUCED = [
    synth.WORKLOADS[0].replace(d_model=512, d_ff=256, n_expert=8, k=2, T=13, seed=101),
    synth.WORKLOADS[1].replace(d_model=768, d_ff=512, n_expert=16, k=6, T=21, seed=102),
    synth.WORKLOADS[2].replace(d_model=1024, d_ff=256, n_expert=5, k=3, T=40, seed=103),
    synth.WORKLOADS[3].replace(d_model=512, d_ff=768, n_expert=12, k=4, T=97, seed=104),
    # shapes whose rows split into 16-byte bulk copies (tensor-core decode path)
    synth.WORKLOADS[1].replace(d_model=1024, d_ff=1024, n_expert=12, k=4, T=37, seed=105),
    synth.WORKLOADS[2].replace(d_model=2048, d_ff=1024, n_expert=10, k=3, T=50, seed=106),
    synth.WORKLOADS[0].replace(d_model=2048, d_ff=1024, n_expert=6, k=2, T=19, seed=107,
                               gate=synth.Q2K, up=synth.Q41_4BIT),
    synth.WORKLOADS[3].replace(d_model=4096, d_ff=2048, n_expert=9, k=6, T=11, seed=108),
]


@pytest.mark.parametrize("prefill", [False, True])
@pytest.mark.parametrize("wi", range(len(REDUCED)))
def test_reduced_layers_all_tokens(M, wi, prefill):
    w = REDUCED[wi]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    out, idx, wt, st = gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill)
    assert st == M.DS4MOE_OK
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx, ridx)
    ref = oracle_out(L, x, ridx, rw)
    assert rel_err(out, ref) <= TOL


@pytest.mark.parametrize("wi", range(len(REDUCED)))
def test_fused_decode_entry_point(M, wi):
    w = REDUCED[wi]
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    out, idx, wt, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
    assert st == M.DS4MOE_OK
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx, ridx)
    assert np.abs(wt.view(np.int32).astype(np.int64) - rw.view(np.int32)).max() <= 2
    assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL
    # and twice in a row on the same workspace-free call pattern gives the same bits
    out2, idx2, _, _ = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
    assert np.array_equal(out2.view(np.uint32), out.view(np.uint32)) and np.array_equal(idx2, idx)


@pytest.mark.parametrize("wi", [0, 4])
def test_one_expert_takes_every_token_and_k_1(M, wi):
    # n_e = T for one expert (many token groups); k = 1
    w = REDUCED[wi].replace(T=45, k=1)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    idx = np.full((w.T, 1), 3, np.int32)
    wt = np.ones((w.T, 1), np.float32)
    for prefill in (False, True):
        out, _, _, st = gpu_forward(M, dev, x, L.Wr, None, 1, prefill, idx, wt)
        assert st == M.DS4MOE_OK
        assert rel_err(out, oracle_out(L, x, idx, wt)) <= TOL


def test_out_of_range_expert_ids_are_flagged_and_skipped(M):
    w = REDUCED[0].replace(T=6, k=2)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    idx = np.array([[0, 1], [2, 99], [3, -1], [4, 5], [6, 7], [1, 0]], np.int32)
    wt = np.full((6, 2), 0.5, np.float32)
    out, _, _, st = gpu_forward(M, dev, x, L.Wr, None, 2, False, idx, wt)
    assert st == M.DS4MOE_EDEVICE
    ok = [0, 3, 4, 5]
    assert rel_err(out[ok], oracle_out(L, x[ok], idx[ok], wt[ok])) <= TOL
    # the valid half of a partly invalid token is still combined
    ref1 = oracle_out(L, x[1:2], np.array([[2, 2]], np.int32), np.array([[0.5, 0.0]], np.float32))
    assert rel_err(out[1:2], ref1) <= TOL


def test_zero_tokens_is_a_noop(M):
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    w = REDUCED[0]
    dev = to_device(build_layer(w, experts=[]))
    ws = workspace(dev, 1, 2)
    for fn in (M.ds4moe_ffn_decode, M.ds4moe_ffn_prefill):
        fn(dev.abi, torch.empty((0, w.d_model), dtype=torch.int16, device="cuda"),
           torch.empty((0, 2), dtype=torch.int32, device="cuda"),
           torch.empty((0, 2), dtype=torch.float32, device="cuda"),
           torch.empty((0, w.d_model), dtype=torch.float32, device="cuda"), ws)
    assert M.ds4moe_stream_status(ws) == M.DS4MOE_OK


# ------------------------------------------------------ full workload sizes
def _sample_tokens(idx, n_expert, n):
    """Tokens for the oracle: the first few plus every token of the two
    lightest used experts."""
    counts = np.bincount(idx.ravel(), minlength=n_expert)
    used = np.nonzero(counts)[0]
    light = used[np.argsort(counts[used], kind="stable")[:2]]
    pick = set(range(min(n, idx.shape[0])))
    for e in light:
        pick |= set(np.nonzero((idx == e).any(1))[0][:4].tolist())
    return np.array(sorted(pick))


def test_full_workload_fused_decode_t1(M):
    w = synth.WORKLOADS[1]
    L, dev = cached_layer(w)
    for batch in (0, 1, 2):
        x = synth.activations(w, batch=batch)
        out, idx, wt, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        assert st == M.DS4MOE_OK
        ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
        assert np.array_equal(idx, ridx)
        assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL


@pytest.mark.parametrize("wid,prefill", [(0, False), (1, False), (2, False), (3, True)])
def test_full_workloads(M, wid, prefill):
    w = synth.WORKLOADS[wid]
    L, dev = cached_layer(w)
    x = synth.activations(w)
    out, idx, wt, st = gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill)
    assert st == M.DS4MOE_OK
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx, ridx)
    sel = np.arange(w.T) if w.T <= 8 else _sample_tokens(ridx, w.n_expert, 6)
    ref = oracle_out(L, x[sel], ridx[sel], rw[sel])
    assert rel_err(out[sel], ref) <= TOL
    assert np.isfinite(out).all()
