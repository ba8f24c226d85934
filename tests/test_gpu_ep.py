"""Expert parallelism on the GPU with the library's kernels: R ranks emulated
in one process (each rank's experts in their own device layer; the exchanges
move the buffers between the emulated ranks, so no kernel waits on another
rank), and ep_layer under a one-rank NCCL group; every rank's output against
the oracle layer on its tokens.  Also the two data-plane kernels
(ds4moe_gather_rows bit-exact, ds4moe_combine_pairs)."""
import os
import socket

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err
from tests.layers import build_layer

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _rank_layers(M, L, R):
    """DeviceLayers holding each rank's contiguous expert range."""
    import torch
    from bit_quantized_moe_q2_gb300.device import DeviceLayer
    from bit_quantized_moe_q2_gb300.ep import expert_ranges
    w = L.w
    qid = {synth.Q4_1: M.DS4MOE_Q4_1, synth.Q2_K: M.DS4MOE_Q2_K, synth.Q4_K: M.DS4MOE_Q4_K}
    out = []
    for lo, hi in expert_ranges(w.n_expert, R):
        parts = []
        for name in ("gate", "up", "down"):
            buf = getattr(L, name)
            per = buf.size // w.n_expert
            parts.append(buf[lo * per:hi * per])
        out.append(DeviceLayer.from_host(w.d_model, w.d_ff, hi - lo, qid[w.gate.qtype], qid[w.up.qtype],
                                         qid[w.down.qtype], *parts))
    return out


def _backends(M, L, R):
    import torch
    from bit_quantized_moe_q2_gb300.ep import DeviceBackend
    Wr = torch.from_numpy(L.Wr).cuda()
    bias = None if L.bias is None else torch.from_numpy(L.bias).cuda()
    return [DeviceBackend(layer, Wr, bias, L.w.k) for layer in _rank_layers(M, L, R)]


CASES = [
    # decode-sized batches per rank (the owners' FFN takes the decode kernels)
    (synth.WORKLOADS[1].replace(d_model=1024, d_ff=512, n_expert=8, k=2, T=5, seed=71), 2),
    (synth.WORKLOADS[0].replace(d_model=1024, d_ff=1024, n_expert=16, k=3, T=7, seed=72), 4),
    # prefill-sized batches (the owners' FFN takes the tensor-core prefill kernels), router bias
    (synth.WORKLOADS[3].replace(d_model=1024, d_ff=1024, n_expert=8, k=2, T=150, seed=73), 2),
]


@pytest.mark.parametrize("wi", range(len(CASES)))
def test_emulated_ranks_match_the_oracle_layer(M, wi):
    import torch
    from bit_quantized_moe_q2_gb300.ep import run_local_ranks
    w, R = CASES[wi]
    L = build_layer(w)
    xs_host = [synth.activations(w, batch=200 + r) for r in range(R)]
    xs = [torch.from_numpy(x.view(np.int16).copy()).cuda() for x in xs_host]
    res = run_local_ranks(xs, _backends(M, L, R), w.n_expert)
    moved = 0
    for r, (out, idx, wt) in enumerate(res):
        x = xs_host[r]
        ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
        assert np.array_equal(idx.cpu().numpy(), ridx)
        ref = oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, x, ridx, rw)
        assert rel_err(out.cpu().numpy(), ref) <= TOL
        moved += int((ridx // (w.n_expert // R) != r).sum())
    assert moved > 0


def test_ep_layer_under_a_one_rank_nccl_group(M):
    import torch
    import torch.distributed as dist
    from bit_quantized_moe_q2_gb300 import ep
    w = CASES[0][0]
    L = build_layer(w)
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        x = synth.activations(w, batch=300)
        xt = torch.from_numpy(x.view(np.int16).copy()).cuda()
        out, idx, _ = ep.ep_layer(xt, _backends(M, L, 1)[0], w.n_expert, ep.DistExchange())
    finally:
        dist.destroy_process_group()
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    ref = oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, x, ridx, rw)
    assert rel_err(out.cpu().numpy(), ref) <= TOL


def test_gather_rows_and_combine_pairs(M):
    import torch
    rng = np.random.default_rng(9)
    x = rng.integers(0, 1 << 16, size=(37, 264), dtype=np.uint16)
    rows = rng.integers(0, 37, size=53).astype(np.int32)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    dst = torch.empty((53, 264), dtype=torch.int16, device="cuda")
    M.ds4moe_gather_rows(xd, torch.from_numpy(rows).cuda(), dst)
    assert np.array_equal(dst.cpu().numpy().view(np.uint16), x[rows])
    T, k, D = 11, 3, 200
    y = rng.standard_normal((20, D)).astype(np.float32)
    pos = rng.integers(-1, 20, size=(T, k)).astype(np.int32)
    wt = rng.random((T, k)).astype(np.float32)
    out = torch.empty((T, D), dtype=torch.float32, device="cuda")
    M.ds4moe_combine_pairs(torch.from_numpy(y).cuda(), torch.from_numpy(pos).cuda(), torch.from_numpy(wt).cuda(), out)
    ref = np.zeros((T, D))
    for t in range(T):
        for i in range(k):
            if pos[t, i] >= 0:
                ref[t] += float(wt[t, i]) * y[pos[t, i]].astype(np.float64)
    assert np.abs(out.cpu().numpy() - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
