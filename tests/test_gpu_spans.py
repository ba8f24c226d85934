"""Device-side kernel spans (ds4moe_profile_span): each instrumented kernel
records one span per launch while recording is on, nothing while it is off,
and records inside a replayed CUDA graph, where events cannot bracket a
kernel.  The spans are a timing aid; the outputs are checked elsewhere."""
import pytest

import synth
from tests.layers import build_layer, to_device
from tests.test_gpu_ffn import gpu_forward, gpu_moe_decode

pytestmark = pytest.mark.gpu

Q2 = synth.WORKLOADS[1]


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _spans(M, fn, reps):
    M.ds4moe_profile_span(1)
    try:
        for _ in range(reps):
            fn()
        return M.ds4moe_profile_span(0)
    finally:
        M.ds4moe_profile_span(0)


def _check(spans, names, reps):
    assert names <= set(spans), (names, spans)
    for name in names:
        ns, n = spans[name]
        assert n == reps, (name, n)
        assert 1e2 < ns / n < 1e8, (name, ns / n)  # 0.1 us .. 100 ms per launch


def test_single_token_merged_grid_and_router(M):
    w = Q2.replace(d_model=2048, d_ff=1024, n_expert=8, k=3, seed=901)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w, T=1)
    spans = _spans(M, lambda: gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k), 3)
    _check(spans, {"route", "ffn_t1"}, 3)


def test_multi_token_decode_kernels(M):
    w = Q2.replace(d_model=1024, d_ff=1024, n_expert=8, k=2, T=4, seed=902)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w, T=4)
    spans = _spans(M, lambda: gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k), 2)
    _check(spans, {"route", "gate_up_mma", "down_mma"}, 2)


def test_prefill_tensor_core_kernels(M):
    w = synth.WORKLOADS[3].replace(d_model=1024, d_ff=1024, n_expert=8, k=2, T=20, seed=903)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w)
    spans = _spans(M, lambda: gpu_forward(M, dev, x, L.Wr, L.bias, w.k, prefill=True), 2)
    _check(spans, {"gate_up_tc", "down_tc"}, 2)


def test_off_records_nothing_and_graph_replays_record(M):
    import numpy as np
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    w = Q2.replace(d_model=2048, d_ff=1024, n_expert=8, k=3, seed=904)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w, T=1)
    M.ds4moe_profile_span(0)
    gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
    assert M.ds4moe_profile_span(-1) == {}
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()
    Wr = torch.from_numpy(L.Wr).cuda()
    idx = torch.empty((1, w.k), dtype=torch.int32, device="cuda")
    wt = torch.empty((1, w.k), dtype=torch.float32, device="cuda")
    out = torch.empty((1, w.d_model), dtype=torch.float32, device="cuda")
    ws = workspace(dev, 1, w.k)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        M.ds4moe_moe_decode(dev.abi, xd, Wr, None, w.k, out, idx, wt, ws, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        M.ds4moe_moe_decode(dev.abi, xd, Wr, None, w.k, out, idx, wt, ws, s)
    spans = _spans(M, lambda: (g.replay(), torch.cuda.synchronize()), 4)
    _check(spans, {"route", "ffn_t1"}, 4)


def test_single_token_separate_kernels(M):
    # Q4_K experts at T = 1: the separate single-token gate/up and down kernels
    w = synth.WORKLOADS[5].replace(d_model=1024, d_ff=1024, n_expert=8, k=2, seed=905)
    L = build_layer(w)
    dev = to_device(L)
    x = synth.activations(w, T=1)
    spans = _spans(M, lambda: gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k), 2)
    _check(spans, {"route", "gate_up_t1", "down_t1"}, 2)
