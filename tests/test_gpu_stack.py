"""GPU parity of the decode stack: ds4moe_residual_norm and
ds4moe_stack_decode over several full-size layers (d_model 4096, d_ff 2048,
Q2_K experts, each layer with its own router and experts), T = 1 and 16.

Layer by layer, the oracle is fed the GPU's own bf16 input of that layer
(so that a routing flip at a near-tie cannot compound across layers): the
routing must match bit for bit and the layer output within 2e-3 * max |ref|.
The residual add must match exactly (one fp32 rounding); the normalised
bf16 input may differ from the fp64 oracle by one bf16 ulp on a few values
(fp32 sum of squares).  The one-call stack must reproduce the layer-by-layer
calls bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err
from tests.layers import build_layer, to_device

pytestmark = pytest.mark.gpu
TOL = 2e-3
N_LAYERS = 5


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


@pytest.fixture(scope="module")
def stack():
    w = synth.WORKLOADS[4].replace(n_expert=16, n_layers=N_LAYERS)
    Ls = [build_layer(w, layer=l) for l in range(N_LAYERS)]
    return w, Ls, [to_device(L) for L in Ls]


def _check_norm(xb, x_res):
    got = xb.cpu().numpy().view(np.uint16)
    ref = oracle.rmsnorm_bf16(x_res.cpu().numpy(), 1e-6)
    d = np.abs(got.astype(np.int32) - ref.astype(np.int32))  # same-sign bf16 patterns: ulp distance
    assert d.max() <= 1 and (d > 0).mean() <= 1e-3


@pytest.mark.parametrize("T", [1, 16])
def test_stack_layer_by_layer_matches_oracle(M, stack, T):
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    w, Ls, devs = stack
    D, k = w.d_model, w.k
    x0 = synth.activations(w, T=T, batch=T)
    x_res = torch.from_numpy(oracle.bf16_to_f32(x0).copy()).cuda()
    xb = torch.empty((T, D), dtype=torch.int16, device="cuda")
    out = torch.empty((T, D), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = workspace(devs[0], T, k)
    M.ds4moe_residual_norm(x_res, None, xb)
    _check_norm(xb, x_res)
    trace = {"x_res": [x_res.clone()], "idx": [], "w": []}
    for l, (L, dev) in enumerate(zip(Ls, devs)):
        xin = xb.cpu().numpy().view(np.uint16).copy()
        bias = None if L.bias is None else torch.from_numpy(L.bias).cuda()
        M.ds4moe_moe_decode(dev.abi, xb, torch.from_numpy(L.Wr).cuda(), bias, k, out, idx, wt, ws)
        st = M.ds4moe_stream_status(ws)
        assert st == M.DS4MOE_OK, f"layer {l}: status {st}, max |x| {np.abs(oracle.bf16_to_f32(xin)).max()}"
        ridx, rw, _ = oracle.route(xin, L.Wr, L.bias, k)
        assert np.array_equal(idx.cpu().numpy(), ridx), f"layer {l}"
        ref = oracle.moe_ffn(D, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, xin, ridx, rw)
        o = out.cpu().numpy()
        assert rel_err(o, ref) <= TOL, f"layer {l}"
        prev = x_res.cpu().numpy()
        M.ds4moe_residual_norm(x_res, out, xb)
        torch.cuda.synchronize()
        nxt = x_res.cpu().numpy()
        assert np.array_equal(nxt, (prev + o).astype(np.float32))           # one fp32 rounding
        _check_norm(xb, x_res)
        trace["x_res"].append(x_res.clone())
        trace["idx"].append(idx.clone())
        trace["w"].append(wt.clone())

    # the one-call stack gives the same bits
    xs = torch.from_numpy(oracle.bf16_to_f32(x0).copy()).cuda()
    ldk = M.stack_ldk(T, k)
    idx_all = torch.empty((N_LAYERS, ldk), dtype=torch.int32, device="cuda")
    w_all = torch.empty((N_LAYERS, ldk), dtype=torch.float32, device="cuda")
    Wr = [torch.from_numpy(L.Wr).cuda() for L in Ls]
    M.ds4moe_stack_decode([d.abi for d in devs], Wr, None, k, xs, xb, out, idx_all, w_all, ws)
    assert M.ds4moe_stream_status(ws) == M.DS4MOE_OK
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), trace["x_res"][-1].cpu().numpy().view(np.uint32))
    for l in range(N_LAYERS):
        assert np.array_equal(idx_all[l, :T * k].cpu().numpy().reshape(T, k), trace["idx"][l].cpu().numpy())
        assert np.array_equal(w_all[l, :T * k].cpu().numpy().reshape(T, k).view(np.uint32),
                              trace["w"][l].cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("n_layers", [1, 2, 5])
def test_tile_order_stack_forms_inputs_in_the_router(M, stack, n_layers):
    """One token over tile-order layers: every layer after the first forms
    its input (residual add + RMS norm of the previous output) inside its
    router grid, the residual alternating between the caller's buffer and a
    workspace buffer.  The results must be the bits of the layer-by-layer
    calls (ds4moe_moe_decode then ds4moe_residual_norm), for an odd and an
    even number of layers."""
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    w, Ls, devs = stack
    r16 = [d.repacked_r16() for d in devs[:n_layers]]
    T, D, k = 1, w.d_model, w.k
    x0 = synth.activations(w, T=T, batch=7)
    Wr = [torch.from_numpy(L.Wr).cuda() for L in Ls[:n_layers]]
    ws = workspace(r16[0], T, k)
    # layer by layer
    x_res = torch.from_numpy(oracle.bf16_to_f32(x0).copy()).cuda()
    xb = torch.empty((T, D), dtype=torch.int16, device="cuda")
    out = torch.empty((T, D), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    M.ds4moe_residual_norm(x_res, None, xb)
    ref_idx, ref_w = [], []
    for l in range(n_layers):
        M.ds4moe_moe_decode(r16[l].abi, xb, Wr[l], None, k, out, idx, wt, ws)
        M.ds4moe_residual_norm(x_res, out, xb)
        ref_idx.append(idx.clone())
        ref_w.append(wt.clone())
    assert M.ds4moe_stream_status(ws) == M.DS4MOE_OK
    ref_res, ref_xb = x_res.clone(), xb.clone()
    # one call
    xs = torch.from_numpy(oracle.bf16_to_f32(x0).copy()).cuda()
    xb2 = torch.empty_like(xb)
    ldk = M.stack_ldk(T, k)
    idx_all = torch.empty((n_layers, ldk), dtype=torch.int32, device="cuda")
    w_all = torch.empty((n_layers, ldk), dtype=torch.float32, device="cuda")
    M.ds4moe_profile_enable(True)
    try:
        M.ds4moe_stack_decode([d.abi for d in r16], Wr, None, k, xs, xb2, out, idx_all, w_all, ws)
        names = M.ds4moe_profile_read()
    finally:
        M.ds4moe_profile_enable(False)
    assert M.ds4moe_stream_status(ws) == M.DS4MOE_OK
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), ref_res.cpu().numpy().view(np.uint32))
    assert np.array_equal(xb2.cpu().numpy(), ref_xb.cpu().numpy())
    for l in range(n_layers):
        assert np.array_equal(idx_all[l, :k].cpu().numpy(), ref_idx[l].cpu().numpy().ravel()), l
        assert np.array_equal(w_all[l, :k].cpu().numpy().view(np.uint32), ref_w[l].cpu().numpy().ravel().view(np.uint32)), l
    # one residual grid for the whole stack besides the input's (the layers' are in the routers)
    assert names["residual_norm"][1] == 2


def test_stack_rejects_bad_arguments_before_launching(M, stack):
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    w, Ls, devs = stack
    T, D, k = 4, w.d_model, w.k
    x = torch.zeros((T, D), dtype=torch.float32, device="cuda")
    xb = torch.zeros((T, D), dtype=torch.int16, device="cuda")
    out = torch.zeros_like(x)
    idx = torch.zeros((N_LAYERS, M.stack_ldk(T, k)), dtype=torch.int32, device="cuda")
    wt = torch.zeros((N_LAYERS, M.stack_ldk(T, k)), dtype=torch.float32, device="cuda")
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    Wr = [torch.from_numpy(L.Wr).cuda() for L in Ls]
    with pytest.raises(M.Ds4moeError):
        M.ds4moe_stack_decode([d.abi for d in devs], Wr, None, k, x, xb, out, idx, wt, small)
    ws = workspace(devs[0], T, k)
    with pytest.raises(M.Ds4moeError):  # k > n_expert
        M.ds4moe_stack_decode([d.abi for d in devs], Wr, None, w.n_expert + 1, x, xb, out, idx, wt, ws)
    with pytest.raises(M.Ds4moeError):  # d_model not a multiple of 4
        M.ds4moe_residual_norm(x[:, :D - 2].contiguous(), None, xb)
    with pytest.raises(M.Ds4moeError):  # negative eps
        M.ds4moe_residual_norm(x, None, xb, eps=-1.0)
