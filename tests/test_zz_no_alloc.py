"""GPU test of ds4moe_ffn_decode_noalloc, the decode FFN entry point that
allocates nothing and takes no workspace.

It exists for callers that cannot allocate device memory themselves: an
application whose GPU memory is owned by a framework's pool (an allocation
behind its back breaks the pool's accounting), a per-token decode loop that
cannot pay for cudaMalloc's implicit synchronisation, or a fixed plug-in
interface with nowhere to pass a workspace.  Its scratch is a fixed array
inside the library, shared by every call on the device.

The test calls it through the C ABI and checks it against the workspace
entry point ds4moe_ffn_decode on two calls in a row (different tokens, so
the second call runs over the first call's leftover scratch), within the
same tolerance as the other FFN parity tests.  This file is collected last
so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err, torch_bf16_bits
from tests.layers import build_layer, to_device

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _route(M, torch, L, x, ws):
    w = L.w
    idx = torch.empty((x.shape[0], w.k), dtype=torch.int32, device="cuda")
    wt = torch.empty((x.shape[0], w.k), dtype=torch.float32, device="cuda")
    bias = None if L.bias is None else torch.from_numpy(L.bias).cuda()
    M.ds4moe_route_topk(torch_bf16_bits(x), torch.from_numpy(L.Wr).cuda(), bias, w.k, idx, wt, None, ws)
    return idx, wt


@pytest.mark.parametrize("w", [
    synth.WORKLOADS[1].replace(n_expert=12, T=3, seed=211),                              # Flash dims, Q2_K
    synth.WORKLOADS[0].replace(d_model=1024, d_ff=512, n_expert=8, k=2, T=9, seed=212),  # Q4_1 gate/up
])
def test_noalloc_matches_workspace_entry_point_twice(M, w):
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    L = build_layer(w)
    dev = to_device(L)
    lib = M.lib()
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):   # second call: different tokens over the first call's scratch
        x = synth.activations(w, batch=77 + call)
        ws = workspace(dev, w.T, w.k)
        idx, wt = _route(M, torch, L, x, ws)
        xd = torch_bf16_bits(x)
        ref = torch.full((w.T, w.d_model), float("nan"), dtype=torch.float32, device="cuda")
        M.ds4moe_ffn_decode(dev.abi, xd, idx, wt, ref, ws)
        got = torch.full_like(ref, float("nan"))
        layer = dev.abi
        st = lib.ds4moe_ffn_decode_noalloc(ctypes.byref(layer), xd.data_ptr(), idx.data_ptr(), wt.data_ptr(),
                                           w.T, w.k, got.data_ptr(), status.data_ptr(), ctypes.c_void_p(stream))
        assert st == M.DS4MOE_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.isfinite(g).all()
        assert rel_err(g, r) <= TOL, f"call {call}"
        # and both agree with the oracle
        ri, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
        o = oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, x, ri, rw)
        assert rel_err(g, o) <= TOL


def test_noalloc_rejects_sizes_beyond_its_scratch_and_flags_bad_ids(M):
    import torch
    w = synth.WORKLOADS[1].replace(n_expert=8, T=64, seed=213)
    L = build_layer(w, experts=[0])
    dev = to_device(L)
    lib = M.lib()
    # 64 tokens x top-6 on the 4096 x 2048 shape needs more than the fixed array
    need = M.ds4moe_workspace_bytes(dev.abi, 64, 6, False)
    assert need > M.NOALLOC_SCRATCH_BYTES
    x = torch.zeros((64, w.d_model), dtype=torch.int16, device="cuda")
    idx = torch.zeros((64, 6), dtype=torch.int32, device="cuda")
    wt = torch.zeros((64, 6), dtype=torch.float32, device="cuda")
    out = torch.zeros((64, w.d_model), dtype=torch.float32, device="cuda")
    layer = dev.abi
    st = lib.ds4moe_ffn_decode_noalloc(ctypes.byref(layer), x.data_ptr(), idx.data_ptr(), wt.data_ptr(), 64, 6,
                                       out.data_ptr(), None, None)
    assert st == M.DS4MOE_ESPACE
    # an out-of-range expert id is reported through status_out
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    idx2 = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")
    wt2 = torch.tensor([[1.0, 0.0]], dtype=torch.float32, device="cuda")
    st = lib.ds4moe_ffn_decode_noalloc(ctypes.byref(layer), x.data_ptr(), idx2.data_ptr(), wt2.data_ptr(), 1, 2,
                                       out.data_ptr(), status.data_ptr(),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == M.DS4MOE_OK
    torch.cuda.synchronize()
    assert int(status.item()) == M.DS4MOE_EDEVICE
