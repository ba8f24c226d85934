"""GPU parity when one workspace (or the no-allocation scratch array) serves
a sequence of calls of different sizes and paths, as in a serving loop whose
batch changes from step to step, and with a token routed to the same expert
more than once (caller-supplied routing).  Every call is checked against the
oracle: max |err| <= 2e-3 * max |ref|.

The combine of the tensor-core decode kernels counts arrivals per output
tile in the workspace; the regions of the workspace move with the sizes, so
these cases catch counters that do not start at zero in a call."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err, torch_bf16_bits
from tests.layers import build_layer, to_device
from tests.test_gpu_ffn import oracle_out

pytestmark = pytest.mark.gpu
TOL = 2e-3

LAYERS = [
    # Q2_K everywhere: single-token kernels at T = 1, multi-token kernels above
    synth.WORKLOADS[1].replace(d_model=1024, d_ff=1024, n_expert=12, k=6, seed=701),
    # Q4_1 gate/up, Q2_K down
    synth.WORKLOADS[2].replace(d_model=2048, d_ff=1024, n_expert=9, k=3, seed=702),
    # Q4_K everywhere
    synth.WORKLOADS[5].replace(d_model=1024, d_ff=1024, n_expert=8, k=4, seed=703),
]
TS = [7, 1, 3, 12, 1, 5, 2, 1, 9]


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _run(M, dev, x, idx, wt, ws, prefill=False):
    import torch
    T = x.shape[0]
    out = torch.full((T, dev.d_model), float("nan"), dtype=torch.float32, device="cuda")
    fn = M.ds4moe_ffn_prefill if prefill else M.ds4moe_ffn_decode
    fn(dev.abi, torch_bf16_bits(x), torch.from_numpy(idx).cuda(), torch.from_numpy(wt).cuda(), out, ws)
    return out.cpu().numpy(), M.ds4moe_stream_status(ws)


@pytest.mark.parametrize("li", range(len(LAYERS)))
def test_one_workspace_many_sizes(M, li):
    import torch
    w = LAYERS[li]
    L = build_layer(w)
    dev = to_device(L)
    n = max(M.ds4moe_workspace_bytes(dev.abi, T, w.k, p) for T in TS for p in (0, 1))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    M.ds4moe_workspace_init(ws)
    for i, T in enumerate(TS):
        x = synth.activations(w, T=T, batch=i)
        idx, wt, _ = oracle.route(x, L.Wr, L.bias, w.k)
        out, st = _run(M, dev, x, idx, wt, ws, prefill=(i % 3 == 2))
        assert st == M.DS4MOE_OK, (T, st)
        assert rel_err(out, oracle_out(L, x, idx, wt)) <= TOL, T


@pytest.mark.parametrize("li", range(len(LAYERS)))
def test_noalloc_scratch_many_sizes(M, li):
    import torch
    w = LAYERS[li]
    L = build_layer(w)
    dev = to_device(L)
    for i, T in enumerate(TS):
        x = synth.activations(w, T=T, batch=100 + i)
        idx, wt, _ = oracle.route(x, L.Wr, L.bias, w.k)
        out = torch.full((T, dev.d_model), float("nan"), dtype=torch.float32, device="cuda")
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        M.ds4moe_ffn_decode_noalloc(dev.abi, torch_bf16_bits(x), torch.from_numpy(idx).cuda(),
                                    torch.from_numpy(wt).cuda(), out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == M.DS4MOE_OK, T
        assert rel_err(out.cpu().numpy(), oracle_out(L, x, idx, wt)) <= TOL, T


@pytest.mark.parametrize("li", range(len(LAYERS)))
@pytest.mark.parametrize("T", [1, 4])
def test_repeated_expert_in_a_token(M, li, T):
    """Caller routing that names one expert twice (or three times) for a
    token: the expert's output enters the combine once per slot."""
    import torch
    w = LAYERS[li]
    L = build_layer(w)
    dev = to_device(L)
    rng = np.random.default_rng(50 + li * 7 + T)
    x = synth.activations(w, T=T)
    idx = np.stack([rng.choice(w.n_expert, w.k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[:, 1] = idx[:, 0]
    if w.k >= 4:
        idx[0, 3] = idx[0, 0]
    wt = rng.uniform(0.05, 1.0, (T, w.k)).astype(np.float32)
    ws = torch.empty(M.ds4moe_workspace_bytes(dev.abi, T, w.k, 1), dtype=torch.uint8, device="cuda")
    M.ds4moe_workspace_init(ws)
    ref = oracle_out(L, x, idx, wt)
    for prefill in (False, True):
        out, st = _run(M, dev, x, idx, wt, ws, prefill)
        assert st == M.DS4MOE_OK
        assert rel_err(out, ref) <= TOL, prefill
