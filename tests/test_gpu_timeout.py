"""Failure detection on the GPU without a fault: a bounded cross-CTA wait is
made to run out, and the host reads the status.

The single-token fused decode on all-Q2_K layers with d_model = 2 d_ff runs
the expert FFN as one grid whose CTAs wait on each other: a CTA's down work
on an expert waits until every gate/up unit of that expert has published h.
The library's fault-injection hook raises the count that wait needs by one,
so nothing can ever satisfy it, and gives it a small poll budget.  The wait
must give up, the call must report DS4MOE_ETIMEOUT through
ds4moe_stream_status, and the context must stay usable: the next call with
the defaults restored matches the oracle.  No GPU is trapped, faulted or
hung (the kernel finishes on its own once the budget is spent).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err
from tests.layers import build_layer, to_device
from tests.test_gpu_ffn import gpu_moe_decode, oracle_out

pytestmark = pytest.mark.gpu
TOL = 2e-3
W = synth.WORKLOADS[1].replace(d_model=2048, d_ff=1024, n_expert=7, k=3, seed=421)


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def test_wait_that_cannot_succeed_gives_up_and_reports_etimeout(M):
    L = build_layer(W)
    dev = to_device(L)
    x = synth.activations(W, T=1)
    M.ds4moe_profile_enable(True)
    try:
        M.ds4moe_debug_sync_wait(2000, 1)
        _, _, _, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, W.k)
        names = set(M.ds4moe_profile_read())
    finally:
        M.ds4moe_debug_sync_wait()
        M.ds4moe_profile_enable(False)
    assert "ffn_t1" in names  # the merged grid (the wait under test) ran
    assert st == M.DS4MOE_ETIMEOUT
    # the status word was cleared by the read, the context is usable and the
    # next call (defaults restored) is right
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, W.k)
    out, idx, _, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, W.k)
    assert st == M.DS4MOE_OK
    assert np.array_equal(idx, ridx)
    assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL
