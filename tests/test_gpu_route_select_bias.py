"""GPU parity of the routing variant with the bias used for selection only
(ds4moe_route_topk_select_bias) against the oracle: indices bit-exact,
weights within 2 fp32 ulp, the unbiased logits equal to the plain router's
bit for bit; a zero bias gives the plain route."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import torch_bf16_bits

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(4242)


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _run(M, x, Wr, bias, k, fn="select"):
    import torch
    T, D = x.shape
    E = Wr.shape[0]
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    xd = torch_bf16_bits(x)
    Wd = torch.from_numpy(Wr).cuda()
    bd = None if bias is None else torch.from_numpy(bias).cuda()
    if fn == "select":
        M.ds4moe_route_topk_select_bias(xd, Wd, bd, k, idx, w, lg, ws)
    else:
        M.ds4moe_route_topk(xd, Wd, bd, k, idx, w, lg, ws)
    return idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()


def _inputs(T, D, E):
    x = (RNG.standard_normal((T, D))).astype(np.float32)
    xb = ((x.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    Wr = (RNG.standard_normal((E, D)) * 0.02).astype(np.float32)
    return xb, Wr


@pytest.mark.parametrize("T,D,E,k", [(1, 4096, 256, 6), (7, 1024, 64, 8), (300, 2048, 256, 6), (33, 512, 16, 1)])
def test_select_bias_matches_oracle(M, T, D, E, k):
    xb, Wr = _inputs(T, D, E)
    bias = RNG.standard_normal(E).astype(np.float32) * 0.5
    idx, w, lu = _run(M, xb, Wr, bias, k)
    ridx, rw, rlu, _ = oracle.route_select_bias(xb, Wr, bias, k)
    assert np.array_equal(idx, ridx)
    assert np.abs(w.view(np.int32).astype(np.int64) - rw.view(np.int32)).max() <= 2
    # unbiased logits: the plain router's, bit for bit
    _, _, plain = _run(M, xb, Wr, None, k, fn="plain")
    assert np.array_equal(lu.view(np.uint32), plain.view(np.uint32))


def test_zero_bias_is_the_plain_route(M):
    xb, Wr = _inputs(12, 1024, 32)
    idx, w, _ = _run(M, xb, Wr, np.zeros(32, np.float32), 4)
    pidx, pw, _ = _run(M, xb, Wr, None, 4, fn="plain")
    assert np.array_equal(idx, pidx)
    assert np.array_equal(w.view(np.uint32), pw.view(np.uint32))


def test_rejects_missing_bias_and_large_expert_counts(M):
    xb, Wr = _inputs(2, 256, 300)
    with pytest.raises(M.Ds4moeError):
        _run(M, xb, Wr, RNG.standard_normal(300).astype(np.float32), 2)
    xb, Wr = _inputs(2, 256, 16)
    with pytest.raises(M.Ds4moeError):
        _run(M, xb, Wr, None, 2)
