"""GPU parity of the float-input quantizer (ds4moe_quantize_f32) against the
oracle: the block bytes -- codes, sub-block scales and mins, binary16 d and
dmin / d and m -- must match bit for bit, with and without importance, on
ordinary, heavy-tailed, one-signed, tiny, huge and degenerate inputs; a
non-finite value zeroes its block and is reported.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(9090)


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _ws():
    import torch
    from bit_quantized_moe_q2_gb300 import ds4moe_workspace_init
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    ds4moe_workspace_init(ws)
    return ws


def _gpu(M, qtype, x, imp=None, cols=None):
    import torch
    bv, bb = oracle.block_values(qtype), oracle.block_bytes(qtype)
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    out = torch.full((x.size // bv * bb,), 0xAB, dtype=torch.uint8, device="cuda")
    ws = _ws()
    idev = None if imp is None else torch.from_numpy(np.ascontiguousarray(imp, np.float32)).cuda()
    M.ds4moe_quantize_f32(qtype, xd.reshape(-1), idev, out, ws, cols=cols if cols else x.size)
    return out.cpu().numpy(), M.ds4moe_stream_status(ws)


def _inputs(kind, n):
    if kind == "normal":
        return RNG.standard_normal(n).astype(np.float32)
    if kind == "heavy":
        return (RNG.standard_t(2, n) * 0.05).astype(np.float32)
    if kind == "positive":
        return np.abs(RNG.standard_normal(n) * 7.0).astype(np.float32)
    if kind == "negative":
        return (-np.abs(RNG.standard_normal(n)) - 3.0).astype(np.float32)
    if kind == "tiny":
        return (RNG.standard_normal(n) * 1e-6).astype(np.float32)
    if kind == "huge":
        return (RNG.standard_normal(n) * 3e4).astype(np.float32)
    if kind == "steps":  # constant sub-blocks and exact zeros mixed in
        x = np.repeat(RNG.standard_normal(n // 16), 16).astype(np.float32)
        x[RNG.random(n) < 0.2] = 0.0
        return x
    raise ValueError(kind)


KINDS = ["normal", "heavy", "positive", "negative", "tiny", "huge", "steps"]


@pytest.mark.parametrize("qtype", [oracle.Q2_K, oracle.Q4_1])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("weighted", [False, True])
def test_quantize_matches_oracle_bit_for_bit(M, qtype, kind, weighted):
    cols = 1024
    x = _inputs(kind, cols * 9)
    imp = (RNG.exponential(1.0, cols) ** 2).astype(np.float32) if weighted else None
    got, st = _gpu(M, qtype, x, imp, cols)
    assert st == M.DS4MOE_OK
    ref = oracle.quantize_f32(qtype, x, imp, cols)
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} bytes differ"


def test_quantize_full_expert_matrix(M):
    """One Q2_K expert matrix at the flash layer's size (2048 x 4096) with
    importance, and its Q4_1 twin."""
    rows, cols = 2048, 4096
    x = (RNG.standard_normal(rows * cols) * 0.02).astype(np.float32)
    imp = (RNG.exponential(1.0, cols) ** 2).astype(np.float32)
    for qtype in (oracle.Q2_K, oracle.Q4_1):
        got, st = _gpu(M, qtype, x, imp, cols)
        assert st == M.DS4MOE_OK
        assert np.array_equal(got, oracle.quantize_f32(qtype, x, imp, cols))


def test_non_finite_block_is_zeroed_and_reported(M):
    x = RNG.standard_normal(256 * 3).astype(np.float32)
    x[300] = np.nan
    got, st = _gpu(M, oracle.Q2_K, x)
    assert st == M.DS4MOE_EDEVICE
    assert not got[84:168].any()
    ok = np.concatenate([x[:256], x[512:]])
    assert np.array_equal(np.concatenate([got[:84], got[168:]]), oracle.quantize_f32(oracle.Q2_K, ok))


def test_argument_errors(M):
    import torch
    x = torch.zeros(100, dtype=torch.float32, device="cuda")
    out = torch.zeros(1000, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.Ds4moeError):
        M.ds4moe_quantize_f32(oracle.Q2_K, x, None, out, _ws())
    x = torch.zeros(512, dtype=torch.float32, device="cuda")
    with pytest.raises(M.Ds4moeError):  # too little output space
        M.ds4moe_quantize_f32(oracle.Q2_K, x, None, out[:100], _ws())
    with pytest.raises(M.Ds4moeError):  # importance columns not whole blocks
        M.ds4moe_quantize_f32(oracle.Q4_1, x, torch.ones(48, device="cuda"), out, _ws(), cols=48)
