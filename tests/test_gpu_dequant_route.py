"""GPU parity: block dequantisation and routing (CUDA path through the C ABI)
against the CPU oracle.  Dequantised weights and routing indices must match
bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import torch_bf16_bits, ulp_diff_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _gpu_dequant(M, qtype, blocks, n):
    import torch
    b = torch.from_numpy(np.ascontiguousarray(blocks)).cuda()
    out = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    M.ds4moe_dequant(qtype, b, n, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _same_bits(a, b):
    a = a.view(np.uint32)
    b = b.view(np.uint32)
    nan_a = np.isnan(a.view(np.float32))
    nan_b = np.isnan(b.view(np.float32))
    return np.array_equal(nan_a, nan_b) and np.array_equal(a[~nan_a], b[~nan_b])


@pytest.mark.parametrize("nb", [1, 7, 1000, 40001])
def test_dequant_q4_1_bit_exact(M, nb):
    rng = np.random.default_rng(nb)
    codes = rng.integers(0, 16, nb * 32).astype(np.uint8)
    d = rng.integers(0, 0x7C00, nb).astype(np.uint16) | (rng.integers(0, 2, nb) << 15).astype(np.uint16)
    m = rng.integers(0, 0x7C00, nb).astype(np.uint16) | (rng.integers(0, 2, nb) << 15).astype(np.uint16)
    blk = oracle.q41_pack(codes, d, m)
    assert _same_bits(_gpu_dequant(M, M.DS4MOE_Q4_1, blk, nb * 32), oracle.dequant(oracle.Q4_1, blk, nb * 32))


@pytest.mark.parametrize("nb", [1, 5, 333, 20001])
def test_dequant_q2_k_bit_exact(M, nb):
    rng = np.random.default_rng(nb + 1)
    blk = oracle.q2k_pack(rng.integers(0, 4, nb * 256).astype(np.uint8), rng.integers(0, 16, nb * 16).astype(np.uint8),
                          rng.integers(0, 16, nb * 16).astype(np.uint8), rng.integers(0, 0x7C00, nb).astype(np.uint16),
                          rng.integers(0, 0xFC00, nb).astype(np.uint16))
    assert _same_bits(_gpu_dequant(M, M.DS4MOE_Q2_K, blk, nb * 256), oracle.dequant(oracle.Q2_K, blk, nb * 256))


@pytest.mark.parametrize("qtype", ["q4_1", "q2_k"])
def test_dequant_arbitrary_bytes_incl_inf_nan(M, qtype):
    # every byte pattern is a valid block: fp16 fields may be inf / NaN / subnormal
    q = oracle.QTYPES[qtype]
    nb = 5000
    blk = np.random.default_rng(9).integers(0, 256, nb * oracle.block_bytes(q), dtype=np.uint8)
    n = nb * oracle.block_values(q)
    assert _same_bits(_gpu_dequant(M, q, blk, n), oracle.dequant(q, blk, n))


@pytest.mark.parametrize("wid,tensor", [(1, synth.T_GATE), (3, synth.T_UP), (2, synth.T_GATE), (0, synth.T_DOWN)])
def test_dequant_full_expert_matrix(M, wid, tensor):
    w = synth.WORKLOADS[wid]
    f = synth.matrix_fields(w, 0, tensor, 11)
    blk = oracle.pack_fields(f)
    q = oracle.QTYPES[f.qtype]
    n = f.rows * f.cols
    assert _same_bits(_gpu_dequant(M, q, blk, n), oracle.dequant(q, blk, n))


# ------------------------------------------------------------------ routing
def _gpu_route(M, x, Wr, bias, k):
    import torch
    T = x.shape[0]
    E = Wr.shape[0]
    xd = torch_bf16_bits(x)
    Wd = torch.from_numpy(np.ascontiguousarray(Wr)).cuda()
    bd = None if bias is None else torch.from_numpy(bias).cuda()
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    lg = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    M.ds4moe_route_topk(xd, Wd, bd, k, idx, w, lg, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()


def _check_route(M, x, Wr, bias, k):
    idx, w, lg = _gpu_route(M, x, Wr, bias, k)
    ridx, rw, rlg = oracle.route(x, Wr, bias, k)
    # logits: compensated fp32 vs double -> same fp32 value up to the final rounding
    nan = np.isnan(rlg)
    assert np.array_equal(np.isnan(lg), nan)
    assert ulp_diff_f32(lg[~nan], rlg[~nan]).max() <= 1
    mism = np.nonzero((idx != ridx).any(1))[0]
    if mism.size:
        # report the oracle gap between the disagreeing experts (must be a near tie)
        t = mism[0]
        pytest.fail(f"{mism.size} tokens route differently; token {t}: gpu {idx[t]} oracle {ridx[t]} "
                    f"logits {rlg[t, ridx[t]]}")
    assert ulp_diff_f32(w, rw).max() <= 2
    return idx


@pytest.mark.parametrize("wid", [0, 1, 2, 3])
def test_route_matches_oracle_on_workloads(M, wid):
    w = synth.WORKLOADS[wid]
    Wr, bias = synth.router(w)
    x = synth.activations(w)
    idx = _check_route(M, x, Wr, bias, w.k)
    if wid == 3:  # the bias skews expert load
        counts = np.bincount(idx.ravel(), minlength=w.n_expert)
        assert counts.max() > 4 * counts.mean()


def test_route_ties_nan_and_k_extremes(M):
    rng = np.random.default_rng(5)
    E, D, T = 40, 256, 37
    Wr = (rng.standard_normal((E, D)) * 0.02).astype(np.float32)
    Wr[7] = Wr[3]            # exact tie: 3 ranks before 7
    Wr[11] = np.nan          # NaN logit ranks last
    x = oracle.round_bf16(rng.standard_normal((T, D)))
    for k in (1, 2, 6, 32):
        idx = _check_route(M, x, Wr, None, k)
        assert not np.any(idx == 11) or k > E - 1
        both = (idx == 3).any(1) & (idx == 7).any(1)
        for t in np.nonzero(both)[0]:
            r = idx[t].tolist()
            assert r.index(3) < r.index(7)
    # all logits equal -> ids 0..k-1, uniform weights
    idx, w, _ = _gpu_route(M, x[:4], np.zeros((E, D), np.float32), None, 6)
    assert np.array_equal(idx, np.tile(np.arange(6), (4, 1)))
    assert np.all(w == np.float32(1 / 6))


def test_route_with_bias_large_t(M):
    w = synth.WORKLOADS[3].replace(T=1000, seed=31)
    Wr, bias = synth.router(w)
    _check_route(M, synth.activations(w), Wr, bias, 6)


# ------------------------------------------- routing without a logits output
# Batches above 256 tokens then take the certified fast path: approximate
# fp32 logits with a rigorous error bound select the top-k; only the selected
# logits are recomputed exactly, and tokens whose boundary is within the
# bound are recomputed exactly in full.  Indices must still match bit for bit.
def _gpu_route_no_logits(M, x, Wr, bias, k):
    import torch
    T = x.shape[0]
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(T * Wr.shape[0] * 4 + 8 * (T + Wr.shape[0]) + (1 << 20), dtype=torch.uint8, device="cuda")
    M.ds4moe_route_topk(torch_bf16_bits(x), torch.from_numpy(np.ascontiguousarray(Wr)).cuda(),
                        None if bias is None else torch.from_numpy(bias).cuda(), k, idx, w, None, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("wid", [2, 3])
def test_route_without_logits_output_matches_oracle(M, wid):
    w = synth.WORKLOADS[wid]
    Wr, bias = synth.router(w)
    x = synth.activations(w)
    idx, wt = _gpu_route_no_logits(M, x, Wr, bias, w.k)
    ridx, rw, _ = oracle.route(x, Wr, bias, w.k)
    assert np.array_equal(idx, ridx)
    assert ulp_diff_f32(wt, rw).max() <= 2


def test_route_fast_path_hands_back_tied_tokens(M):
    """Half the tokens carry a large x[0]; experts 0-4 weigh x[0] heavily and
    experts 9, 17, 21 share one row that weighs it less, so for those tokens
    the 6th choice is an exact three-way tie (resolved to expert 9), which no
    error bound can certify: those tokens must go through the exact pass."""
    rng = np.random.default_rng(41)
    E, D, T, k = 32, 1024, 300, 6
    Wr = (rng.standard_normal((E, D)) * 0.02).astype(np.float32)
    Wr[0:5, 0] = 1.0
    Wr[9, 0] = 0.5
    Wr[17] = Wr[9]
    Wr[21] = Wr[9]
    xf = rng.standard_normal((T, D))
    xf[::2, 0] = 8.0
    x = oracle.round_bf16(xf)
    idx, wt = _gpu_route_no_logits(M, x, Wr, None, k)
    ridx, rw, _ = oracle.route(x, Wr, None, k)
    assert np.array_equal(idx, ridx)
    assert (ridx[::2, 5] == 9).all() and set(ridx[::2, :5].ravel().tolist()) == {0, 1, 2, 3, 4}
    assert ulp_diff_f32(wt, rw).max() <= 2
