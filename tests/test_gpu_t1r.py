"""GPU parity of the single-token FFN over Q2_K weights in the 16-row tile
order (DS4MOE_Q2_K_R16), against the CPU oracle, through the C ABI.

The weights are the oracle-packed plain Q2_K blocks of the layer, rewritten
on the device by ds4moe_repack; the reference is the oracle's FFN over the
plain blocks.  Covers: the repacking (bit-exact against the oracle's own
tile order, both directions); every d_model the kernel takes (512 .. 4096,
d_model = 2 d_ff) with k = 1 .. 32 and a router bias; the fused entry
(router logits ranked in every CTA) and ds4moe_ffn_decode with the caller's
routing (an expert id out of range is flagged and skipped); the
allocation-free entry; run-to-run bit equality; the device-side span
record; the formats and shapes the path refuses; the full Flash layer (256
experts, top-6).  Bar as for every FFN test: max |err| <= 2e-3 * max |ref|,
routing bit-exact.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import rel_err, torch_bf16_bits, ulp_diff_f32
from tests.layers import build_layer, cached_layer, to_device
from tests.test_gpu_ffn import gpu_forward, gpu_moe_decode, oracle_out

pytestmark = pytest.mark.gpu
TOL = 2e-3

Q2 = synth.WORKLOADS[1]
SHAPES = [
    Q2.replace(d_model=4096, d_ff=2048, n_expert=12, k=6, seed=501),
    Q2.replace(d_model=2048, d_ff=1024, n_expert=7, k=3, seed=502, bias_sigma=1.0),
    Q2.replace(d_model=1024, d_ff=512, n_expert=5, k=1, seed=503),
    Q2.replace(d_model=3072, d_ff=1536, n_expert=9, k=8, seed=504),
    Q2.replace(d_model=512, d_ff=256, n_expert=40, k=32, seed=505),
    # 256 experts: more than one router CTA per SM
    Q2.replace(d_model=2048, d_ff=1024, n_expert=256, k=8, seed=506),
]


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    return M


def _r16(L):
    return to_device(L).repacked_r16()


def test_repack_matches_the_oracle_tile_order(M):
    import torch
    rng = np.random.default_rng(77)
    for rows, cols in ((16, 256), (48, 768), (2048, 4096)):
        src = rng.integers(0, 256, size=rows * cols // 256 * 84, dtype=np.uint8)
        s = torch.from_numpy(src).cuda()
        d = torch.empty_like(s)
        M.ds4moe_repack(M.DS4MOE_Q2_K, M.DS4MOE_Q2_K_R16, s, rows, cols, d)
        assert np.array_equal(d.cpu().numpy(), oracle.q2k_to_r16(src, rows, cols))
        back = torch.empty_like(s)
        M.ds4moe_repack(M.DS4MOE_Q2_K_R16, M.DS4MOE_Q2_K, d, rows, cols, back)
        assert np.array_equal(back.cpu().numpy(), src)


def test_repack_refuses_bad_arguments(M):
    import torch
    s = torch.zeros(16 * 84, dtype=torch.uint8, device="cuda")
    d = torch.empty_like(s)
    for args in ((M.DS4MOE_Q2_K, M.DS4MOE_Q2_K_R16, s, 8, 256, d),     # partial tile
                 (M.DS4MOE_Q2_K, M.DS4MOE_Q2_K_R16, s, 16, 128, d),    # partial block
                 (M.DS4MOE_Q2_K, M.DS4MOE_Q2_K_R16, s, 16, 256, s)):   # in place
        with pytest.raises(M.Ds4moeError) as ei:
            M.ds4moe_repack(*args)
        assert ei.value.status == M.DS4MOE_EINVAL
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_repack(M.DS4MOE_Q4_1, M.DS4MOE_Q2_K_R16, s, 16, 256, d)
    assert ei.value.status == M.DS4MOE_EUNSUPPORTED


@pytest.mark.parametrize("wi", range(len(SHAPES)))
def test_r16_fused_decode_matches_oracle(M, wi):
    w = SHAPES[wi]
    L = build_layer(w)
    dev = _r16(L)
    for batch in (0, 1):
        x = synth.activations(w, T=1, batch=batch)
        ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
        ref = oracle_out(L, x, ridx, rw)
        out, idx, wt, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        assert st == M.DS4MOE_OK
        assert np.array_equal(idx, ridx)
        assert ulp_diff_f32(wt, rw).max() <= 2
        assert rel_err(out, ref) <= TOL
        # the caller's routing through ds4moe_ffn_decode: same kernel, same bits
        out2, idx2, wt2, st2 = gpu_forward(M, dev, x, L.Wr, L.bias, w.k)
        assert st2 == M.DS4MOE_OK and np.array_equal(idx2, ridx)
        assert rel_err(out2, ref) <= TOL
        if np.array_equal(wt.view(np.uint32), wt2.view(np.uint32)):
            assert np.array_equal(out.view(np.uint32), out2.view(np.uint32))
        # same inputs, same bits (the combine sums in rank order)
        out3, _, _, _ = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        assert np.array_equal(out3.view(np.uint32), out.view(np.uint32))


def test_r16_large_activations_take_the_scaled_operand(M):
    """|x| up to ~3000: the kernel lowers its operand scale per 256-value
    block (exact while no value leaves the binary16 range)."""
    w = SHAPES[1]
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=1)
    xf = oracle.bf16_to_f32(x) * 700.0
    xb = oracle.round_bf16(xf.astype(np.float64))
    ridx, rw, _ = oracle.route(xb, L.Wr, L.bias, w.k)
    out, idx, _, st = gpu_moe_decode(M, dev, xb, L.Wr, L.bias, w.k)
    assert st == M.DS4MOE_OK and np.array_equal(idx, ridx)
    assert rel_err(out, oracle_out(L, xb, ridx, rw)) <= TOL


@pytest.mark.parametrize("wi", [0, 2])
def test_r16_kernel_is_the_one_launched(M, wi):
    w = SHAPES[wi]
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=1)
    M.ds4moe_profile_enable(True)
    try:
        gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        names = set(M.ds4moe_profile_read())
    finally:
        M.ds4moe_profile_enable(False)
    assert "ffn_t1r" in names
    assert "route" in names  # the logits' grid, then the tile-order grid
    assert not {"ffn_t1", "gate_up", "down", "combine", "bucket", "gate_up_simt", "down_simt"} & names


def test_r16_out_of_range_expert(M):
    w = SHAPES[1].replace(k=3)
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=1)
    idx = np.array([[2, 99, 5]], np.int32)
    wt = np.array([[0.5, 0.3, 0.2]], np.float32)
    out, _, _, st = gpu_forward(M, dev, x, L.Wr, None, 3, False, idx, wt)
    assert st == M.DS4MOE_EDEVICE
    ref = oracle_out(L, x, np.array([[2, 5, 5]], np.int32), np.array([[0.5, 0.2, 0.0]], np.float32))
    assert rel_err(out, ref) <= TOL
    # no valid expert at all: the combine of nothing is zero
    out0, _, _, st0 = gpu_forward(M, dev, x, L.Wr, None, 3, False, np.array([[-1, 99, 7]], np.int32), wt)
    assert st0 == M.DS4MOE_EDEVICE
    assert not out0.any()


def test_r16_allocation_free_entry(M):
    import torch
    w = SHAPES[1]
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=1)
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    out = torch.empty((1, w.d_model), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        M.ds4moe_ffn_decode_noalloc(dev.abi, torch_bf16_bits(x), torch.from_numpy(ridx).cuda(),
                                    torch.from_numpy(rw).cuda(), out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == M.DS4MOE_OK
        assert rel_err(out.cpu().numpy(), oracle_out(L, x, ridx, rw)) <= TOL


def test_r16_refused_shapes_and_calls(M):
    import torch
    from bit_quantized_moe_q2_gb300.device import workspace
    w = SHAPES[2]
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=2)
    ws = workspace(dev, 2, w.k, True)
    idx = torch.zeros((2, w.k), dtype=torch.int32, device="cuda")
    wt = torch.ones((2, w.k), dtype=torch.float32, device="cuda")
    out = torch.empty((2, w.d_model), dtype=torch.float32, device="cuda")
    for fn in (M.ds4moe_ffn_decode, M.ds4moe_ffn_prefill):   # T = 2, and prefill
        with pytest.raises(M.Ds4moeError) as ei:
            fn(dev.abi, torch_bf16_bits(x), idx, wt, out, ws)
        assert ei.value.status == M.DS4MOE_EUNSUPPORTED
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_dequant(M.DS4MOE_Q2_K_R16, dev.gate, 256, out)
    assert ei.value.status == M.DS4MOE_EUNSUPPORTED
    # one matrix in the tile order, the others plain
    plain = to_device(L)
    mixed = M.make_layer(w.d_model, w.d_ff, w.n_expert, M.DS4MOE_Q2_K_R16, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K,
                         dev.gate, plain.up, plain.down)
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_ffn_decode(mixed, torch_bf16_bits(x[:1]), idx[:1], wt[:1], out[:1], ws)
    assert ei.value.status == M.DS4MOE_EUNSUPPORTED
    assert M.ds4moe_stream_status(ws) == M.DS4MOE_OK


def test_r16_wait_gives_up_and_reports_etimeout(M):
    """The grid's cross-CTA h-ready wait made unsatisfiable (fault-injection
    hook): it gives up, the call reports DS4MOE_ETIMEOUT, the next call with
    the defaults restored is right.  No GPU fault or hang."""
    w = SHAPES[1]
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=1)
    try:
        M.ds4moe_debug_sync_wait(2000, 1)
        _, _, _, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
    finally:
        M.ds4moe_debug_sync_wait()
    assert st == M.DS4MOE_ETIMEOUT
    ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
    out, idx, _, st = gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
    assert st == M.DS4MOE_OK and np.array_equal(idx, ridx)
    assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL


def test_r16_span_record(M):
    w = SHAPES[0]
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=1)
    M.ds4moe_profile_span(1)
    try:
        for _ in range(3):
            gpu_moe_decode(M, dev, x, L.Wr, L.bias, w.k)
        spans = M.ds4moe_profile_span(0)
    finally:
        M.ds4moe_profile_span(0)
    assert set(spans) == {"route", "ffn_t1r"}
    for name, (ns, n) in spans.items():
        assert n == 3, name
        assert 1e2 < ns / n < 1e7, name  # between 0.1 us and 10 ms per launch


def test_r16_full_flash_layer(M):
    """The Flash layer itself (256 experts, top-6, 4096 x 2048): every output
    against the oracle for three tokens."""
    w = synth.WORKLOADS[1]
    L, dev = cached_layer(w)
    r16 = dev.repacked_r16()
    for batch in (0, 1, 2):
        x = synth.activations(w, batch=batch)
        out, idx, wt, st = gpu_moe_decode(M, r16, x, L.Wr, L.bias, w.k)
        assert st == M.DS4MOE_OK
        ridx, rw, _ = oracle.route(x, L.Wr, L.bias, w.k)
        assert np.array_equal(idx, ridx)
        assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL


@pytest.mark.parametrize("case", ["all_tie", "tie_nan"])
def test_r16_routing_ties_and_nan(M, case):
    """Every CTA ranks the logits itself: exact ties go to the lower expert
    id, a NaN logit ranks below every number."""
    w = SHAPES[1]
    L = build_layer(w)
    dev = _r16(L)
    x = synth.activations(w, T=1)
    Wr = np.repeat(L.Wr[:1], w.n_expert, axis=0).copy()  # every logit equal
    if case == "tie_nan":
        Wr[4] = L.Wr[4] * 3.0   # one distinct expert
        Wr[0, 0] = np.nan       # expert 0: NaN logit
    ridx, rw, _ = oracle.route(x, Wr, None, w.k)
    out, idx, wt, st = gpu_moe_decode(M, dev, x, Wr, None, w.k)
    assert st == M.DS4MOE_OK
    assert np.array_equal(idx, ridx)
    assert ulp_diff_f32(wt, rw).max() <= 2
    assert rel_err(out, oracle_out(L, x, ridx, rw)) <= TOL
