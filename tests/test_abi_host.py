"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every symbol include/ds4moe.h declares, its host packer matches the oracle
byte for byte, and the device entry points reject bad arguments before
launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    M.lib()
    return M


def test_library_exports_every_declared_symbol(M):
    hdr = open(os.path.join(ROOT, "include", "ds4moe.h"), encoding="utf-8").read()
    declared = set(re.findall(r"\b(ds4moe_[a-z0-9_]+)\s*\(", hdr))
    assert declared, "no declarations found"
    assert declared == set(M.EXPORTS)
    L = ctypes.CDLL(M.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), name


def test_block_traits(M):
    assert (M.block_values(M.DS4MOE_Q4_1), M.block_bytes(M.DS4MOE_Q4_1)) == (32, 20)
    assert (M.block_values(M.DS4MOE_Q2_K), M.block_bytes(M.DS4MOE_Q2_K)) == (256, 84)
    assert M.block_values(M.DS4MOE_IQ2_XXS) == 0
    assert M.status_string(M.DS4MOE_EBLOCKER).startswith("lossless")


@pytest.mark.parametrize("bits,group", [(3, 32), (4, 64), (3, 64), (4, 32), (2, 128)])
def test_quantize_ref_q4_1_equals_oracle_reencode(M, bits, group):
    rng = np.random.default_rng(bits * 100 + group)
    n = group * 96
    codes = rng.integers(0, 1 << bits, n).astype(np.uint8)
    scale = rng.integers(0, 0x7C00, n // group).astype(np.uint16)
    mins = rng.integers(0, 0xFC00, n // group).astype(np.uint16)
    st, ref = oracle.q41_reencode(bits, group, codes, scale, mins)
    assert st == oracle.OK
    got = M.ds4moe_quantize_ref(M.DS4MOE_Q4_1, bits, group, codes, scale, mins)
    assert np.array_equal(got, ref)


def test_quantize_ref_q2_k_equals_oracle_pack(M):
    w = synth.WORKLOADS[1]
    f = synth.matrix_fields(w, 0, synth.T_DOWN, 5, row0=0, nrows=64)
    ref = oracle.pack_fields(f)
    got = M.ds4moe_quantize_ref(M.DS4MOE_Q2_K, 2, 256, f.codes, f.scale, f.minv, f.sc, f.mn)
    assert np.array_equal(got, ref)


def test_quantize_ref_q4_k_equals_oracle_pack(M):
    w = synth.WORKLOADS[5]
    f = synth.matrix_fields(w, 0, synth.T_UP, 9, row0=5, nrows=32)
    got = M.ds4moe_quantize_ref(M.DS4MOE_Q4_K, 4, 256, f.codes, f.scale, f.minv, f.sc, f.mn)
    assert np.array_equal(got, oracle.pack_fields(f))
    rng = np.random.default_rng(44)
    codes = rng.integers(0, 16, 256 * 7).astype(np.uint8)
    sc, mn = rng.integers(0, 64, 56).astype(np.uint8), rng.integers(0, 64, 56).astype(np.uint8)
    d, dm = rng.integers(0, 0x7C00, 7).astype(np.uint16), rng.integers(0, 0x7C00, 7).astype(np.uint16)
    assert np.array_equal(M.ds4moe_quantize_ref(M.DS4MOE_Q4_K, 4, 256, codes, d, dm, sc, mn),
                          oracle.q4k_pack(codes, sc, mn, d, dm))
    with pytest.raises(M.Ds4moeError) as ei:  # a 7-bit scale
        M.ds4moe_quantize_ref(M.DS4MOE_Q4_K, 4, 256, codes, d, dm, np.full(56, 64, np.uint8), mn)
    assert ei.value.status == M.DS4MOE_EBLOCKER


def test_quantize_ref_workload_fields_equal_oracle(M):
    for wid, tensor in ((0, synth.T_GATE), (2, synth.T_UP), (3, synth.T_GATE)):
        f = synth.matrix_fields(synth.WORKLOADS[wid], 0, tensor, 7, row0=3, nrows=8)
        got = M.ds4moe_quantize_ref(M.DS4MOE_Q4_1, f.bits, f.group, f.codes, f.scale, f.minv)
        assert np.array_equal(got, oracle.pack_fields(f))


@pytest.mark.parametrize("bits,group,bad,expect", [
    (4, 48, None, "EBLOCKER"), (5, 32, None, "EBLOCKER"), (4, 32, 16, "EBLOCKER"),
    (3, 32, 8, "EBLOCKER"), (0, 32, None, "EINVAL"), (4, 0, None, "EINVAL"),
])
def test_quantize_ref_q4_1_rejections(M, bits, group, bad, expect):
    n = 32 * 6
    codes = np.zeros(n, np.uint8)
    if bad is not None:
        codes[5] = bad
    ng = max(n // max(group, 1), 1)
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_quantize_ref(M.DS4MOE_Q4_1, bits, group, codes, np.zeros(ng, np.uint16), np.zeros(ng, np.uint16))
    assert ei.value.status == getattr(M, "DS4MOE_" + expect)


def test_quantize_ref_q2_k_rejections_and_unsupported(M):
    z = np.zeros
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_quantize_ref(M.DS4MOE_Q2_K, 2, 256, np.full(256, 4, np.uint8), z(1, np.uint16), z(1, np.uint16),
                              z(16, np.uint8), z(16, np.uint8))
    assert ei.value.status == M.DS4MOE_EBLOCKER
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_quantize_ref(M.DS4MOE_Q2_K, 2, 256, z(256, np.uint8), z(1, np.uint16), z(1, np.uint16),
                              np.full(16, 16, np.uint8), z(16, np.uint8))
    assert ei.value.status == M.DS4MOE_EBLOCKER
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_quantize_ref(M.DS4MOE_Q2_K, 3, 256, z(256, np.uint8), z(1, np.uint16), z(1, np.uint16),
                              z(16, np.uint8), z(16, np.uint8))
    assert ei.value.status == M.DS4MOE_EINVAL
    with pytest.raises(M.Ds4moeError) as ei:
        M.ds4moe_quantize_ref(M.DS4MOE_IQ2_XXS, 2, 256, z(256, np.uint8), z(1, np.uint16), z(1, np.uint16))
    assert ei.value.status == M.DS4MOE_EUNSUPPORTED
    # too small an output buffer
    L = M.lib()
    out = np.zeros(10, np.uint8)
    codes = z(32, np.uint8)
    st = L.ds4moe_quantize_ref(M.DS4MOE_Q4_1, 4, 32, codes.ctypes.data, z(1, np.uint16).ctypes.data,
                               z(1, np.uint16).ctypes.data, None, None, 32, out.ctypes.data, out.nbytes)
    assert st == M.DS4MOE_ESPACE


def test_device_entry_points_reject_bad_arguments_before_launch(M):
    L = M.lib()
    fake = 0x10000  # 16-byte aligned, never dereferenced: validation fails first
    # dequant: unsupported format, ragged size, misaligned pointer
    assert L.ds4moe_dequant(M.DS4MOE_IQ2_XXS, fake, 256, fake, None) == M.DS4MOE_EUNSUPPORTED
    assert L.ds4moe_dequant(9, fake, 256, fake, None) == M.DS4MOE_EUNSUPPORTED
    assert L.ds4moe_dequant(M.DS4MOE_Q2_K, fake, 255, fake, None) == M.DS4MOE_EINVAL
    assert L.ds4moe_dequant(M.DS4MOE_Q4_1, fake + 4, 64, fake, None) == M.DS4MOE_EINVAL
    assert L.ds4moe_dequant(M.DS4MOE_Q4_1, fake, 0, fake, None) == M.DS4MOE_OK   # empty: no-op
    lay = M.Layer(4096, 2048, 256, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K, fake, fake, fake)
    ws_need = M.ds4moe_workspace_bytes(lay, 4, 6, False)
    assert ws_need > 0
    args = lambda T, k, ws_bytes=ws_need: (ctypes.byref(lay), fake, fake, fake, T, k, fake, fake, ws_bytes, None)
    assert L.ds4moe_ffn_decode(*args(0, 6)) == M.DS4MOE_OK                  # T = 0: no-op
    assert L.ds4moe_ffn_decode(*args(4, 0)) == M.DS4MOE_EINVAL              # k < 1
    assert L.ds4moe_ffn_decode(*args(4, 257)) == M.DS4MOE_EINVAL            # k > E
    assert L.ds4moe_ffn_decode(*args(-1, 6)) == M.DS4MOE_EINVAL             # T < 0
    assert L.ds4moe_ffn_prefill(*args(4, 6, ws_need - 1)) == M.DS4MOE_ESPACE
    bad = M.Layer(4096, 2048, 256, M.DS4MOE_IQ2_XXS, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K, fake, fake, fake)
    assert L.ds4moe_ffn_decode(ctypes.byref(bad), fake, fake, fake, 4, 6, fake, fake, ws_need, None) == \
        M.DS4MOE_EUNSUPPORTED
    ragged = M.Layer(4000, 2048, 256, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K, fake, fake, fake)
    assert L.ds4moe_ffn_decode(ctypes.byref(ragged), fake, fake, fake, 4, 6, fake, fake, ws_need, None) == \
        M.DS4MOE_EINVAL
    mis = M.Layer(4096, 2048, 256, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K, M.DS4MOE_Q2_K, fake + 8, fake, fake)
    assert L.ds4moe_ffn_decode(ctypes.byref(mis), fake, fake, fake, 4, 6, fake, fake, ws_need, None) == \
        M.DS4MOE_EINVAL
    # router: k above 32 or above E, d_model not a multiple of 4
    assert L.ds4moe_route_topk(fake, fake, None, 4, 4096, 256, 33, fake, fake, None, fake, ws_need, None) == \
        M.DS4MOE_EINVAL
    assert L.ds4moe_route_topk(fake, fake, None, 4, 4096, 4, 6, fake, fake, None, fake, ws_need, None) == \
        M.DS4MOE_EINVAL
    assert L.ds4moe_route_topk(fake, fake, None, 4, 4094, 256, 6, fake, fake, None, fake, ws_need, None) == \
        M.DS4MOE_EINVAL
    assert L.ds4moe_route_topk(fake, fake, None, 0, 4096, 256, 6, fake, fake, None, fake, ws_need, None) == \
        M.DS4MOE_OK
    assert M.ds4moe_workspace_bytes(M.Layer(0, 0, 0, 0, 0, 0, None, None, None), 4, 6) == 0
    # prefill split threshold: an invalid layer is -1 before any device query
    assert M.ds4moe_prefill_small_pairs(bad) == -1
    assert M.ds4moe_prefill_small_pairs(ragged) == -1
    assert M.ds4moe_prefill_small_pairs(lay) in (0, 16)  # 0 without a tensor-core device
    # fault-injection hook: a budget below one poll or a negative offset
    assert L.ds4moe_debug_sync_wait(0, 0) == M.DS4MOE_EINVAL
    assert L.ds4moe_debug_sync_wait(100, -1) == M.DS4MOE_EINVAL


def test_shared_ffn_rejects_bad_arguments_before_launch(M):
    """ds4moe_shared_ffn validates on the host (fake, aligned pointers: nothing
    is dereferenced when a check fails)."""
    L = M.lib()
    A = 1 << 20  # aligned fake addresses
    D, Fs, T = 256, 128, 4
    need = M.ds4moe_shared_workspace_bytes(D, Fs, T)
    assert need >= 256 + T * Fs * 2
    assert M.ds4moe_shared_workspace_bytes(0, Fs, T) == 0
    assert M.ds4moe_shared_workspace_bytes(D, -1, T) == 0

    def call(w1=A, w3=A, w2=A, d=D, fs=Fs, x=A, t=T, out=A, acc=0, ws=A, nws=None):
        return L.ds4moe_shared_ffn(w1, w3, w2, d, fs, x, t, out, acc, ws, need if nws is None else nws, None)

    assert call(d=260) == M.DS4MOE_EINVAL          # d_model not a multiple of 8
    assert call(fs=-8) == M.DS4MOE_EINVAL
    assert call(fs=12) == M.DS4MOE_EINVAL          # d_shared not a multiple of 8
    assert call(acc=2) == M.DS4MOE_EINVAL
    assert call(x=A + 4) == M.DS4MOE_EINVAL        # misaligned
    assert call(out=None) == M.DS4MOE_EINVAL
    assert call(w2=None) == M.DS4MOE_EINVAL
    assert call(nws=need - 1) == M.DS4MOE_ESPACE
    assert call(t=0, x=None, out=None) == M.DS4MOE_OK  # zero tokens: nothing to do
