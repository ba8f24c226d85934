"""Python binding of libds4moe (the C ABI declared in include/ds4moe.h).

Argument marshalling only: every step of the routed-MoE path runs in the
library's sm_103a kernels.  Tensors are PyTorch CUDA tensors (PyTorch is
used for device memory and streams); host-side packing takes numpy arrays.
There is no fallback: if the compiled library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libds4moe.so")

DS4MOE_OK, DS4MOE_EINVAL, DS4MOE_EBLOCKER, DS4MOE_EUNSUPPORTED = 0, 1, 2, 3
DS4MOE_ECUDA, DS4MOE_ETIMEOUT, DS4MOE_EDEVICE, DS4MOE_ESPACE = 4, 5, 6, 7
DS4MOE_Q4_1, DS4MOE_Q2_K, DS4MOE_IQ2_XXS, DS4MOE_Q4_K, DS4MOE_Q2_K_R16 = 1, 2, 3, 4, 5
QTYPES = {"q4_1": DS4MOE_Q4_1, "q2_k": DS4MOE_Q2_K, "iq2_xxs": DS4MOE_IQ2_XXS, "q4_k": DS4MOE_Q4_K,
          "q2_k_r16": DS4MOE_Q2_K_R16}

# Every symbol include/ds4moe.h declares.
EXPORTS = (
    "ds4moe_block_values", "ds4moe_block_bytes", "ds4moe_status_string", "ds4moe_quantize_ref",
    "ds4moe_prefill_small_pairs",
    "ds4moe_dequant", "ds4moe_workspace_bytes", "ds4moe_workspace_init", "ds4moe_route_topk",
    "ds4moe_ffn_decode", "ds4moe_ffn_prefill", "ds4moe_stream_status",
    "ds4moe_profile_enable", "ds4moe_profile_count", "ds4moe_profile_entry",
    "ds4moe_ffn_decode_noalloc", "ds4moe_moe_decode", "ds4moe_residual_norm", "ds4moe_stack_decode",
    "ds4moe_quantize_f32", "ds4moe_route_topk_select_bias", "ds4moe_debug_sync_wait",
    "ds4moe_repack", "ds4moe_profile_span", "ds4moe_shared_workspace_bytes", "ds4moe_shared_ffn",
    "ds4moe_gather_rows", "ds4moe_combine_pairs",
)
NOALLOC_SCRATCH_BYTES = 4 << 20


class Ds4moeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Layer(ctypes.Structure):
    """Mirror of ds4moe_layer."""
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_expert", ctypes.c_int32),
                ("q_gate", ctypes.c_int32), ("q_up", ctypes.c_int32), ("q_down", ctypes.c_int32),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded library; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libds4moe.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.ds4moe_block_values.argtypes = [i32]
        L.ds4moe_block_values.restype = i32
        L.ds4moe_block_bytes.argtypes = [i32]
        L.ds4moe_block_bytes.restype = i32
        L.ds4moe_status_string.argtypes = [i32]
        L.ds4moe_status_string.restype = ctypes.c_char_p
        L.ds4moe_quantize_ref.argtypes = [i32, i32, i32, p, p, p, p, p, i64, p, sz]
        L.ds4moe_dequant.argtypes = [i32, p, i64, p, p]
        L.ds4moe_repack.argtypes = [i32, i32, p, i64, i64, p, p]
        L.ds4moe_profile_span.argtypes = [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
        L.ds4moe_shared_workspace_bytes.argtypes = [i32, i32, i32]
        L.ds4moe_shared_workspace_bytes.restype = sz
        L.ds4moe_shared_ffn.argtypes = [p, p, p, i32, i32, p, i32, p, i32, p, sz, p]
        L.ds4moe_gather_rows.argtypes = [p, p, i32, i32, p, p]
        L.ds4moe_combine_pairs.argtypes = [p, p, p, i32, i32, i32, p, p]
        L.ds4moe_quantize_f32.argtypes = [i32, p, p, i64, i64, p, ctypes.c_size_t, p, ctypes.c_size_t, p]
        L.ds4moe_workspace_bytes.argtypes = [ctypes.POINTER(Layer), i32, i32, i32]
        L.ds4moe_workspace_bytes.restype = sz
        L.ds4moe_workspace_init.argtypes = [p, sz, p]
        L.ds4moe_prefill_small_pairs.argtypes = [ctypes.POINTER(Layer)]
        L.ds4moe_route_topk.argtypes = [p, p, p, i32, i32, i32, i32, p, p, p, p, sz, p]
        L.ds4moe_route_topk_select_bias.argtypes = [p, p, p, i32, i32, i32, i32, p, p, p, p, sz, p]
        L.ds4moe_ffn_decode.argtypes = [ctypes.POINTER(Layer), p, p, p, i32, i32, p, p, sz, p]
        L.ds4moe_ffn_prefill.argtypes = [ctypes.POINTER(Layer), p, p, p, i32, i32, p, p, sz, p]
        L.ds4moe_stream_status.argtypes = [p, p]
        L.ds4moe_ffn_decode_noalloc.argtypes = [ctypes.POINTER(Layer), p, p, p, i32, i32, p, p, p]
        L.ds4moe_moe_decode.argtypes = [ctypes.POINTER(Layer), p, p, p, i32, i32, p, p, p, p, sz, p]
        L.ds4moe_residual_norm.argtypes = [p, p, p, i32, i32, ctypes.c_float, p]
        L.ds4moe_stack_decode.argtypes = [ctypes.POINTER(Layer), ctypes.POINTER(p), ctypes.POINTER(p), i32, i32,
                                          i32, ctypes.c_float, p, p, p, p, p, p, sz, p]
        L.ds4moe_profile_enable.argtypes = [i32]
        L.ds4moe_debug_sync_wait.argtypes = [i32, i32]
        L.ds4moe_profile_count.argtypes = []
        L.ds4moe_profile_entry.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_int64)]
        for name in EXPORTS:
            if name not in ("ds4moe_block_values", "ds4moe_block_bytes", "ds4moe_status_string",
                            "ds4moe_workspace_bytes"):
                getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ds4moe_status_string(status).decode()


def _check(status: int, what: str):
    if status != DS4MOE_OK:
        raise Ds4moeError(status, what)


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def block_values(qtype: int) -> int:
    return lib().ds4moe_block_values(qtype)


def block_bytes(qtype: int) -> int:
    return lib().ds4moe_block_bytes(qtype)


def make_layer(d_model, d_ff, n_expert, q_gate, q_up, q_down, gate, up, down) -> Layer:
    """Layer descriptor over three device tensors of experts-major block bytes."""
    return Layer(d_model, d_ff, n_expert, q_gate, q_up, q_down, _ptr(gate), _ptr(up), _ptr(down))


# ------------------------------------------------------------- entry points
def ds4moe_quantize_ref(out_type, bits, group, codes, scale_f16, min_f16, sub_sc=None, sub_mn=None):
    """Host packing (numpy in, numpy uint8 block bytes out)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scale_f16 = np.ascontiguousarray(scale_f16, dtype=np.uint16)
    min_f16 = np.ascontiguousarray(min_f16, dtype=np.uint16)
    sub_sc = None if sub_sc is None else np.ascontiguousarray(sub_sc, dtype=np.uint8)
    sub_mn = None if sub_mn is None else np.ascontiguousarray(sub_mn, dtype=np.uint8)
    n = codes.size
    bv = max(block_values(out_type), 1)
    out = np.zeros(n // bv * max(block_bytes(out_type), 0), dtype=np.uint8)
    st = lib().ds4moe_quantize_ref(out_type, bits, group, codes.ctypes.data, scale_f16.ctypes.data,
                                   min_f16.ctypes.data, None if sub_sc is None else sub_sc.ctypes.data,
                                   None if sub_mn is None else sub_mn.ctypes.data, n,
                                   out.ctypes.data if out.size else None, out.nbytes)
    _check(st, "ds4moe_quantize_ref")
    return out


def ds4moe_dequant(qtype, blocks, n_values, out, stream=None):
    _check(lib().ds4moe_dequant(qtype, _ptr(blocks), n_values, _ptr(out), _stream(stream)), "ds4moe_dequant")


def ds4moe_repack(src_type, dst_type, src, rows, cols, dst, stream=None):
    """Rewrite a Q2_K matrix (rows x cols values, device uint8 tensors) between
    the plain block layout and the 16-row tile order, either way."""
    _check(lib().ds4moe_repack(src_type, dst_type, _ptr(src), int(rows), int(cols), _ptr(dst), _stream(stream)),
           "ds4moe_repack")


def ds4moe_shared_workspace_bytes(d_model: int, d_shared: int, T: int) -> int:
    return int(lib().ds4moe_shared_workspace_bytes(int(d_model), int(d_shared), int(T)))


def ds4moe_shared_ffn(w1, w3, w2, x, out, ws, accumulate=False, stream=None):
    """Shared expert: out (+)= w2 bf16(silu(w1 x) * (w3 x)).  w1, w3 [Fs, D]
    and w2 [D, Fs] bf16 bit patterns (16-bit device tensors), x [T, D] bf16
    bits, out [T, D] float32, ws a uint8 device tensor of at least
    ds4moe_shared_workspace_bytes(D, Fs, T) bytes."""
    Fs, D = w1.shape
    T = x.shape[0]
    _check(lib().ds4moe_shared_ffn(_ptr(w1), _ptr(w3), _ptr(w2), D, Fs, _ptr(x), T, _ptr(out), int(bool(accumulate)),
                                   _ptr(ws), ws.numel(), _stream(stream)), "ds4moe_shared_ffn")


def ds4moe_gather_rows(x, rows, dst, stream=None):
    """dst[j] = x[rows[j]]: x, dst bf16-bit device tensors [., D]; rows int32 [n]."""
    _check(lib().ds4moe_gather_rows(_ptr(x), _ptr(rows), rows.numel(), x.shape[1], _ptr(dst), _stream(stream)),
           "ds4moe_gather_rows")


def ds4moe_combine_pairs(y, pos, w, out, stream=None):
    """out[t] = sum_i w[t, i] * y[pos[t, i]] in rank order (pos < 0 skipped):
    y float32 [., D], pos int32 [T, k], w float32 [T, k], out float32 [T, D]."""
    T, k = pos.shape
    _check(lib().ds4moe_combine_pairs(_ptr(y), _ptr(pos), _ptr(w), T, k, out.shape[1], _ptr(out), _stream(stream)),
           "ds4moe_combine_pairs")


# ds4moe_span_kernel order
SPAN_KERNELS = ("route", "ffn_t1", "ffn_t1r", "gate_up_mma", "down_mma", "gate_up_tc", "down_tc",
                "shared_gate_up_tc", "shared_down_tc", "gate_up_t1", "down_t1")


def ds4moe_profile_span(on: int = -1) -> dict:
    """{kernel: (total_ns, launches)} of the device-side span record so far
    (kernels with no recorded launch omitted); on = 1 / 0 then clears it and
    switches recording on / off (-1: read only)."""
    n = len(SPAN_KERNELS)
    ns, cnt = (ctypes.c_double * n)(), (ctypes.c_int64 * n)()
    _check(lib().ds4moe_profile_span(int(on), ns, cnt), "ds4moe_profile_span")
    return {k: (ns[i], cnt[i]) for i, k in enumerate(SPAN_KERNELS) if cnt[i]}


def ds4moe_quantize_f32(qtype, x, importance, out, ws, cols=None, stream=None):
    """x: float32 device tensor (rows of `cols` values; the last dimension by
    default), importance: None or `cols` float32 weights, out: uint8 device
    tensor of the block bytes, ws: workspace (device status word)."""
    n = x.numel()
    c = int(cols if cols is not None else (x.shape[-1] if x.dim() else n))
    _check(lib().ds4moe_quantize_f32(qtype, _ptr(x), _ptr(importance), n, c, _ptr(out),
                                     out.numel() * out.element_size(), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)), "ds4moe_quantize_f32")


def ds4moe_workspace_bytes(layer: Layer, T: int, k: int, prefill: bool = False) -> int:
    return int(lib().ds4moe_workspace_bytes(ctypes.byref(layer), T, k, int(bool(prefill))))


def ds4moe_prefill_small_pairs(layer: Layer) -> int:
    return int(lib().ds4moe_prefill_small_pairs(ctypes.byref(layer)))


def ds4moe_workspace_init(ws, stream=None):
    _check(lib().ds4moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "ds4moe_workspace_init")


def ds4moe_route_topk_select_bias(x, Wr, bias, k, idx, w, logits, ws, stream=None):
    T, D = x.shape
    E = Wr.shape[0]
    _check(lib().ds4moe_route_topk_select_bias(_ptr(x), _ptr(Wr), _ptr(bias), T, D, E, k, _ptr(idx), _ptr(w),
                                               _ptr(logits), _ptr(ws), ws.numel() * ws.element_size(),
                                               _stream(stream)), "ds4moe_route_topk_select_bias")


def ds4moe_route_topk(x, Wr, bias, k, idx, w, logits, ws, stream=None):
    T, D = x.shape
    E = Wr.shape[0]
    _check(lib().ds4moe_route_topk(_ptr(x), _ptr(Wr), _ptr(bias), T, D, E, k, _ptr(idx), _ptr(w),
                                   _ptr(logits), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "ds4moe_route_topk")


def ds4moe_ffn_decode(layer: Layer, x, idx, w, out, ws, stream=None):
    T, k = idx.shape
    _check(lib().ds4moe_ffn_decode(ctypes.byref(layer), _ptr(x), _ptr(idx), _ptr(w), T, k, _ptr(out),
                                   _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "ds4moe_ffn_decode")


def ds4moe_ffn_prefill(layer: Layer, x, idx, w, out, ws, stream=None):
    T, k = idx.shape
    _check(lib().ds4moe_ffn_prefill(ctypes.byref(layer), _ptr(x), _ptr(idx), _ptr(w), T, k, _ptr(out),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "ds4moe_ffn_prefill")


def ds4moe_moe_decode(layer: Layer, x, Wr, bias, k, out, idx, w, ws, stream=None):
    """Route + expert FFN + combine of one decode step (writes idx, w, out)."""
    T = x.shape[0]
    _check(lib().ds4moe_moe_decode(ctypes.byref(layer), _ptr(x), _ptr(Wr), _ptr(bias), T, k, _ptr(out), _ptr(idx),
                                   _ptr(w), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "ds4moe_moe_decode")


STACK_RMS_EPS = 1e-6


def ds4moe_residual_norm(x_res, out, x_next, eps=STACK_RMS_EPS, stream=None):
    """x_res += out (fp32; out None: skip), x_next = bf16(x_res / rms(x_res))."""
    T, D = x_res.shape
    _check(lib().ds4moe_residual_norm(_ptr(x_res), _ptr(out), _ptr(x_next), T, D, float(eps), _stream(stream)),
           "ds4moe_residual_norm")


def stack_ldk(T: int, k: int) -> int:
    """Per-layer stride of ds4moe_stack_decode's idx / w outputs."""
    return (T * k + 3) // 4 * 4


def ds4moe_stack_decode(layers, Wr, bias, k, x_res, x_bf16, out, idx, w, ws, eps=STACK_RMS_EPS, stream=None):
    """One decode step through len(layers) layers (x_res updated in place;
    idx / w [n_layers, stack_ldk(T, k)] receive every layer's routing)."""
    n = len(layers)
    T = x_res.shape[0]
    arr = (Layer * n)(*layers)
    wr = (ctypes.c_void_p * n)(*[_ptr(t) for t in Wr])
    bs = None if bias is None else (ctypes.c_void_p * n)(*[_ptr(t) for t in bias])
    _check(lib().ds4moe_stack_decode(arr, wr, bs, n, T, k, float(eps), _ptr(x_res), _ptr(x_bf16), _ptr(out),
                                     _ptr(idx), _ptr(w), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "ds4moe_stack_decode")


def ds4moe_ffn_decode_noalloc(layer: Layer, x, idx, w, out, status_out=None, stream=None):
    """ds4moe_ffn_decode without a workspace: the library's fixed scratch array
    is used instead (see include/ds4moe.h for who needs this and its limits)."""
    T, k = idx.shape
    _check(lib().ds4moe_ffn_decode_noalloc(ctypes.byref(layer), _ptr(x), _ptr(idx), _ptr(w), T, k, _ptr(out),
                                           _ptr(status_out), _stream(stream)), "ds4moe_ffn_decode_noalloc")


def ds4moe_debug_sync_wait(budget_polls: int = 1 << 24, extra_target: int = 0):
    """Fault-injection hook for failure-detection tests: the poll budget and
    target offset of the merged single-token grid's cross-CTA h-ready wait
    (defaults restore normal operation)."""
    _check(lib().ds4moe_debug_sync_wait(int(budget_polls), int(extra_target)), "ds4moe_debug_sync_wait")


def ds4moe_profile_enable(on: bool):
    _check(lib().ds4moe_profile_enable(int(bool(on))), "ds4moe_profile_enable")


def ds4moe_profile_read() -> dict:
    """{kernel name: (total_ms, launches)} since the last ds4moe_profile_enable."""
    L = lib()
    out = {}
    for i in range(L.ds4moe_profile_count()):
        name, ms, n = ctypes.c_char_p(), ctypes.c_double(), ctypes.c_int64()
        _check(L.ds4moe_profile_entry(i, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(n)), "ds4moe_profile_entry")
        out[name.value.decode()] = (ms.value, n.value)
    return out


def ds4moe_stream_status(ws, stream=None) -> int:
    """Synchronizes and returns (and clears) the workspace's device status."""
    return int(lib().ds4moe_stream_status(_ptr(ws), _stream(stream)))
