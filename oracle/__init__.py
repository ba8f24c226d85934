"""CPU oracle for the routed-MoE expert FFN (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``; never by the product package.
The arithmetic lives in ``oracle.c`` (plain C, fp64), whose header lists the
pages each function follows and the readings taken where they are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, EINVAL, EBLOCKER, EUNSUPPORTED = 0, 1, 2, 3
Q4_1, Q2_K, Q4_K = 1, 2, 4
QTYPES = {"q4_1": Q4_1, "q2_k": Q2_K, "q4_k": Q4_K}


def build(force: bool = False) -> str:
    """Compile the oracle in place (gcc -O2, OpenMP, no FP contraction so the
    results are the same on every host architecture)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.orc_block_values.argtypes = [i32]
        lib.orc_block_bytes.argtypes = [i32]
        lib.orc_f16.restype = ctypes.c_double
        lib.orc_f16.argtypes = [ctypes.c_uint16]
        lib.orc_bf16.restype = ctypes.c_double
        lib.orc_bf16.argtypes = [ctypes.c_uint16]
        lib.orc_round_bf16.restype = ctypes.c_uint16
        lib.orc_round_bf16.argtypes = [ctypes.c_double]
        lib.orc_round_bf16_array.argtypes = [p, i64, p]
        lib.orc_rmsnorm_bf16.argtypes = [p, i64, i64, ctypes.c_double, p]
        lib.orc_q41_pack.argtypes = [p, p, p, i64, p]
        lib.orc_q41_unpack.argtypes = [p, i64, p, p, p]
        lib.orc_q41_dequant.argtypes = [p, i64, p]
        lib.orc_q41_reencode.argtypes = [i32, i32, p, p, p, i64, p]
        lib.orc_q2k_pack.argtypes = [p, p, p, p, p, i64, p]
        lib.orc_q2k_unpack.argtypes = [p, i64, p, p, p, p, p]
        lib.orc_q2k_dequant.argtypes = [p, i64, p]
        lib.orc_q2k_to_r16.argtypes = [p, i64, i64, p]
        lib.orc_q2k_from_r16.argtypes = [p, i64, i64, p]
        lib.orc_r16_dequant.argtypes = [p, i64, i64, p]
        lib.orc_dequant.argtypes = [i32, p, i64, p]
        lib.orc_router_logits.argtypes = [p, p, p, i32, i32, i32, p]
        lib.orc_topk_softmax.argtypes = [p, i32, i32, i32, p, p]
        lib.orc_matvec_rows.argtypes = [i32, p, i32, i32, i32, i32, p, p]
        lib.orc_expert_ffn.argtypes = [i32, i32, i32, p, i32, p, i32, p, i32, p, p, p, p, p]
        lib.orc_moe_ffn.argtypes = [i32, i32, i32, i32, p, i32, p, i32, p, p, p, p, i32, i32, p]
        lib.orc_topk_softmax_selbias.argtypes = [p, p, i32, i32, i32, p, p]
        lib.orc_q4k_pack.argtypes = [p, p, p, p, p, i64, p]
        lib.orc_q4k_unpack.argtypes = [p, i64, p, p, p, p, p]
        lib.orc_q4k_dequant.argtypes = [p, i64, p]
        lib.orc_f32_to_f16.restype = ctypes.c_uint16
        lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
        lib.orc_quantize_f32.argtypes = [i32, p, p, i64, i64, p]
        lib.orc_weighted_sq_error.restype = ctypes.c_double
        lib.orc_weighted_sq_error.argtypes = [i32, p, p, i64, i64, p]
        lib.orc_shared_ffn.argtypes = [i32, i32, p, p, p, i32, p, p, p]
        _lib = lib
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return a.ctypes.data if a is not None else None


class OracleError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: oracle status {status}")
        self.status = status


def block_values(qtype: int) -> int:
    return _L().orc_block_values(qtype)


def block_bytes(qtype: int) -> int:
    return _L().orc_block_bytes(qtype)


def f16(h: int) -> float:
    return _L().orc_f16(h)


def bf16(b: int) -> float:
    return _L().orc_bf16(b)


def round_bf16(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _L().orc_round_bf16_array(v.ctypes.data, v.size, out.ctypes.data)
    return out


def rmsnorm_bf16(x_res, eps: float) -> np.ndarray:
    """Layer input of the decode stack: bf16 bits of x / sqrt(mean(x^2) + eps)
    per row of the fp32 residual x_res [T, D] (fp64 arithmetic)."""
    x = _c(x_res, np.float32)
    T, D = x.shape
    out = np.empty((T, D), dtype=np.uint16)
    _L().orc_rmsnorm_bf16(x.ctypes.data, T, D, float(eps), out.ctypes.data)
    return out


def bf16_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a plain bit shift)."""
    b = _c(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ formats
def q41_pack(codes, d, m) -> np.ndarray:
    codes, d, m = _c(codes, np.uint8), _c(d, np.uint16), _c(m, np.uint16)
    nb = codes.size // 32
    out = np.zeros(nb * 20, dtype=np.uint8)
    st = _L().orc_q41_pack(codes.ctypes.data, d.ctypes.data, m.ctypes.data, nb, out.ctypes.data)
    if st:
        raise OracleError(st, "q41_pack")
    return out


def q41_unpack(blocks):
    blocks = _c(blocks, np.uint8)
    nb = blocks.size // 20
    codes = np.empty(nb * 32, np.uint8)
    d = np.empty(nb, np.uint16)
    m = np.empty(nb, np.uint16)
    _L().orc_q41_unpack(blocks.ctypes.data, nb, codes.ctypes.data, d.ctypes.data, m.ctypes.data)
    return codes, d, m


def q41_reencode(bits: int, group: int, codes, scale, mins):
    """Returns (status, blocks)."""
    codes, scale, mins = _c(codes, np.uint8), _c(scale, np.uint16), _c(mins, np.uint16)
    n = codes.size
    out = np.zeros(n // 32 * 20, dtype=np.uint8)
    st = _L().orc_q41_reencode(bits, group, codes.ctypes.data, scale.ctypes.data,
                               mins.ctypes.data, n, out.ctypes.data)
    return st, out


def q2k_pack(codes, sc, mn, d, dmin) -> np.ndarray:
    codes, sc, mn = _c(codes, np.uint8), _c(sc, np.uint8), _c(mn, np.uint8)
    d, dmin = _c(d, np.uint16), _c(dmin, np.uint16)
    nb = codes.size // 256
    out = np.zeros(nb * 84, dtype=np.uint8)
    st = _L().orc_q2k_pack(codes.ctypes.data, sc.ctypes.data, mn.ctypes.data, d.ctypes.data,
                           dmin.ctypes.data, nb, out.ctypes.data)
    if st:
        raise OracleError(st, "q2k_pack")
    return out


def q2k_unpack(blocks):
    blocks = _c(blocks, np.uint8)
    nb = blocks.size // 84
    codes = np.empty(nb * 256, np.uint8)
    sc = np.empty(nb * 16, np.uint8)
    mn = np.empty(nb * 16, np.uint8)
    d = np.empty(nb, np.uint16)
    dmin = np.empty(nb, np.uint16)
    _L().orc_q2k_unpack(blocks.ctypes.data, nb, codes.ctypes.data, sc.ctypes.data, mn.ctypes.data,
                        d.ctypes.data, dmin.ctypes.data)
    return codes, sc, mn, d, dmin


def q2k_to_r16(blocks, rows: int, cols: int) -> np.ndarray:
    """Plain Q2_K matrix bytes (rows x cols values) -> the 16-row tile order."""
    src = _c(blocks, np.uint8)
    out = np.zeros(src.size, dtype=np.uint8)
    st = _L().orc_q2k_to_r16(_ptr(src), rows, cols, _ptr(out))
    if st != OK:
        raise ValueError(f"q2k_to_r16: status {st}")
    return out


def q2k_from_r16(blocks, rows: int, cols: int) -> np.ndarray:
    """The inverse of q2k_to_r16."""
    src = _c(blocks, np.uint8)
    out = np.zeros(src.size, dtype=np.uint8)
    st = _L().orc_q2k_from_r16(_ptr(src), rows, cols, _ptr(out))
    if st != OK:
        raise ValueError(f"q2k_from_r16: status {st}")
    return out


def r16_dequant(blocks, rows: int, cols: int) -> np.ndarray:
    """fp32 values [rows, cols] of a tile-order matrix, read in place."""
    src = _c(blocks, np.uint8)
    out = np.zeros((rows, cols), dtype=np.float32)
    st = _L().orc_r16_dequant(_ptr(src), rows, cols, _ptr(out))
    if st != OK:
        raise ValueError(f"r16_dequant: status {st}")
    return out


def dequant(qtype: int, blocks, n_values: int) -> np.ndarray:
    blocks = _c(blocks, np.uint8)
    out = np.empty(n_values, dtype=np.float32)
    st = _L().orc_dequant(qtype, blocks.ctypes.data, n_values, out.ctypes.data)
    if st:
        raise OracleError(st, "dequant")
    return out


def pack_fields(f) -> np.ndarray:
    """Block bytes of a ``synth.Fields`` matrix (Q4_1 via the lossless
    re-encode with the fields' explicit bits/group; Q2_K / Q4_K via the
    packers)."""
    if f.qtype == "q4_1":
        st, out = q41_reencode(f.bits, f.group, f.codes, f.scale, f.minv)
        if st:
            raise OracleError(st, "q41_reencode")
        return out
    if f.qtype == "q4_k":
        return q4k_pack(f.codes, f.sc, f.mn, f.scale, f.minv)
    return q2k_pack(f.codes, f.sc, f.mn, f.scale, f.minv)


# ------------------------------------------------------------------ routing
def router_logits(x_bf16, Wr, bias=None) -> np.ndarray:
    x, Wr = _c(x_bf16, np.uint16), _c(Wr, np.float32)
    T, D = x.shape
    E = Wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _L().orc_router_logits(x.ctypes.data, Wr.ctypes.data, _ptr(b), T, D, E, out.ctypes.data)
    return out


def topk_softmax(logits, k: int):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _L().orc_topk_softmax(logits.ctypes.data, T, E, k, idx.ctypes.data, w.ctypes.data)
    return idx, w


def route(x_bf16, Wr, bias, k: int):
    logits = router_logits(x_bf16, Wr, bias)
    idx, w = topk_softmax(logits, k)
    return idx, w, logits


# ---------------------------------------------------------------------- FFN
def matvec_rows(qtype, mat, rows, cols, row0, nrows, vec) -> np.ndarray:
    """Rows [row0, row0+nrows) of W @ vec for one [rows x cols] block matrix."""
    mat = _c(mat, np.uint8)
    vec = _c(vec, np.float64)
    out = np.empty(nrows, np.float64)
    st = _L().orc_matvec_rows(qtype, mat.ctypes.data, rows, cols, row0, nrows, vec.ctypes.data, out.ctypes.data)
    if st:
        raise OracleError(st, "matvec_rows")
    return out


def expert_ffn(D, F, qg, gate, qu, up, qd, down, e, x_bf16):
    """One (token, expert): returns (y fp64 [D], h bf16 [F], g fp64 [F], u fp64 [F])."""
    x = _c(x_bf16, np.uint16)
    gate, up, down = _c(gate, np.uint8), _c(up, np.uint8), _c(down, np.uint8)
    y = np.empty(D, np.float64)
    h = np.empty(F, np.uint16)
    g = np.empty(F, np.float64)
    u = np.empty(F, np.float64)
    st = _L().orc_expert_ffn(D, F, qg, gate.ctypes.data, qu, up.ctypes.data, qd, down.ctypes.data, e,
                             x.ctypes.data, y.ctypes.data, h.ctypes.data, g.ctypes.data, u.ctypes.data)
    if st:
        raise OracleError(st, "expert_ffn")
    return y, h, g, u


def moe_ffn(D, F, E, qg, gate, qu, up, qd, down, x_bf16, idx, w) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    idx, w = _c(idx, np.int32), _c(w, np.float32)
    T, k = idx.shape
    gate, up, down = _c(gate, np.uint8), _c(up, np.uint8), _c(down, np.uint8)
    out = np.empty((T, D), np.float32)
    st = _L().orc_moe_ffn(D, F, E, qg, gate.ctypes.data, qu, up.ctypes.data, qd, down.ctypes.data,
                          x.ctypes.data, idx.ctypes.data, w.ctypes.data, T, k, out.ctypes.data)
    if st:
        raise OracleError(st, "moe_ffn")
    return out


def shared_ffn(w1, w3, w2, x_bf16, base=None) -> np.ndarray:
    """Shared expert ([DS4-2]: kept unquantised): bf16 w1, w3 [Fs, D] and
    w2 [D, Fs] (bit patterns), x bf16 [T, D]; returns fp32 [T, D] =
    base + w2 bf16(silu(w1 x) * (w3 x)), one rounding (base may be None)."""
    w1, w3, w2 = _c(w1, np.uint16), _c(w3, np.uint16), _c(w2, np.uint16)
    x = _c(x_bf16, np.uint16)
    Fs, D = w1.shape
    if w3.shape != (Fs, D) or w2.shape != (D, Fs) or x.ndim != 2 or x.shape[1] != D:
        raise ValueError("shared_ffn: shapes")
    T = x.shape[0]
    b = None if base is None else _c(base, np.float32)
    if b is not None and b.shape != (T, D):
        raise ValueError("shared_ffn: base shape")
    out = np.empty((T, D), np.float32)
    st = _L().orc_shared_ffn(D, Fs, _ptr(w1), _ptr(w3), _ptr(w2), T, _ptr(x), _ptr(b), out.ctypes.data)
    if st:
        raise OracleError(st, "shared_ffn")
    return out


# ------------------------------------------------------ float-input quantizer
def f32_to_f16(v) -> np.ndarray:
    """binary32 -> binary16 bit patterns, round to nearest even (own encoder)."""
    v = np.asarray(v, dtype=np.float32).ravel()
    return np.array([_L().orc_f32_to_f16(float(a)) for a in v], dtype=np.uint16)


def quantize_f32(qtype: int, x, importance=None, cols: int | None = None) -> np.ndarray:
    """Float-input quantizer ([DS4-2] Q2_K block writer reading; Q4_1 likewise):
    per-block (Q4_1) or per-sub-block (Q2_K) min / max scales, nearest codes,
    and with per-column `importance` a small search over neighbouring scales
    that minimises the weighted squared error.  Returns the block bytes."""
    x = _c(x, np.float32).ravel()
    n = x.size
    bv, bb = block_values(qtype), block_bytes(qtype)
    out = np.zeros(n // bv * bb if bv else 0, dtype=np.uint8)
    imp = None if importance is None else _c(importance, np.float32).ravel()
    c = cols if cols is not None else (imp.size if imp is not None else n)
    st = _L().orc_quantize_f32(qtype, _ptr(x), _ptr(imp), n, c, _ptr(out))
    if st != OK:
        raise OracleError(st, "quantize_f32")
    return out


def weighted_sq_error(qtype: int, x, importance, cols: int, blocks) -> float:
    """sum over values of importance[col] * (x - dequant)^2 (unit weights when
    importance is None), in double."""
    x = _c(x, np.float32).ravel()
    imp = None if importance is None else _c(importance, np.float32).ravel()
    return _L().orc_weighted_sq_error(qtype, _ptr(x), _ptr(imp), x.size, cols, _ptr(_c(blocks, np.uint8)))


# ----------------------------------------------- routing: selection-only bias
def route_select_bias(x_bf16, Wr, bias, k: int):
    """Experts ranked by the biased logit, weights = softmax of the selected
    experts' unbiased logits (bias used for selection only).  Returns
    (idx, w, unbiased logits, biased logits)."""
    lu = router_logits(x_bf16, Wr, None)
    lb = router_logits(x_bf16, Wr, bias)
    T, E = lu.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _L().orc_topk_softmax_selbias(_ptr(_c(lb, np.float32)), _ptr(_c(lu, np.float32)), T, E, k, _ptr(idx), _ptr(w))
    return idx, w, lu, lb


# ------------------------------------------------------------------- Q4_K
def q4k_pack(codes, sc, mn, d, dmin) -> np.ndarray:
    """codes: 256 per block (0..15); sc, mn: 8 per block (0..63); d, dmin:
    binary16 bit patterns per block."""
    codes, sc, mn = _c(codes, np.uint8), _c(sc, np.uint8), _c(mn, np.uint8)
    d, dmin = _c(d, np.uint16), _c(dmin, np.uint16)
    nb = codes.size // 256
    out = np.zeros(nb * 144, dtype=np.uint8)
    st = _L().orc_q4k_pack(_ptr(codes), _ptr(sc), _ptr(mn), _ptr(d), _ptr(dmin), nb, _ptr(out))
    if st:
        raise OracleError(st, "q4k_pack")
    return out


def q4k_unpack(blocks):
    blocks = _c(blocks, np.uint8)
    nb = blocks.size // 144
    codes = np.empty(nb * 256, np.uint8)
    sc = np.empty(nb * 8, np.uint8)
    mn = np.empty(nb * 8, np.uint8)
    d = np.empty(nb, np.uint16)
    dmin = np.empty(nb, np.uint16)
    _L().orc_q4k_unpack(_ptr(blocks), nb, _ptr(codes), _ptr(sc), _ptr(mn), _ptr(d), _ptr(dmin))
    return codes, sc, mn, d, dmin
