"""Seeded synthetic workloads for the routed-MoE expert FFN.

This module is shared by the tests (oracle side and CUDA side) and by
``bench.py``.  It generates the raw fields of a workload -- integer codes,
4-bit sub-block scales and mins, fp16 scale patterns, bf16 activations, fp32
router weights and biases -- and holds none of the method's arithmetic: no
block packing, no dequantisation, no routing, no FFN.  The C core
(``synth.c``) is a counter-based SplitMix64 stream, so any element can be
regenerated on demand.

Workload recipes (shapes and value distributions) follow the five workloads
the library is measured on: a tiny 8-expert layer, a Flash-shaped 256-expert
layer at decode batch 1 and 64, a 4096-token prefill chunk with a skewing
router bias, and a 43-layer all-Q2_K decode stack.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

# Stream identifiers (tensor, field) -- part of the workload definition.
T_ROUTER, T_BIAS, T_X, T_GATE, T_UP, T_DOWN = 0, 1, 2, 3, 4, 5
F_CODES, F_SC, F_MN, F_D, F_DMIN = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile the generator core (plain C, OpenMP) in place."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_u64.restype = u64
        lib.synth_u64.argtypes = [u64, u64]
        lib.synth_key.restype = u64
        lib.synth_key.argtypes = [u64] * 5
        lib.synth_normal.restype = ctypes.c_double
        lib.synth_normal.argtypes = [u64, u64]
        lib.synth_codes.argtypes = [u64, i64, i64, ctypes.c_int, p]
        lib.synth_abs_normal_f16.argtypes = [u64, i64, i64, ctypes.c_double, p]
        lib.synth_normal_bf16.argtypes = [u64, i64, i64, ctypes.c_double, p]
        lib.synth_normal_f32.argtypes = [u64, i64, i64, ctypes.c_double, p]
        lib.synth_f16_scale_pow2.argtypes = [p, i64, ctypes.c_double, p]
        lib.synth_round_f16.restype = ctypes.c_uint16
        lib.synth_round_f16.argtypes = [ctypes.c_double]
        lib.synth_round_bf16.restype = ctypes.c_uint16
        lib.synth_round_bf16.argtypes = [ctypes.c_double]
        _lib = lib
    return _lib


def key(seed: int, layer: int, tensor: int, expert: int, fld: int) -> int:
    return int(_L().synth_key(seed, layer, tensor, expert, fld))


def u64(k: int, i: int) -> int:
    return int(_L().synth_u64(k, i))


def codes(k: int, n: int, bits: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    if n:
        _L().synth_codes(k, start, n, bits, out.ctypes.data)
    return out


def abs_normal_f16(k: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    if n:
        _L().synth_abs_normal_f16(k, start, n, sigma, out.ctypes.data)
    return out


def normal_bf16(k: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    if n:
        _L().synth_normal_bf16(k, start, n, sigma, out.ctypes.data)
    return out


def normal_f32(k: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    if n:
        _L().synth_normal_f32(k, start, n, sigma, out.ctypes.data)
    return out


def f16_scale_pow2(h: np.ndarray, mult: float) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty_like(h)
    if h.size:
        _L().synth_f16_scale_pow2(h.ctypes.data, h.size, mult, out.ctypes.data)
    return out


# --------------------------------------------------------------------------
# Workload recipes
# --------------------------------------------------------------------------

Q4_1, Q2_K, Q4_K = "q4_1", "q2_k", "q4_k"


@dataclass(frozen=True)
class MatrixRecipe:
    """How one expert matrix is drawn.

    qtype   block format the matrix is stored in.
    bits    code width of the source codes (Q4_1 sources: 3 or 4; Q2_K: 2).
    group   values sharing one (scale, min) pair in the source (Q4_1: 32;
            Q2_K: 256 for d/dmin, with 4-bit sc/mn per 16 values).
    sigma   std-dev of the |N(0, sigma)| fp16 scales.
    min_mult  Q4_1 sources: min = min_mult * scale (power of two, exact).
    """
    qtype: str
    bits: int
    group: int
    sigma: float
    min_mult: float = 0.0


Q41_4BIT = MatrixRecipe(Q4_1, 4, 32, 0.01, -8.0)   # codes U[0,15], m = -8 d
Q41_3BIT = MatrixRecipe(Q4_1, 3, 32, 0.01, -4.0)   # codes U[0,7], min = -4 scale
Q2K = MatrixRecipe(Q2_K, 2, 256, 0.002)             # codes U[0,3], sc/mn U[0,15]
Q4K = MatrixRecipe(Q4_K, 4, 256, 0.0002)            # codes U[0,15], sc/mn U[0,63] per 32 values


@dataclass(frozen=True)
class Workload:
    name: str
    d_model: int
    d_ff: int
    n_expert: int
    k: int
    T: int
    seed: int
    gate: MatrixRecipe
    up: MatrixRecipe
    down: MatrixRecipe
    router_sigma: float = 0.02
    bias_sigma: float = 0.0      # 0: no router bias
    n_layers: int = 1
    path: str = "decode"

    def replace(self, **kw) -> "Workload":
        d = {f: getattr(self, f) for f in self.__dataclass_fields__}
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    0: Workload("tiny-moe-e8-top2-t4", 4096, 2048, 8, 2, 4, 0, Q41_4BIT, Q41_4BIT, Q2K),
    1: Workload("flash-layer-decode-t1-q2k", 4096, 2048, 256, 6, 1, 1, Q2K, Q2K, Q2K),
    2: Workload("flash-layer-decode-t64-q41-q2k", 4096, 2048, 256, 6, 64, 2, Q41_3BIT, Q41_3BIT, Q2K),
    3: Workload("flash-layer-prefill-t4096-q41-q2k", 4096, 2048, 256, 6, 4096, 3, Q41_4BIT, Q41_4BIT, Q2K,
                bias_sigma=1.0, path="prefill"),
    4: Workload("flash-stack43-decode-q2k", 4096, 2048, 256, 6, 1, 4, Q2K, Q2K, Q2K, n_layers=43),
    # the mixed recipe's Q4_K routed experts (its last six layers)
    5: Workload("flash-layer-decode-t1-q4k", 4096, 2048, 256, 6, 1, 5, Q4K, Q4K, Q4K),
}


def matrix_shape(w: Workload, tensor: int):
    """(rows, cols) of an expert matrix: rows = output features, blocks run
    along cols (the input / contraction axis)."""
    if tensor in (T_GATE, T_UP):
        return w.d_ff, w.d_model
    return w.d_model, w.d_ff


def recipe(w: Workload, tensor: int) -> MatrixRecipe:
    return {T_GATE: w.gate, T_UP: w.up, T_DOWN: w.down}[tensor]


@dataclass
class Fields:
    """Raw fields of one matrix (row-major values, rows x cols)."""
    qtype: str
    rows: int
    cols: int
    codes: np.ndarray                 # uint8 [rows*cols]
    bits: int
    group: int
    scale: np.ndarray                 # uint16 fp16: Q4_1 per group; Q2_K d per 256
    minv: np.ndarray                  # uint16 fp16: Q4_1 min per group; Q2_K dmin per 256
    sc: np.ndarray | None = None      # uint8 [n/16] (Q2_K) or [n/32] 6-bit (Q4_K)
    mn: np.ndarray | None = None      # uint8 [n/16] (Q2_K) or [n/32] 6-bit (Q4_K)


def matrix_fields(w: Workload, layer: int, tensor: int, expert: int,
                  row0: int = 0, nrows: int | None = None) -> Fields:
    """Fields of rows [row0, row0+nrows) of one expert matrix."""
    rows, cols = matrix_shape(w, tensor)
    nrows = rows - row0 if nrows is None else nrows
    r = recipe(w, tensor)
    s = w.seed
    v0, n = row0 * cols, nrows * cols
    c = codes(key(s, layer, tensor, expert, F_CODES), n, r.bits, start=v0)
    if r.qtype == Q2_K:
        sc = codes(key(s, layer, tensor, expert, F_SC), n // 16, 4, start=v0 // 16)
        mn = codes(key(s, layer, tensor, expert, F_MN), n // 16, 4, start=v0 // 16)
        d = abs_normal_f16(key(s, layer, tensor, expert, F_D), n // 256, r.sigma, start=v0 // 256)
        dm = abs_normal_f16(key(s, layer, tensor, expert, F_DMIN), n // 256, r.sigma, start=v0 // 256)
        return Fields(Q2_K, nrows, cols, c, 2, 256, d, dm, sc, mn)
    if r.qtype == Q4_K:
        sc = codes(key(s, layer, tensor, expert, F_SC), n // 32, 6, start=v0 // 32)
        mn = codes(key(s, layer, tensor, expert, F_MN), n // 32, 6, start=v0 // 32)
        d = abs_normal_f16(key(s, layer, tensor, expert, F_D), n // 256, r.sigma, start=v0 // 256)
        dm = abs_normal_f16(key(s, layer, tensor, expert, F_DMIN), n // 256, r.sigma, start=v0 // 256)
        return Fields(Q4_K, nrows, cols, c, 4, 256, d, dm, sc, mn)
    g = r.group
    sc16 = abs_normal_f16(key(s, layer, tensor, expert, F_D), n // g, r.sigma, start=v0 // g)
    mn16 = f16_scale_pow2(sc16, r.min_mult)
    return Fields(Q4_1, nrows, cols, c, r.bits, g, sc16, mn16)


def router(w: Workload, layer: int = 0):
    """Router weight fp32 [E, d_model] ~ N(0, router_sigma) and optional bias fp32 [E]."""
    W = normal_f32(key(w.seed, layer, T_ROUTER, 0, 0), w.n_expert * w.d_model, w.router_sigma)
    b = None
    if w.bias_sigma:
        b = normal_f32(key(w.seed, layer, T_BIAS, 0, 0), w.n_expert, w.bias_sigma)
    return W.reshape(w.n_expert, w.d_model), b


def activations(w: Workload, T: int | None = None, batch: int = 0) -> np.ndarray:
    """x bf16 bit patterns [T, d_model] ~ N(0, 1); `batch` selects an
    independent draw (used to give every timed step fresh tokens)."""
    T = w.T if T is None else T
    x = normal_bf16(key(w.seed, batch, T_X, 0, 0), T * w.d_model, 1.0)
    return x.reshape(T, w.d_model)
