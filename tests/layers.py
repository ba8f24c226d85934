"""Test-side assembly of synthetic MoE layers: synth fields -> block bytes
packed by the oracle's packer.  Used by the oracle pins and, as the input
source, by the GPU parity tests (the CUDA path only ever receives bytes made
here, never the other way round)."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
import synth


@dataclass
class Layer:
    w: synth.Workload
    layer: int
    gate: np.ndarray   # uint8, experts-major block bytes
    up: np.ndarray
    down: np.ndarray
    Wr: np.ndarray     # fp32 [E, D]
    bias: np.ndarray | None

    @property
    def qg(self):
        return oracle.QTYPES[self.w.gate.qtype]

    @property
    def qu(self):
        return oracle.QTYPES[self.w.up.qtype]

    @property
    def qd(self):
        return oracle.QTYPES[self.w.down.qtype]


def expert_matrix(w: synth.Workload, layer: int, tensor: int, e: int) -> np.ndarray:
    return oracle.pack_fields(synth.matrix_fields(w, layer, tensor, e))


def build_layer(w: synth.Workload, layer: int = 0, experts=None) -> Layer:
    """All experts (or the listed ones; unlisted experts are left as zero
    bytes) of one layer."""
    E = w.n_expert
    experts = range(E) if experts is None else experts
    mats = {}
    for t in (synth.T_GATE, synth.T_UP, synth.T_DOWN):
        rows, cols = synth.matrix_shape(w, t)
        q = oracle.QTYPES[synth.recipe(w, t).qtype]
        per = rows * (cols // oracle.block_values(q)) * oracle.block_bytes(q)
        buf = np.zeros(E * per, np.uint8)
        for e in experts:
            buf[e * per:(e + 1) * per] = expert_matrix(w, layer, t, e)
        mats[t] = buf
    Wr, b = synth.router(w, layer)
    return Layer(w, layer, mats[synth.T_GATE], mats[synth.T_UP], mats[synth.T_DOWN], Wr, b)


def oracle_forward(L: Layer, x_bf16: np.ndarray):
    """Route + FFN on the oracle. Returns (out fp32 [T, D], idx, w, logits)."""
    w = L.w
    idx, wt, logits = oracle.route(x_bf16, L.Wr, L.bias, w.k)
    out = oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down,
                         x_bf16, idx, wt)
    return out, idx, wt, logits


# ---------------------------------------------------------------- GPU side
def to_device(L: Layer):
    """Upload a host layer's block bytes (made by the oracle's packer) for
    the CUDA path."""
    import bit_quantized_moe_q2_gb300 as M
    from bit_quantized_moe_q2_gb300.device import DeviceLayer
    w = L.w
    return DeviceLayer.from_host(w.d_model, w.d_ff, w.n_expert, M.QTYPES[w.gate.qtype], M.QTYPES[w.up.qtype],
                                 M.QTYPES[w.down.qtype], L.gate, L.up, L.down)


_cache = {}


def cached_layer(w: synth.Workload, layer: int = 0):
    """(host Layer, DeviceLayer) built once per test session."""
    key = (w, layer)
    if key not in _cache:
        L = build_layer(w, layer)
        _cache.clear()          # keep at most one full layer resident
        _cache[key] = (L, to_device(L))
    return _cache[key]
