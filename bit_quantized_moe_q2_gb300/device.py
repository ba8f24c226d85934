"""Device-side holders used by callers of the binding: a routed-MoE layer's
expert weights and the shared workspace, as PyTorch CUDA tensors."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import (DS4MOE_OK, Ds4moeError, Layer, block_bytes, block_values, ds4moe_stream_status,
               ds4moe_workspace_bytes, ds4moe_workspace_init, make_layer)


def matrix_bytes(qtype: int, rows: int, cols: int) -> int:
    return rows * (cols // block_values(qtype)) * block_bytes(qtype)


@dataclass
class DeviceLayer:
    d_model: int
    d_ff: int
    n_expert: int
    q_gate: int
    q_up: int
    q_down: int
    gate: "object"   # torch uint8 cuda tensors, experts-major block bytes
    up: "object"
    down: "object"

    @classmethod
    def empty(cls, d_model, d_ff, n_expert, q_gate, q_up, q_down, device="cuda"):
        import torch
        g = torch.empty(n_expert * matrix_bytes(q_gate, d_ff, d_model), dtype=torch.uint8, device=device)
        u = torch.empty(n_expert * matrix_bytes(q_up, d_ff, d_model), dtype=torch.uint8, device=device)
        d = torch.empty(n_expert * matrix_bytes(q_down, d_model, d_ff), dtype=torch.uint8, device=device)
        return cls(d_model, d_ff, n_expert, q_gate, q_up, q_down, g, u, d)

    @classmethod
    def from_host(cls, d_model, d_ff, n_expert, q_gate, q_up, q_down, gate, up, down, device="cuda"):
        import torch
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(device)
        return cls(d_model, d_ff, n_expert, q_gate, q_up, q_down, t(gate), t(up), t(down))

    def expert_slice(self, tensor: str, e: int):
        """View of expert e's bytes of 'gate' | 'up' | 'down'."""
        buf = getattr(self, tensor)
        per = buf.numel() // self.n_expert
        return buf[e * per:(e + 1) * per]

    @property
    def abi(self) -> Layer:
        return make_layer(self.d_model, self.d_ff, self.n_expert, self.q_gate, self.q_up, self.q_down,
                          self.gate, self.up, self.down)

    def repacked_r16(self) -> "DeviceLayer":
        """A copy of an all-Q2_K layer with every matrix in the 16-row tile
        order (ds4moe_repack), for the single-token decode kernel."""
        import torch
        from . import DS4MOE_Q2_K, DS4MOE_Q2_K_R16, ds4moe_repack
        assert self.q_gate == self.q_up == self.q_down == DS4MOE_Q2_K, "repacking takes Q2_K matrices"
        out = {}
        for name, rows, cols in (("gate", self.d_ff, self.d_model), ("up", self.d_ff, self.d_model),
                                 ("down", self.d_model, self.d_ff)):
            src = getattr(self, name)
            dst = torch.empty_like(src)
            ds4moe_repack(DS4MOE_Q2_K, DS4MOE_Q2_K_R16, src, self.n_expert * rows, cols, dst)
            out[name] = dst
        return DeviceLayer(self.d_model, self.d_ff, self.n_expert, DS4MOE_Q2_K_R16, DS4MOE_Q2_K_R16,
                           DS4MOE_Q2_K_R16, out["gate"], out["up"], out["down"])

    def weight_bytes_per_expert(self) -> int:
        return (matrix_bytes(self.q_gate, self.d_ff, self.d_model) + matrix_bytes(self.q_up, self.d_ff, self.d_model)
                + matrix_bytes(self.q_down, self.d_model, self.d_ff))


def workspace(layer: DeviceLayer, T: int, k: int, prefill: bool = False, device="cuda"):
    """Allocate and initialise the workspace for route + FFN of T tokens."""
    import torch
    n = ds4moe_workspace_bytes(layer.abi, T, k, prefill)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    ds4moe_workspace_init(ws)
    return ws


def check_status(ws, stream=None):
    st = ds4moe_stream_status(ws, stream)
    if st != DS4MOE_OK:
        raise Ds4moeError(st, "device status")
