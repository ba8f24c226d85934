"""Expert parallelism for one routed-MoE layer across R ranks.

The experts of a layer are split into R contiguous ranges: rank r owns
experts [r E / R, (r + 1) E / R) and holds only their weights.  Every rank
keeps its own tokens.  One layer on rank r:

  1. route its tokens (top-k of E, softmax over the selected);
  2. dispatch: the (token, slot) pairs, ordered by owner rank (stable, so
     pairs keep token order within a destination), send their activation
     rows and local expert ids to the owners (all-to-all, counts first);
  3. the owner runs its experts on the rows it received, one expert per row
     with weight 1 (the FFN entry points with k = 1);
  4. the outputs go back by the reverse all-to-all;
  5. combine on the token's rank: out[t] = sum_i w[t, i] y[t, i] in rank
     order i, pairs whose expert id is out of range skipped.

The pages' engine splits a model across machines by layer slices ("【#6】
ds4.c 분석하기"); this is the expert-wise split of the same layer, its
exchange the all-to-all above.  The arithmetic stays in the backend: on a
GPU the library's kernels (`DeviceBackend`); the exchange goes through
`torch.distributed` (NCCL across GPUs, gloo on CPU) or, for R ranks emulated
in one process, through `run_local_ranks`, which moves the buffers between
the emulated ranks directly (no kernel ever waits on another rank).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def expert_ranges(E: int, R: int):
    """[(first, last + 1)] of the experts each rank owns."""
    if R < 1 or E % R:
        raise ValueError(f"{E} experts do not split evenly over {R} ranks")
    n = E // R
    return [(r * n, (r + 1) * n) for r in range(R)]


@dataclass
class Dispatch:
    """Plan of one rank's pairs: the pair indices p = t k + i in send order,
    the owner of each, per-destination counts, and the local expert id of
    each sent pair on its owner."""
    order: np.ndarray        # int64 [n_send]: pair index in send order
    counts: np.ndarray       # int64 [R]
    local_ids: np.ndarray    # int32 [n_send]
    pos: np.ndarray          # int32 [T, k]: row of each pair in the send (= return) order, -1 if skipped


def plan_dispatch(idx: np.ndarray, E: int, R: int) -> Dispatch:
    """Host-side plan from the routing indices idx [T, k] (int32)."""
    T, k = idx.shape
    per = E // R
    flat = idx.reshape(-1).astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    owner = np.where(valid, flat // per, R)           # invalid pairs sort last and are not sent
    order = np.argsort(owner, kind="stable")
    order = order[: int(valid.sum())]
    counts = np.bincount(owner[valid], minlength=R).astype(np.int64)
    local_ids = (flat[order] - owner[order] * per).astype(np.int32)
    pos = np.full(T * k, -1, np.int32)
    pos[order] = np.arange(order.size, dtype=np.int32)
    return Dispatch(order, counts, local_ids, pos.reshape(T, k))


class DistExchange:
    """All-to-all over a torch.distributed process group (one rank per process)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.R = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

    def counts(self, send_counts):
        import torch
        s = torch.as_tensor(np.asarray(send_counts, np.int64))
        r = torch.empty_like(s)
        dev = self._device()
        s, r = s.to(dev), r.to(dev)
        self.dist.all_to_all_single(r, s, group=self.group)
        return r.cpu().numpy()

    def rows(self, send, send_counts, recv_counts):
        """send [sum(send_counts), ...] -> [sum(recv_counts), ...] (torch tensors),
        moved as raw bytes so that any element type crosses any backend."""
        import torch
        send = send.contiguous()
        tail = tuple(send.shape[1:])
        row_bytes = send[:1].numel() * send.element_size() if send.shape[0] else \
            int(np.prod(tail, dtype=np.int64)) * send.element_size()
        sb = send.view(torch.uint8).reshape(send.shape[0], row_bytes)
        rb = torch.empty((int(np.sum(recv_counts)), row_bytes), dtype=torch.uint8, device=send.device)
        self.dist.all_to_all_single(rb, sb, [int(c) for c in recv_counts], [int(c) for c in send_counts],
                                    group=self.group)
        return rb.view(send.dtype).reshape((rb.shape[0],) + tail)

    def _device(self):
        return "cuda" if self.dist.get_backend(self.group) == "nccl" else "cpu"


def ep_layer(x, backend, E: int, exchange):
    """One layer on this rank: returns (out, idx, w) for its tokens.  x is the
    backend's activation tensor [T, D]; `exchange` a DistExchange."""
    idx, w = backend.route(x)
    plan = plan_dispatch(backend.to_host_int(idx), E, exchange.R)
    recv_counts = exchange.counts(plan.counts)
    xs = backend.gather(x, plan.order // idx.shape[1])
    ids = backend.from_host_int(plan.local_ids)
    recv_x = exchange.rows(xs, plan.counts, recv_counts)
    recv_ids = exchange.rows(ids, plan.counts, recv_counts)
    y_recv = backend.ffn_pairs(recv_x, recv_ids)
    y = exchange.rows(y_recv, recv_counts, plan.counts)
    out = backend.combine(y, backend.from_host_int(plan.pos), w, x.shape[0])
    return out, idx, w


def run_local_ranks(xs, backends, E: int):
    """R ranks emulated in one process: each step of ep_layer runs for every
    rank, and the exchanges move the buffers between the emulated ranks.
    Returns [(out, idx, w)] per rank."""
    R = len(backends)
    routed = [b.route(x) for b, x in zip(backends, xs)]
    plans = [plan_dispatch(b.to_host_int(idx), E, R) for b, (idx, _) in zip(backends, routed)]
    sent_x = [b.gather(x, p.order // idx.shape[1]) for b, x, p, (idx, _) in zip(backends, xs, plans, routed)]
    sent_ids = [b.from_host_int(p.local_ids) for b, p in zip(backends, plans)]
    offs = [np.concatenate([[0], np.cumsum(p.counts)]) for p in plans]
    y_back = [[None] * R for _ in range(R)]  # [src][dst] rows computed by dst for src
    for dst in range(R):
        parts_x = [sent_x[src][offs[src][dst]:offs[src][dst + 1]] for src in range(R)]
        parts_i = [sent_ids[src][offs[src][dst]:offs[src][dst + 1]] for src in range(R)]
        y = backends[dst].ffn_pairs(backends[dst].cat(parts_x), backends[dst].cat(parts_i))
        o = 0
        for src in range(R):
            n = int(plans[src].counts[dst])
            y_back[src][dst] = y[o:o + n]
            o += n
    outs = []
    for src in range(R):
        b = backends[src]
        y = b.cat([y_back[src][dst] for dst in range(R)])
        idx, w = routed[src]
        outs.append((b.combine(y, b.from_host_int(plans[src].pos), w, xs[src].shape[0]), idx, w))
    return outs


class DeviceBackend:
    """The library's kernels on one GPU for the experts this rank owns:
    `layer` is a DeviceLayer holding only those experts (local ids 0 ..),
    `Wr` / `bias` the full router (every rank ranks all E = Wr.shape[0]
    experts)."""

    def __init__(self, layer, Wr, bias, k: int, stream=None):
        self.layer, self.Wr, self.bias, self.k, self.stream = layer, Wr, bias, k, stream

    def _route_workspace(self, T):
        """Workspace sized for ranking all E experts (the local layer holds fewer)."""
        import torch
        from . import ds4moe_workspace_bytes, ds4moe_workspace_init, make_layer
        L = self.layer
        shape = make_layer(L.d_model, L.d_ff, int(self.Wr.shape[0]), L.q_gate, L.q_up, L.q_down, None, None, None)
        ws = torch.empty(max(ds4moe_workspace_bytes(shape, T, self.k, T > 64), 256), dtype=torch.uint8,
                         device="cuda")
        ds4moe_workspace_init(ws)
        return ws

    def route(self, x):
        import torch
        from . import ds4moe_route_topk
        T = x.shape[0]
        idx = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=x.device)
        ws = self._route_workspace(T)
        ds4moe_route_topk(x, self.Wr, self.bias, self.k, idx, w, None, ws, self.stream)
        self._check(ws)
        return idx, w

    def to_host_int(self, t):
        return t.cpu().numpy()

    def from_host_int(self, a):
        import torch
        return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()

    def gather(self, x, rows):
        import torch
        from . import ds4moe_gather_rows
        r = self.from_host_int(rows)
        dst = torch.empty((r.numel(), x.shape[1]), dtype=x.dtype, device=x.device)
        ds4moe_gather_rows(x, r, dst, self.stream)
        return dst

    def cat(self, parts):
        import torch
        return torch.cat(parts) if parts else parts

    def ffn_pairs(self, xr, ids):
        """y[j] = expert ids[j]'s FFN of row xr[j] (k = 1, weight 1)."""
        import torch
        from .device import workspace
        from . import ds4moe_ffn_decode, ds4moe_ffn_prefill
        n = xr.shape[0]
        y = torch.empty((n, self.layer.d_model), dtype=torch.float32, device=xr.device)
        if n == 0:
            return y
        prefill = n > 64
        ws = workspace(self.layer, n, 1, prefill=prefill)
        ones = torch.ones((n, 1), dtype=torch.float32, device=xr.device)
        fn = ds4moe_ffn_prefill if prefill else ds4moe_ffn_decode
        fn(self.layer.abi, xr, ids.view(n, 1), ones, y, ws, self.stream)
        self._check(ws)
        return y

    def combine(self, y, pos, w, T):
        import torch
        from . import ds4moe_combine_pairs
        out = torch.empty((T, self.layer.d_model), dtype=torch.float32, device=w.device)
        ds4moe_combine_pairs(y, pos.view(T, -1), w, out, self.stream)
        return out

    def _check(self, ws):
        from .device import check_status
        check_status(ws, self.stream)
