"""Expert parallelism across two ranks (gloo, CPU): each rank owns half of
the layer's experts and keeps its own tokens; bit_quantized_moe_q2_gb300.ep
routes, dispatches the (token, expert) pairs to the owners with all-to-all,
runs the owners' experts and combines the returned outputs.  The expert
arithmetic here is the oracle's (a test backend); the test checks the
partition, the exchange and the reassembly: every rank's output equals the
single-rank oracle layer on its tokens."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import synth

W = synth.WORKLOADS[0].replace(d_model=512, d_ff=256, n_expert=8, k=2, T=6, seed=61)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


class OracleBackend:
    """Test backend: the oracle's expert FFN on the experts [lo, hi) only
    (their blocks sliced out of the layer), numpy for the data movement."""

    def __init__(self, L, lo, hi):
        import oracle
        self.o, self.L, self.lo, self.hi = oracle, L, lo, hi
        E = L.w.n_expert
        self.mats = {}
        for name in ("gate", "up", "down"):
            buf = getattr(L, name)
            per = buf.size // E
            self.mats[name] = buf[lo * per:hi * per]

    def route(self, x):
        import torch
        idx, w, _ = self.o.route(x.numpy().view(np.uint16), self.L.Wr, self.L.bias, self.L.w.k)
        return torch.from_numpy(idx.astype(np.int32)), torch.from_numpy(w.astype(np.float32))

    def to_host_int(self, t):
        return t.numpy()

    def from_host_int(self, a):
        import torch
        return torch.from_numpy(np.ascontiguousarray(a, np.int32))

    def gather(self, x, rows):
        return x[np.asarray(rows, np.int64)]

    def cat(self, parts):
        import torch
        return torch.cat(parts)

    def ffn_pairs(self, xr, ids):
        import torch
        L, w = self.L, self.L.w
        out = np.empty((xr.shape[0], w.d_model), np.float32)
        xa = xr.numpy().view(np.uint16)
        for j, e in enumerate(ids.numpy().tolist()):
            assert 0 <= e < self.hi - self.lo
            y, _, _, _ = self.o.expert_ffn(w.d_model, w.d_ff, L.qg, self.mats["gate"], L.qu, self.mats["up"], L.qd,
                                           self.mats["down"], e, xa[j])
            out[j] = y
        return torch.from_numpy(out)

    def combine(self, y, pos, w, T):
        import torch
        yv, p, wv = y.numpy().astype(np.float64), pos.numpy(), w.numpy().astype(np.float64)
        out = np.zeros((T, yv.shape[1] if yv.size else self.L.w.d_model))
        for t in range(T):
            for i in range(p.shape[1]):
                if p[t, i] >= 0:
                    out[t] += wv[t, i] * yv[p[t, i]]
        return torch.from_numpy(out.astype(np.float32))


def _worker(rank, world, port, q):
    import traceback
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from bit_quantized_moe_q2_gb300 import ep
        from tests.layers import build_layer
        L = build_layer(W)
        lo, hi = ep.expert_ranges(W.n_expert, world)[rank]
        x = synth.activations(W, batch=100 + rank)
        xt = torch.from_numpy(x.view(np.int16).copy())
        out, idx, w = ep.ep_layer(xt, OracleBackend(L, lo, hi), W.n_expert, ep.DistExchange())
        q.put((rank, out.numpy(), idx.numpy()))
    except Exception:  # report at once instead of leaving the parent waiting
        q.put((rank, None, traceback.format_exc()))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_ranks_each_owning_half_the_experts():
    import oracle
    from tests.layers import build_layer
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
    for rank, out, err in res:
        assert out is not None, f"rank {rank}:\n{err}"
    assert all(p.exitcode == 0 for p in procs)
    L = build_layer(W)
    crossing = 0
    for rank, out, idx in res:
        x = synth.activations(W, batch=100 + rank)
        ridx, rw, _ = oracle.route(x, L.Wr, L.bias, W.k)
        assert np.array_equal(idx, ridx)
        ref = oracle.moe_ffn(W.d_model, W.d_ff, W.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, x, ridx, rw)
        # the same arithmetic, one more fp32 rounding per expert output
        assert np.abs(out - ref).max() <= 1e-6 * np.abs(ref).max()
        crossing += int(((ridx // (W.n_expert // 2)) != rank).sum())
    assert crossing > 0  # pairs really travelled to the other rank


def test_plan_dispatch_orders_pairs_by_owner():
    from bit_quantized_moe_q2_gb300.ep import plan_dispatch, expert_ranges
    idx = np.array([[5, 0], [2, 7], [9, 3], [-1, 4]], np.int32)  # 9 and -1: out of range for E = 8
    p = plan_dispatch(idx, 8, 2)
    assert p.counts.tolist() == [3, 3]
    assert p.order.tolist() == [1, 2, 5, 0, 3, 7]            # owner 0 first, stable within an owner
    assert p.local_ids.tolist() == [0, 2, 3, 1, 3, 0]
    assert p.pos.tolist() == [[3, 0], [1, 4], [-1, 2], [-1, 5]]
    assert expert_ranges(8, 2) == [(0, 4), (4, 8)]
    with pytest.raises(ValueError):
        expert_ranges(8, 3)


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_emulated_ranks_reproduce_the_single_rank_layer(R):
    """R ranks emulated in one process (run_local_ranks): every rank's output
    equals the single-rank oracle layer on its tokens, including ranks whose
    experts receive no pair (at R = 8 each rank owns one expert)."""
    import torch
    import oracle
    from bit_quantized_moe_q2_gb300 import ep
    from tests.layers import build_layer
    L = build_layer(W)
    xs = [torch.from_numpy(synth.activations(W, batch=200 + r).view(np.int16).copy()) for r in range(R)]
    backends = [OracleBackend(L, lo, hi) for lo, hi in ep.expert_ranges(W.n_expert, R)]
    outs = ep.run_local_ranks(xs, backends, W.n_expert)
    for r, (out, idx, w) in enumerate(outs):
        x = xs[r].numpy().view(np.uint16)
        ridx, rw, _ = oracle.route(x, L.Wr, L.bias, W.k)
        assert np.array_equal(idx.numpy(), ridx)
        ref = oracle.moe_ffn(W.d_model, W.d_ff, W.n_expert, L.qg, L.gate, L.qu, L.up, L.qd, L.down, x, ridx, rw)
        assert np.max(np.abs(out.numpy() - ref)) <= 1e-5 * max(np.max(np.abs(ref)), 1e-30)
