"""Host-side logic of bench.py's multi-process path on CPU (gloo, world size 2):
the slowest rank sets the job time, every rank draws its own tokens, and the
whole-job value counts every rank's tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    elapsed = 10.0 + 5.0 * rank            # rank 1 is slower
    ms = bench.reduce_max(elapsed, w)
    bench.barrier(w)
    q.put((r, w, lr, ms, bench.rank_batch_offset(r)))
    dist.destroy_process_group()


def test_two_rank_timing_and_token_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == 15.0 for r in res)          # max over ranks on every rank
    assert res[0][4] != res[1][4]                   # distinct token draws per rank
    import synth
    w = synth.WORKLOADS[1]
    a = synth.activations(w, batch=res[0][4])
    b = synth.activations(w, batch=res[1][4])
    assert not (a == b).all()
