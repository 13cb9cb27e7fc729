"""Token-data-parallel replicas on CPU ranks (gloo, world size 2).

With the batch's tokens split across replicas, the only exchange the method needs is
the sum of the per-expert loads before the end-of-step bias update (the bias update
uses the load of the whole batch).  Each rank routes its shard with the CPU oracle,
the loads are all-reduced, and every rank must reach the whole-batch load and the
same updated bias.  A rank that never joins must surface as an error on the host.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(0)
    T, N_r, K_r = 64, 16, 4
    s = (1 / (1 + np.exp(-rng.standard_normal((T, N_r))))).astype(np.float32)
    b = rng.uniform(-0.01, 0.01, N_r).astype(np.float32)
    shard = slice(rank * T // world, (rank + 1) * T // world)
    idx = oracle.select_experts(s[shard], b, K_r)
    load = torch.from_numpy(oracle.dispatch(idx, N_r)["load"].astype(np.int64))
    dist.all_reduce(load)
    new_b = oracle.bias_update(b, load.numpy(), T, K_r, 0.001)
    whole = oracle.dispatch(oracle.select_experts(s, b, K_r), N_r)["load"]
    q.put((rank, load.numpy().tolist(), whole.tolist(), new_b.tolist()))
    dist.destroy_process_group()


def test_sharded_loads_sum_to_whole_batch_load():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, l0, w0, b0), (_, l1, w1, b1) = res
    assert l0 == l1 == w0 == w1
    assert b0 == b1


def _lonely_rank(port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        import datetime
        dist.init_process_group("gloo", rank=0, world_size=2,
                                timeout=datetime.timedelta(seconds=3))
        q.put("joined")
    except Exception as exc:  # the missing peer is reported on the host
        q.put("error:" + type(exc).__name__)


def test_missing_rank_is_reported_not_hung():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_lonely_rank, args=(_free_port(), q))
    p.start()
    msg = q.get(timeout=120)
    p.join(timeout=60)
    assert msg.startswith("error:")
