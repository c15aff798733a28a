"""Multi-rank host logic on CPU: two gloo ranks partition a batch's requests,
gather their shards, and aggregate timings the way bench.py does under torchrun."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from generative_recommender_ranking_gb300 import sharding
from generative_recommender_ranking_gb300 import workloads as W


def test_partition_covers_every_request_once_and_balances():
    rng = np.random.default_rng(0)
    costs = rng.integers(1, 1000, size=101).astype(float)
    for world in (1, 2, 3, 8):
        parts = sharding.partition(costs, world)
        allr = np.sort(np.concatenate(parts))
        assert np.array_equal(allr, np.arange(101))
        loads = [costs[p].sum() for p in parts]
        assert max(loads) <= costs.sum() / world + costs.max()


def test_gather_keeps_request_contents():
    w = W.mtgr(batch=5, hist=(20, 40), rt=(5, 9), cand=(3, 6))
    off, t, ty, q = sharding.gather(w.offsets, [1, 3], w.t, w.types, w.q)
    assert off[0] == 0 and len(off) == 3
    for i, b in enumerate([1, 3]):
        s, e = w.offsets[b], w.offsets[b + 1]
        assert np.array_equal(t[off[i]:off[i + 1]], w.t[s:e])
        assert np.array_equal(q[off[i]:off[i + 1]], w.q[s:e])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.sort(batch=6, n_special=4, n_hist=50, n_cand=5)
    parts = sharding.partition(sharding.causal_cost(w.offsets), world)
    mine = parts[rank]
    off, t, ty = sharding.gather(w.offsets, mine, w.t, w.types)
    got = [None] * world
    dist.all_gather_object(got, (rank, mine.tolist(), int(off[-1])))
    (ms,), (flops, toks) = sharding.aggregate([10.0 + rank], [100.0 * (rank + 1), float(off[-1])])
    out.put((rank, got, ms, flops, toks, int(w.offsets[-1])))
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, ms, flops, toks, total in res:
        reqs = sorted(r for _, mine, _ in got for r in mine)
        assert reqs == list(range(6))
        assert ms == 11.0                      # slowest rank
        assert flops == 300.0                  # sum of work
        assert toks == total                   # every token once
