"""Request-level sharding across GPUs (host logic only).

Requests of a packed batch never see each other, so the path shards by request with
no data-path collective: each rank plans and runs its own requests.  The partition
is greedy longest-processing-time (heaviest request to the least loaded rank) on a
per-request cost such as its visible-pair count.  Timing aggregation for a run over
ranks takes the slowest rank's time and the sum of the work.
"""
from __future__ import annotations

import heapq

import numpy as np


def partition(costs, world: int) -> list[np.ndarray]:
    """Split request indices over `world` ranks (greedy LPT).  Each rank's list is
    sorted ascending; together they cover every request exactly once."""
    costs = np.asarray(costs, dtype=np.float64)
    if world < 1:
        raise ValueError("world must be >= 1")
    heap = [(0.0, r) for r in range(world)]
    owned: list[list[int]] = [[] for _ in range(world)]
    for idx in np.argsort(-costs, kind="stable"):
        load, r = heapq.heappop(heap)
        owned[r].append(int(idx))
        heapq.heappush(heap, (load + float(costs[idx]), r))
    return [np.array(sorted(o), dtype=np.int64) for o in owned]


def causal_cost(offsets) -> np.ndarray:
    """Upper-bound cost per request (L(L+1)/2 pairs) when exact counts are not at hand."""
    L = np.diff(np.asarray(offsets, dtype=np.int64)).astype(np.float64)
    return L * (L + 1) / 2


def gather(offsets, requests, *arrays):
    """Pack the tokens of `requests` (sorted indices) into new contiguous arrays.
    Returns (new offsets, *gathered arrays); arrays are indexed by token on axis 0."""
    offsets = np.asarray(offsets, dtype=np.int64)
    req = np.asarray(requests, dtype=np.int64)
    lens = offsets[req + 1] - offsets[req]
    new_off = np.zeros(len(req) + 1, dtype=np.int64)
    new_off[1:] = np.cumsum(lens)
    idx = np.concatenate([np.arange(offsets[r], offsets[r + 1]) for r in req]) if len(req) else \
        np.zeros(0, dtype=np.int64)
    return (new_off, *[np.asarray(a)[idx] for a in arrays])


def aggregate(times, works, device=None):
    """Slowest rank's value of each time and the total of each work quantity over the
    initialised process group (the local values when torch.distributed is not
    initialised).  Returns (list of max times, list of summed works)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(times), dtype=torch.float64, device=device)
    w = torch.tensor(list(works), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return t.tolist(), w.tolist()
