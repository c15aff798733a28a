"""Helpers shared by the GPU tests: move a seeded workload to the device, run the
C-ABI path, and compare with the CPU oracle."""
import numpy as np
import torch

import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import build as bld
from generative_recommender_ranking_gb300 import workloads as W

# tolerances the tests hold the CUDA path to (outputs vs the fp64 oracle)
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
FP32_MAX_ABS = 1e-4


def ensure_built():
    bld.build()
    oracle.build()


def device_inputs(w: W.Workload, dev="cuda"):
    tens = {}
    tens["off_h"] = np.ascontiguousarray(w.offsets, dtype=np.int64)
    tens["off_d"] = torch.from_numpy(tens["off_h"]).to(dev)
    tens["t"] = torch.from_numpy(np.ascontiguousarray(w.t)).to(dev)
    tens["ty"] = torch.from_numpy(np.ascontiguousarray(w.types)).to(dev)
    if w.dtype == "bf16":
        conv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        conv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    tens["q"], tens["k"], tens["v"] = conv(w.q), conv(w.k), conv(w.v)
    return tens


def params_for(w: W.Workload, **over):
    kw = dict(w.mask)
    kw.update(w.rope)
    kw.update(over)
    return bd.make_params(w.num_heads, w.head_dim, dtype=w.dtype, **kw)


def oracle_params(w: W.Workload, **over):
    kw = dict(w.mask)
    kw.update(w.rope)
    kw.update(over)
    return oracle.Params(w.num_heads, w.head_dim, **kw)


def run_gpu(w: W.Workload, tens=None, with_lse=False, poison=True, **over):
    """plan + fwd through the C-ABI; returns (out tensor, lse tensor or None, plan)."""
    tens = tens or device_inputs(w)
    p = params_for(w, **over)
    plan = bd.rec_attn_plan(p, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    out = torch.empty_like(tens["q"])
    if poison:
        out.fill_(float("nan"))
    lse = torch.full((w.total_tokens, w.num_heads), float("nan"), device=out.device) if with_lse else None
    bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out, lse)
    torch.cuda.synchronize()
    return out, lse, plan


def to_f64(x: torch.Tensor) -> np.ndarray:
    return x.float().cpu().numpy().astype(np.float64)


def errors(gpu: np.ndarray, ref: np.ndarray):
    d = np.abs(gpu - ref)
    return float(np.nanmax(d)) if d.size else 0.0, float(np.mean(d)) if d.size else 0.0


def assert_close(w: W.Workload, gpu: np.ndarray, ref: np.ndarray, what=""):
    assert not np.isnan(gpu).any(), f"{what}: NaN in the CUDA output (unwritten or invalid rows)"
    mx, mean = errors(gpu, ref)
    if w.dtype == "bf16":
        assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, f"{what}: max {mx:.3e} mean {mean:.3e}"
    else:
        assert mx <= FP32_MAX_ABS, f"{what}: max {mx:.3e}"
    return mx, mean


def sample_rows(w: W.Workload, per_request=48, max_requests=6, seed=0):
    """Sorted global rows: first/last rows, tile edges and random rows of a few requests."""
    rng = np.random.default_rng(seed)
    B = w.batch
    reqs = sorted(set([0, B - 1] + list(rng.choice(B, size=min(B, max_requests), replace=False))))
    rows = []
    for b in reqs:
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        L = e - s
        if L == 0:
            continue
        cand = {0, L - 1, min(L - 1, 127), min(L - 1, 128), L // 2}
        cand |= set(int(x) for x in rng.integers(0, L, size=per_request))
        rows += [s + c for c in sorted(cand)]
    return np.array(sorted(set(rows)), dtype=np.int64)
