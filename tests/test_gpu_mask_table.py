"""The plan's mask table beyond its capacity (8 slots per tile + 1024): one request
whose history and candidate tokens are interleaved makes every (query tile, key tile)
pair PARTIAL (candidates see every history token, history tokens see causal history,
candidates see only themselves), so the table fills and the remaining pairs fall back
to the kernels building their visibility bits themselves.  Forward and backward must
agree with the fp64 oracle on both kinds of tile."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TILE = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    gu.ensure_built()


def _interleaved(n_tokens=4901, heads=2, seed=7):
    rng = np.random.default_rng(seed)
    t0 = 1_700_000_000 + int(rng.integers(0, 10_000_000))
    t = t0 + np.cumsum(rng.integers(1, 3600, size=n_tokens)).astype(np.int64)
    ty = np.where(rng.random(n_tokens) < 0.3, W.CAND, W.HIST).astype(np.int8)
    d = 64
    q, k, v = (W.round_to_bf16_bits(rng.standard_normal((n_tokens, heads, d)).astype(np.float32) / np.sqrt(d))
               for _ in range(3))
    return W.Workload("interleaved", heads, d, "bf16", np.array([0, n_tokens], dtype=np.int64), t, ty, q, k, v,
                      dict(use_delay=False, delay_s=0, window=0, hist_bidirectional=False),
                      dict(use_rope=True, phi_min=1e-4, dt_max_s=31536000.0, rope_base=6e5))


def test_mask_table_overflow_forward_and_backward():
    w = _interleaved()
    tens = gu.device_inputs(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        cls = bd.rec_attn_tile_classes(plan)
        n_tiles = (w.total_tokens + TILE - 1) // TILE
        n_partial = int((cls == 1).sum())
        assert n_partial > 8 * n_tiles + 1024, "the workload must overflow the mask table"
        out = torch.full_like(tens["q"], float("nan"))
        lse = torch.empty((w.total_tokens, w.num_heads), dtype=torch.float32, device=out.device)
        bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out, lse)
        g_host = W.round_to_bf16_bits(np.random.default_rng(3).standard_normal(w.q.shape).astype(np.float32))
        dout = gu.device_inputs(W.Workload(**{**w.__dict__, "q": g_host}))["q"]
        dq, dk, dv = (torch.full_like(tens["q"], float("nan")) for _ in range(3))
        bd.rec_attn_bwd(plan, tens["q"], tens["k"], tens["v"], out, lse, dout, dq, dk, dv)
        torch.cuda.synchronize()
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
    op = gu.oracle_params(w)
    ref = oracle.attention(op, w.offsets, w.t, w.types, w.q, w.k, w.v)
    gu.assert_close(w, gu.to_f64(out), ref, "forward")
    grads = oracle.attention_bwd(op, w.offsets, w.t, w.types, w.q, w.k, w.v, g_host)
    for what, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), grads):
        x = gu.to_f64(got)
        assert np.isfinite(x).all(), what
        rel = np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-30)
        assert rel <= 1e-2 and np.max(np.abs(x - r)) <= 2e-2 * max(np.max(np.abs(r)), 1e-30), (what, rel)
