"""Fused QK-RMSNorm, Q/K sigmoid gates and attention output gate on the GPU
(rec_attn_fwd_fused) vs the fp64 oracle, through the C-ABI.

Reduced sizes with every row checked, each step alone and all together, plans with
and without the time-RoPE, and one full-size workload on sampled rows.  Same
tolerances as the plain path: max-abs 2e-2 and mean-abs 2e-3 for bf16, 1e-4 for fp32.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gu.ensure_built()


SMALL = {
    "tiny_fp32": lambda: W.tiny_fp32(batch=3, n_hist=150, n_cand=20),
    "cadet": lambda: W.cadet(batch=4, n_pairs=150),
    "sort": lambda: W.sort(batch=2, n_hist=400, n_cand=40, window=96),
    "mtgr": lambda: W.mtgr(batch=3, hist=(150, 300), rt=(20, 60), cand=(10, 30)),
    "sort_d128": lambda: W.sort(batch=2, n_hist=260, n_cand=30, window=100, heads=2, head_dim=128),
}

STEPS = {
    "all": ("q_norm_w", "k_norm_w", "q_gate", "k_gate", "out_gate"),
    "norm": ("q_norm_w", "k_norm_w"),
    "qk_gates": ("q_gate", "k_gate"),
    "out_gate": ("out_gate",),
}


def _device(a, w):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(w, fi, steps, rows=None, **over):
    tens = gu.device_inputs(w)
    p = gu.params_for(w, **over)
    plan = bd.rec_attn_plan(p, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        out = torch.full_like(tens["q"], float("nan"))
        dev = {n: _device(getattr(fi, n), w) for n in steps}
        bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], out, None, None,
                              q_norm_weight=dev.get("q_norm_w"), k_norm_weight=dev.get("k_norm_w"),
                              norm_eps=fi.norm_eps, q_gate=dev.get("q_gate"), k_gate=dev.get("k_gate"),
                              out_gate=dev.get("out_gate"))
        torch.cuda.synchronize()
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
    f = oracle.Fused(norm_eps=fi.norm_eps, **{n: (getattr(fi, n).astype(np.float64) if n.endswith("_w")
                                                  else getattr(fi, n)) for n in steps})
    ref = oracle.attention(gu.oracle_params(w, **over), w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows,
                           fused=f)
    got = out if rows is None else out[torch.from_numpy(rows).cuda()]
    return gu.to_f64(got), ref


@pytest.mark.parametrize("steps", sorted(STEPS))
@pytest.mark.parametrize("name", sorted(SMALL))
def test_fused_parity_all_rows(name, steps):
    w = SMALL[name]()
    got, ref = _run(w, W.fused_inputs(w), STEPS[steps])
    gu.assert_close(w, got, ref, f"{name}/{steps}")


@pytest.mark.parametrize("name", ["cadet", "tiny_fp32"])
def test_fused_on_a_plan_without_rope(name):
    # the Q/K steps then need their own Q'/K' buffers, taken on the first fused call
    w = SMALL[name]()
    got, ref = _run(w, W.fused_inputs(w), STEPS["all"], use_rope=False)
    gu.assert_close(w, got, ref, f"{name}/no-rope")


def test_fused_with_no_step_equals_plain_forward():
    w = SMALL["mtgr"]()
    tens = gu.device_inputs(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        a = torch.empty_like(tens["q"])
        b = torch.empty_like(tens["q"])
        bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], a)
        bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], b)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    finally:
        bd.rec_attn_free(plan)


def test_fused_full_size_sampled():
    w = W.make("mtgr")
    rows = gu.sample_rows(w)
    got, ref = _run(w, W.fused_inputs(w), STEPS["all"], rows=rows)
    gu.assert_close(w, got, ref, "mtgr full size")


def test_fused_rejects_bad_arguments():
    w = SMALL["cadet"]()
    tens = gu.device_inputs(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        out = torch.empty_like(tens["q"])
        with pytest.raises(bd.RecAttnError):
            bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], out, norm_eps=-1.0)
        with pytest.raises(bd.RecAttnError):
            bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], out, out_gate=out)
        g = torch.zeros(out.numel() + 8, dtype=out.dtype, device=out.device)[1:1 + out.numel()].view_as(out)
        with pytest.raises(bd.RecAttnError):  # misaligned gate
            bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], out, q_gate=g)
    finally:
        bd.rec_attn_free(plan)
