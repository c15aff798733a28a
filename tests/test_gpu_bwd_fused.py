"""Backward through the fused steps on the GPU (rec_attn_bwd_fused) vs the oracle's
fused backward (chain rule through the output gate, the attention, the rotation, the
Q/K gates and QK-RMSNorm; SORT review page 3.3.2, TM20K QK Norm, CADET self-gating).

Every gradient -- dq, dk, dv, the three gate pre-activations and both norm gains -- is
held to the backward's tolerances: relative Frobenius error <= 1e-2 and max-abs <= 2e-2
of the reference's largest value for bf16 (one more bf16 rounding than the plain
backward: the gradient of the gated, normalised rows), 1e-4 / 1e-3 for fp32."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import workloads as W
from test_gpu_fused import STEPS, _device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gu.ensure_built()


CASES = {
    "tiny_fp32": lambda: W.tiny_fp32(batch=3, n_hist=150, n_cand=20),
    "cadet": lambda: W.cadet(batch=4, n_pairs=150, heads=2),
    "sort": lambda: W.sort(batch=2, n_hist=400, n_cand=40, window=96, heads=2),
    "mtgr": lambda: W.mtgr(batch=3, hist=(150, 300), rt=(20, 60), cand=(10, 30), heads=2),
    "sort_d128": lambda: W.sort(batch=2, n_hist=260, n_cand=30, window=100, heads=2, head_dim=128),
}


def _tol(w):
    return (1e-2, 2e-2) if w.dtype == "bf16" else (1e-4, 1e-3)


@pytest.mark.parametrize("steps", sorted(STEPS))
@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_backward_matches_oracle(name, steps):
    w = CASES[name]()
    fi = W.fused_inputs(w)
    on = STEPS[steps]
    tens = gu.device_inputs(w)
    dev = {n: _device(getattr(fi, n), w) for n in on}
    kw = dict(q_norm_weight=dev.get("q_norm_w"), k_norm_weight=dev.get("k_norm_w"), norm_eps=fi.norm_eps,
              q_gate=dev.get("q_gate"), k_gate=dev.get("k_gate"), out_gate=dev.get("out_gate"))
    g_host = (W.round_to_bf16_bits(np.random.default_rng(13).standard_normal(w.q.shape).astype(np.float32))
              if w.dtype == "bf16" else np.random.default_rng(13).standard_normal(w.q.shape).astype(np.float32))
    dout = _device(g_host, w)
    nan = lambda x: torch.full_like(x, float("nan"))
    grads = {"dq": nan(tens["q"]), "dk": nan(tens["q"]), "dv": nan(tens["q"])}
    if "q_gate" in on:
        grads["dq_gate"] = nan(tens["q"])
    if "k_gate" in on:
        grads["dk_gate"] = nan(tens["q"])
    if "out_gate" in on:
        grads["dout_gate"] = nan(tens["q"])
    if "q_norm_w" in on:
        grads["dq_norm_weight"] = torch.full((w.num_heads, w.head_dim), float("nan"), device="cuda")
    if "k_norm_w" in on:
        grads["dk_norm_weight"] = torch.full((w.num_heads, w.head_dim), float("nan"), device="cuda")
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        out = nan(tens["q"])
        lse = torch.empty((w.total_tokens, w.num_heads), dtype=torch.float32, device="cuda")
        bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], out, lse, None, **kw)
        bd.rec_attn_bwd_fused(plan, tens["q"], tens["k"], tens["v"], out, lse, dout, grads["dq"], grads["dk"],
                              grads["dv"], None, **kw, **{n: x for n, x in grads.items() if n not in ("dq", "dk", "dv")})
        torch.cuda.synchronize()
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
    f = oracle.Fused(q_norm_w=fi.q_norm_w.astype(np.float64) if "q_norm_w" in on else None,
                     k_norm_w=fi.k_norm_w.astype(np.float64) if "k_norm_w" in on else None, norm_eps=fi.norm_eps,
                     q_gate=fi.q_gate if "q_gate" in on else None, k_gate=fi.k_gate if "k_gate" in on else None,
                     out_gate=fi.out_gate if "out_gate" in on else None)
    ref = oracle.attention_bwd_fused(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v, f, g_host)
    rel_tol, max_tol = _tol(w)
    for n, got in grads.items():
        r = ref[{"dq_norm_weight": "dq_norm_w", "dk_norm_weight": "dk_norm_w"}.get(n, n)]
        x = got.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(x).all(), f"{n}: unwritten or non-finite values"
        rel = np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-30)
        mx = np.max(np.abs(x - r))
        assert rel <= rel_tol and mx <= max_tol * max(np.max(np.abs(r)), 1e-30), (name, steps, n, rel, mx)


def test_fused_backward_requires_the_gradients_of_its_steps():
    w = CASES["cadet"]()
    fi = W.fused_inputs(w)
    tens = gu.device_inputs(w)
    g = _device(fi.q_gate, w)
    x = torch.empty_like(tens["q"])
    lse = torch.empty((w.total_tokens, w.num_heads), dtype=torch.float32, device="cuda")
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        with pytest.raises(bd.RecAttnError) as e:  # a q gate without its gradient
            bd.rec_attn_bwd_fused(plan, tens["q"], tens["k"], tens["v"], x, lse, x, torch.empty_like(x),
                                  torch.empty_like(x), torch.empty_like(x), None, q_gate=g)
        assert e.value.code == bd.ERR_INVALID_ARG
    finally:
        bd.rec_attn_free(plan)
