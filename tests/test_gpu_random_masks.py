"""Seeded random mask layouts on the GPU against the oracle: token types in random runs
(GLOBAL, HIST, RT, CAND), times sorted, perturbed or repeated, and random mask
parameters (delay, window, bidirectional history).  Each case checks the tile classes
and visible-pair count bit for bit, every output row and lse within the bf16
tolerances, and, for a third of the cases, the gradients.  Further variants run the same
layouts with head_dim 128, through the fp32 path, through query-pruned plans and through
the fused QK-RMSNorm and gates."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N_CASES = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    gu.ensure_built()


def _case(seed, dtype="bf16", d=64):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 5))
    lengths = [int(x) for x in rng.integers(1, 700, size=B)]
    if rng.random() < 0.3:
        lengths[int(rng.integers(0, B))] = 0
    T = sum(lengths)
    types = np.empty(T, dtype=np.int8)
    t = np.empty(T, dtype=np.int64)
    s = 0
    for n in lengths:
        # random runs of types, GLOBAL more likely first and CAND last
        pos = 0
        while pos < n:
            run = int(rng.integers(1, 80))
            frac = pos / max(n, 1)
            p = np.array([0.3 * (1 - frac), 0.4, 0.15, 0.15 + 0.3 * frac])
            types[s + pos:s + min(n, pos + run)] = rng.choice(4, p=p / p.sum())
            pos += run
        span = int(rng.choice([3600, 86400, 30 * 86400, 365 * 86400]))
        tt = W.EPOCH + np.sort(rng.integers(0, span, size=n)).astype(np.int64)
        mode = rng.integers(0, 3)
        if mode == 1 and n > 2:  # a few swapped neighbours: runs no longer time-sorted
            for i in rng.integers(0, n - 1, size=max(1, n // 50)):
                tt[i], tt[i + 1] = tt[i + 1], tt[i]
        elif mode == 2 and n > 0:  # candidates stamped at one request time
            c = types[s:s + n] == W.CAND
            tt[c] = tt.max()
        t[s:s + n] = tt
        s += n
    mask = dict(use_delay=bool(rng.random() < 0.6), delay_s=int(rng.choice([0, 60, 3600, 86400])),
                window=int(rng.choice([0, 0, 16, 100, 256])), hist_bidirectional=bool(rng.random() < 0.25))
    x = [rng.standard_normal((T, 2, d)).astype(np.float32) * 0.5 for _ in range(3)]
    if dtype == "bf16":
        x = [W.round_to_bf16_bits(a) for a in x]
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return W.Workload(f"random{seed}", 2, d, dtype, off, t, types, *x, mask,
                      dict(use_rope=True, phi_min=1e-4, dt_max_s=float(W.YEAR), rope_base=6e5))


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_mask_layouts(seed):
    w = _case(seed)
    out, lse, plan = gu.run_gpu(w, with_lse=True)
    try:
        op = gu.oracle_params(w)
        np.testing.assert_array_equal(bd.rec_attn_tile_classes(plan),
                                      oracle.tile_classes(op, w.offsets, w.t, w.types))
        assert bd.rec_attn_visible_pairs(plan) == oracle.visible_pairs(op, w.offsets, w.t, w.types)
        ref, ref_lse = oracle.attention(op, w.offsets, w.t, w.types, w.q, w.k, w.v, with_lse=True)
        gu.assert_close(w, gu.to_f64(out), ref, w.name)
        lg = lse.cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lg), fin)
        assert np.max(np.abs(lg[fin] - ref_lse[fin]), initial=0.0) <= 2e-2
        if seed % 3 == 0 and w.total_tokens > 0:
            rng = np.random.default_rng(seed)
            g = W.round_to_bf16_bits(rng.standard_normal(w.q.shape).astype(np.float32))
            tens = gu.device_inputs(w)
            dout = gu.device_inputs(W.Workload(**{**w.__dict__, "q": g}))["q"]
            grads = [torch.full_like(tens["q"], float("nan")) for _ in range(3)]
            bd.rec_attn_bwd(plan, tens["q"], tens["k"], tens["v"], out, lse, dout, *grads)
            torch.cuda.synchronize()
            refg = oracle.attention_bwd(op, w.offsets, w.t, w.types, w.q, w.k, w.v, g)
            for what, got, r in zip(("dq", "dk", "dv"), grads, refg):
                xg = gu.to_f64(got)
                assert np.isfinite(xg).all(), what
                rel = np.linalg.norm(xg - r) / max(np.linalg.norm(r), 1e-30)
                mx = np.max(np.abs(xg - r))
                assert rel <= 1e-2 and mx <= 2e-2 * max(np.max(np.abs(r)), 1e-30), (w.name, what, rel, mx)
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)


VARIANTS = ("d128", "fp32", "pruned", "fused")


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("variant", VARIANTS)
def test_random_mask_layouts_variants(variant, seed):
    w = _case(100 + seed, dtype="fp32" if variant == "fp32" else "bf16",
              d=128 if variant == "d128" else (32 if variant == "fp32" else 64))
    if w.total_tokens == 0:
        pytest.skip("empty batch (the edge tests cover it)")
    op = gu.oracle_params(w)
    tens = gu.device_inputs(w)
    p = gu.params_for(w)
    keep = int(np.random.default_rng(seed).integers(0, 400)) if variant == "pruned" else -1
    if variant == "pruned":
        plan = bd.rec_attn_plan_query_pruned(p, keep, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    else:
        plan = bd.rec_attn_plan(p, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    fused = None
    try:
        out = torch.full_like(tens["q"], float("nan"))
        if variant == "fused":
            fi = W.fused_inputs(w)
            dev = {n: torch.from_numpy(np.ascontiguousarray(getattr(fi, n).view(np.int16)
                                                            if getattr(fi, n).dtype == np.uint16
                                                            else getattr(fi, n))).cuda()
                   for n in ("q_norm_w", "k_norm_w", "q_gate", "k_gate", "out_gate")}
            for n in ("q_gate", "k_gate", "out_gate"):
                dev[n] = dev[n].view(torch.bfloat16)
            bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], out, None, None,
                                  q_norm_weight=dev["q_norm_w"], k_norm_weight=dev["k_norm_w"],
                                  norm_eps=fi.norm_eps, q_gate=dev["q_gate"], k_gate=dev["k_gate"],
                                  out_gate=dev["out_gate"])
            fused = oracle.Fused(norm_eps=fi.norm_eps, q_norm_w=fi.q_norm_w.astype(np.float64),
                                 k_norm_w=fi.k_norm_w.astype(np.float64), q_gate=fi.q_gate, k_gate=fi.k_gate,
                                 out_gate=fi.out_gate)
        else:
            bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out)
        torch.cuda.synchronize()
        assert bd.rec_attn_device_status(plan) == bd.OK
        np.testing.assert_array_equal(bd.rec_attn_tile_classes(plan),
                                      oracle.tile_classes(op, w.offsets, w.t, w.types))
    finally:
        bd.rec_attn_free(plan)
    rows = oracle.kept_rows(w.offsets, w.types, keep) if variant == "pruned" else None
    ref = oracle.attention(op, w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows, fused=fused)
    o = gu.to_f64(out)
    if rows is not None:
        written = np.zeros(w.total_tokens, dtype=bool)
        written[rows] = True
        assert np.isnan(o[~written]).all(), "a pruned row was written"
        o = o[rows]
    gu.assert_close(w, o, ref, f"{w.name}/{variant}")
