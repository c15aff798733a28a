"""Query pruning on the GPU (rec_attn_plan_query_pruned) vs the oracle: computed rows
match the oracle row by row, pruned rows are left untouched, and the visible-pair
count covers computed rows only.  Includes target attention (keep = 0) on the CADET
serving workload at full size."""
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
    "tiny_fp32": lambda: W.tiny_fp32(batch=3, n_hist=300, n_cand=20),
    "cadet": lambda: W.cadet(batch=3, n_pairs=180),
    "sort": lambda: W.sort(batch=2, n_hist=500, n_cand=40, window=96),
    "mtgr": lambda: W.mtgr(batch=3, hist=(150, 400), rt=(20, 80), cand=(10, 40)),
    "tm20k_window": lambda: W.tm20k("window", batch=2, n_hist=1100),
    "serving": lambda: W.cadet_serving(batch=2, n_hist=700, n_cand=90),
}


def _pairs_of_rows(w, rows):
    op = gu.oracle_params(w)
    n = 0
    for b in range(w.batch):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        m = oracle.mask(op, w.t[s:e], w.types[s:e])
        sel = rows[(rows >= s) & (rows < e)] - s
        n += int(m[sel].sum())
    return n


def _run(w, keep, sample=None):
    tens = gu.device_inputs(w)
    plan = bd.rec_attn_plan_query_pruned(gu.params_for(w), keep, tens["off_h"], tens["off_d"], tens["t"],
                                         tens["ty"])
    try:
        out = torch.full_like(tens["q"], float("nan"))
        lse = torch.full((w.total_tokens, w.num_heads), float("nan"), device=out.device)
        bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out, lse)
        torch.cuda.synchronize()
        assert bd.rec_attn_device_status(plan) == bd.OK
        pairs = bd.rec_attn_visible_pairs(plan)
    finally:
        bd.rec_attn_free(plan)
    kept = oracle.kept_rows(w.offsets, w.types, keep)
    mask = np.zeros(w.total_tokens, dtype=bool)
    mask[kept] = True
    o = gu.to_f64(out)
    # pruned rows: untouched
    assert np.isnan(o[~mask]).all(), "a pruned row was written"
    assert torch.isnan(lse[torch.from_numpy(~mask).to(lse.device)]).all()
    rows = kept if sample is None else np.intersect1d(kept, sample)
    ref, ref_lse = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows,
                                    with_lse=True)
    gu.assert_close(w, o[rows], ref, f"{w.name}/keep={keep}")
    lg = lse.cpu().numpy().astype(np.float64)[rows]
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.max(np.abs(lg[fin] - ref_lse[fin]), initial=0.0) <= (1e-4 if w.dtype == "fp32" else 2e-2)
    return pairs, kept


@pytest.mark.parametrize("keep", [0, 37, 300, -1])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_pruned_parity(name, keep):
    w = SMALL[name]()
    pairs, kept = _run(w, keep)
    assert pairs == _pairs_of_rows(w, kept)


def test_lazformer_schedule_layers():
    # the history queries of a four-layer stack on a LazFormer-like request (history
    # with its last 64 tokens typed GLOBAL, one target), Eq. 22 with N_min = 128
    w = W.tm20k("window", batch=2, n_hist=1100)
    n_user = int(np.sum(w.types[: int(w.offsets[1])] != W.CAND))
    for layer in range(1, 5):
        keep = bd.rec_attn_query_keep(n_user, 128, layer, 4)
        pairs, kept = _run(w, keep)
        assert len(kept) == 2 * (keep + 1)


def test_target_attention_full_size_serving():
    # CADET serving at full size: 4096 history events + 500 candidates per request,
    # only the candidates query (keep = 0)
    w = W.make("cadet_serving")
    rows = gu.sample_rows(w)
    pairs, kept = _run(w, 0, sample=rows)
    # each candidate sees every history event older than t_req - 1 h, and itself
    assert len(kept) == w.batch * 500
    assert pairs == _pairs_of_rows(w, kept)


@pytest.mark.parametrize("keep", [0, 37, 3000, -1])
def test_pruned_parity_split_planner(keep):
    # requests of 40 tiles: the planner splits each request's query tiles over several
    # blocks, every one of which finds the first kept position for itself
    w = W.tm20k("window", batch=2, n_hist=5000, heads=2)
    n_tiles = sum((int(n) + 127) // 128 for n in np.diff(w.offsets))
    assert -(-n_tiles // w.batch) >= 32
    rows = gu.sample_rows(w, per_request=200)
    pairs, kept = _run(w, keep, sample=rows)
    assert len(kept) == (w.total_tokens if keep < 0 else w.batch * (min(keep, 5000) + 1))


def test_target_attention_ignores_stale_rotated_queries():
    """In a plan where no user token queries, the prologue leaves the rotated-Q rows of
    user tokens unwritten, and query tiles that mix user tokens and candidates still pass
    those rows through the tensor cores.  A previous forward with NaN queries leaves NaN
    in the pool memory the next plan's rotated-Q buffer takes; the candidates' outputs
    must still match the oracle and be finite (rows of the score and output tiles are
    independent)."""
    w = W.cadet_serving(batch=3, n_hist=700, n_cand=90)
    tens = gu.device_inputs(w)
    p = gu.params_for(w)
    poison = bd.rec_attn_plan(p, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    out = torch.empty_like(tens["q"])
    bd.rec_attn_fwd(poison, torch.full_like(tens["q"], float("nan")), tens["k"], tens["v"], out)
    torch.cuda.synchronize()
    bd.rec_attn_free(poison)
    torch.cuda.synchronize()
    plan = bd.rec_attn_plan_query_pruned(p, 0, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        out = torch.full_like(tens["q"], float("nan"))
        bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out)
        torch.cuda.synchronize()
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
    rows = oracle.kept_rows(w.offsets, w.types, 0)
    ref = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows)
    got = gu.to_f64(out)[rows]
    assert np.isfinite(got).all()
    gu.assert_close(w, got, ref, "target attention after a NaN forward")
