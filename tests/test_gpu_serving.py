"""Serving with a cached history (M-FALCON, HSTU notes on the blog index page; CADET's
scoring of hundreds of candidates per request): rec_attn_cache_create keeps each
request's rotated history keys and values, rec_attn_cache_score scores micro-batches
of candidates against them.

By candidate isolation a candidate's output does not depend on which other
candidates share its micro-batch, so every micro-batch size must reproduce the
oracle's outputs for the candidate rows of the whole request [history, all
candidates] (bf16: max-abs 2e-2, mean-abs 2e-3; fp32: 1e-4), lse included."""
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


def _split(w: W.Workload):
    """History rows (every non-candidate) and candidate rows of each request; the
    candidates of every workload family come last in their request."""
    hist_rows, cand_rows, hoff, coff = [], [], [0], [0]
    for b in range(w.batch):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        c = np.nonzero(w.types[s:e] == W.CAND)[0]
        n_h = (e - s) - len(c)
        assert (c == np.arange(n_h, e - s)).all(), "candidates must close the request"
        hist_rows += list(range(s, s + n_h))
        cand_rows += list(range(s + n_h, e))
        hoff.append(hoff[-1] + n_h)
        coff.append(coff[-1] + len(c))
    return np.array(hist_rows, dtype=np.int64), np.array(cand_rows, dtype=np.int64), np.array(hoff), np.array(coff)


def _dev(a, dtype):
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


CASES = {
    "cadet_serving": lambda: W.cadet_serving(batch=3, n_hist=700, n_cand=90),
    "mtgr": lambda: W.mtgr(batch=3, hist=(150, 300), rt=(20, 60), cand=(30, 70)),
    "cadet_serving_d128": lambda: W.cadet_serving(batch=2, n_hist=300, n_cand=40, heads=2, head_dim=128),
    "tiny_fp32": lambda: W.tiny_fp32(batch=3, n_hist=200, n_cand=37),
}


@pytest.mark.parametrize("micro", [1, 16, 29, None])
@pytest.mark.parametrize("name", sorted(CASES))
def test_cached_history_matches_oracle(name, micro):
    w = CASES[name]()
    hr, cr, hoff, coff = _split(w)
    n_c = np.diff(coff)
    bm = int(n_c.max()) if micro is None else micro
    op = gu.oracle_params(w)
    ref, ref_lse = oracle.attention(op, w.offsets, w.t, w.types, w.q, w.k, w.v, rows=cr, with_lse=True)
    cache = bd.rec_attn_cache_create(gu.params_for(w), hoff, torch.from_numpy(w.t[hr]).cuda(),
                                     torch.from_numpy(w.types[hr]).cuda(), _dev(w.k[hr], w.dtype),
                                     _dev(w.v[hr], w.dtype), bm)
    try:
        got = np.full(ref.shape, np.nan)
        got_lse = np.full(ref_lse.shape, np.nan)
        first = None
        for i0 in range(0, int(n_c.max()), bm):
            # micro-batch: candidates i0 .. i0 + bm of every request (fewer, or none, at the end)
            take = [np.arange(coff[b] + min(i0, n_c[b]), coff[b] + min(i0 + bm, n_c[b])) for b in range(w.batch)]
            mb_off = np.concatenate([[0], np.cumsum([len(x) for x in take])])
            idx = np.concatenate(take)
            rows = cr[idx]
            out = torch.full((len(rows), w.num_heads, w.head_dim), float("nan"),
                             dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float32, device="cuda")
            lse = torch.full((len(rows), w.num_heads), float("nan"), device="cuda")
            args = (mb_off, torch.from_numpy(w.t[rows]).cuda(), _dev(w.q[rows], w.dtype), _dev(w.k[rows], w.dtype),
                    _dev(w.v[rows], w.dtype), out, lse)
            bd.rec_attn_cache_score(cache, *args)
            torch.cuda.synchronize()
            got[idx] = gu.to_f64(out)
            got_lse[idx] = lse.cpu().numpy()
            if first is None:  # the same micro-batch again: identical results
                first = out.clone()
                bd.rec_attn_cache_score(cache, *args)
                torch.cuda.synchronize()
                assert torch.equal(first, out)
        gu.assert_close(w, got, ref, f"{name} micro-batch {bm}")
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(got_lse), fin)
        tol = 1e-4 if w.dtype == "fp32" else 2e-2
        assert np.max(np.abs(got_lse[fin] - ref_lse[fin]), initial=0.0) <= tol
    finally:
        bd.rec_attn_cache_free(cache)


def test_cached_history_empty_history_and_rejects_overfull_batches():
    w = W.cadet_serving(batch=2, n_hist=0, n_cand=20)
    hr, cr, hoff, coff = _split(w)
    cache = bd.rec_attn_cache_create(gu.params_for(w), hoff, torch.zeros(1, dtype=torch.int64, device="cuda"),
                                     torch.zeros(1, dtype=torch.int8, device="cuda"), None, None, 20)
    try:
        out = torch.full((len(cr), w.num_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
        args = [torch.from_numpy(w.t[cr]).cuda(), _dev(w.q[cr], "bf16"), _dev(w.k[cr], "bf16"), _dev(w.v[cr], "bf16")]
        bd.rec_attn_cache_score(cache, coff, *args, out)
        torch.cuda.synchronize()
        ref = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v, rows=cr)
        gu.assert_close(w, gu.to_f64(out), ref, "empty history")
        with pytest.raises(bd.RecAttnError) as e:
            bd.rec_attn_cache_score(cache, np.array([0, 21, 21]), *args, out)
        assert e.value.code == bd.ERR_INVALID_ARG
    finally:
        bd.rec_attn_cache_free(cache)
