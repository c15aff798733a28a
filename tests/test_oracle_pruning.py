"""Pins of the oracle's query pruning: the LazFormer Eq. 22 per-layer budget and the
rule that picks the computed rows (SORT section 3.2.2: only the user side is pruned;
LazFormer: the most recent N_l history tokens and every target; TA: targets only)."""
import numpy as np
import pytest

from golden_io import load_json

G, H, R, C = 0, 1, 2, 3


def test_eq22_schedule_on_the_page_defaults(orc):
    g = load_json("query_pruning_lazformer.json")
    # the compressed history length the schedule starts from
    assert g["short_term_kept"] + (g["raw_history"] - g["short_term_kept"]) // g["merge_group"] == \
        g["compressed_history"]
    sched = [orc.query_keep(g["compressed_history"], g["n_min"], l, 4) for l in range(1, 5)]
    assert sched == g["four_layer_schedule"]


def test_eq22_closed_forms(orc):
    for Lh, nmin, L in [(1152, 128, 6), (2048, 512, 3), (300, 128, 12), (20000, 128, 8)]:
        s = [orc.query_keep(Lh, nmin, l, L) for l in range(1, L + 1)]
        assert s[0] == Lh and s[-1] == nmin
        assert all(a >= b for a, b in zip(s, s[1:]))
        # linear: consecutive steps differ by at most one from the exact step
        step = (Lh - nmin) / (L - 1)
        assert all(abs((a - b) - step) <= 1.0 for a, b in zip(s, s[1:]))
    # a history shorter than N_min is never cut; one layer keeps everything
    assert [orc.query_keep(100, 128, l, 5) for l in range(1, 6)] == [100] * 5
    assert orc.query_keep(777, 128, 1, 1) == 777
    # round half away from zero: Lh = 129, N_min = 128, L = 3 -> 129, 128.5 -> 129, 128
    assert [orc.query_keep(129, 128, l, 3) for l in (1, 2, 3)] == [129, 129, 128]
    assert orc.query_keep(10, 2, 0, 3) == -1 and orc.query_keep(10, 2, 4, 3) == -1


def _rows(orc, types, keep, offsets=None):
    ty = np.array(types, dtype=np.int8)
    off = offsets if offsets is not None else [0, len(types)]
    return list(orc.kept_rows(off, ty, keep))


def test_kept_rows_hand_cases(orc):
    sort_like = [G, G, H, H, H, H, H, C, C, C]
    assert _rows(orc, sort_like, -1) == list(range(10))
    assert _rows(orc, sort_like, 3) == [4, 5, 6, 7, 8, 9]
    assert _rows(orc, sort_like, 6) == [1, 2, 3, 4, 5, 6, 7, 8, 9]  # the user side counts profile tokens
    assert _rows(orc, sort_like, 0) == [7, 8, 9]                    # target attention
    assert _rows(orc, sort_like, 50) == list(range(10))
    # MTGR: real-time events are never pruned
    mtgr_like = [G, G, H, H, H, R, R, C, C]
    assert _rows(orc, mtgr_like, 1) == [4, 5, 6, 7, 8]
    assert _rows(orc, mtgr_like, 0) == [5, 6, 7, 8]
    # LazFormer: the last history tokens (here typed GLOBAL) are the most recent ones
    laz_like = [H, H, H, H, G, G, C]
    assert _rows(orc, laz_like, 2) == [4, 5, 6]
    # several requests, one empty, each pruned on its own
    types = [H, H, C] + [] + [G, H, H, H, C, C]
    assert _rows(orc, types, 1, offsets=[0, 3, 3, 9]) == [1, 2, 6, 7, 8]


def test_kept_rows_do_not_change_the_outputs_of_kept_queries(orc):
    # pruning removes queries, never keys: the oracle's output for a kept row is the
    # same as in the unpruned layer (row by row definition), checked on a workload
    from generative_recommender_ranking_gb300 import workloads as W
    w = W.sort(batch=2, n_special=8, n_hist=200, n_cand=16, window=48)
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    full = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v)
    rows = orc.kept_rows(w.offsets, w.types, 40)
    assert len(rows) == 2 * (40 + 16)
    sub = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows)
    assert np.array_equal(sub, full[rows])
