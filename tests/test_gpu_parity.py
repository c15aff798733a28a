"""CUDA path vs the fp64 CPU oracle, element by element, through the C-ABI.

Reduced sizes (several tiles and a ragged tail, every row checked) and the five
full-size workloads (sampled rows; tile classes and visible-pair counts in full).
Outputs: max-abs 2e-2 and mean-abs 2e-3 for bf16, 1e-4 for fp32.  Tile classes
and visible-pair counts: bit-exact.
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
    "tiny_fp32": lambda: W.tiny_fp32(),
    "tiny_fp32_long": lambda: W.tiny_fp32(batch=3, n_hist=300, n_cand=37),
    "cadet": lambda: W.cadet(batch=6, n_pairs=200),
    "sort": lambda: W.sort(batch=3, n_hist=500, n_cand=50),
    "mtgr": lambda: W.mtgr(batch=4, hist=(150, 400), rt=(20, 80), cand=(10, 40)),
    "tm20k_full": lambda: W.tm20k("full", batch=2, n_hist=1500),
    "tm20k_window": lambda: W.tm20k("window", batch=2, n_hist=1500),
    # 33 tiles with no window: long enough for the softmax's lazy maximum (requests of
    # at least 32 tiles on average), every row checked
    "tm20k_full_long": lambda: W.tm20k("full", batch=2, n_hist=4150, heads=2),
    "cadet_d128": lambda: W.cadet(batch=3, n_pairs=170, heads=2, head_dim=128),
    "sort_d128": lambda: W.sort(batch=2, n_hist=300, n_cand=40, window=100, heads=2, head_dim=128),
}


def _classes_and_pairs(w, plan, full_pairs=True):
    op = gu.oracle_params(w)
    cls = bd.rec_attn_tile_classes(plan)
    np.testing.assert_array_equal(cls, oracle.tile_classes(op, w.offsets, w.t, w.types))
    if full_pairs:
        assert bd.rec_attn_visible_pairs(plan) == oracle.visible_pairs(op, w.offsets, w.t, w.types)
    assert bd.rec_attn_device_status(plan) == bd.OK


@pytest.mark.parametrize("name", sorted(SMALL))
def test_parity_all_rows(name):
    w = SMALL[name]()
    out, lse, plan = gu.run_gpu(w, with_lse=True)
    try:
        ref, ref_lse = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v,
                                        with_lse=True)
        gu.assert_close(w, gu.to_f64(out), ref, name)
        lg = lse.cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lg), fin)
        tol = 1e-4 if w.dtype == "fp32" else 2e-2
        assert np.max(np.abs(lg[fin] - ref_lse[fin]), initial=0.0) <= tol
        _classes_and_pairs(w, plan)
    finally:
        bd.rec_attn_free(plan)


def _closed_form_pairs(w):
    """Visible pairs of the TM20K workloads without the oracle: causal over globals
    then history, the target sees all user tokens and itself."""
    n_hist = int(w.offsets[1] - w.offsets[0]) - 1
    n_glob = int(np.sum(w.types[:n_hist] == W.GLOBAL))
    W_ = w.mask["window"]
    p = np.arange(n_hist, dtype=np.int64)
    if W_ == 0:
        per_req = int(np.sum(p + 1)) + n_hist + 1
    else:
        glob = p < n_glob
        hist_cnt = np.where(glob, p + 1, n_glob + (p - np.maximum(n_glob, p - W_ + 1) + 1))
        per_req = int(hist_cnt.sum()) + n_hist + 1
    return per_req * w.batch


@pytest.mark.parametrize("name", W.NAMES)
def test_parity_full_size_sampled(name):
    w = W.make(name)
    out, _, plan = gu.run_gpu(w)
    try:
        assert not torch.isnan(out).any(), "unwritten output rows"
        rows = gu.sample_rows(w)
        ref = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows)
        gu.assert_close(w, gu.to_f64(out[torch.from_numpy(rows).to(out.device)]), ref, name)
        op = gu.oracle_params(w)
        np.testing.assert_array_equal(bd.rec_attn_tile_classes(plan),
                                      oracle.tile_classes(op, w.offsets, w.t, w.types))
        if name.startswith("tm20k"):
            expect = _closed_form_pairs(w)
        else:
            expect = oracle.visible_pairs(op, w.offsets, w.t, w.types)
        assert bd.rec_attn_visible_pairs(plan) == expect
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)


RISING = {
    # 33 tiles a request with no window: the long-item softmax (lazy maximum)
    "tm20k_long": lambda: W.tm20k("full", batch=2, n_hist=4150, heads=2),
    # short requests: the plain softmax, whose reference moves past 2^8 jumps (O rescaled)
    "cadet": lambda: W.cadet(batch=4, n_pairs=300, heads=2),
    # head_dim 128: the chunked layout's rescale
    "cadet_d128": lambda: W.cadet(batch=3, n_pairs=300, heads=2, head_dim=128),
    # bidirectional history and real-time events
    "mtgr": lambda: W.mtgr(batch=3, hist=(300, 600), rt=(40, 80), cand=(10, 30), heads=2),
}


@pytest.mark.parametrize("name", sorted(RISING))
def test_parity_rising_scores(name):
    """Rows whose running maximum keeps moving: keys gain a component along a fixed
    direction that the queries share, growing with the key's position within its
    request (head 0 steeply, so most key tiles exceed the reference and O is rescaled
    or the chunk formed again; head 1 gently, with bumps, so some do and some do not).
    The time-RoPE is off so the alignment survives; every row against the oracle."""
    w = gu.rising_scores(RISING[name]())
    out, lse, plan = gu.run_gpu(w, with_lse=True)
    try:
        ref, ref_lse = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v,
                                        with_lse=True)
        gu.assert_close(w, gu.to_f64(out), ref, f"rising scores, {name}")
        lg = lse.cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lg), fin)
        assert np.max(np.abs(lg[fin] - ref_lse[fin]) / np.maximum(1.0, np.abs(ref_lse[fin])), initial=0.0) <= 2e-2
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
