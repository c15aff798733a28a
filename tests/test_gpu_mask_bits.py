"""The visibility bits the attention kernels apply, bit for bit against the oracle's
mask (masked pairs get -inf, not a small constant: LazFormer review page, section 2.3,
Eq. 19-21; CADET delay rule; SORT section 3.1; MTGR hybrid mask).

rec_attn_applied_masks copies out, per (request, query tile, key tile), the 128 x 128
bits the kernels use: the mask-table rows or the in-kernel construction (tensor-core
path) and the per-pair predicate (CUDA-core path).  They are compared with
oracle.mask_block on every tile pair of the full-size workloads (sampled query tiles of
the 20K-token ones), the seeded random layouts and the table-overflow case.

The strict-masking test checks the same property through the outputs: for one query
row per request, every key it must not see gets a value row of 1e4 and a key row
aligned with the query, and the row's output must stay bit-identical."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import workloads as W
from test_gpu_mask_table import _interleaved
from test_gpu_random_masks import _case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gu.ensure_built()


def _sampled_pairs(w: W.Workload, q_tiles_per_request: int, seed: int):
    """Every key tile against the first, last and a few random query tiles of each request."""
    rng = np.random.default_rng(seed)
    out = []
    for b in range(w.batch):
        nt = (int(w.offsets[b + 1] - w.offsets[b]) + 127) // 128
        if nt == 0:
            continue
        qts = sorted({0, nt - 1, nt // 2} | set(rng.integers(0, nt, size=q_tiles_per_request).tolist()))
        for qt in qts:
            out += [(b, qt, kt) for kt in range(nt)]
    return np.array(out, dtype=np.int32)


FULL_SIZE = ("tiny_fp32", "cadet", "sort", "mtgr", "tm20k_full", "tm20k_window")


@pytest.mark.parametrize("name", FULL_SIZE)
def test_applied_masks_full_size(name):
    w = W.make(name)
    tens = gu.device_inputs(w)
    op = gu.oracle_params(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        if name.startswith("tm20k"):
            pairs = _sampled_pairs(w, 3, seed=11)
            tile_cls = None  # the planner's classes are compared in full by the parity tests
        else:
            pairs = gu.all_pairs(w)
            tile_cls = gu.tile_class_map(w, oracle.tile_classes(op, w.offsets, w.t, w.types))
        stats = gu.check_applied_masks(w, plan, pairs, op, tile_cls=tile_cls)
        assert stats[0][2] > 0, "no PARTIAL pair was checked"
        print(name, stats)
    finally:
        bd.rec_attn_free(plan)


def test_applied_masks_query_pruned_plan():
    """A target-attention plan (no user token queries): the masks are those of the full
    mask; query tiles with no computed row are never loaded."""
    w = W.cadet_serving(batch=3, n_hist=700, n_cand=90)
    tens = gu.device_inputs(w)
    op = gu.oracle_params(w)
    plan = bd.rec_attn_plan_query_pruned(gu.params_for(w), 0, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        pairs = gu.all_pairs(w)
        bits, lcls, _ = bd.rec_attn_applied_masks(plan, pairs, bd.MASK_APPLIED)
        got = gu.unpack_bits(bits)
        kept = set(oracle.kept_rows(w.offsets, w.types, 0).tolist())
        for n, (b, qt, kt) in enumerate(pairs.tolist()):
            s, e = int(w.offsets[b]), int(w.offsets[b + 1])
            rows = [r for r in range(128) if s + 128 * qt + r in kept and 128 * qt + r < e - s]
            if not rows:
                assert lcls[n] == 0xFF and not got[n].any()  # a tile of pruned queries
                continue
            blk = oracle.mask_block(op, w.t[s:e], w.types[s:e], 128 * qt, 128, 128 * kt, 128)
            if lcls[n] == 0xFF:
                assert not blk.any()
            elif lcls[n] == bd.TILE_FULL:
                assert blk[rows].all()
            else:
                assert np.array_equal(got[n][rows], blk[rows]), (b, qt, kt)
    finally:
        bd.rec_attn_free(plan)


@pytest.mark.parametrize("seed", range(64))
def test_applied_masks_random_layouts(seed):
    w = _case(seed)
    if w.total_tokens == 0:
        pytest.skip("empty batch")
    tens = gu.device_inputs(w)
    op = gu.oracle_params(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        tile_cls = gu.tile_class_map(w, oracle.tile_classes(op, w.offsets, w.t, w.types))
        gu.check_applied_masks(w, plan, gu.all_pairs(w), op, tile_cls=tile_cls)
    finally:
        bd.rec_attn_free(plan)


def test_applied_masks_table_overflow():
    """Past the table's capacity the kernels build the rows themselves: both kinds of
    PARTIAL pair are present and both match the mask."""
    w = _interleaved()
    tens = gu.device_inputs(w)
    op = gu.oracle_params(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        pairs = gu.all_pairs(w)
        _, lcls, slot = bd.rec_attn_applied_masks(plan, pairs, bd.MASK_APPLIED)
        partial = lcls == bd.TILE_PARTIAL
        assert (slot[partial] >= 0).any() and (slot[partial] < 0).any()
        gu.check_applied_masks(w, plan, pairs, op, modes=(0, 1))
    finally:
        bd.rec_attn_free(plan)


def test_applied_masks_rejects_bad_pairs():
    w = W.cadet(batch=2, n_pairs=100)
    tens = gu.device_inputs(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        for bad in ((2, 0, 0), (0, 2, 0), (0, 0, -1), (-1, 0, 0)):
            with pytest.raises(bd.RecAttnError) as ei:
                bd.rec_attn_applied_masks(plan, [bad])
            assert ei.value.code == bd.ERR_INVALID_ARG
        with pytest.raises(bd.RecAttnError):
            bd.rec_attn_applied_masks(plan, [(0, 0, 0)], mode=3)
    finally:
        bd.rec_attn_free(plan)


STRICT = ("cadet", "sort", "mtgr", "tm20k_window", "tiny_fp32")


@pytest.mark.parametrize("name", STRICT)
def test_strict_masking_outputs_bit_identical(name):
    """One query row per request: every key hidden from it gets V = 1e4 and K = 4 Q_row
    (a large score were it visible).  The row's output and lse must not change at all:
    hidden keys enter its softmax as exact zeros."""
    w = W.make(name)
    if name == "tm20k_window":
        w = W.tm20k("window", batch=4)
    rng = np.random.default_rng(5)
    op = gu.oracle_params(w)
    k2, v2 = w.k.copy(), w.v.copy()
    big = W.round_to_bf16_bits(np.full(w.v.shape[1:], 1e4, dtype=np.float32)) if w.dtype == "bf16" else 1e4
    rows, n_hidden = [], 0
    for b in range(w.batch):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        if e == s:
            continue
        i = int(rng.integers(0, e - s))
        vis = oracle.mask_block(op, w.t[s:e], w.types[s:e], i, 1, 0, e - s)[0].astype(bool)
        hid = np.nonzero(~vis)[0]
        if w.dtype == "bf16":
            qf = W.bf16_bits_to_float32(w.q[s + i])
            k2[s + hid] = W.round_to_bf16_bits(4.0 * qf)
        else:
            k2[s + hid] = 4.0 * w.q[s + i]
        v2[s + hid] = big
        rows.append(s + i)
        n_hidden += len(hid)
    assert n_hidden > 0
    outs = []
    for kk, vv in ((w.k, w.v), (k2, v2)):
        ww = W.Workload(**{**w.__dict__, "k": kk, "v": vv})
        out, lse, plan = gu.run_gpu(ww, with_lse=True)
        bd.rec_attn_free(plan)
        outs.append((out[rows].cpu(), lse[rows].cpu()))
    assert torch.equal(outs[0][0], outs[1][0]), f"{name}: an output row moved when only hidden keys changed"
    assert torch.equal(outs[0][1], outs[1][1]), f"{name}: an lse moved when only hidden keys changed"
