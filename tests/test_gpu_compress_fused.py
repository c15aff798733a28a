"""History compression fused into the attention epilogue (rec_attn_fwd_compress) vs the
oracle: oracle.compress applied to oracle.attention's output (TM20K review page, LPTM
and PATM; LazFormer review page, Eq. 16-18).  Times and types exact; each output row
within its group's summed per-row attention tolerance (max-abs 2e-2 per member row,
mean-abs 2e-3 per member row) plus one bf16 rounding of the sum."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import workloads as W
from test_gpu_compress import _hist_ranges

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gu.ensure_built()


CASES = {
    "lazformer_keep300_g8": (lambda: W.tm20k("window", batch=2, n_hist=1500, heads=2), [(300, 1), (-1, 8)]),
    "sort_keep256_g8": (lambda: W.sort(batch=2, n_hist=900, n_cand=40, window=96, heads=2), [(256, 1), (-1, 8)]),
    "mtgr_lptm": (lambda: W.mtgr(batch=3, hist=(150, 300), rt=(20, 60), cand=(10, 30), heads=2), [(-1, 2)]),
    "cadet_lptm": (lambda: W.cadet(batch=4, n_pairs=150, heads=2), [(-1, 2)]),
    "sort_g3_g32": (lambda: W.sort(batch=2, n_hist=700, n_cand=30, window=64, heads=2), [(100, 3), (-1, 32)]),
    "patm_bands": (lambda: W.tm20k("full", batch=1, n_hist=3000, heads=2), [(500, 1), (900, 2), (700, 3), (-1, 4)]),
    "cadet_d128_lptm": (lambda: W.cadet(batch=3, n_pairs=130, heads=2, head_dim=128), [(64, 1), (-1, 2)]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_compression_matches_oracle(name):
    make, segs = CASES[name]
    w = make()
    hb, hl = _hist_ranges(w)
    tens = gu.device_inputs(w)
    H, d = w.num_heads, w.head_dim
    out_off = bd.rec_attn_compress_lengths(w.offsets, hb, hl, segs)
    n = int(out_off[-1])
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        outs = []
        for _ in range(2):  # twice: the result is deterministic
            x_out = torch.full((n, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
            t_out = torch.full((n,), -1, dtype=torch.int64, device="cuda")
            ty_out = torch.full((n,), -1, dtype=torch.int8, device="cuda")
            bd.rec_attn_fwd_compress(plan, tens["q"], tens["k"], tens["v"], hb, hl, segs, x_out, t_out, ty_out)
            torch.cuda.synchronize()
            outs.append((x_out, t_out, ty_out))
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
    assert torch.equal(outs[0][0], outs[1][0])
    x_out, t_out, ty_out = outs[0]
    attn = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v)
    T = w.total_tokens
    ref_off, ref_x, ref_t, ref_ty = oracle.compress(w.offsets, hb, hl, segs, attn.reshape(T, H * d).astype(np.float32),
                                                    w.t, w.types)
    _, sizes, _, _ = oracle.compress(w.offsets, hb, hl, segs, np.ones((T, 4), dtype=np.float32), w.t, w.types)
    g = sizes[:, 0][:, None, None]  # members of each output row
    assert np.array_equal(out_off, ref_off)
    assert np.array_equal(t_out.cpu().numpy(), ref_t)
    assert np.array_equal(ty_out.cpu().numpy(), ref_ty)
    got = gu.to_f64(x_out)
    ref = ref_x.reshape(n, H, d)
    assert np.isfinite(got).all(), "unwritten output rows"
    err = np.abs(got - ref)
    assert np.all(err <= g * gu.BF16_MAX_ABS + 2.0 ** -8 * np.abs(ref)), (name, float(err.max()))
    assert float(np.mean(err / g)) <= gu.BF16_MEAN_ABS, (name, float(np.mean(err / g)))
    assert g.max() > 1, "the case merges no rows"


def test_fused_compression_rejects_unsupported():
    w = W.cadet(batch=2, n_pairs=100, heads=2)
    tens = gu.device_inputs(w)
    hb, hl = _hist_ranges(w)
    x = torch.empty((w.total_tokens, 2, 64), dtype=torch.bfloat16, device="cuda")
    t = torch.empty(w.total_tokens, dtype=torch.int64, device="cuda")
    ty = torch.empty(w.total_tokens, dtype=torch.int8, device="cuda")
    plan = bd.rec_attn_plan_query_pruned(gu.params_for(w), 10, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        with pytest.raises(bd.RecAttnError) as e:
            bd.rec_attn_fwd_compress(plan, tens["q"], tens["k"], tens["v"], hb, hl, [(-1, 2)], x, t, ty)
        assert e.value.code == bd.ERR_UNSUPPORTED
    finally:
        bd.rec_attn_free(plan)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        with pytest.raises(bd.RecAttnError) as e:
            bd.rec_attn_fwd_compress(plan, tens["q"], tens["k"], tens["v"], hb, hl, [(-1, 33)], x, t, ty)
        assert e.value.code == bd.ERR_UNSUPPORTED
    finally:
        bd.rec_attn_free(plan)
