"""History compression on the GPU (rec_attn_compress) vs the oracle: every output row,
timestamps and types exactly, values within one bf16 rounding of the fp32 sum."""
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


def _hist_ranges(w):
    hb, hl = [], []
    for b in range(w.batch):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        idx = np.nonzero(w.types[s:e] == W.HIST)[0]
        hb.append(int(idx[0]) if len(idx) else 0)
        hl.append(len(idx))
    return np.array(hb), np.array(hl)


CASES = {
    "lazformer_keep1024_g8": (lambda: W.tm20k("full", batch=2, n_hist=3000), [(1024, 1), (-1, 8)]),
    "lazformer_keep256_g8": (lambda: W.sort(batch=3, n_hist=2048, n_cand=40), [(256, 1), (-1, 8)]),
    "lptm_pairs": (lambda: W.mtgr(batch=4), [(-1, 2)]),
    "patm_bands": (lambda: W.tm20k("window", batch=1, n_hist=20000), [(1000, 1), (4000, 2), (5000, 3), (-1, 4)]),
    "fp32_groups": (lambda: W.tiny_fp32(batch=3, n_hist=300, n_cand=9), [(17, 1), (-1, 5)]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_compress_parity(name):
    make, segs = CASES[name]
    w = make()
    hb, hl = _hist_ranges(w)
    T = w.total_tokens
    x_host = w.k.reshape(T, -1)
    tens = gu.device_inputs(w)
    x = tens["k"].reshape(T, -1)
    out_off = bd.rec_attn_compress_lengths(w.offsets, hb, hl, segs)
    n = int(out_off[-1])
    x_out = torch.full((n, x.shape[1]), float("nan"), dtype=x.dtype, device=x.device)
    t_out = torch.full((n,), -1, dtype=torch.int64, device=x.device)
    ty_out = torch.full((n,), -1, dtype=torch.int8, device=x.device)
    bd.rec_attn_compress(w.offsets, hb, hl, segs, x, tens["t"], tens["ty"], x_out, t_out, ty_out)
    torch.cuda.synchronize()
    ref_off, ref_x, ref_t, ref_ty = oracle.compress(w.offsets, hb, hl, segs, x_host, w.t, w.types)
    assert np.array_equal(out_off, ref_off)
    assert np.array_equal(t_out.cpu().numpy(), ref_t)
    assert np.array_equal(ty_out.cpu().numpy(), ref_ty)
    got = x_out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref_x)
    if w.dtype == "bf16":
        # one rounding of the fp32 sum to bf16 (2^-9 relative) plus fp32 summation error
        assert np.all(err <= 2.0 ** -8 * np.abs(ref_x) + 1e-5), float(err.max())
    else:
        assert np.all(err <= 1e-6 * np.maximum(1.0, np.abs(ref_x))), float(err.max())
