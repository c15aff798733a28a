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


def _random_case(seed):
    rng = np.random.default_rng(3000 + seed)
    B = int(rng.integers(1, 6))
    lengths = [int(x) for x in rng.integers(0, 600, size=B)]
    hb = np.zeros(B, dtype=np.int64)
    hl = np.zeros(B, dtype=np.int64)
    for b, n in enumerate(lengths):
        if n and rng.random() < 0.85:
            lo = int(rng.integers(0, max(1, n // 4)))
            hi = int(rng.integers(lo, n + 1))
            hb[b], hl[b] = lo, hi - lo
    segs = [(int(rng.integers(1, 300)), int(rng.integers(1, 10))) for _ in range(int(rng.integers(1, 5)))]
    if rng.random() < 0.7:
        segs[-1] = (-1, segs[-1][1])
    else:  # bounded segments only: the last one reaches past the longest history
        covered = sum(n for n, _ in segs[:-1])
        segs[-1] = (max(segs[-1][0], int(hl.max()) - covered + int(rng.integers(0, 5)), 1), segs[-1][1])
    dtype = "fp32" if rng.random() < 0.25 else "bf16"
    width = int(rng.choice([64, 128, 256, 512])) if dtype == "bf16" else int(rng.choice([32, 64, 128]))
    T = sum(lengths)
    x = rng.standard_normal((T, width)).astype(np.float32)
    if dtype == "bf16":
        x = W.round_to_bf16_bits(x)
    t = W.EPOCH + np.sort(rng.integers(0, 10**7, size=T)).astype(np.int64)
    ty = rng.integers(0, 4, size=T).astype(np.int8)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return off, hb, hl, segs, x, t, ty, dtype


@pytest.mark.parametrize("seed", range(40))
def test_compress_random_segments(seed):
    """Seeded random batches (empty requests and histories included), history ranges and
    recency segments (1 to 4, bounded or not, groups of 1 to 9), bf16 and fp32 rows."""
    off, hb, hl, segs, x_host, t_host, ty_host, dtype = _random_case(seed)
    out_off = bd.rec_attn_compress_lengths(off, hb, hl, segs)
    ref_off, ref_x, ref_t, ref_ty = oracle.compress(off, hb, hl, segs, x_host, t_host, ty_host)
    assert np.array_equal(out_off, ref_off)
    n = int(out_off[-1])
    if n == 0:
        return
    if dtype == "bf16":
        x = torch.from_numpy(x_host.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        x = torch.from_numpy(x_host).cuda()
    x_out = torch.full((n, x.shape[1]), float("nan"), dtype=x.dtype, device=x.device)
    t_out = torch.full((n,), -1, dtype=torch.int64, device=x.device)
    ty_out = torch.full((n,), -1, dtype=torch.int8, device=x.device)
    bd.rec_attn_compress(off, hb, hl, segs, x, torch.from_numpy(t_host).cuda(), torch.from_numpy(ty_host).cuda(),
                         x_out, t_out, ty_out)
    torch.cuda.synchronize()
    assert np.array_equal(t_out.cpu().numpy(), ref_t)
    assert np.array_equal(ty_out.cpu().numpy(), ref_ty)
    got = x_out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref_x)
    if dtype == "bf16":
        assert np.all(err <= 2.0 ** -8 * np.abs(ref_x) + 1e-5), float(err.max())
    else:
        assert np.all(err <= 1e-6 * np.maximum(1.0, np.abs(ref_x))), float(err.max())
