"""Pins of the CPU oracle against what the pages and mathematics fix.

Every check here compares the oracle with something other than itself: numbers
printed on the pages (tests/golden), hand-enumerated masks, closed forms, brute
force, invariants and a library routine (torch SDPA in float64).
"""
import math

import numpy as np
import pytest
import torch

from golden_io import load_json, load_mask, mask_files

YEAR = 365 * 86400
DAY = 86400


def _params(orc, **kw):
    base = dict(num_heads=1, head_dim=2)
    base.update(kw)
    return orc.Params(**base)


def _angle(orc, p, t, pair):
    """Rotation angle the oracle applies to component pair `pair` at time t."""
    x = np.zeros(p.head_dim)
    x[2 * pair] = 1.0
    y = orc.rope(p, t, x)
    return math.atan2(y[2 * pair + 1], y[2 * pair])


# --------------------------------------------------------------------------- RoPE

def test_rope_clock_hands_match_page(orc):
    g = load_json("time_rope_clock.json")
    # The fastest hand of the page: phi_min * base rad per year.  A d = 2 head whose
    # only pair turns at that speed (phi_min := 60 rad over dt_max = 1 year).
    fast = g["fastest_rad_per_year"]["value"]
    assert abs(g["phi_min"] * g["rope_base"] - fast) <= g["fastest_rad_per_year"]["abs_tol"]
    p = _params(orc, phi_min=g["phi_min"] * g["rope_base"], dt_max_s=float(YEAR), rope_base=2.0)
    per_day = _angle(orc, p, DAY, 0)
    per_hour = _angle(orc, p, 3600, 0)
    assert abs(per_day - g["fastest_rad_per_day"]["value"]) <= g["fastest_rad_per_day"]["abs_tol"]
    assert abs(per_hour - g["fastest_rad_per_hour"]["value"]) <= g["fastest_rad_per_hour"]["abs_tol"]
    # one full turn in ~38.2 days: angle(turn) = 2*pi
    turn_days = 2 * math.pi / per_day
    assert abs(turn_days - g["fastest_turn_days"]["value"]) <= g["fastest_turn_days"]["abs_tol"]


def test_rope_clock_example_scores(orc):
    """Query and key aligned on one pair, 38.0 days apart: the pair's score is the
    cosine of the angle difference (1.00 for the 60 rad/yr hand, 0.81 for 6 rad/yr)."""
    g = load_json("time_rope_clock.json")["clock_example"]
    dt = int(round(g["delta_days"] * DAY))
    for speed, key in ((g["fast_hand_rad_per_year"], "fast_hand_cos"),
                       (g["slow_hand_rad_per_year"], "slow_hand_cos")):
        p = _params(orc, phi_min=float(speed), dt_max_s=float(YEAR), rope_base=3.0)
        t_k = 1_700_000_000
        qr = orc.rope(p, t_k + dt, np.array([1.0, 0.0]))
        kr = orc.rope(p, t_k, np.array([1.0, 0.0]))
        score = float(qr @ kr)
        assert abs(score - g[key]["value"]) <= g[key]["abs_tol"], (speed, score)
    p = _params(orc, phi_min=float(g["slow_hand_rad_per_year"]), dt_max_s=float(YEAR), rope_base=3.0)
    ang = _angle(orc, p, dt, 0)
    assert abs(ang - g["slow_hand_angle_rad"]["value"]) <= g["slow_hand_angle_rad"]["abs_tol"]


def test_rope_pair_frequencies_closed_form(orc):
    """Slowest pair turns exactly phi_min over dt_max; consecutive pairs are base^(2/d)
    apart; extrapolating one pair past the last reaches phi_min * base (the page's
    approximate fastest hand)."""
    g = load_json("time_rope_clock.json")
    d = 64
    p = _params(orc, head_dim=d, phi_min=1e-4, dt_max_s=float(YEAR), rope_base=6e5)
    a0 = _angle(orc, p, YEAR, 0)
    assert abs(a0 - g["slowest_pair_rad_over_dt_max"]["value"]) <= 1e-12 * 1e-4 + 1e-18
    # use a short interval so no angle wraps: rates in rad/s
    t = 1000
    rates = [_angle(orc, p, t, i) / t for i in range(d // 2)]
    ratio = 6e5 ** (2.0 / d)
    for i in range(d // 2 - 1):
        assert rates[i + 1] / rates[i] == pytest.approx(ratio, rel=1e-9)
    assert rates[-1] * ratio * YEAR == pytest.approx(1e-4 * 6e5, rel=1e-9)
    # the exact fastest pair at d = 64 is phi_min * base^((d-2)/d) rad per year
    assert rates[-1] * YEAR == pytest.approx(1e-4 * 6e5 ** ((d - 2) / d), rel=1e-9)


def test_rope_is_a_rotation_and_pairs_are_adjacent(orc):
    rng = np.random.default_rng(0)
    p = _params(orc, head_dim=8, phi_min=1e-4, dt_max_s=float(YEAR), rope_base=6e5)
    x = rng.standard_normal(8)
    y = orc.rope(p, 123456789, x)
    for i in range(4):  # each adjacent pair keeps its norm
        assert np.hypot(*y[2 * i:2 * i + 2]) == pytest.approx(np.hypot(*x[2 * i:2 * i + 2]), rel=1e-12)
    # t = 0 is the identity
    assert np.array_equal(orc.rope(p, 0, x), x)


# --------------------------------------------------------------------------- mask

@pytest.mark.parametrize("fname", mask_files())
def test_mask_matches_hand_enumeration(orc, fname):
    types, times, prm, expect = load_mask(fname)
    p = _params(orc, window=int(prm["window"]),
                use_delay=prm["delay"] != "none",
                delay_s=0 if prm["delay"] == "none" else int(prm["delay"]),
                hist_bidirectional=bool(int(prm["bidirectional"])))
    got = orc.mask(p, times, types)
    assert np.array_equal(got, expect), f"\n{got}\n!=\n{expect}"


@pytest.mark.parametrize("fname", mask_files())
def test_mask_block_matches_hand_enumeration(orc, fname):
    """Every block of the hand-enumerated masks, with indices running past the request
    end (those entries are 0: there is no such token)."""
    types, times, prm, expect = load_mask(fname)
    p = _params(orc, window=int(prm["window"]),
                use_delay=prm["delay"] != "none",
                delay_s=0 if prm["delay"] == "none" else int(prm["delay"]),
                hist_bidirectional=bool(int(prm["bidirectional"])))
    L = len(types)
    padded = np.zeros((L + 3, L + 3), dtype=np.uint8)
    padded[:L, :L] = expect
    for i0 in range(L + 1):
        for j0 in range(L + 1):
            for ni, nj in ((1, 1), (2, 3), (L, 1), (3, L + 3 - j0)):
                ni = min(ni, L + 3 - i0)
                got = orc.mask_block(p, times, types, i0, ni, j0, nj)
                assert np.array_equal(got, padded[i0:i0 + ni, j0:j0 + nj]), (fname, i0, j0, ni, nj)


def test_mask_block_causal_closed_form(orc):
    """A causal history of L tokens: the block of rows [i0, i0+n) x keys [j0, j0+n)
    holds #{(i, j): j <= i} (counted in closed form), here for 128-token tiles."""
    L = 1000
    t = np.zeros(L, dtype=np.int64)
    ty = np.ones(L, dtype=np.int8)
    p = _params(orc)
    for qt, kt in ((0, 0), (3, 1), (2, 5), (7, 7), (7, 3)):
        i0, j0, n = 128 * qt, 128 * kt, 128
        blk = orc.mask_block(p, t, ty, i0, n, j0, n)
        expect = 0
        for i in range(i0, min(i0 + n, L)):
            lo, hi = j0, min(j0 + n, L, i + 1)
            expect += max(0, hi - lo)
        assert int(blk.sum()) == expect, (qt, kt)


def test_pair_counts_match_page(orc):
    g = load_json("pair_counts.json")
    L, N = g["L"], g["N"]
    types = np.array([1] * L + [3] * N, dtype=np.int8)
    t = np.zeros(L + N, dtype=np.int64)
    off = np.array([0, L + N], dtype=np.int64)
    p = _params(orc)
    n_iso = orc.visible_pairs(p, off, t, types)
    assert n_iso == L * (L + 1) // 2 + L * N + N
    assert abs(n_iso / 1e6 - g["isolated_pairs_millions"]["value"]) <= g["isolated_pairs_millions"]["abs_tol"]
    # full visibility over all L + N tokens gives the page's (L + N)^2
    pb = _params(orc, hist_bidirectional=True)
    n_full = orc.visible_pairs(pb, off, t, np.ones(L + N, dtype=np.int8))
    assert n_full == (L + N) ** 2
    assert abs(n_full / 1e6 - g["full_pairs_millions"]["value"]) <= g["full_pairs_millions"]["abs_tol"]
    # plain causal over L tokens: L(L+1)/2
    assert orc.visible_pairs(p, np.array([0, L]), t[:L], types[:L]) == L * (L + 1) // 2


def test_requests_never_see_each_other(orc):
    p = _params(orc, hist_bidirectional=True)
    t = np.zeros(10, dtype=np.int64)
    ty = np.ones(10, dtype=np.int8)
    assert orc.visible_pairs(p, np.array([0, 3, 10]), t, ty) == 9 + 49
    assert orc.visible_pairs(p, np.array([0, 0, 10, 10]), t, ty) == 100  # empty requests


def test_delay_boundary_and_overflow(orc):
    p = _params(orc, use_delay=True, delay_s=3600)
    # t_j = t_i - delta stays visible, one second later is masked
    assert orc.visible(p, 5, 10_000, 1, 4, 10_000 - 3600, 1)
    assert not orc.visible(p, 5, 10_000, 1, 4, 10_000 - 3599, 1)
    # non-candidate self pair is masked under delay; candidate self pair is exempt
    assert not orc.visible(p, 5, 10_000, 1, 5, 10_000, 1)
    assert orc.visible(p, 5, 10_000, 3, 5, 10_000, 3)
    # extreme timestamps: t_i - delta below INT64_MIN means nothing is old enough
    i64min = -(2 ** 63)
    assert not orc.visible(p, 5, i64min + 10, 1, 4, i64min, 1)
    assert orc.visible(_params(orc, use_delay=True, delay_s=0), 5, i64min, 1, 4, i64min, 1)


# --------------------------------------------------------------------------- attention

def _single_request(orc, types, t, H, d, rng, dtype=np.float32):
    L = len(types)
    q = rng.standard_normal((L, H, d)).astype(dtype)
    k = rng.standard_normal((L, H, d)).astype(dtype)
    v = rng.standard_normal((L, H, d)).astype(dtype)
    return np.array([0, L], dtype=np.int64), np.asarray(t, dtype=np.int64), np.asarray(types, np.int8), q, k, v


def test_attention_equals_sdpa_without_mask_or_rope(orc):
    rng = np.random.default_rng(1)
    H, d, L = 2, 16, 37
    off, t, ty, q, k, v = _single_request(orc, [1] * L, rng.integers(0, 10**9, L), H, d, rng)
    p = _params(orc, num_heads=H, head_dim=d, hist_bidirectional=True, use_rope=False)
    got = orc.attention(p, off, t, ty, q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(a.astype(np.float64)).permute(1, 0, 2) for a in (q, k, v))).permute(1, 0, 2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)
    # plain causal history equals SDPA with is_causal
    pc = _params(orc, num_heads=H, head_dim=d, use_rope=False)
    got = orc.attention(pc, off, t, ty, q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(a.astype(np.float64)).permute(1, 0, 2) for a in (q, k, v)),
        is_causal=True).permute(1, 0, 2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_attention_equals_sdpa_with_explicit_mask_and_rotation(orc):
    """Any mask: SDPA with the hand-enumerated boolean mask, on keys/queries the
    oracle rotated (rotation pinned separately above)."""
    rng = np.random.default_rng(2)
    types, times, prm, expect = load_mask("mask_sort_u2u_c2u_c2c.txt")
    H, d = 2, 8
    times = times + rng.integers(0, 10**6, len(times))
    off, t, ty, q, k, v = _single_request(orc, types, times, H, d, rng)
    p = _params(orc, num_heads=H, head_dim=d, window=2)
    got = orc.attention(p, off, t, ty, q, k, v)
    rot = lambda x: np.stack([[orc.rope(p, t[i], x[i, h]) for h in range(H)] for i in range(len(t))])
    qr, kr = rot(q.astype(np.float64)), rot(k.astype(np.float64))
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(a).permute(1, 0, 2) for a in (qr, kr, v.astype(np.float64))),
        attn_mask=torch.from_numpy(expect.astype(bool))).permute(1, 0, 2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_softmax_special_cases(orc):
    rng = np.random.default_rng(3)
    types, times, prm, expect = load_mask("mask_cadet_delay.txt")
    H, d = 1, 4
    off, t, ty, q, k, v = _single_request(orc, types, times, H, d, rng)
    p = _params(orc, num_heads=H, head_dim=d, use_delay=True, delay_s=3600)
    out, lse = orc.attention(p, off, t, ty, q, k, v, with_lse=True)
    # row 0 sees nothing: zero output, lse = -inf
    assert np.all(out[0] == 0.0) and lse[0, 0] == -np.inf
    # rows 1 and 2 see exactly one key (token 0): the output is that value row
    np.testing.assert_array_equal(out[1], v[0].astype(np.float64))
    np.testing.assert_array_equal(out[2], v[0].astype(np.float64))
    # uniform scores (q = 0): mean of the visible values
    q0 = np.zeros_like(q)
    out = orc.attention(p, off, t, ty, q0, k, v)
    np.testing.assert_allclose(out[3], (v[0].astype(np.float64) + v[3].astype(np.float64)) / 2,
                               rtol=1e-14)
    # lse of a row with one visible key is its scaled score
    p2 = _params(orc, num_heads=H, head_dim=d, use_delay=True, delay_s=3600, use_rope=False)
    _, lse = orc.attention(p2, off, t, ty, q, k, v, with_lse=True)
    s = float(q[1, 0].astype(np.float64) @ k[0, 0].astype(np.float64)) / math.sqrt(d)
    assert lse[1, 0] == pytest.approx(s, rel=1e-14, abs=1e-14)


def test_rows_subset_and_threads_agree_with_full(orc):
    from generative_recommender_ranking_gb300 import workloads
    w = workloads.sort(batch=2, n_special=4, n_hist=150, n_cand=12, window=32)
    p = orc.Params(w.num_heads, w.head_dim, window=32)
    full = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v, threads=1)
    rows = np.array([0, 5, 77, 165, 166, 200, 331], dtype=np.int64)
    sub = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows, threads=4)
    np.testing.assert_array_equal(sub, full[rows])


def test_bf16_inputs_are_widened_exactly(orc):
    from generative_recommender_ranking_gb300 import workloads as W
    rng = np.random.default_rng(4)
    x = rng.standard_normal((20, 1, 4)).astype(np.float32)
    bits = W.round_to_bf16_bits(x)
    xf = W.bf16_bits_to_float32(bits)
    assert np.array_equal(xf, torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    off = np.array([0, 20])
    t = np.arange(20, dtype=np.int64) * 100
    ty = np.ones(20, dtype=np.int8)
    p = _params(orc, num_heads=1, head_dim=4)
    np.testing.assert_array_equal(orc.attention(p, off, t, ty, bits, bits, bits),
                                  orc.attention(p, off, t, ty, xf, xf, xf))
