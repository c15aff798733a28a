"""The oracle's tile classification (bounding-box interval rule) against the
brute-force mask: SKIP tiles hold no visible pair, FULL tiles hold only visible
pairs over a complete key tile, and where the rule is exact (one token type per
tile, causal or windowed positions only) the classes equal the brute-force ones.
"""
import numpy as np
import pytest

from generative_recommender_ranking_gb300 import workloads as W

T = 128


def _brute_classes(orc, p, offsets, t, ty):
    out = []
    for b in range(len(offsets) - 1):
        s, e = int(offsets[b]), int(offsets[b + 1])
        L = e - s
        m = orc.mask(p, t[s:e], ty[s:e])
        nt = (L + T - 1) // T
        for qt in range(nt):
            for kt in range(nt):
                blk = m[qt * T:(qt + 1) * T, kt * T:(kt + 1) * T]
                k_full = (kt + 1) * T <= L
                if not blk.any():
                    out.append(0)
                elif blk.all() and k_full:
                    out.append(2)
                else:
                    out.append(1)
    return np.array(out, dtype=np.uint8)


MID = {
    "tiny_fp32": lambda: W.tiny_fp32(batch=3, n_hist=300, n_cand=20),
    "cadet": lambda: W.cadet(batch=3, n_pairs=300),
    "sort": lambda: W.sort(batch=2, n_special=16, n_hist=700, n_cand=60, window=200),
    "mtgr": lambda: W.mtgr(batch=3, n_profile=32, hist=(200, 400), rt=(30, 150), cand=(20, 60)),
    "tm20k_full": lambda: W.tm20k("full", batch=2, n_hist=900, n_global=64),
    "tm20k_window": lambda: W.tm20k("window", batch=2, n_hist=900, n_global=64, window=200),
}


@pytest.mark.parametrize("name", sorted(MID))
def test_rule_is_sound(orc, name):
    w = MID[name]()
    p = orc.Params(w.num_heads, w.head_dim, **w.mask)
    rule = orc.tile_classes(p, w.offsets, w.t, w.types)
    brute = _brute_classes(orc, p, w.offsets, w.t, w.types)
    assert rule.shape == brute.shape
    # SKIP => brute SKIP; FULL => brute FULL
    assert np.all(brute[rule == 0] == 0)
    assert np.all(brute[rule == 2] == 2)
    # a tile with visible pairs is never skipped
    assert np.all(rule[brute != 0] != 0)


@pytest.mark.parametrize("window", [0, 100, 300])
def test_rule_exact_for_single_type_positions(orc, window):
    L = 1000
    t = np.arange(L, dtype=np.int64)
    ty = np.full(L, W.HIST, dtype=np.int8)
    off = np.array([0, 600, L], dtype=np.int64)
    p = orc.Params(1, 2, window=window)
    np.testing.assert_array_equal(orc.tile_classes(p, off, t, ty), _brute_classes(orc, p, off, t, ty))


def test_causal_tile_pattern_by_hand(orc):
    """Four full tiles of plain causal history: below the diagonal FULL, on it
    PARTIAL, above it SKIP."""
    L = 4 * T
    p = orc.Params(1, 2)
    cls = orc.tile_classes(p, np.array([0, L]), np.zeros(L, np.int64), np.ones(L, np.int8))
    expect = np.array([[1, 0, 0, 0], [2, 1, 0, 0], [2, 2, 1, 0], [2, 2, 2, 1]], dtype=np.uint8)
    np.testing.assert_array_equal(cls.reshape(4, 4), expect)
    # ragged last tile: a FULL-looking pair whose key tile is ragged is PARTIAL; the
    # ragged query tile may still be FULL against complete key tiles
    L = 3 * T + 5
    cls = orc.tile_classes(p, np.array([0, L]), np.zeros(L, np.int64), np.ones(L, np.int8)).reshape(4, 4)
    assert cls[3, 0] == 2 and cls[3, 3] == 1 and cls[2, 3] == 0


def test_delay_makes_old_tiles_full_and_recent_tiles_partial(orc):
    # two tiles one day apart, then a tile inside the delay window
    t = np.concatenate([np.full(T, 0), np.full(T, 86400), np.full(T, 86400 + 10)]).astype(np.int64)
    ty = np.ones(3 * T, dtype=np.int8)
    p = orc.Params(1, 2, use_delay=True, delay_s=3600)
    cls = orc.tile_classes(p, np.array([0, 3 * T]), t, ty).reshape(3, 3)
    assert cls[1, 0] == 2  # all keys a day older and earlier: FULL
    assert cls[2, 1] == 0  # keys 10 s older: inside the delay window -> SKIP
    assert cls[2, 0] == 2
    assert cls[0, 0] == 0  # equal times on the diagonal: nothing is old enough
