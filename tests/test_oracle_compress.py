"""Pins of the oracle's history compression: the LazFormer Table 6 lengths, the
TM20K PATM example, LPTM pair sums, a hand-computed case, and the invariants of
summing groups (totals kept, latest member time, untouched non-history tokens)."""
import numpy as np

from golden_io import load_json

from generative_recommender_ranking_gb300 import workloads as W


def test_table6_and_patm_lengths(orc):
    g = load_json("history_compression.json")
    L = g["history"]
    for row in g["table6"]:
        segs = ([(row["keep"], 1)] if row["keep"] else []) + [(-1, row["group"])]
        assert orc.compress([0, L], [0], [L], segs)[1] == row["length"], row
    pa = g["patm"]
    n = orc.compress([0, pa["history"]], [0], [pa["history"]], [tuple(s) for s in pa["segments"]])[1]
    assert abs(n - pa["approx_length"]) <= pa["abs_tol"]
    # exactly: 1000 + 4000/2 + ceil(5000/3) + 10000/4
    assert n == 1000 + 2000 + 1667 + 2500


def test_hand_case_and_times(orc):
    x = np.arange(1, 6, dtype=np.float32)[:, None]  # history values 1..5, oldest first
    off, ox, ot, oty = orc.compress([0, 5], [0], [5], [(1, 1), (-1, 2)], x, np.array([10, 20, 30, 40, 50]),
                                    np.ones(5, np.int8))
    assert list(off) == [0, 3]
    assert ox[:, 0].tolist() == [1 + 2, 3 + 4, 5]  # four long-term tokens: two full groups
    assert ot.tolist() == [20, 40, 50]
    # three long-term tokens in groups of two: the oldest group is the partial one
    off, ox, ot, _ = orc.compress([0, 4], [0], [4], [(1, 1), (-1, 2)], x[:4], np.arange(4), np.ones(4, np.int8))
    assert ox[:, 0].tolist() == [1, 2 + 3, 4] and ot.tolist() == [0, 2, 3]


def test_lptm_pair_sums_leave_targets_alone(orc):
    w = W.tiny_fp32(batch=2, n_hist=64, n_cand=8)
    T = w.total_tokens
    x = w.q.reshape(T, -1)
    hb = np.zeros(2, dtype=np.int64)
    hl = np.full(2, 64, dtype=np.int64)
    off, ox, ot, oty = orc.compress(w.offsets, hb, hl, [(-1, 2)], x, w.t, w.types)
    assert list(np.diff(off)) == [32 + 8, 32 + 8]
    for b in range(2):
        s, o = int(w.offsets[b]), int(off[b])
        xs = x[s:s + 64].astype(np.float64)
        assert np.allclose(ox[o:o + 32], xs[0::2] + xs[1::2], rtol=0, atol=1e-12)
        assert np.array_equal(ox[o + 32:o + 40], x[s + 64:s + 72].astype(np.float64))  # candidates
        assert np.array_equal(oty[o + 32:o + 40], w.types[s + 64:s + 72])
        assert np.array_equal(ot[o:o + 32], np.maximum(w.t[s:s + 64:2], w.t[s + 1:s + 64:2]))


def test_sums_are_kept_and_specials_untouched(orc):
    w = W.sort(batch=2, n_special=16, n_hist=700, n_cand=20, window=64)
    T = w.total_tokens
    x = w.k.reshape(T, -1)
    hb = np.full(2, 16, dtype=np.int64)
    hl = np.full(2, 700, dtype=np.int64)
    segs = [(128, 1), (300, 4), (-1, 16)]
    off, ox, ot, oty = orc.compress(w.offsets, hb, hl, segs, x, w.t, w.types)
    xf = W.bf16_bits_to_float32(x).astype(np.float64)
    for b in range(2):
        s, e, o, oe = int(w.offsets[b]), int(w.offsets[b + 1]), int(off[b]), int(off[b + 1])
        n_groups = (oe - o) - 16 - 20
        assert n_groups == 128 + 300 // 4 + (700 - 428 + 15) // 16
        assert np.allclose(ox[o + 16:o + 16 + n_groups].sum(0), xf[s + 16:s + 716].sum(0), rtol=0, atol=1e-9)
        assert np.array_equal(ox[o:o + 16], xf[s:s + 16])
        assert np.array_equal(ox[oe - 20:oe], xf[e - 20:e])
        assert np.all(np.diff(ot[o + 16:o + 16 + n_groups]) >= 0)  # time order kept
