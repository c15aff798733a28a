"""Host-side history-compression layout (no GPU): the library's output lengths against
the oracle's on many segment specs, and argument checks."""
import numpy as np
import pytest

from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import build as bld

SPECS = [[(-1, 4)], [(256, 1), (-1, 8)], [(512, 1), (-1, 16)], [(-1, 2)], [(1024, 1), (-1, 16)],
         [(1024, 1), (-1, 8)], [(-1, 1)], [(1000, 1), (4000, 2), (5000, 3), (-1, 4)], [(3, 1), (5, 2), (-1, 7)]]


@pytest.fixture(scope="module")
def L():
    bld.build()
    return bd.lib()


@pytest.mark.parametrize("spec", range(len(SPECS)))
def test_lengths_match_the_oracle(L, orc, spec):
    rng = np.random.default_rng(spec)
    lens = rng.integers(0, 3000, size=7)
    off = np.concatenate([[0], np.cumsum(lens)])
    hb = np.array([rng.integers(0, max(1, n // 4)) if n else 0 for n in lens])
    hl = np.array([rng.integers(0, n - b + 1) for n, b in zip(lens, hb)])
    got = bd.rec_attn_compress_lengths(off, hb, hl, SPECS[spec])
    assert np.array_equal(got, orc.compress(off, hb, hl, SPECS[spec]))


def test_bad_layouts_are_rejected(L):
    off = np.array([0, 100])
    for hb, hl, segs in [([0], [101], [(-1, 2)]), ([-1], [10], [(-1, 2)]), ([0], [50], [(10, 2)]),
                         ([0], [50], [(-1, 0)]), ([0], [50], [(1, 1)] * 9)]:
        with pytest.raises(bd.RecAttnError):
            bd.rec_attn_compress_lengths(off, hb, hl, segs)
