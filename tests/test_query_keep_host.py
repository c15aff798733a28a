"""Host-side parts of query pruning, no GPU: the library's LazFormer Eq. 22 helper
(exact integer arithmetic) against the oracle's (floating point), and argument checks
of rec_attn_plan_query_pruned."""
import ctypes

import numpy as np
import pytest

from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import build as bld


@pytest.fixture(scope="module")
def L():
    bld.build()
    return bd.lib()


def test_query_keep_matches_the_oracle(L, orc):
    for Lh in (0, 1, 100, 127, 128, 129, 1152, 2048, 20000):
        for nmin in (0, 1, 64, 128, 512):
            for n_layers in (1, 2, 3, 4, 6, 8, 12):
                for layer in range(1, n_layers + 1):
                    assert bd.rec_attn_query_keep(Lh, nmin, layer, n_layers) == \
                        orc.query_keep(Lh, nmin, layer, n_layers), (Lh, nmin, layer, n_layers)


def test_query_keep_rejects_bad_arguments(L):
    for args in [(-1, 0, 1, 1), (10, -1, 1, 1), (10, 2, 0, 3), (10, 2, 4, 3), (10, 2, 1, 0)]:
        assert bd.rec_attn_query_keep(*args) == -1


def test_pruned_plan_rejects_bad_keep(L):
    p = bd.make_params(4, 64)
    off = np.array([0, 100], dtype=np.int64)
    h = ctypes.c_void_p(123)
    code = L.rec_attn_plan_query_pruned(ctypes.byref(p), -2, 1, off.ctypes.data, 1, 1, 1, None, ctypes.byref(h))
    assert code == bd.ERR_INVALID_ARG and h.value is None
