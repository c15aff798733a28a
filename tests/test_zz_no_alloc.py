"""rec_attn_fwd_noalloc: the entry point for callers that cannot allocate device
memory (a process whose inference runtime has reserved the GPU's memory for its own
allocator, or a serving loop that cannot pay cudaMalloc's latency per request).

It keeps its workspace in one static device array, so these checks call it through
the C-ABI twice in a row and compare each result with the plan-based entry points
(rec_attn_plan + rec_attn_fwd) on the same inputs, within the tolerance the other
GPU tests use and, since both run the same kernels on the same mask bits, bit for
bit; a second, different batch then checks that nothing from the first call leaks
into the next.  The device's free memory must not change across the later calls.  The file is named to be collected last, and it passes
both alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gu.ensure_built()


def _reference(w, tens):
    out, _, plan = gu.run_gpu(w, tens=tens, poison=True)
    bd.rec_attn_free(plan)
    return out


def _noalloc(w, tens):
    out = torch.full_like(tens["q"], float("nan"))
    bd.rec_attn_fwd_noalloc(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"],
                            tens["q"], tens["k"], tens["v"], out)
    torch.cuda.synchronize()
    return out


def _close(w, a, b):
    assert torch.equal(a, b), "the no-allocation path differs from the plan API"
    a64, b64 = gu.to_f64(a), gu.to_f64(b)
    assert not np.isnan(a64).any()
    d = np.abs(a64 - b64)
    if w.dtype == "bf16":
        assert d.max() <= gu.BF16_MAX_ABS and d.mean() <= gu.BF16_MEAN_ABS
    else:
        assert d.max() <= gu.FP32_MAX_ABS


@pytest.mark.parametrize("make", [
    lambda: W.sort(batch=2, n_special=16, n_hist=500, n_cand=50, window=128),
    lambda: W.cadet(batch=4, n_pairs=200),
    lambda: W.tiny_fp32(),
    # requests of 36 tiles: the planner splits their query tiles over several blocks
    lambda: W.tm20k("window", batch=2, n_hist=4500, heads=2),
])
def test_noalloc_matches_plan_api_twice_in_a_row(make):
    w = make()
    tens = gu.device_inputs(w)
    ref = _reference(w, tens)
    out = torch.full_like(tens["q"], float("nan"))
    free = []
    for _ in range(3):
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        bd.rec_attn_fwd_noalloc(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"],
                                tens["q"], tens["k"], tens["v"], out)
        torch.cuda.synchronize()
        _close(w, out, ref)
    free.append(torch.cuda.mem_get_info()[0])
    # the first call may load the library's kernels; later calls take no device memory
    assert free[1] == free[2] == free[3], free


def test_noalloc_state_does_not_leak_between_batches():
    a = W.mtgr(batch=3, hist=(200, 400), rt=(20, 60), cand=(10, 30))
    b = W.sort(batch=1, n_hist=300, n_cand=20, window=64)
    ta, tb = gu.device_inputs(a), gu.device_inputs(b)
    ra, rb = _reference(a, ta), _reference(b, tb)
    _close(a, _noalloc(a, ta), ra)
    _close(b, _noalloc(b, tb), rb)
    _close(a, _noalloc(a, ta), ra)


def test_noalloc_rejects_batches_beyond_its_workspace():
    # the rotated K alone (T x H x d x 2 bytes) exceeds the static array
    T = bd.NOALLOC_SCRATCH_BYTES // (8 * 64 * 2) + 1024
    w = W.Workload("big", 8, 64, "bf16", np.array([0, T], dtype=np.int64),
                   np.zeros(T, np.int64), np.ones(T, np.int8), None, None, None)
    dev = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(bd.RecAttnError) as e:
        bd.rec_attn_fwd_noalloc(gu.params_for(w, **dict(use_delay=False, delay_s=0, window=0,
                                                        hist_bidirectional=False, use_rope=True)),
                                w.offsets, dev, dev, dev, dev, dev, dev, dev)
    assert e.value.code == bd.ERR_UNSUPPORTED
