"""Edge cases of the CUDA path: empty batches and requests, ragged lengths around
the tile size, rows with no visible key, plan reuse and determinism, the
time-shift invariance (bit-identical on the GPU, since the library works on
int64 time differences), invalid device data (reported, never a fault) and the
largest accepted request."""
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


def _custom(lengths, H=2, d=64, dtype="bf16", seed=7, types=None, t=None, mask=None):
    rng = np.random.default_rng(seed)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lengths)
    T = int(off[-1])
    if t is None:
        t = W.EPOCH + np.sort(rng.integers(0, 10**7, size=T)).astype(np.int64)
    if types is None:
        types = np.full(T, W.HIST, dtype=np.int8)
    x = [rng.standard_normal((T, H, d), dtype=np.float32) for _ in range(3)]
    if dtype == "bf16":
        x = [W.round_to_bf16_bits(a) for a in x]
    return W.Workload("custom", H, d, dtype, off, np.asarray(t, np.int64), np.asarray(types, np.int8),
                      *x, mask or dict(use_delay=False, delay_s=0, window=0, hist_bidirectional=False),
                      dict(use_rope=True, phi_min=1e-4, dt_max_s=float(W.YEAR), rope_base=6e5))


def _check_all(w):
    out, lse, plan = gu.run_gpu(w, with_lse=True)
    try:
        ref = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v)
        gu.assert_close(w, gu.to_f64(out), ref, "custom")
        op = gu.oracle_params(w)
        np.testing.assert_array_equal(bd.rec_attn_tile_classes(plan),
                                      oracle.tile_classes(op, w.offsets, w.t, w.types))
        assert bd.rec_attn_visible_pairs(plan) == oracle.visible_pairs(op, w.offsets, w.t, w.types)
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
    return out


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("fp32", 32)])
def test_ragged_lengths_and_empty_requests(dtype, d):
    _check_all(_custom([1, 0, 127, 128, 129, 0, 255, 256, 257, 3], d=d, dtype=dtype))


def test_empty_batch_and_all_empty_requests():
    for lengths in ([], [0, 0, 0]):
        w = _custom(lengths)
        tens = gu.device_inputs(w)
        plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
        out = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
        bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out)
        assert bd.rec_attn_tile_classes(plan).size == 0
        assert bd.rec_attn_visible_pairs(plan) == 0
        bd.rec_attn_free(plan)


def test_rows_without_visible_keys_are_zero():
    # every timestamp equal and a one-hour delay: nothing is old enough, except the
    # candidates' self pairs
    L = 300
    ty = np.full(L, W.HIST, dtype=np.int8)
    ty[-20:] = W.CAND
    w = _custom([L, 170], types=np.concatenate([ty, np.full(170, W.HIST, np.int8)]),
                t=np.full(L + 170, W.EPOCH, dtype=np.int64),
                mask=dict(use_delay=True, delay_s=3600, window=0, hist_bidirectional=False))
    out = _check_all(w)
    o = out.float().cpu().numpy()
    assert np.all(o[:L - 20] == 0.0) and np.all(o[L:] == 0.0)
    np.testing.assert_array_equal(o[L - 20:L], W.bf16_bits_to_float32(w.v[L - 20:L]))


def test_time_shift_is_bit_identical_and_plan_reuse_is_deterministic():
    w = W.sort(batch=3, n_hist=400, n_cand=30)
    tens = gu.device_inputs(w)
    out1, _, plan = gu.run_gpu(w, tens=tens)
    out2 = torch.empty_like(out1)
    bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out2)   # same plan, second call
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    bd.rec_attn_free(plan)
    tens["t"] = tens["t"] + 123_456_789
    out3, _, plan = gu.run_gpu(w, tens=tens)
    bd.rec_attn_free(plan)
    assert torch.equal(out1, out3)


def test_invalid_device_types_are_reported_not_faulted():
    w = _custom([200, 100])
    tens = gu.device_inputs(w)
    tens["ty"][5] = 7
    tens["ty"][250] = -3
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    out = torch.empty_like(tens["q"])
    bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out)
    assert bd.rec_attn_device_status(plan) == bd.ERR_DEVICE_INPUT
    bd.rec_attn_free(plan)
    # offsets on the device that disagree with the host copy are reported too
    w = _custom([200, 100])
    tens = gu.device_inputs(w)
    tens["off_d"][1] = 150
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    assert bd.rec_attn_device_status(plan) == bd.ERR_DEVICE_INPUT
    bd.rec_attn_free(plan)


def test_host_argument_errors_on_gpu():
    w = _custom([130])
    tens = gu.device_inputs(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    with pytest.raises(bd.RecAttnError) as e:   # output aliasing an input
        bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], tens["q"])
    assert e.value.code == bd.ERR_INVALID_ARG
    with pytest.raises(bd.RecAttnError):       # misaligned pointer
        bd.rec_attn_fwd(plan, tens["q"].data_ptr() + 2, tens["k"], tens["v"], torch.empty_like(tens["q"]))
    bd.rec_attn_free(plan)


def test_longest_request_sampled():
    L = bd.MAX_REQUEST_LEN
    rng = np.random.default_rng(11)
    t = W.EPOCH + np.cumsum(rng.integers(1, 100, size=L)).astype(np.int64)
    ty = np.full(L, W.HIST, dtype=np.int8)
    ty[:64] = W.GLOBAL
    ty[-8:] = W.CAND
    w = _custom([L], H=1, t=t, types=ty, mask=dict(use_delay=False, delay_s=0, window=1024,
                                                    hist_bidirectional=False))
    out, _, plan = gu.run_gpu(w)
    try:
        rows = np.array([0, 63, 64, 1000, 131071, 131072, L - 9, L - 8, L - 1], dtype=np.int64)
        ref = oracle.attention(gu.oracle_params(w), w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows)
        gu.assert_close(w, gu.to_f64(out[torch.from_numpy(rows).cuda()]), ref, "max length")
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)


def test_bounded_wait_times_out_and_the_device_stays_usable():
    # the kernels' bounded mbarrier wait, on a barrier nothing arrives at, must give up
    # with REC_ATTN_ERR_TIMEOUT in the status word after its limit (50 ms here)
    assert bd.rec_attn_check_wait_timeout(50) == bd.ERR_TIMEOUT
    w = W.sort(batch=1, n_hist=200, n_cand=10, window=64)
    out, _, plan = gu.run_gpu(w)
    try:
        assert bd.rec_attn_device_status(plan) == bd.OK
        assert not torch.isnan(out).any()
    finally:
        bd.rec_attn_free(plan)


@pytest.mark.parametrize("case", ["sorted", "unsorted_within_tile", "unsorted_across_tiles", "interleaved_types"])
def test_time_clauses_with_and_without_sorted_runs(case):
    # The planner turns a time clause into a position bound only when the key type's
    # tokens form one contiguous run with non-decreasing times; every other layout
    # must take the per-key time path and give the same result as the oracle.
    rng = np.random.default_rng(21)
    lengths = [300, 260]
    T = sum(lengths)
    t = W.EPOCH + np.sort(rng.integers(0, 30 * 86400, size=T)).astype(np.int64)
    types = np.full(T, W.HIST, dtype=np.int8)
    for b, (s, n) in enumerate(zip([0, 300], lengths)):
        types[s + n - 40:s + n - 20] = W.RT
        types[s + n - 20:s + n] = W.CAND
        t[s + n - 20:s + n] = t[s + n - 21] + 10
    if case == "unsorted_within_tile":
        t[10], t[11] = t[11] + 7200, t[10]
    elif case == "unsorted_across_tiles":
        t[127], t[128] = t[128] + 7200, t[127]
    elif case == "interleaved_types":
        types[50:60] = W.RT  # real-time events inside the history: RT no longer one run
    w = _custom(lengths, t=t, types=types, mask=dict(use_delay=True, delay_s=3600, window=0,
                                                     hist_bidirectional=False))
    _check_all(w)


def test_split_planner_with_empty_and_tiny_requests():
    """Requests averaging 32 tiles or more: the planner splits each request's query tiles
    over several blocks.  Empty and one-token requests sit between the long ones."""
    lengths = [8000, 0, 1, 9000, 0, 7000]
    rng = np.random.default_rng(23)
    T = sum(lengths)
    t = W.EPOCH + np.sort(rng.integers(0, 10**7, size=T)).astype(np.int64)
    ty = np.full(T, W.HIST, dtype=np.int8)
    s = 0
    for n in lengths:  # a few GLOBAL tokens first and candidates last in each request
        if n > 100:
            ty[s:s + 16] = W.GLOBAL
            ty[s + n - 40:s + n] = W.CAND
            t[s + n - 40:s + n] = t[s + n - 41]
        s += n
    w = _custom(lengths, t=t, types=ty, mask=dict(use_delay=True, delay_s=3600, window=700,
                                                   hist_bidirectional=False))
    n_tiles = sum((n + 127) // 128 for n in lengths)
    assert -(-n_tiles // len(lengths)) >= 32  # the split planner
    out, lse, plan = gu.run_gpu(w, with_lse=True)
    try:
        op = gu.oracle_params(w)
        np.testing.assert_array_equal(bd.rec_attn_tile_classes(plan),
                                      oracle.tile_classes(op, w.offsets, w.t, w.types))
        assert bd.rec_attn_visible_pairs(plan) == oracle.visible_pairs(op, w.offsets, w.t, w.types)
        rows = gu.sample_rows(w, per_request=64, max_requests=len(lengths))
        ref = oracle.attention(op, w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows)
        gu.assert_close(w, gu.to_f64(out[torch.from_numpy(rows).cuda()]), ref, "split planner")
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)


@pytest.mark.parametrize("case", ["cadet", "tm20k_long", "cadet_gated", "sort_d128"])
def test_output_at_16_byte_offset_is_identical(case):
    """O goes out as 32-byte stores when out is 32-byte aligned and as 16-byte stores
    otherwise (the interface promises 16); a buffer 16 bytes past a 32-byte boundary gets
    exactly the aligned result (plain, long-item, gated and head_dim 128 kernels)."""
    make = {"cadet": lambda: W.cadet(batch=3, n_pairs=150), "cadet_gated": lambda: W.cadet(batch=3, n_pairs=150),
            "tm20k_long": lambda: W.tm20k("full", batch=1, n_hist=4150, heads=2),
            "sort_d128": lambda: W.sort(batch=2, n_hist=300, n_cand=40, window=100, heads=2, head_dim=128)}[case]
    w = make()
    tens = gu.device_inputs(w)
    plan = bd.rec_attn_plan(gu.params_for(w), tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    try:
        n = tens["q"].numel()
        aligned = torch.full_like(tens["q"], float("nan"))
        buf = torch.full((n + 64,), float("nan"), dtype=tens["q"].dtype, device=aligned.device)
        lead = (-buf.data_ptr() % 32) // buf.element_size() + 16 // buf.element_size()
        offset = buf[lead:lead + n].view(tens["q"].shape)
        assert offset.data_ptr() % 32 == 16 and aligned.data_ptr() % 32 == 0
        outs = (aligned, offset)
        if case == "cadet_gated":
            g = gu.device_inputs(W.Workload(**{**w.__dict__, "q": W.fused_inputs(w).out_gate}))["q"]
            for o in outs:
                bd.rec_attn_fwd_fused(plan, tens["q"], tens["k"], tens["v"], o, None, None, out_gate=g)
        else:
            for o in outs:
                bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], o)
        torch.cuda.synchronize()
        assert bd.rec_attn_device_status(plan) == bd.OK
    finally:
        bd.rec_attn_free(plan)
    assert not torch.isnan(aligned).any()
    assert torch.equal(aligned, offset)
