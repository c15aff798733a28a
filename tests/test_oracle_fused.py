"""Pins of the oracle's fused steps: QK-RMSNorm, the Q/K sigmoid gates and the
attention output gate (CADET self-gating; SORT "Attention Gate & QK Norm"; TM20K
QK Norm).

Each check compares the oracle with a value the pages print, a closed form, a
limit of the definition or an invariant, never with itself.
"""
import math

import numpy as np
import pytest

from golden_io import load_json

from generative_recommender_ranking_gb300 import workloads as W


def test_sigmoid_matches_the_page_example(orc):
    g = load_json("self_gate_cadet.json")
    s = orc.sigmoid(g["gate_input"])
    assert abs(s - g["sigmoid"]["value"]) <= g["sigmoid"]["abs_tol"]
    assert abs(s - g["kept_fraction"]["value"]) <= g["kept_fraction"]["abs_tol"]


def test_sigmoid_closed_forms(orc):
    assert orc.sigmoid(0.0) == 0.5
    for x in (0.3, 1.7, 5.0, -4.2):
        assert abs(orc.sigmoid(x) + orc.sigmoid(-x) - 1.0) < 1e-15
        assert abs(orc.sigmoid(x) - math.exp(x) / (1.0 + math.exp(x))) < 1e-15


def test_rmsnorm_closed_forms(orc):
    # (3, 4): mean square 12.5
    y = orc.rmsnorm([3.0, 4.0], [1.0, 1.0], 0.0)
    assert np.allclose(y, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    # epsilon enters under the root: (1, 1), eps = 1 -> 1 / sqrt(2)
    y = orc.rmsnorm([1.0, 1.0], [1.0, 1.0], 1.0)
    assert np.allclose(y, [2 ** -0.5] * 2, rtol=0, atol=1e-15)
    # a constant vector maps to the gains (eps = 0), with its sign
    w = np.array([0.5, 2.0, -1.0, 3.0])
    assert np.allclose(orc.rmsnorm([-7.0] * 4, w, 0.0), -w, rtol=0, atol=1e-14)
    # gains scale each output component
    y1 = orc.rmsnorm([1.0, -2.0, 3.0, 0.5], [1.0] * 4, 0.0)
    y2 = orc.rmsnorm([1.0, -2.0, 3.0, 0.5], w, 0.0)
    assert np.allclose(y2, y1 * w, rtol=0, atol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance(orc):
    rng = np.random.default_rng(7)
    for d in (2, 32, 64, 128):
        x = rng.normal(size=d) * 3.0
        y = orc.rmsnorm(x, np.ones(d), 0.0)
        assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-13
        for c in (1e-3, 0.25, 40.0):
            assert np.allclose(orc.rmsnorm(c * x, np.ones(d), 0.0), y, rtol=0, atol=1e-12)


def _small(name="sort"):
    return W.make(name, batch=2) if name != "sort" else W.sort(batch=2, n_special=8, n_hist=120, n_cand=12, window=32)


def _run(orc, w, fused=None, rows=None, with_lse=False):
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    return orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows, fused=fused,
                         with_lse=with_lse)


def _bf16(x):
    """Round fp32 values to bf16 bit patterns (round to nearest even)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def test_open_gates_and_no_norm_reduce_to_plain_attention(orc):
    w = _small()
    T, H, d = w.q.shape
    big = _bf16(np.full((T, H, d), 40.0))  # sigmoid(40) = 1 - 4e-18
    f = orc.Fused(q_gate=big, k_gate=big, out_gate=big)
    assert np.allclose(_run(orc, w, f), _run(orc, w), rtol=0, atol=1e-12)


def test_zero_output_gate_halves_the_output(orc):
    w = _small()
    zero = np.zeros(w.q.shape, dtype=np.uint16)  # bf16 +0.0
    base = _run(orc, w)
    assert np.array_equal(_run(orc, w, orc.Fused(out_gate=zero)), 0.5 * base)


def test_closed_key_gates_give_the_mean_of_visible_values(orc):
    # sigmoid(-80) ~ 1.8e-35: every key vector vanishes, all scores are 0 and each
    # row's output is the plain mean of the value rows it sees
    w = _small()
    closed = _bf16(np.full(w.q.shape, -80.0))
    out = _run(orc, w, orc.Fused(k_gate=closed))
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    vf = (w.v.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for b in range(len(w.offsets) - 1):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        m = orc.mask(p, w.t[s:e], w.types[s:e]).astype(np.float64)
        n = m.sum(1)
        for h in range(w.num_heads):
            ref = np.where(n[:, None] > 0, (m @ vf[s:e, h]) / np.maximum(n, 1)[:, None], 0.0)
            assert np.allclose(out[s:e, h], ref, rtol=0, atol=1e-12)


def test_qk_norm_bounds_every_score(orc):
    # unit gains: |q'| = |k'| = sqrt(d), RoPE keeps norms, so |score| <= scale * d =
    # sqrt(d), which bounds the log-sum-exp of every row with n visible keys by
    # [-sqrt(d) + log n, sqrt(d) + log n]
    w = _small("cadet")
    T, H, d = w.q.shape
    ones = np.ones((H, d))
    f = orc.Fused(q_norm_w=ones, k_norm_w=ones, norm_eps=0.0)
    _, lse = _run(orc, w, f, with_lse=True)
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    for b in range(len(w.offsets) - 1):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        n = orc.mask(p, w.t[s:e], w.types[s:e]).sum(1)
        for h in range(H):
            vis = n > 0
            bound = math.sqrt(d)
            assert np.all(lse[s:e, h][vis] <= bound + np.log(n[vis]) + 1e-9)
            assert np.all(lse[s:e, h][vis] >= -bound + np.log(n[vis]) - 1e-9)
            assert np.all(np.isneginf(lse[s:e, h][~vis]))


def test_qk_norm_makes_scores_independent_of_input_scale(orc):
    w = _small("mtgr")
    H, d = w.num_heads, w.head_dim
    rng = np.random.default_rng(3)
    f = orc.Fused(q_norm_w=rng.uniform(0.5, 1.5, (H, d)), k_norm_w=rng.uniform(0.5, 1.5, (H, d)), norm_eps=0.0)
    qf = (w.q.astype(np.uint32) << 16).view(np.float32)
    kf = (w.k.astype(np.uint32) << 16).view(np.float32)
    w2 = W.Workload(**{**w.__dict__, "q": _bf16(qf * 4.0), "k": _bf16(kf * 0.125)})
    # scaling by powers of two is exact in bf16, and RMSNorm removes it
    assert np.allclose(_run(orc, w2, f), _run(orc, w, f), rtol=0, atol=1e-12)


def test_norm_then_gate_then_rotation(orc):
    # Two tokens of one request, d = 4, every pair turning 1 rad per second.  With a
    # 1 s delay the query at t = 1 sees only the key at t = 0, so its log-sum-exp is
    # that one score: scale * <R(1) g_q * norm(q), g_k * norm(k)>, written out by hand.
    p = orc.Params(1, 4, use_delay=True, delay_s=1, use_rope=True, phi_min=1.0, dt_max_s=1.0,
                   rope_base=1.0)
    xq = np.array([1.0, 2.0, -0.5, 0.25], dtype=np.float32)
    xk = np.array([0.5, -1.0, 2.0, 1.5], dtype=np.float32)
    gq = np.array([0.3, -1.2, 2.0, 0.0], dtype=np.float32)
    wq = np.array([1.0, 3.0, 0.5, 2.0])
    wk = np.array([2.0, 0.5, 1.0, 1.5])
    q = np.stack([xk, xq])[:, None, :]
    k = np.stack([xk, xq])[:, None, :]
    v = np.ones_like(q)
    gate = np.stack([np.zeros(4, np.float32), gq])[:, None, :]
    f = orc.Fused(q_norm_w=wq[None], k_norm_w=wk[None], norm_eps=0.0, q_gate=gate)
    _, lse = orc.attention(p, [0, 2], np.array([0, 1]), np.array([1, 1], np.int8), q, k, v,
                           fused=f, with_lse=True)
    xq64, xk64 = xq.astype(np.float64), xk.astype(np.float64)
    nq = xq64 / math.sqrt(np.mean(xq64 ** 2)) * wq
    nq = nq / (1.0 + np.exp(-gq.astype(np.float64)))
    nk = xk64 / math.sqrt(np.mean(xk64 ** 2)) * wk
    c, sn = math.cos(1.0), math.sin(1.0)
    rq = np.array([nq[0] * c - nq[1] * sn, nq[0] * sn + nq[1] * c, nq[2] * c - nq[3] * sn, nq[2] * sn + nq[3] * c])
    ref = 0.5 * float(rq @ nk)
    assert abs(lse[1, 0] - ref) < 1e-12
    # rotating before the norm gives another score: the order is pinned
    rx = np.array([xq64[0] * c - xq64[1] * sn, xq64[0] * sn + xq64[1] * c, xq64[2] * c - xq64[3] * sn,
                   xq64[2] * sn + xq64[3] * c])
    alt = rx / math.sqrt(np.mean(rx ** 2)) * wq / (1.0 + np.exp(-gq.astype(np.float64)))
    assert abs(0.5 * float(alt @ nk) - ref) > 1e-3
