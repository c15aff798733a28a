"""Pins of the oracle's backward pass: central finite differences of the oracle's own
forward (masks and time-RoPE included), torch autograd on float64 SDPA where the
method reduces to plain attention, and closed-form properties of the gradients."""
import numpy as np
import pytest
import torch

from generative_recommender_ranking_gb300 import workloads as W


def _tiny(name):
    if name == "cadet":
        w = W.cadet(batch=2, n_pairs=6, heads=2, head_dim=64)
    elif name == "sort":
        w = W.sort(batch=2, n_special=2, n_hist=9, n_cand=3, window=4, heads=2, head_dim=64)
    elif name == "mtgr":
        w = W.mtgr(batch=2, n_profile=2, hist=(4, 6), rt=(2, 4), cand=(2, 3), heads=1, head_dim=64)
    else:
        w = W.tiny_fp32(batch=2, n_hist=10, n_cand=3)
    # fp32 copies of the inputs: finite differences need exactly known perturbations
    f32 = (lambda a: W.bf16_bits_to_float32(a)) if w.dtype == "bf16" else (lambda a: a.copy())
    return w, f32(w.q), f32(w.k), f32(w.v)


def _loss(orc, p, w, q, k, v, g):
    out = orc.attention(p, w.offsets, w.t, w.types, q, k, v, threads=1)
    return float(np.sum(out * g.astype(np.float64)))


@pytest.mark.parametrize("name", ["cadet", "sort", "mtgr", "tiny"])
def test_backward_matches_finite_differences(orc, name):
    w, q, k, v = _tiny(name)
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    rng = np.random.default_rng(5)
    g = rng.standard_normal(q.shape).astype(np.float32)
    dq, dk, dv = orc.attention_bwd(p, w.offsets, w.t, w.types, q, k, v, g, threads=1)
    T, H, d = q.shape
    for which, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = (int(rng.integers(T)), int(rng.integers(H)), int(rng.integers(d)))
            eps = np.float32(1e-3)
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += eps
            minus[idx] -= eps
            h = float(plus[idx]) - float(minus[idx])  # exact step after fp32 rounding
            args = {"q": q, "k": k, "v": v}
            fp = _loss(orc, p, w, **{**args, which: plus}, g=g)
            fm = _loss(orc, p, w, **{**args, which: minus}, g=g)
            fd = (fp - fm) / h
            assert abs(fd - grad[idx]) <= 1e-5 * max(1.0, abs(grad[idx])), (which, idx, fd, grad[idx])


def test_backward_matches_torch_autograd_on_plain_attention(orc):
    # all tokens mutually visible and no RoPE: the method is plain softmax attention
    T, H, d = 40, 2, 64
    rng = np.random.default_rng(9)
    q, k, v, g = (rng.standard_normal((T, H, d)).astype(np.float32) for _ in range(4))
    off = np.array([0, 17, 40])
    t = np.zeros(T, dtype=np.int64)
    ty = np.full(T, W.HIST, dtype=np.int8)
    p = orc.Params(H, d, use_rope=False, hist_bidirectional=True)
    dq, dk, dv = orc.attention_bwd(p, off, t, ty, q, k, v, g)
    for b in range(2):
        s, e = off[b], off[b + 1]
        tq, tk, tv = (torch.tensor(a[s:e], dtype=torch.float64).permute(1, 0, 2).requires_grad_() for a in (q, k, v))
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)
        o.backward(torch.tensor(g[s:e], dtype=torch.float64).permute(1, 0, 2))
        for ref, got in ((tq.grad, dq), (tk.grad, dk), (tv.grad, dv)):
            assert np.allclose(ref.permute(1, 0, 2).numpy(), got[s:e], rtol=0, atol=1e-12)


def test_value_gradients_sum_to_the_upstream_gradient(orc):
    # every probability row sums to one, so sum_j dV_j = sum over rows with a visible
    # key of dO_i, per head
    w, q, k, v = _tiny("cadet")
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    g = np.random.default_rng(2).standard_normal(q.shape).astype(np.float32)
    _, _, dv = orc.attention_bwd(p, w.offsets, w.t, w.types, q, k, v, g)
    for b in range(w.batch):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        seen = orc.mask(p, w.t[s:e], w.types[s:e]).sum(1) > 0
        assert np.allclose(dv[s:e].sum(0), g[s:e][seen].astype(np.float64).sum(0), rtol=0, atol=1e-12)


def test_masked_keys_and_blind_rows_get_no_gradient(orc):
    # with the delay rule the first events of a request see nothing (their dQ is 0)
    # and events within the last hour before every query are read by none (dK = dV = 0)
    w, q, k, v = _tiny("cadet")
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    g = np.random.default_rng(4).standard_normal(q.shape).astype(np.float32)
    dq, dk, dv = orc.attention_bwd(p, w.offsets, w.t, w.types, q, k, v, g)
    n_blind = n_unread = 0
    for b in range(w.batch):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        m = orc.mask(p, w.t[s:e], w.types[s:e])
        blind, unread = m.sum(1) == 0, m.sum(0) == 0
        n_blind += int(blind.sum()); n_unread += int(unread.sum())
        assert np.all(dq[s:e][blind] == 0.0)
        assert np.all(dk[s:e][unread] == 0.0) and np.all(dv[s:e][unread] == 0.0)
    assert n_blind > 0 and n_unread > 0
