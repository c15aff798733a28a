"""Pins of the oracle's backward through the fused steps (QK-RMSNorm, Q/K sigmoid
gates, output gate): central finite differences of the oracle's own fused forward
for every input (q, k, v, the three gate pre-activations and both norm gains), and
the plain backward when every fused step is off."""
import numpy as np
import pytest

from generative_recommender_ranking_gb300 import workloads as W


def _case(name):
    if name == "cadet":
        w = W.cadet(batch=2, n_pairs=6, heads=2, head_dim=64)
    elif name == "sort":
        w = W.sort(batch=2, n_special=2, n_hist=9, n_cand=3, window=4, heads=2, head_dim=64)
    elif name == "mtgr":
        w = W.mtgr(batch=2, n_profile=2, hist=(4, 6), rt=(2, 4), cand=(2, 3), heads=1, head_dim=64)
    else:
        w = W.tiny_fp32(batch=2, n_hist=10, n_cand=3)
    fi = W.fused_inputs(w)
    f32 = (lambda a: W.bf16_bits_to_float32(a)) if w.dtype == "bf16" else (lambda a: np.array(a, dtype=np.float32))
    x = {"q": f32(w.q), "k": f32(w.k), "v": f32(w.v), "q_gate": f32(fi.q_gate), "k_gate": f32(fi.k_gate),
         "out_gate": f32(fi.out_gate), "q_norm_w": fi.q_norm_w.astype(np.float64),
         "k_norm_w": fi.k_norm_w.astype(np.float64)}
    return w, x, fi.norm_eps


def _fused(orc, x, eps, on=("q_norm_w", "k_norm_w", "q_gate", "k_gate", "out_gate")):
    return orc.Fused(q_norm_w=x["q_norm_w"] if "q_norm_w" in on else None,
                     k_norm_w=x["k_norm_w"] if "k_norm_w" in on else None, norm_eps=eps,
                     q_gate=x["q_gate"] if "q_gate" in on else None, k_gate=x["k_gate"] if "k_gate" in on else None,
                     out_gate=x["out_gate"] if "out_gate" in on else None)


def _loss(orc, p, w, x, eps, g):
    out = orc.attention(p, w.offsets, w.t, w.types, x["q"], x["k"], x["v"], threads=1, fused=_fused(orc, x, eps))
    return float(np.sum(out * g))


@pytest.mark.parametrize("name", ["cadet", "sort", "mtgr", "tiny"])
def test_fused_backward_matches_finite_differences(orc, name):
    w, x, eps = _case(name)
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    rng = np.random.default_rng(7)
    g = rng.standard_normal(x["q"].shape).astype(np.float32)
    grads = orc.attention_bwd_fused(p, w.offsets, w.t, w.types, x["q"], x["k"], x["v"], _fused(orc, x, eps), g,
                                    threads=1)
    names = {"q": "dq", "k": "dk", "v": "dv", "q_gate": "dq_gate", "k_gate": "dk_gate", "out_gate": "dout_gate",
             "q_norm_w": "dq_norm_w", "k_norm_w": "dk_norm_w"}
    g64 = g.astype(np.float64)
    for which, gname in names.items():
        arr, grad = x[which], grads[gname]
        for _ in range(8):
            idx = tuple(int(rng.integers(n)) for n in arr.shape)
            step = arr.dtype.type(1e-3)
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += step
            minus[idx] -= step
            h = float(plus[idx]) - float(minus[idx])  # the exact step after rounding
            fp = _loss(orc, p, w, {**x, which: plus}, eps, g64)
            fm = _loss(orc, p, w, {**x, which: minus}, eps, g64)
            fd = (fp - fm) / h
            assert abs(fd - grad[idx]) <= 2e-5 * max(1.0, abs(grad[idx])), (name, which, idx, fd, grad[idx])


def test_fused_backward_with_every_step_off_is_the_plain_backward(orc):
    w, x, eps = _case("sort")
    p = orc.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    g = np.random.default_rng(3).standard_normal(x["q"].shape).astype(np.float32)
    grads = orc.attention_bwd_fused(p, w.offsets, w.t, w.types, x["q"], x["k"], x["v"], _fused(orc, x, eps, on=()),
                                    g, threads=2)
    dq, dk, dv = orc.attention_bwd(p, w.offsets, w.t, w.types, x["q"], x["k"], x["v"], g, threads=2)
    for a, b in ((grads["dq"], dq), (grads["dk"], dk), (grads["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    for n in ("dq_gate", "dk_gate", "dout_gate", "dq_norm_w", "dk_norm_w"):
        assert not grads[n].any()
