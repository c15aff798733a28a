"""Invariants the pages fix, checked on the CPU oracle over every workload family.

- only time differences matter (CADET time-RoPE section): shifting every timestamp
  of a request by a constant leaves every output unchanged;
- candidates are independent (CADET candidate isolation, SORT C2C, LazFormer
  Eq. 19-21, M-FALCON appendix H): permuting candidates permutes their outputs,
  removing one leaves the rest unchanged, and a candidate scored alongside others
  equals a separate pass over the user tokens plus that one candidate;
- -inf masking is strict (LazFormer section 2.3): changing K/V at masked
  positions leaves the output unchanged.
"""
import numpy as np
import pytest

from generative_recommender_ranking_gb300 import workloads as W


def _p(orc, w, **kw):
    args = dict(w.mask)
    args.update(kw)
    return orc.Params(w.num_heads, w.head_dim, **args)


SMALL = {
    "tiny_fp32": lambda: W.tiny_fp32(batch=2),
    "cadet": lambda: W.cadet(batch=2, n_pairs=40),
    "sort": lambda: W.sort(batch=2, n_special=4, n_hist=60, n_cand=10, window=16),
    "mtgr": lambda: W.mtgr(batch=2, n_profile=4, hist=(20, 40), rt=(5, 12), cand=(3, 8)),
    "tm20k_full": lambda: W.tm20k("full", batch=2, n_hist=90, n_global=8),
    "tm20k_window": lambda: W.tm20k("window", batch=2, n_hist=90, n_global=8, window=16),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_time_shift_invariance(orc, name):
    w = SMALL[name]()
    p = _p(orc, w)
    base = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v)
    for c in (-1_700_000_000, 12345, 3 * 10**10):
        shifted = orc.attention(p, w.offsets, w.t + c, w.types, w.q, w.k, w.v)
        np.testing.assert_allclose(shifted, base, rtol=1e-9, atol=1e-11)
    # per-request shifts too
    cs = np.repeat(np.array([7, -99999], dtype=np.int64), np.diff(w.offsets))
    shifted = orc.attention(p, w.offsets, w.t + cs, w.types, w.q, w.k, w.v)
    np.testing.assert_allclose(shifted, base, rtol=1e-9, atol=1e-11)


def _cand_slice(w, b):
    s, e = int(w.offsets[b]), int(w.offsets[b + 1])
    idx = np.nonzero(w.types[s:e] == W.CAND)[0] + s
    return s, e, idx


@pytest.mark.parametrize("name", ["tiny_fp32", "sort", "mtgr"])
def test_candidate_permutation(orc, name):
    w = SMALL[name]()
    p = _p(orc, w)
    base = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v)
    rng = np.random.default_rng(5)
    perm = np.arange(w.total_tokens)
    for b in range(w.batch):
        _, _, idx = _cand_slice(w, b)
        perm[idx] = rng.permutation(idx)
    q, k, v, t = w.q[perm], w.k[perm], w.v[perm], w.t[perm]
    out = orc.attention(p, w.offsets, t, w.types[perm], q, k, v)
    np.testing.assert_allclose(out, base[perm], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("name", ["tiny_fp32", "sort", "mtgr", "tm20k_window"])
def test_candidate_removal_and_mfalcon_equivalence(orc, name):
    """Scoring one candidate next to the others equals a separate pass over the
    user tokens and that candidate alone (M-FALCON batched inference)."""
    w = SMALL[name]()
    p = _p(orc, w)
    base = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v)
    b = 1
    s, e, cands = _cand_slice(w, b)
    user = np.arange(s, cands[0])
    for c in cands[[0, -1]]:
        keep = np.concatenate([user, [c]])
        off = np.array([0, len(keep)], dtype=np.int64)
        out = orc.attention(p, off, w.t[keep], w.types[keep], w.q[keep], w.k[keep], w.v[keep])
        np.testing.assert_allclose(out[-1], base[c], rtol=1e-12, atol=1e-13)
        # the user tokens never read candidates, so they are unchanged as well
        np.testing.assert_allclose(out[:-1], base[user], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_masked_keys_do_not_matter(orc, name):
    w = SMALL[name]()
    p = _p(orc, w)
    b = 1
    s, e = int(w.offsets[b]), int(w.offsets[b + 1])
    L = e - s
    m = orc.mask(p, w.t[s:e], w.types[s:e])
    rows = [0, L // 3, L // 2, L - 1]
    rng = np.random.default_rng(6)
    base = orc.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v)
    for i in rows:
        hidden = np.nonzero(m[i] == 0)[0] + s
        if len(hidden) == 0:
            continue
        k, v = w.k.copy(), w.v.copy()
        if w.dtype == "bf16":
            k[hidden] = rng.integers(0, 0x7F00, size=k[hidden].shape, dtype=np.uint16)
            v[hidden] = rng.integers(0, 0x7F00, size=v[hidden].shape, dtype=np.uint16)
        else:
            k[hidden] = rng.standard_normal(k[hidden].shape).astype(np.float32) * 100
            v[hidden] = rng.standard_normal(v[hidden].shape).astype(np.float32) * 100
        out = orc.attention(p, w.offsets, w.t, w.types, w.q, k, v, rows=[s + i])
        np.testing.assert_array_equal(out[0], base[s + i])


@pytest.mark.parametrize("name", sorted(SMALL))
def test_brute_force_softmax_on_tiny_cases(orc, name):
    """A pure-Python softmax over the oracle's own mask for a 4-8 token prefix of
    each workload (rotation via the pinned oracle rope)."""
    import math
    w = SMALL[name]()
    p = _p(orc, w)
    L = 8
    idx = np.arange(L)
    off = np.array([0, L], dtype=np.int64)
    t, ty = w.t[idx], w.types[idx].copy()
    ty[-2:] = W.CAND  # make sure candidates take part
    toF = (lambda a: W.bf16_bits_to_float32(a).astype(np.float64)) if w.dtype == "bf16" else (
        lambda a: a.astype(np.float64))
    q, k, v = (toF(a[idx]) for a in (w.q, w.k, w.v))
    out = orc.attention(p, off, t, ty, w.q[idx], w.k[idx], w.v[idx])
    m = orc.mask(p, t, ty)
    d = w.head_dim
    for h in range(w.num_heads):
        for i in range(L):
            qi = orc.rope(p, t[i], q[i, h])
            sc = [math.fsum(qi * orc.rope(p, t[j], k[j, h])) / math.sqrt(d) if m[i, j] else None
                  for j in range(L)]
            vis = [j for j in range(L) if m[i, j]]
            if not vis:
                assert np.all(out[i, h] == 0)
                continue
            mx = max(sc[j] for j in vis)
            wts = {j: math.exp(sc[j] - mx) for j in vis}
            den = math.fsum(wts.values())
            ref = sum(wts[j] / den * v[j, h] for j in vis)
            np.testing.assert_allclose(out[i, h], ref, rtol=1e-11, atol=1e-12)
