"""Seeded synthetic inputs for the five ranking-attention workloads.

This module only draws inputs: packed jagged offsets, int64 timestamps, int8
token types and Q/K/V.  It contains none of the attention, mask or RoPE
arithmetic, and it is the one module that both the CUDA path's tests/bench and
the CPU oracle's tests consume.

The shapes follow the workloads the pages describe (CADET impression/action
sequences, SORT request-centric samples, MTGR hybrid user-day samples, TM20K /
LazFormer 20K histories); the pages' data are private logs, so these seeded
generators stand in for them.  Every generator uses
``numpy.random.default_rng(1000 + config_id)`` unless a seed is given.

Token types: 0 GLOBAL (profile / special / global summary), 1 HIST (history),
2 RT (real-time block), 3 CAND (candidate / target).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GLOBAL, HIST, RT, CAND = 0, 1, 2, 3
DAY = 86400
YEAR = 365 * DAY
EPOCH = 1_700_000_000


@dataclass
class Workload:
    name: str
    num_heads: int
    head_dim: int
    dtype: str                   # "bf16" (q/k/v hold bf16 bit patterns as uint16) or "fp32"
    offsets: np.ndarray          # int64 [B+1]
    t: np.ndarray                # int64 [T], seconds
    types: np.ndarray            # int8  [T]
    q: np.ndarray                # [T, H, d]
    k: np.ndarray
    v: np.ndarray
    mask: dict = field(default_factory=dict)  # use_delay, delay_s, window, hist_bidirectional
    rope: dict = field(default_factory=dict)  # use_rope, phi_min, dt_max_s, rope_base

    @property
    def batch(self) -> int:
        return len(self.offsets) - 1

    @property
    def total_tokens(self) -> int:
        return int(self.offsets[-1])


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the bit
    patterns as uint16.  Inputs are finite normals, so no NaN handling."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def _qkv(rng, T, H, d, dtype, scale=1.0):
    out = []
    for _ in range(3):
        x = rng.standard_normal((T, H, d), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out.append(round_to_bf16_bits(x) if dtype == "bf16" else x)
    return out


def _lognormal_gaps(rng, n, median_s, sigma, max_span, clip=None):
    g = rng.lognormal(np.log(median_s), sigma, size=n)
    if clip is not None:
        g = np.clip(g, clip[0], clip[1])
    s = g.sum()
    if s > max_span:
        g *= max_span / s
    return g


def _epoch(rng):
    return EPOCH + int(rng.integers(0, 10_000_000))


def _pack(lengths):
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lengths)
    return off


_ROPE = dict(use_rope=True, phi_min=1e-4, dt_max_s=float(YEAR), rope_base=6e5)


def tiny_fp32(batch=4, n_hist=64, n_cand=8, seed=1001):
    """B requests of n_hist history tokens + n_cand candidates, H=2, d=32, fp32.
    History gaps log-normal (median 10 min), span <= 30 days; candidates are
    stamped at request time (one more gap after the last history event)."""
    rng = np.random.default_rng(seed)
    H, d = 2, 32
    ts, tys = [], []
    for _ in range(batch):
        t0 = _epoch(rng)
        g = _lognormal_gaps(rng, n_hist + 1, 600.0, 2.0, 30 * DAY)
        c = t0 + np.round(np.cumsum(g)).astype(np.int64)
        ts.append(np.concatenate([c[:n_hist], np.full(n_cand, c[n_hist], dtype=np.int64)]))
        tys.append(np.array([HIST] * n_hist + [CAND] * n_cand, dtype=np.int8))
    t, ty = np.concatenate(ts), np.concatenate(tys)
    q, k, v = _qkv(rng, len(t), H, d, "fp32")
    return Workload("tiny_fp32", H, d, "fp32", _pack([n_hist + n_cand] * batch), t, ty, q, k, v,
                    dict(use_delay=True, delay_s=3600, window=0, hist_bidirectional=False),
                    dict(_ROPE))


def cadet(batch=256, n_pairs=256, seed=1002, heads=4, head_dim=64):
    """CADET-style interleaved impression/action sequences: 2*n_pairs tokens per
    request, both tokens of a pair share a timestamp; pair gaps log-normal
    (median 3 h) clipped to [1 s, 28 d], span <= 1 year.  All HIST; causal +
    delta_delay = 3600 s.  Q/K/V ~ N(0,1)/sqrt(d), bf16."""
    rng = np.random.default_rng(seed)
    H, d = heads, head_dim
    ts = []
    for _ in range(batch):
        t0 = _epoch(rng)
        g = _lognormal_gaps(rng, n_pairs, 10800.0, 2.5, YEAR, clip=(1.0, 28 * DAY))
        c = t0 + np.round(np.cumsum(g)).astype(np.int64)
        ts.append(np.repeat(c, 2))
    t = np.concatenate(ts)
    ty = np.full(len(t), HIST, dtype=np.int8)
    q, k, v = _qkv(rng, len(t), H, d, "bf16", scale=1.0 / np.sqrt(d))
    return Workload("cadet", H, d, "bf16", _pack([2 * n_pairs] * batch), t, ty, q, k, v,
                    dict(use_delay=True, delay_s=3600, window=0, hist_bidirectional=False),
                    dict(_ROPE))


def sort(batch=128, n_special=16, n_hist=2048, n_cand=200, window=256, seed=1003,
         heads=8, head_dim=64):
    """SORT-style request-centric samples: n_special GLOBAL tokens, n_hist HIST
    tokens (gaps log-normal, median 10 min, span <= 1 year), n_cand CAND tokens.
    Special tokens and candidates are stamped at request time.  U2U causal with
    a local window over history, C2U full, C2C diagonal.  Q/K/V ~ N(0,1), bf16."""
    rng = np.random.default_rng(seed)
    H, d = heads, head_dim
    ts, tys = [], []
    for _ in range(batch):
        t0 = _epoch(rng)
        g = _lognormal_gaps(rng, n_hist + 1, 600.0, 2.0, YEAR)
        c = t0 + np.round(np.cumsum(g)).astype(np.int64)
        treq = c[n_hist]
        ts.append(np.concatenate([np.full(n_special, treq, dtype=np.int64), c[:n_hist],
                                  np.full(n_cand, treq, dtype=np.int64)]))
        tys.append(np.array([GLOBAL] * n_special + [HIST] * n_hist + [CAND] * n_cand,
                            dtype=np.int8))
    t, ty = np.concatenate(ts), np.concatenate(tys)
    q, k, v = _qkv(rng, len(t), H, d, "bf16")
    L = n_special + n_hist + n_cand
    return Workload("sort", H, d, "bf16", _pack([L] * batch), t, ty, q, k, v,
                    dict(use_delay=False, delay_s=0, window=window, hist_bidirectional=False),
                    dict(_ROPE))


def mtgr(batch=64, n_profile=32, hist=(500, 1500), rt=(50, 250), cand=(20, 100), seed=1004,
         heads=8, head_dim=64):
    """MTGR-style user-day samples (jagged): n_profile GLOBAL tokens stamped at
    the start of the request day, U[hist] HIST tokens spread over the previous
    180 days, U[rt] RT tokens and U[cand] CAND tokens, each sorted uniform
    seconds inside the request day.  Static part bidirectional, RT causal,
    targets see real-time events strictly before them and only themselves."""
    rng = np.random.default_rng(seed)
    H, d = heads, head_dim
    ts, tys, lens = [], [], []
    for _ in range(batch):
        day = (_epoch(rng) // DAY) * DAY
        nh = int(rng.integers(hist[0], hist[1] + 1))
        nr = int(rng.integers(rt[0], rt[1] + 1))
        nc = int(rng.integers(cand[0], cand[1] + 1))
        th = np.sort(rng.integers(day - 180 * DAY, day, size=nh))
        tr = np.sort(rng.integers(day, day + DAY, size=nr))
        tc = np.sort(rng.integers(day, day + DAY, size=nc))
        ts.append(np.concatenate([np.full(n_profile, day, dtype=np.int64), th, tr, tc]).astype(
            np.int64))
        tys.append(np.array([GLOBAL] * n_profile + [HIST] * nh + [RT] * nr + [CAND] * nc,
                            dtype=np.int8))
        lens.append(n_profile + nh + nr + nc)
    t, ty = np.concatenate(ts), np.concatenate(tys)
    q, k, v = _qkv(rng, len(t), H, d, "bf16")
    return Workload("mtgr", H, d, "bf16", _pack(lens), t, ty, q, k, v,
                    dict(use_delay=False, delay_s=0, window=0, hist_bidirectional=True),
                    dict(_ROPE))


def tm20k(variant="full", batch=16, n_hist=20000, n_global=64, window=512, seed=1005,
          heads=8, head_dim=64):
    """TM20K / LazFormer long histories: n_hist history tokens (the first
    n_global typed GLOBAL) + 1 target at request time; gaps log-normal (median
    10 min), span <= 1 year.  variant "full": plain causal (window 0, which with
    the globals first equals full causal attention over all tokens); variant
    "window": local window plus the global summary tokens everyone sees."""
    rng = np.random.default_rng(seed)
    H, d = heads, head_dim
    ts, tys = [], []
    for _ in range(batch):
        t0 = _epoch(rng)
        g = _lognormal_gaps(rng, n_hist + 1, 600.0, 2.0, YEAR)
        c = t0 + np.round(np.cumsum(g)).astype(np.int64)
        ts.append(np.concatenate([c[:n_hist], c[n_hist:n_hist + 1]]))
        ng = min(n_global, n_hist)
        tys.append(np.array([GLOBAL] * ng + [HIST] * (n_hist - ng) + [CAND], dtype=np.int8))
    t, ty = np.concatenate(ts), np.concatenate(tys)
    q, k, v = _qkv(rng, len(t), H, d, "bf16")
    w = 0 if variant == "full" else window
    return Workload(f"tm20k_{variant}", H, d, "bf16", _pack([n_hist + 1] * batch), t, ty, q, k, v,
                    dict(use_delay=False, delay_s=0, window=w, hist_bidirectional=False),
                    dict(_ROPE))


def cadet_serving(batch=16, n_hist=4096, n_cand=500, seed=1006, heads=4, head_dim=64):
    """CADET serving: one user history of n_hist events (gaps log-normal, median 3 h,
    clipped to [1 s, 28 d], span <= 1 year) with n_cand candidates appended, stamped
    at request time.  History causal + delta_delay = 3600 s, candidates see the
    history and themselves only.  Q/K/V ~ N(0,1)/sqrt(d), bf16."""
    rng = np.random.default_rng(seed)
    H, d = heads, head_dim
    ts, tys = [], []
    for _ in range(batch):
        t0 = _epoch(rng)
        g = _lognormal_gaps(rng, n_hist + 1, 10800.0, 2.5, YEAR, clip=(1.0, 28 * DAY))
        c = t0 + np.round(np.cumsum(g)).astype(np.int64)
        ts.append(np.concatenate([c[:n_hist], np.full(n_cand, c[n_hist], dtype=np.int64)]))
        tys.append(np.array([HIST] * n_hist + [CAND] * n_cand, dtype=np.int8))
    t, ty = np.concatenate(ts), np.concatenate(tys)
    q, k, v = _qkv(rng, len(t), H, d, "bf16", scale=1.0 / np.sqrt(d))
    return Workload("cadet_serving", H, d, "bf16", _pack([n_hist + n_cand] * batch), t, ty, q, k, v,
                    dict(use_delay=True, delay_s=3600, window=0, hist_bidirectional=False),
                    dict(_ROPE))


def make(name: str, **kw) -> Workload:
    """Workload by name: tiny_fp32, cadet, sort, mtgr, tm20k_full, tm20k_window,
    cadet_serving."""
    if name == "tiny_fp32":
        return tiny_fp32(**kw)
    if name == "cadet":
        return cadet(**kw)
    if name == "sort":
        return sort(**kw)
    if name == "mtgr":
        return mtgr(**kw)
    if name == "tm20k_full":
        return tm20k("full", **kw)
    if name == "tm20k_window":
        return tm20k("window", **kw)
    if name == "cadet_serving":
        return cadet_serving(**kw)
    raise KeyError(name)


NAMES = ("tiny_fp32", "cadet", "sort", "mtgr", "tm20k_full", "tm20k_window")
# serving-side workloads (query pruning / target attention), outside the five configs
EXTRA_NAMES = ("cadet_serving",)


@dataclass
class FusedInputs:
    """Inputs of the fused steps: QK-RMSNorm gains [H, d] (float32) and sigmoid-gate
    pre-activations [T, H, d] (bf16 bits or float32, like Q/K/V)."""

    q_norm_w: np.ndarray
    k_norm_w: np.ndarray
    q_gate: np.ndarray
    k_gate: np.ndarray
    out_gate: np.ndarray
    norm_eps: float = 1e-6


def fused_inputs(w: Workload, seed: int = 2001) -> FusedInputs:
    """Seeded gains ~ U(0.5, 1.5) and gate pre-activations ~ N(0, 1.5^2) for a workload."""
    rng = np.random.default_rng(seed)
    T, H, d = w.total_tokens, w.num_heads, w.head_dim
    gains = lambda: rng.uniform(0.5, 1.5, size=(H, d)).astype(np.float32)
    qn, kn = gains(), gains()

    def gate():
        g = (rng.standard_normal(size=(T, H, d)) * 1.5).astype(np.float32)
        return round_to_bf16_bits(g) if w.dtype == "bf16" else g

    return FusedInputs(qn, kn, gate(), gate(), gate())
