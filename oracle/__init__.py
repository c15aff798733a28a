"""fp64 CPU oracle for masked time-RoPE attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and has no CPU fallback.

The arithmetic lives in ``rec_attn_oracle.c`` (plain C, fp64, one row at a
time); this module compiles it with gcc into ``oracle/_build`` and wraps it with
ctypes.  Citations for each function are in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rec_attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "librec_attn_oracle.so")

SKIP, PARTIAL, FULL = 0, 1, 2
TILE = 128
GLOBAL, HIST, RT, CAND = 0, 1, 2, 3


class OrcParams(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("use_delay", ctypes.c_int32),
        ("delay_s", ctypes.c_int64),
        ("window", ctypes.c_int32),
        ("hist_bidirectional", ctypes.c_int32),
        ("use_rope", ctypes.c_int32),
        ("phi_min", ctypes.c_double),
        ("dt_max_s", ctypes.c_double),
        ("rope_base", ctypes.c_double),
        ("softmax_scale", ctypes.c_double),
    ]


@dataclass
class Params:
    """Mask and RoPE parameters (CADET defaults: delta = 1 h, phi_min = 1e-4,
    dt_max = 365 days, base = 6e5)."""

    num_heads: int
    head_dim: int
    use_delay: bool = False
    delay_s: int = 3600
    window: int = 0
    hist_bidirectional: bool = False
    use_rope: bool = True
    phi_min: float = 1e-4
    dt_max_s: float = 365.0 * 86400.0
    rope_base: float = 6e5
    softmax_scale: float = 0.0

    def c(self) -> OrcParams:
        return OrcParams(self.num_heads, self.head_dim, int(self.use_delay), int(self.delay_s),
                         int(self.window), int(self.hist_bidirectional), int(self.use_rope),
                         float(self.phi_min), float(self.dt_max_s), float(self.rope_base),
                         float(self.softmax_scale))


class OrcFused(ctypes.Structure):
    _fields_ = [
        ("q_norm_w", ctypes.c_void_p),
        ("k_norm_w", ctypes.c_void_p),
        ("norm_eps", ctypes.c_double),
        ("q_gate", ctypes.c_void_p),
        ("k_gate", ctypes.c_void_p),
        ("out_gate", ctypes.c_void_p),
    ]


@dataclass
class Fused:
    """Fused prologue/epilogue inputs: QK-RMSNorm gains [H, d] (None = no norm on
    that side), its epsilon, and sigmoid-gate pre-activations [T, H, d] in the I/O
    dtype (None = no gate) for Q, K and the attention output."""

    q_norm_w: np.ndarray | None = None
    k_norm_w: np.ndarray | None = None
    norm_eps: float = 1e-6
    q_gate: np.ndarray | None = None
    k_gate: np.ndarray | None = None
    out_gate: np.ndarray | None = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA); returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "rec_attn_oracle.h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts agree.
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.POINTER(OrcParams)
        vp = ctypes.c_void_p
        L.orc_visible.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
        L.orc_visible.restype = ctypes.c_int
        L.orc_mask.argtypes = [P, ctypes.c_int64, vp, vp, vp]
        L.orc_mask.restype = None
        L.orc_mask_block.argtypes = [P, ctypes.c_int64, vp, vp, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int64, vp]
        L.orc_mask_block.restype = None
        L.orc_visible_pairs.argtypes = [P, ctypes.c_int32, vp, vp, vp]
        L.orc_visible_pairs.restype = ctypes.c_uint64
        L.orc_rope.argtypes = [P, ctypes.c_int64, vp, vp]
        L.orc_rope.restype = None
        L.orc_attention.argtypes = [P, ctypes.c_int32, vp, vp, vp, ctypes.c_int32, vp, vp, vp,
                                    ctypes.c_int64, vp, vp, vp, ctypes.c_int32]
        L.orc_attention.restype = ctypes.c_int
        L.orc_attention_fused.argtypes = [P, ctypes.c_int32, vp, vp, vp, ctypes.c_int32, vp, vp, vp,
                                          ctypes.POINTER(OrcFused), ctypes.c_int64, vp, vp, vp,
                                          ctypes.c_int32]
        L.orc_attention_fused.restype = ctypes.c_int
        L.orc_rmsnorm.argtypes = [vp, vp, ctypes.c_int, ctypes.c_double, vp]
        L.orc_rmsnorm.restype = None
        L.orc_sigmoid.argtypes = [ctypes.c_double]
        L.orc_sigmoid.restype = ctypes.c_double
        L.orc_attention_bwd.argtypes = [P, ctypes.c_int32, vp, vp, vp, ctypes.c_int32, vp, vp, vp, vp,
                                        vp, vp, vp, ctypes.c_int32]
        L.orc_attention_bwd.restype = ctypes.c_int
        L.orc_attention_bwd_fused.argtypes = [P, ctypes.c_int32, vp, vp, vp, ctypes.c_int32, vp, vp, vp,
                                              ctypes.POINTER(OrcFused), vp] + [vp] * 8 + [ctypes.c_int32]
        L.orc_attention_bwd_fused.restype = ctypes.c_int
        L.orc_compress.argtypes = [ctypes.c_int32, vp, vp, vp, ctypes.c_int32, vp, vp, ctypes.c_int32,
                                   ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp]
        L.orc_compress.restype = ctypes.c_int64
        L.orc_query_keep.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
        L.orc_query_keep.restype = ctypes.c_int64
        L.orc_kept_rows.argtypes = [ctypes.c_int32, vp, vp, ctypes.c_int64, vp]
        L.orc_kept_rows.restype = ctypes.c_int64
        L.orc_tile_classes.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp]
        L.orc_tile_classes.restype = ctypes.c_int64
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _c8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int8)


def visible(p: Params, pi, ti, ty_i, pj, tj, ty_j) -> bool:
    cp = p.c()
    return bool(lib().orc_visible(ctypes.byref(cp), int(pi), int(ti), int(ty_i),
                                  int(pj), int(tj), int(ty_j)))


def mask(p: Params, t, ty) -> np.ndarray:
    """L x L visibility mask (uint8, 1 = visible) of a single request."""
    t, ty = _c64(t), _c8(ty)
    L = t.shape[0]
    out = np.zeros((L, L), dtype=np.uint8)
    cp = p.c()
    lib().orc_mask(ctypes.byref(cp), L, _ptr(t), _ptr(ty), _ptr(out))
    return out


def mask_block(p: Params, t, ty, i0: int, ni: int, j0: int, nj: int) -> np.ndarray:
    """Rows [i0, i0+ni) x keys [j0, j0+nj) of the mask of a single request (uint8,
    1 = visible; 0 past the request end)."""
    t, ty = _c64(t), _c8(ty)
    out = np.zeros((ni, nj), dtype=np.uint8)
    cp = p.c()
    lib().orc_mask_block(ctypes.byref(cp), t.shape[0], _ptr(t), _ptr(ty), int(i0), int(ni), int(j0), int(nj),
                         _ptr(out))
    return out


def visible_pairs(p: Params, offsets, t, ty) -> int:
    offsets, t, ty = _c64(offsets), _c64(t), _c8(ty)
    cp = p.c()
    return int(lib().orc_visible_pairs(ctypes.byref(cp), len(offsets) - 1, _ptr(offsets),
                                       _ptr(t), _ptr(ty)))


def rope(p: Params, t: int, x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros_like(x)
    cp = p.c()
    lib().orc_rope(ctypes.byref(cp), int(t), _ptr(x), _ptr(y))
    return y


def rmsnorm(x, w, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over one vector."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    assert x.shape == w.shape and x.ndim == 1
    y = np.zeros_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(w), x.shape[0], float(eps), _ptr(y))
    return y


def sigmoid(x: float) -> float:
    return float(lib().orc_sigmoid(float(x)))


def query_keep(hist_len: int, n_min: int, layer: int, n_layers: int) -> int:
    """LazFormer Eq. 22: history queries kept at layer `layer` (1-based) of `n_layers`."""
    return int(lib().orc_query_keep(int(hist_len), int(n_min), int(layer), int(n_layers)))


def kept_rows(offsets, ty, keep: int) -> np.ndarray:
    """Sorted global rows a pruned layer computes: all non-user tokens and the last
    `keep` user tokens of each request (keep < 0: every token)."""
    offsets, ty = _c64(offsets), _c8(ty)
    B = len(offsets) - 1
    n = lib().orc_kept_rows(B, _ptr(offsets), _ptr(ty), int(keep), None)
    rows = np.zeros(max(n, 1), dtype=np.int64)
    lib().orc_kept_rows(B, _ptr(offsets), _ptr(ty), int(keep), _ptr(rows))
    return rows[:n]


def tile_classes(p: Params, offsets, t, ty) -> np.ndarray:
    offsets, t, ty = _c64(offsets), _c64(t), _c8(ty)
    cp = p.c()
    B = len(offsets) - 1
    n = lib().orc_tile_classes(ctypes.byref(cp), B, _ptr(offsets), _ptr(t), _ptr(ty), None)
    out = np.zeros(max(n, 1), dtype=np.uint8)
    lib().orc_tile_classes(ctypes.byref(cp), B, _ptr(offsets), _ptr(t), _ptr(ty), _ptr(out))
    return out[:n]


def attention(p: Params, offsets, t, ty, q, k, v, rows=None, threads: int | None = None,
              with_lse: bool = False, fused: Fused | None = None):
    """fp64 attention outputs for `rows` (sorted global token indices; None = all).

    q, k, v: [T, H, d] arrays, either float32 or uint16 holding bf16 bit patterns
    (widened exactly to fp64 inside the oracle).  Returns out [n_rows, H, d]
    (float64) and, if requested, lse [n_rows, H].
    """
    offsets, t, ty = _c64(offsets), _c64(t), _c8(ty)
    q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
    if q.dtype == np.uint16:
        dtype = 0
    elif q.dtype == np.float32:
        dtype = 1
    else:
        raise TypeError("q/k/v must be float32 or uint16 (bf16 bits)")
    assert k.dtype == q.dtype and v.dtype == q.dtype
    H, d = p.num_heads, p.head_dim
    if rows is None:
        n_rows = int(offsets[-1] - offsets[0])
        rows_arr = None
    else:
        rows_arr = _c64(rows)
        n_rows = rows_arr.shape[0]
    out = np.zeros((max(n_rows, 1), H, d), dtype=np.float64)
    lse = np.zeros((max(n_rows, 1), H), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    cp = p.c()
    keep = []  # arrays whose buffers the C call reads

    def arr(a, dt, shape):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dt)
        assert a.shape == shape, (a.shape, shape)
        keep.append(a)
        return _ptr(a)

    fp = None
    if fused is not None:
        T = int(offsets[-1])
        gate_dt = np.uint16 if dtype == 0 else np.float32
        fc = OrcFused(arr(fused.q_norm_w, np.float64, (H, d)), arr(fused.k_norm_w, np.float64, (H, d)),
                      float(fused.norm_eps), arr(fused.q_gate, gate_dt, (T, H, d)),
                      arr(fused.k_gate, gate_dt, (T, H, d)), arr(fused.out_gate, gate_dt, (T, H, d)))
        fp = ctypes.byref(fc)
    rc = lib().orc_attention_fused(ctypes.byref(cp), len(offsets) - 1, _ptr(offsets), _ptr(t), _ptr(ty),
                                   dtype, _ptr(q), _ptr(k), _ptr(v), fp, n_rows,
                                   None if rows_arr is None else _ptr(rows_arr), _ptr(out), _ptr(lse),
                                   int(threads))
    if rc != 0:
        raise ValueError(f"orc_attention rejected its arguments (rc={rc})")
    out, lse = out[:n_rows], lse[:n_rows]
    return (out, lse) if with_lse else out


def attention_bwd(p: Params, offsets, t, ty, q, k, v, dout, threads: int | None = None):
    """fp64 gradients (dq, dk, dv), each [T, H, d], of attention() for the upstream
    gradient dout; q, k, v, dout are float32 or uint16 bf16 bits (one dtype)."""
    offsets, t, ty = _c64(offsets), _c64(t), _c8(ty)
    q, k, v, dout = (np.ascontiguousarray(a) for a in (q, k, v, dout))
    if q.dtype == np.uint16:
        dtype = 0
    elif q.dtype == np.float32:
        dtype = 1
    else:
        raise TypeError("q/k/v/dout must be float32 or uint16 (bf16 bits)")
    assert k.dtype == q.dtype and v.dtype == q.dtype and dout.dtype == q.dtype
    assert int(offsets[0]) == 0
    shape = q.shape
    dq, dk, dv = (np.zeros(shape, dtype=np.float64) for _ in range(3))
    cp = p.c()
    rc = lib().orc_attention_bwd(ctypes.byref(cp), len(offsets) - 1, _ptr(offsets), _ptr(t), _ptr(ty), dtype,
                                 _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                 int(threads or os.cpu_count() or 1))
    if rc != 0:
        raise ValueError(f"orc_attention_bwd rejected its arguments (rc={rc})")
    return dq, dk, dv


def attention_bwd_fused(p: Params, offsets, t, ty, q, k, v, fused: Fused, dout, threads: int | None = None):
    """fp64 gradients of attention(..., fused=fused) for the upstream gradient dout:
    a dict with dq, dk, dv, dq_gate, dk_gate, dout_gate ([T, H, d]; zero for a gate that
    is off) and dq_norm_w, dk_norm_w ([H, d]; zero without that norm)."""
    offsets, t, ty = _c64(offsets), _c64(t), _c8(ty)
    q, k, v, dout = (np.ascontiguousarray(a) for a in (q, k, v, dout))
    dtype = 0 if q.dtype == np.uint16 else 1
    assert int(offsets[0]) == 0
    H, d = p.num_heads, p.head_dim
    T = int(offsets[-1])
    keep = []

    def arr(a, dt, shape):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dt)
        assert a.shape == shape, (a.shape, shape)
        keep.append(a)
        return _ptr(a)

    gate_dt = np.uint16 if dtype == 0 else np.float32
    fc = OrcFused(arr(fused.q_norm_w, np.float64, (H, d)), arr(fused.k_norm_w, np.float64, (H, d)),
                  float(fused.norm_eps), arr(fused.q_gate, gate_dt, (T, H, d)),
                  arr(fused.k_gate, gate_dt, (T, H, d)), arr(fused.out_gate, gate_dt, (T, H, d)))
    out = {n: np.zeros((T, H, d)) for n in ("dq", "dk", "dv", "dq_gate", "dk_gate", "dout_gate")}
    out["dq_norm_w"] = np.zeros((H, d))
    out["dk_norm_w"] = np.zeros((H, d))
    cp = p.c()
    rc = lib().orc_attention_bwd_fused(
        ctypes.byref(cp), len(offsets) - 1, _ptr(offsets), _ptr(t), _ptr(ty), dtype, _ptr(q), _ptr(k), _ptr(v),
        ctypes.byref(fc), _ptr(dout), *(_ptr(out[n]) for n in ("dq", "dk", "dv", "dq_gate", "dk_gate", "dout_gate",
                                                               "dq_norm_w", "dk_norm_w")),
        int(threads or os.cpu_count() or 1))
    if rc != 0:
        raise ValueError(f"orc_attention_bwd_fused rejected its arguments (rc={rc})")
    return out


def compress(offsets, hist_begin, hist_len, segments, x=None, t=None, ty=None):
    """History compression.  segments: [(length or -1, group size), ...] from the most
    recent; x: [T, width] float32 or bf16 bits.  Returns (out_offsets, out_x fp64,
    out_t, out_ty), or only out_offsets when x is None."""
    offsets, hb, hl = _c64(offsets), _c64(hist_begin), _c64(hist_len)
    B = len(offsets) - 1
    sl = _c64([s_[0] for s_ in segments])
    sg = np.ascontiguousarray([s_[1] for s_ in segments], dtype=np.int32)
    out_off = np.zeros(B + 1, dtype=np.int64)
    L = lib()
    if x is None:
        n = L.orc_compress(B, _ptr(offsets), _ptr(hb), _ptr(hl), len(segments), _ptr(sl), _ptr(sg), 0, 1,
                           None, None, None, _ptr(out_off), None, None, None)
        if n < 0:
            raise ValueError("orc_compress rejected its arguments")
        return out_off
    x = np.ascontiguousarray(x)
    dtype = 0 if x.dtype == np.uint16 else 1
    width = int(np.prod(x.shape[1:]))
    t, ty = _c64(t), _c8(ty)
    n = L.orc_compress(B, _ptr(offsets), _ptr(hb), _ptr(hl), len(segments), _ptr(sl), _ptr(sg), dtype, width,
                       None, None, None, _ptr(out_off), None, None, None)
    if n < 0:
        raise ValueError("orc_compress rejected its arguments")
    ox = np.zeros((max(n, 1), width), dtype=np.float64)
    ot = np.zeros(max(n, 1), dtype=np.int64)
    oty = np.zeros(max(n, 1), dtype=np.int8)
    L.orc_compress(B, _ptr(offsets), _ptr(hb), _ptr(hl), len(segments), _ptr(sl), _ptr(sg), dtype, width,
                   _ptr(x), _ptr(t), _ptr(ty), _ptr(out_off), _ptr(ox), _ptr(ot), _ptr(oty))
    return out_off, ox[:n].reshape((n,) + x.shape[1:]), ot[:n], oty[:n]
