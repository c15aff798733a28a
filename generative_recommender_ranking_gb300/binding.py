"""ctypes binding of librec_attn.so with the C-ABI's names (include/rec_attn.h).

Argument marshalling only: tensors are passed as raw device pointers, streams as
raw cudaStream_t handles.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU fallback.  If the library has not been built,
loading raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "librec_attn.so")

ABI_VERSION = 1
TILE = 128
MAX_REQUEST_LEN = 262144

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT, ERR_DEVICE_INPUT = range(7)
BF16, FP32 = 0, 1
GLOBAL, HIST, RT, CAND = 0, 1, 2, 3
TILE_SKIP, TILE_PARTIAL, TILE_FULL = 0, 1, 2


class RecAttnParams(ctypes.Structure):
    _fields_ = [
        ("abi_version", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("use_delay", ctypes.c_int32),
        ("delay_s", ctypes.c_int64),
        ("window", ctypes.c_int32),
        ("hist_bidirectional", ctypes.c_int32),
        ("use_rope", ctypes.c_int32),
        ("phi_min", ctypes.c_double),
        ("dt_max_s", ctypes.c_double),
        ("rope_base", ctypes.c_double),
        ("softmax_scale", ctypes.c_float),
    ]


class RecAttnFused(ctypes.Structure):
    """rec_attn_fused: QK-RMSNorm gains, epsilon and sigmoid-gate pre-activations."""
    _fields_ = [
        ("q_norm_weight", ctypes.c_void_p),
        ("k_norm_weight", ctypes.c_void_p),
        ("norm_eps", ctypes.c_float),
        ("q_gate", ctypes.c_void_p),
        ("k_gate", ctypes.c_void_p),
        ("out_gate", ctypes.c_void_p),
    ]


class RecAttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {rec_attn_status_string(code)} (status {code})")


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load librec_attn.so (raises OSError if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise OSError(f"{_LIB_PATH} not found: build it with "
                          "python -m generative_recommender_ranking_gb300.build")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.rec_attn_plan.argtypes = [ctypes.POINTER(RecAttnParams), i32, vp, vp, vp, vp, vp,
                                    ctypes.POINTER(vp)]
        L.rec_attn_plan.restype = ctypes.c_int
        L.rec_attn_plan_query_pruned.argtypes = [ctypes.POINTER(RecAttnParams), i32, i32, vp, vp, vp, vp, vp,
                                                 ctypes.POINTER(vp)]
        L.rec_attn_plan_query_pruned.restype = ctypes.c_int
        L.rec_attn_query_keep.argtypes = [i64, i64, i32, i32]
        L.rec_attn_query_keep.restype = i64
        L.rec_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.rec_attn_fwd.restype = ctypes.c_int
        L.rec_attn_fwd_fused.argtypes = [vp, vp, vp, vp, ctypes.POINTER(RecAttnFused), vp, vp, vp]
        L.rec_attn_fwd_fused.restype = ctypes.c_int
        L.rec_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.rec_attn_bwd.restype = ctypes.c_int
        L.rec_attn_compress_lengths.argtypes = [i32, vp, vp, vp, i32, vp, vp, vp]
        L.rec_attn_compress_lengths.restype = ctypes.c_int
        L.rec_attn_compress.argtypes = [i32, vp, vp, vp, i32, vp, vp, i32, i64, vp, vp, vp, vp, vp, vp, vp]
        L.rec_attn_compress.restype = ctypes.c_int
        L.rec_attn_check_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.POINTER(i32), vp]
        L.rec_attn_check_wait_timeout.restype = ctypes.c_int
        L.rec_attn_free.argtypes = [vp]
        L.rec_attn_free.restype = None
        L.rec_attn_tile_classes.argtypes = [vp, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
        L.rec_attn_tile_classes.restype = ctypes.c_int
        L.rec_attn_visible_pairs.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
        L.rec_attn_visible_pairs.restype = ctypes.c_int
        L.rec_attn_device_status.argtypes = [vp, ctypes.POINTER(i32)]
        L.rec_attn_device_status.restype = ctypes.c_int
        L.rec_attn_status_string.argtypes = [ctypes.c_int]
        L.rec_attn_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def make_params(num_heads: int, head_dim: int, dtype: str = "bf16", use_delay: bool = False,
                delay_s: int = 0, window: int = 0, hist_bidirectional: bool = False,
                use_rope: bool = True, phi_min: float = 1e-4, dt_max_s: float = 365.0 * 86400.0,
                rope_base: float = 6e5, softmax_scale: float = 0.0) -> RecAttnParams:
    return RecAttnParams(ABI_VERSION, int(num_heads), int(head_dim), BF16 if dtype == "bf16" else FP32,
                         int(bool(use_delay)), int(delay_s), int(window), int(bool(hist_bidirectional)),
                         int(bool(use_rope)), float(phi_min), float(dt_max_s), float(rope_base),
                         float(softmax_scale))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()  # torch.Tensor


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, code: int):
    if code != OK:
        raise RecAttnError(fn, code)


@dataclass
class Plan:
    handle: int
    batch: int
    total_tokens: int
    # keep the device arrays the plan reads alive for as long as the plan
    _keep: tuple = ()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        rec_attn_free(self)


def rec_attn_status_string(code: int) -> str:
    return lib().rec_attn_status_string(int(code)).decode()


def rec_attn_plan(params: RecAttnParams, offsets_host, offsets_dev, timestamps_dev, types_dev,
                  stream=None) -> Plan:
    """Plan a packed batch.  offsets_host: host int64 [B+1] (numpy or CPU tensor);
    offsets_dev / timestamps_dev: device int64; types_dev: device int8."""
    off_h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int64))
    B = len(off_h) - 1
    h = ctypes.c_void_p()
    code = lib().rec_attn_plan(ctypes.byref(params), B, _ptr(off_h), _ptr(offsets_dev),
                               _ptr(timestamps_dev), _ptr(types_dev), _stream(stream), ctypes.byref(h))
    _check("rec_attn_plan", code)
    return Plan(h.value, B, int(off_h[-1]) if B > 0 else 0, (offsets_dev, timestamps_dev, types_dev))


def rec_attn_plan_query_pruned(params: RecAttnParams, keep_user_queries: int, offsets_host, offsets_dev,
                               timestamps_dev, types_dev, stream=None) -> Plan:
    """rec_attn_plan for a layer that computes every non-user query and the last
    `keep_user_queries` user queries of each request (-1: all)."""
    off_h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int64))
    B = len(off_h) - 1
    h = ctypes.c_void_p()
    code = lib().rec_attn_plan_query_pruned(ctypes.byref(params), int(keep_user_queries), B, _ptr(off_h),
                                            _ptr(offsets_dev), _ptr(timestamps_dev), _ptr(types_dev),
                                            _stream(stream), ctypes.byref(h))
    _check("rec_attn_plan_query_pruned", code)
    return Plan(h.value, B, int(off_h[-1]) if B > 0 else 0, (offsets_dev, timestamps_dev, types_dev))


def rec_attn_query_keep(hist_len: int, n_min: int, layer: int, n_layers: int) -> int:
    """LazFormer Eq. 22 per-layer query budget (host-only)."""
    return int(lib().rec_attn_query_keep(int(hist_len), int(n_min), int(layer), int(n_layers)))


def rec_attn_fwd(plan: Plan, q, k, v, out, lse=None, stream=None) -> None:
    code = lib().rec_attn_fwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                              _stream(stream))
    _check("rec_attn_fwd", code)


def rec_attn_fwd_fused(plan: Plan, q, k, v, out, lse=None, stream=None, q_norm_weight=None,
                       k_norm_weight=None, norm_eps: float = 1e-6, q_gate=None, k_gate=None,
                       out_gate=None) -> None:
    """rec_attn_fwd with QK-RMSNorm (float32 [H, d] gains), Q/K sigmoid gates and the
    attention output gate ([T, H, d] pre-activations in the I/O dtype); None = off."""
    f = RecAttnFused(_ptr(q_norm_weight), _ptr(k_norm_weight), float(norm_eps), _ptr(q_gate),
                     _ptr(k_gate), _ptr(out_gate))
    code = lib().rec_attn_fwd_fused(plan.handle, _ptr(q), _ptr(k), _ptr(v), ctypes.byref(f), _ptr(out),
                                    _ptr(lse), _stream(stream))
    _check("rec_attn_fwd_fused", code)


def rec_attn_bwd(plan: Plan, q, k, v, out, lse, dout, dq, dk, dv, stream=None) -> None:
    """Gradients dq, dk, dv of rec_attn_fwd for the upstream gradient dout."""
    code = lib().rec_attn_bwd(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                              _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream))
    _check("rec_attn_bwd", code)


class RecAttnFusedGrads(ctypes.Structure):
    _fields_ = [("dq_gate", ctypes.c_void_p), ("dk_gate", ctypes.c_void_p), ("dout_gate", ctypes.c_void_p),
                ("dq_norm_weight", ctypes.c_void_p), ("dk_norm_weight", ctypes.c_void_p)]


def rec_attn_bwd_fused(plan: Plan, q, k, v, out, lse, dout, dq, dk, dv, stream=None, q_norm_weight=None,
                       k_norm_weight=None, norm_eps: float = 1e-6, q_gate=None, k_gate=None, out_gate=None,
                       dq_gate=None, dk_gate=None, dout_gate=None, dq_norm_weight=None, dk_norm_weight=None) -> None:
    """Gradients of rec_attn_fwd_fused (the fused steps' arguments as there) into dq, dk,
    dv and the gate / gain gradients of the steps that are on."""
    L = lib()
    vp = ctypes.c_void_p
    L.rec_attn_bwd_fused.argtypes = [vp, vp, vp, vp, ctypes.POINTER(RecAttnFused), vp, vp, vp, vp, vp, vp,
                                     ctypes.POINTER(RecAttnFusedGrads), vp]
    L.rec_attn_bwd_fused.restype = ctypes.c_int
    f = RecAttnFused(_ptr(q_norm_weight), _ptr(k_norm_weight), float(norm_eps), _ptr(q_gate), _ptr(k_gate),
                     _ptr(out_gate))
    g = RecAttnFusedGrads(_ptr(dq_gate), _ptr(dk_gate), _ptr(dout_gate), _ptr(dq_norm_weight), _ptr(dk_norm_weight))
    _check("rec_attn_bwd_fused", L.rec_attn_bwd_fused(plan.handle, _ptr(q), _ptr(k), _ptr(v), ctypes.byref(f),
                                                      _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                                      ctypes.byref(g), _stream(stream)))


def _segments(segments):
    sl = np.ascontiguousarray([int(a) for a, _ in segments], dtype=np.int64)
    sg = np.ascontiguousarray([int(g) for _, g in segments], dtype=np.int32)
    return sl, sg


def rec_attn_compress_lengths(offsets_host, hist_begin, hist_len, segments) -> np.ndarray:
    """Output offsets of history compression; segments = [(length or -1, group), ...]
    from the most recent."""
    off = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int64))
    hb = np.ascontiguousarray(np.asarray(hist_begin, dtype=np.int64))
    hl = np.ascontiguousarray(np.asarray(hist_len, dtype=np.int64))
    sl, sg = _segments(segments)
    out = np.zeros(len(off), dtype=np.int64)
    _check("rec_attn_compress_lengths",
           lib().rec_attn_compress_lengths(len(off) - 1, _ptr(off), _ptr(hb), _ptr(hl), len(sl), _ptr(sl), _ptr(sg),
                                           _ptr(out)))
    return out


def rec_attn_compress(offsets_host, hist_begin, hist_len, segments, x, timestamps, types, x_out, t_out, ty_out,
                      stream=None) -> None:
    """History compression of device rows x [T, width] (bf16 or float32) into x_out."""
    off = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int64))
    hb = np.ascontiguousarray(np.asarray(hist_begin, dtype=np.int64))
    hl = np.ascontiguousarray(np.asarray(hist_len, dtype=np.int64))
    sl, sg = _segments(segments)
    import torch
    dtype = BF16 if x.dtype == torch.bfloat16 else FP32
    width = x[0].numel() if x.shape[0] > 0 else int(np.prod(x.shape[1:]))
    code = lib().rec_attn_compress(len(off) - 1, _ptr(off), _ptr(hb), _ptr(hl), len(sl), _ptr(sl), _ptr(sg), dtype,
                                   int(width), _ptr(x), _ptr(timestamps), _ptr(types), _ptr(x_out), _ptr(t_out),
                                   _ptr(ty_out), _stream(stream))
    _check("rec_attn_compress", code)


def rec_attn_fwd_compress(plan: Plan, q, k, v, hist_begin, hist_len, segments, x_out, t_out, ty_out,
                          stream=None) -> None:
    """Attention forward whose output is written already history-compressed
    (segments = [(length or -1, group), ...] from the most recent; groups <= 32)."""
    L = lib()
    vp = ctypes.c_void_p
    L.rec_attn_fwd_compress.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp, vp, vp, vp]
    L.rec_attn_fwd_compress.restype = ctypes.c_int
    hb = np.ascontiguousarray(np.asarray(hist_begin, dtype=np.int64))
    hl = np.ascontiguousarray(np.asarray(hist_len, dtype=np.int64))
    sl, sg = _segments(segments)
    _check("rec_attn_fwd_compress", L.rec_attn_fwd_compress(
        plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(hb), _ptr(hl), len(sl), _ptr(sl), _ptr(sg), _ptr(x_out),
        _ptr(t_out), _ptr(ty_out), _stream(stream)))


def rec_attn_check_wait_timeout(limit_ms: int = 50, stream=None) -> int:
    """Run the kernels' bounded wait on a barrier nothing arrives at; returns the
    status word it wrote (ERR_TIMEOUT when the failure detection works)."""
    st = ctypes.c_int32()
    _check("rec_attn_check_wait_timeout", lib().rec_attn_check_wait_timeout(int(limit_ms), ctypes.byref(st),
                                                                             _stream(stream)))
    return int(st.value)


def rec_attn_free(plan: Plan) -> None:
    if plan is not None and plan.handle:
        lib().rec_attn_free(plan.handle)
        plan.handle = 0


def rec_attn_tile_classes(plan: Plan) -> np.ndarray:
    n = ctypes.c_size_t()
    _check("rec_attn_tile_classes", lib().rec_attn_tile_classes(plan.handle, None, 0, ctypes.byref(n)))
    out = np.zeros(max(n.value, 1), dtype=np.uint8)
    _check("rec_attn_tile_classes",
           lib().rec_attn_tile_classes(plan.handle, out.ctypes.data, out.size, ctypes.byref(n)))
    return out[:n.value]


def rec_attn_visible_pairs(plan: Plan) -> int:
    n = ctypes.c_uint64()
    _check("rec_attn_visible_pairs", lib().rec_attn_visible_pairs(plan.handle, ctypes.byref(n)))
    return int(n.value)


@dataclass
class KVCache:
    handle: int
    batch: int
    max_cands: int
    _keep: tuple = ()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        rec_attn_cache_free(self)


def rec_attn_cache_create(params: RecAttnParams, hist_offsets_host, hist_t, hist_types, k_hist, v_hist,
                          max_cands: int, stream=None) -> KVCache:
    """Cache the rotated history keys, values, times and types of a batch of requests
    (serving: candidate micro-batches are then scored against them)."""
    L = lib()
    vp = ctypes.c_void_p
    L.rec_attn_cache_create.argtypes = [ctypes.POINTER(RecAttnParams), ctypes.c_int32, vp, vp, vp, vp, vp,
                                        ctypes.c_int32, vp, ctypes.POINTER(vp)]
    L.rec_attn_cache_create.restype = ctypes.c_int
    off = np.ascontiguousarray(np.asarray(hist_offsets_host, dtype=np.int64))
    h = ctypes.c_void_p()
    _check("rec_attn_cache_create", L.rec_attn_cache_create(
        ctypes.byref(params), len(off) - 1, _ptr(off), _ptr(hist_t), _ptr(hist_types), _ptr(k_hist), _ptr(v_hist),
        int(max_cands), _stream(stream), ctypes.byref(h)))
    return KVCache(h.value, len(off) - 1, int(max_cands))


def rec_attn_cache_score(cache: KVCache, cand_offsets_host, cand_t, q, k, v, out, lse=None, stream=None) -> None:
    """Outputs of one micro-batch of candidates per request against the cached history."""
    L = lib()
    vp = ctypes.c_void_p
    L.rec_attn_cache_score.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.rec_attn_cache_score.restype = ctypes.c_int
    off = np.ascontiguousarray(np.asarray(cand_offsets_host, dtype=np.int64))
    _check("rec_attn_cache_score", L.rec_attn_cache_score(cache.handle, _ptr(off), _ptr(cand_t), _ptr(q), _ptr(k),
                                                          _ptr(v), _ptr(out), _ptr(lse), _stream(stream)))


def rec_attn_cache_free(cache: KVCache) -> None:
    if cache is not None and cache.handle:
        L = lib()
        L.rec_attn_cache_free.argtypes = [ctypes.c_void_p]
        L.rec_attn_cache_free.restype = None
        L.rec_attn_cache_free(cache.handle)
        cache.handle = 0


MASK_APPLIED, MASK_BUILT, MASK_PREDICATE = 0, 1, 2


def rec_attn_applied_masks(plan: Plan, pairs, mode: int = MASK_APPLIED):
    """Visibility bits the attention kernels apply to (request, query tile, key tile)
    pairs: returns (bits uint32 [n, 128, 4], list class uint8 [n] (0xff: not listed),
    mask-table slot int32 [n])."""
    L = lib()
    vp = ctypes.c_void_p
    L.rec_attn_applied_masks.argtypes = [vp, ctypes.c_int32, vp, ctypes.c_int32, vp, vp, vp]
    L.rec_attn_applied_masks.restype = ctypes.c_int
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 3))
    n = pr.shape[0]
    bits = np.zeros((n, TILE, 4), dtype=np.uint32)
    cls = np.zeros(n, dtype=np.uint8)
    slot = np.zeros(n, dtype=np.int32)
    _check("rec_attn_applied_masks", L.rec_attn_applied_masks(plan.handle, n, _ptr(pr), int(mode), _ptr(bits),
                                                              _ptr(cls), _ptr(slot)))
    return bits, cls, slot


def rec_attn_device_status(plan: Plan) -> int:
    s = ctypes.c_int32()
    _check("rec_attn_device_status", lib().rec_attn_device_status(plan.handle, ctypes.byref(s)))
    return int(s.value)


class RecAttnTimings(ctypes.Structure):
    _fields_ = [("rope_ms", ctypes.c_float), ("attn_ms", ctypes.c_float)]


def rec_attn_enable_timing(plan: Plan) -> None:
    L = lib()
    L.rec_attn_enable_timing.argtypes = [ctypes.c_void_p]
    L.rec_attn_enable_timing.restype = ctypes.c_int
    _check("rec_attn_enable_timing", L.rec_attn_enable_timing(plan.handle))


def rec_attn_read_timings(plan: Plan) -> tuple[float, float]:
    """(rope_ms, attn_ms) of the last timed rec_attn_fwd."""
    L = lib()
    L.rec_attn_read_timings.argtypes = [ctypes.c_void_p, ctypes.POINTER(RecAttnTimings)]
    L.rec_attn_read_timings.restype = ctypes.c_int
    t = RecAttnTimings()
    _check("rec_attn_read_timings", L.rec_attn_read_timings(plan.handle, ctypes.byref(t)))
    return float(t.rope_ms), float(t.attn_ms)


NOALLOC_SCRATCH_BYTES = 16 << 20


def rec_attn_fwd_noalloc(params: RecAttnParams, offsets_host, offsets_dev, timestamps_dev, types_dev,
                         q, k, v, out, lse=None, stream=None) -> None:
    """Plan + RoPE + attention without any device allocation (static workspace of
    NOALLOC_SCRATCH_BYTES shared by all calls; calls must not overlap on the GPU)."""
    L = lib()
    vp = ctypes.c_void_p
    L.rec_attn_fwd_noalloc.argtypes = [ctypes.POINTER(RecAttnParams), ctypes.c_int32, vp, vp, vp, vp,
                                       vp, vp, vp, vp, vp, vp]
    L.rec_attn_fwd_noalloc.restype = ctypes.c_int
    off_h = np.ascontiguousarray(np.asarray(offsets_host, dtype=np.int64))
    code = L.rec_attn_fwd_noalloc(ctypes.byref(params), len(off_h) - 1, _ptr(off_h), _ptr(offsets_dev),
                                  _ptr(timestamps_dev), _ptr(types_dev), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(out), _ptr(lse), _stream(stream))
    _check("rec_attn_fwd_noalloc", code)
