"""Helpers shared by the GPU tests: move a seeded workload to the device, run the
C-ABI path, and compare with the CPU oracle."""
import numpy as np
import torch

import oracle
from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import build as bld
from generative_recommender_ranking_gb300 import workloads as W

# tolerances the tests hold the CUDA path to (outputs vs the fp64 oracle)
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
FP32_MAX_ABS = 1e-4


def ensure_built():
    bld.build()
    oracle.build()


def device_inputs(w: W.Workload, dev="cuda"):
    tens = {}
    tens["off_h"] = np.ascontiguousarray(w.offsets, dtype=np.int64)
    tens["off_d"] = torch.from_numpy(tens["off_h"]).to(dev)
    tens["t"] = torch.from_numpy(np.ascontiguousarray(w.t)).to(dev)
    tens["ty"] = torch.from_numpy(np.ascontiguousarray(w.types)).to(dev)
    if w.dtype == "bf16":
        conv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        conv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    tens["q"], tens["k"], tens["v"] = conv(w.q), conv(w.k), conv(w.v)
    return tens


def params_for(w: W.Workload, **over):
    kw = dict(w.mask)
    kw.update(w.rope)
    kw.update(over)
    return bd.make_params(w.num_heads, w.head_dim, dtype=w.dtype, **kw)


def oracle_params(w: W.Workload, **over):
    kw = dict(w.mask)
    kw.update(w.rope)
    kw.update(over)
    return oracle.Params(w.num_heads, w.head_dim, **kw)


def run_gpu(w: W.Workload, tens=None, with_lse=False, poison=True, **over):
    """plan + fwd through the C-ABI; returns (out tensor, lse tensor or None, plan)."""
    tens = tens or device_inputs(w)
    p = params_for(w, **over)
    plan = bd.rec_attn_plan(p, tens["off_h"], tens["off_d"], tens["t"], tens["ty"])
    out = torch.empty_like(tens["q"])
    if poison:
        out.fill_(float("nan"))
    lse = torch.full((w.total_tokens, w.num_heads), float("nan"), device=out.device) if with_lse else None
    bd.rec_attn_fwd(plan, tens["q"], tens["k"], tens["v"], out, lse)
    torch.cuda.synchronize()
    return out, lse, plan


def to_f64(x: torch.Tensor) -> np.ndarray:
    return x.float().cpu().numpy().astype(np.float64)


def errors(gpu: np.ndarray, ref: np.ndarray):
    d = np.abs(gpu - ref)
    return float(np.nanmax(d)) if d.size else 0.0, float(np.mean(d)) if d.size else 0.0


def assert_close(w: W.Workload, gpu: np.ndarray, ref: np.ndarray, what=""):
    assert not np.isnan(gpu).any(), f"{what}: NaN in the CUDA output (unwritten or invalid rows)"
    mx, mean = errors(gpu, ref)
    if w.dtype == "bf16":
        assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, f"{what}: max {mx:.3e} mean {mean:.3e}"
    else:
        assert mx <= FP32_MAX_ABS, f"{what}: max {mx:.3e}"
    return mx, mean


def sample_rows(w: W.Workload, per_request=48, max_requests=6, seed=0):
    """Sorted global rows: first/last rows, tile edges and random rows of a few requests."""
    rng = np.random.default_rng(seed)
    B = w.batch
    reqs = sorted(set([0, B - 1] + list(rng.choice(B, size=min(B, max_requests), replace=False))))
    rows = []
    for b in reqs:
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        L = e - s
        if L == 0:
            continue
        cand = {0, L - 1, min(L - 1, 127), min(L - 1, 128), L // 2}
        cand |= set(int(x) for x in rng.integers(0, L, size=per_request))
        rows += [s + c for c in sorted(cand)]
    return np.array(sorted(set(rows)), dtype=np.int64)


def unpack_bits(bits: np.ndarray) -> np.ndarray:
    """[n, 128, 4] uint32 row words -> [n, 128, 128] uint8 (key c = bit c % 32 of word c / 32)."""
    b = np.ascontiguousarray(bits, dtype="<u4").view(np.uint8)
    return np.unpackbits(b, axis=-1, bitorder="little")


def all_pairs(w: W.Workload, requests=None):
    """(request, query tile, key tile) for every tile pair of the given requests."""
    out = []
    for b in (range(w.batch) if requests is None else requests):
        nt = (int(w.offsets[b + 1] - w.offsets[b]) + 127) // 128
        if nt:
            qt, kt = np.meshgrid(np.arange(nt), np.arange(nt), indexing="ij")
            out.append(np.stack([np.full(nt * nt, b), qt.ravel(), kt.ravel()], axis=1))
    return np.concatenate(out).astype(np.int32) if out else np.zeros((0, 3), dtype=np.int32)


def check_applied_masks(w: W.Workload, plan, pairs, op, modes=(0, 1, 2), tile_cls=None):
    """Hold the visibility bits the kernels apply (rec_attn_applied_masks, every mode)
    bit for bit against the oracle's mask on the same pairs.  A pair missing from the
    key-tile lists must have no visible pair (and is applied as all zero); a FULL pair
    must be all visible over a complete key tile; a PARTIAL pair's bits must equal the
    mask on the request's rows, with zeros for keys past the request end.  tile_cls
    (optional): the oracle's classes as a dict, whose non-SKIP pairs must be exactly the
    listed ones with the same class.  Pairs are checked request by request.  Returns
    {mode: (pairs checked, pairs with a mask-table slot, PARTIAL pairs)}."""
    pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 3)
    stats = {m: [0, 0, 0] for m in modes}
    for b in np.unique(pairs[:, 0]).tolist():
        pb = pairs[pairs[:, 0] == b]
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        L = e - s
        nk = 128 * ((L + 127) // 128)
        ref = {qt: oracle.mask_block(op, w.t[s:e], w.types[s:e], 128 * qt, 128, 0, nk)
               for qt in np.unique(pb[:, 1]).tolist()}
        for mode in modes:
            bits, lcls, slot = bd.rec_attn_applied_masks(plan, pb, mode)
            got = unpack_bits(bits)
            for n, (_, qt, kt) in enumerate(pb.tolist()):
                rows = min(128, L - 128 * qt)
                blk = ref[qt][:, 128 * kt:128 * kt + 128]
                g = got[n]
                where = f"{w.name} mode {mode} pair (b={b}, qt={qt}, kt={kt}) list class {lcls[n]}"
                if lcls[n] == 0xFF:
                    assert not blk.any(), f"{where}: a visible pair in a tile the kernels never load"
                    assert not g.any(), where
                elif lcls[n] == bd.TILE_FULL:
                    assert L - 128 * kt >= 128 and blk[:rows].all(), f"{where}: FULL over a masked pair"
                    assert g.all(), where
                else:
                    assert lcls[n] == bd.TILE_PARTIAL, where
                    bad = np.argwhere(g[:rows] != blk[:rows])
                    assert bad.size == 0, f"{where}: {len(bad)} bits differ, first (row, key) {bad[:4].tolist()}"
                    assert not g[rows:].any(), f"{where}: bits set on rows past the request end"
                    stats[mode][2] += 1
                if tile_cls is not None:
                    c = int(tile_cls[(b, qt, kt)])
                    assert (lcls[n] == 0xFF) == (c == bd.TILE_SKIP) and (c == bd.TILE_SKIP or lcls[n] == c), where
            stats[mode][0] += len(pb)
            stats[mode][1] += int((slot >= 0).sum())
    return {m: tuple(v) for m, v in stats.items()}


def tile_class_map(w: W.Workload, cls: np.ndarray):
    """The flat request-major class array as a dict (b, qt, kt) -> class."""
    out, i = {}, 0
    for b in range(w.batch):
        nt = (int(w.offsets[b + 1] - w.offsets[b]) + 127) // 128
        blk = cls[i:i + nt * nt].reshape(nt, nt)
        for qt in range(nt):
            for kt in range(nt):
                out[(b, qt, kt)] = blk[qt, kt]
        i += nt * nt
    return out


def rising_scores(base: W.Workload, seed=23, steep=0.2) -> W.Workload:
    """The same requests with scores that rise along each row: keys gain a component
    along a fixed per-head direction that the queries share, growing with the key's
    position within its request (head 0 by `steep` per position, head 1 gently with
    bumps, further heads untouched), and the time-RoPE off so the alignment survives."""
    rng = np.random.default_rng(seed)
    T, H, d = base.q.shape
    u = rng.standard_normal((H, d)).astype(np.float32)
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    q = rng.standard_normal((T, H, d)).astype(np.float32) + 2.0 * u[None]
    k = rng.standard_normal((T, H, d)).astype(np.float32)
    for b in range(base.batch):
        s, e = int(base.offsets[b]), int(base.offsets[b + 1])
        j = np.arange(e - s, dtype=np.float32)
        k[s:e, 0] += (steep * j)[:, None] * u[0][None]
        if H > 1:
            k[s:e, 1] += (0.03 * j + 6.0 * np.sin(j / 97.0))[:, None] * u[1][None]
    if base.dtype == "bf16":
        q, k = W.round_to_bf16_bits(q), W.round_to_bf16_bits(k)
    return W.Workload(**{**base.__dict__, "q": q, "k": k, "rope": dict(base.rope, use_rope=False)})

