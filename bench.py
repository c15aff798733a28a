"""Benchmark of the masked time-RoPE attention forward on GB300.

One step = the whole hot path over one batch: plan (tile statistics, tile
classes, key-tile lists, mask table, schedule), time-RoPE prologue, fused masked
attention, plan release.  Default workload: TM20K / LazFormer long histories,
B=16 requests x (20000 history tokens + 1 target), H=8, d=64, bf16, full causal
attention, time-RoPE (the largest single-GPU configuration).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line.  `value` is TFLOP/s counted over visible (query, key) pairs
(4 * d * H per pair) for the whole step (mean over the K timed steps), inputs
resident in HBM; L2 is flushed between timed steps.  The line also carries the
medians of 50 iterations (after 10 warm-ups) of the forward alone and of plan +
forward.  `--impl reference` times the fp64 CPU oracle on the host cores instead
(a bounded sample of the same workload per step).
Under torchrun each rank runs its own batch of the same shape (weak scaling); the
reported value is the total work of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from generative_recommender_ranking_gb300 import workloads as W  # noqa: E402

METRIC = "masked-attn fwd TFLOP/s over visible pairs, % of GB300 bf16 peak; tokens/s"
L2_FLUSH_BYTES = 256 << 20
E2E_RUNS = 5  # runs of the end-to-end leg; the median is reported
# history-compression settings: recency segments (length or -1, group size), newest first
COMPRESS_SPECS = {
    "lazformer_keep1024_g8": [(1024, 1), (-1, 8)],
    "lptm_pairs": [(-1, 2)],
    "patm_bands": [(1000, 1), (4000, 2), (5000, 3), (-1, 4)],
}
# CUDA-core fp32 peak of a GB300 from its unit counts: 152 SMs x 128 FMA lanes x 2 FLOP
# x 2070 MHz (the fp32 backward pass runs there)
FP32_FMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def _traffic(workload: str):
    """DRAM bytes (read + write) of one attention launch from the committed ncu capture
    ("<workload>" or "<workload>/fused"), or None when there is no capture of that case or
    the kernel sources have changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "k_attn_tc_dram_traffic.json")
    try:
        import hashlib
        with open(path) as f:
            d = json.load(f)
        h = hashlib.sha256()
        for src in d["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != d["sources_sha256"] or workload not in d["workloads"]:
            return None
        x = d["workloads"][workload]
        return float(x["dram_bytes_read"] + x["dram_bytes_write"])
    except (OSError, KeyError, ValueError):
        return None


def _compress_traffic(workload: str, spec: str):
    """DRAM bytes of one compression launch from the committed ncu capture, or None (no
    capture for this case, or the kernel sources changed since it was taken)."""
    path = os.path.join(ROOT, "profiles", "k_compress_dram_traffic.json")
    try:
        import hashlib
        with open(path) as f:
            d = json.load(f)
        h = hashlib.sha256()
        for src in d["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        x = d["cases"].get(f"{workload}/{spec}")
        if h.hexdigest() != d["sources_sha256"] or x is None:
            return None
        return float(x["dram_bytes_read"] + x["dram_bytes_write"])
    except (OSError, KeyError, ValueError):
        return None


def _workload(name, rank, batch=None, history=None, heads=None, head_dim=None):
    kw = {}
    if heads:
        kw["heads"] = heads
    if head_dim:
        kw["head_dim"] = head_dim
    if rank:
        base = {"tiny_fp32": 1001, "cadet": 1002, "sort": 1003, "mtgr": 1004}.get(name, 1005)
        kw["seed"] = base + 7919 * rank
    if batch:
        kw["batch"] = batch
    if history:
        if not name.startswith("tm20k"):
            raise SystemExit("--history applies to the tm20k workloads")
        kw["n_hist"] = history
    return W.make(name, **kw)


def _planner_split(w: W.Workload) -> int:
    """1 when the planner runs its per-tile kernel apart (mean tiles per request >= 32)."""
    n_tiles = int(sum((int(n) + 127) // 128 for n in np.diff(w.offsets)))
    return int(w.batch > 0 and -(-n_tiles // w.batch) >= 32)


def _config(w: W.Workload, name: str, parallelism: str):
    lens = np.diff(w.offsets)
    return {"workload": name, "batch": w.batch, "tokens": w.total_tokens,
            "seq_len_mean": float(lens.mean()) if len(lens) else 0.0, "seq_len_max": int(lens.max()),
            "heads": w.num_heads, "head_dim": w.head_dim, "mask": w.mask,
            "time_rope": {k: v for k, v in w.rope.items()}, "parallelism": parallelism,
            "l2": "flushed between timed steps (256 MiB write)"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}",
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[4:8]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- CPU oracle

LONG_REQUEST = 4096  # requests longer than this are sampled by rows for the CPU oracle


def _sample_rows(w: W.Workload, rows_per_request: int, keep: int = -1, seed: int = 4242) -> np.ndarray:
    """Seeded query rows (sorted global indices), up to rows_per_request per request:
    always the first and last rows, the rows at the 128-token tile edges around the
    window and the global-token boundary, the rest uniform.  Under query pruning only
    computed rows are drawn."""
    import oracle
    rng = np.random.default_rng(seed)
    kept = None if keep < 0 else set(oracle.kept_rows(w.offsets, w.types, keep).tolist())
    win = int(w.mask.get("window", 0))
    out = []
    for b in range(w.batch):
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        L = e - s
        cand = np.arange(L) if kept is None else np.array([i for i in range(L) if s + i in kept], dtype=np.int64)
        if len(cand) == 0:
            continue
        if len(cand) <= rows_per_request:
            out.extend((s + cand).tolist())
            continue
        n_glob = int((w.types[s:e] == W.GLOBAL).sum())
        must = {int(cand[0]), int(cand[-1])}
        for x in (127, 128, n_glob - 1, n_glob, win - 1, win, win + 1, n_glob + win - 1, n_glob + win):
            if 0 <= x < L and (kept is None or s + x in kept):
                must.add(int(x))
        rest = np.setdiff1d(cand, np.fromiter(must, dtype=np.int64))
        pick = rng.choice(rest, size=max(0, rows_per_request - len(must)), replace=False)
        out.extend(sorted(s + np.concatenate([np.fromiter(must, dtype=np.int64), pick])))
    return np.array(sorted(out), dtype=np.int64)


def _oracle_rows(w: W.Workload, rows: np.ndarray, threads: int):
    """Time the fp64 oracle on the given query rows (all heads); returns (seconds,
    visible pairs of those rows per head)."""
    import oracle
    p = oracle.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    t0 = time.perf_counter()
    oracle.attention(p, w.offsets, w.t, w.types, w.q, w.k, w.v, rows=rows, threads=threads)
    secs = time.perf_counter() - t0
    pairs = 0
    req = np.searchsorted(w.offsets, rows, side="right") - 1
    for b in np.unique(req).tolist():
        s, e = int(w.offsets[b]), int(w.offsets[b + 1])
        for i in (rows[req == b] - s).tolist():
            pairs += int(oracle.mask_block(p, w.t[s:e], w.types[s:e], i, 1, 0, e - s).sum())
    return secs, pairs


def _oracle_sample(w: W.Workload, budget_s: float, keep: int = -1, rows_per_request: int = 2048, seed: int = 4242):
    """Time the fp64 oracle on a bounded sample of the workload (all heads; with query
    pruning, the computed rows only).  Requests up to LONG_REQUEST tokens: whole
    requests from the first, doubling the count until about `budget_s` seconds of work.
    Longer requests (the 20K-token histories): rows_per_request seeded rows of every
    request.  Returns (seconds, visible pairs per head, description, threads)."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    if w.batch and int(np.diff(w.offsets).max()) > LONG_REQUEST:
        rows = _sample_rows(w, rows_per_request, keep, seed)
        secs, pairs = _oracle_rows(w, rows, threads)
        return secs, pairs, f"{rows_per_request} seeded rows of each of the {w.batch} requests (first, last, tile, " \
                            f"window and global-token boundary rows included), all heads", threads
    p = oracle.Params(w.num_heads, w.head_dim, **w.mask, **w.rope)
    done, secs, pairs = 0, 0.0, 0
    chunk = 1
    while done < w.batch and secs < budget_s:
        n = min(chunk, w.batch - done)
        s, e = int(w.offsets[done]), int(w.offsets[done + n])
        off = w.offsets[done:done + n + 1] - s
        sl = slice(s, e)
        rows = None if keep < 0 else oracle.kept_rows(off, w.types[sl], keep)
        t0 = time.perf_counter()
        oracle.attention(p, off, w.t[sl], w.types[sl], w.q[sl], w.k[sl], w.v[sl], rows=rows, threads=threads)
        secs += time.perf_counter() - t0
        if rows is None:
            pairs += oracle.visible_pairs(p, off, w.t[sl], w.types[sl])
        else:
            for b in range(n):
                bs, be = int(off[b]), int(off[b + 1])
                r = rows[(rows >= bs) & (rows < be)] - bs
                pairs += int(oracle.mask(p, w.t[sl][bs:be], w.types[sl][bs:be])[r].sum())
        done += n
        chunk *= 2
    return secs, pairs, f"first {done} of {w.batch} requests, all heads", threads


def run_reference(args):
    """--impl reference: the fp64 CPU oracle on the host cores, same metric.  Each step
    is a bounded sample of the workload, sized so that warm-up and steps take about a
    minute together."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    w = _workload(args.workload, 0, args.batch, args.history, args.heads, args.head_dim)
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    long_req = w.batch and int(np.diff(w.offsets).max()) > LONG_REQUEST
    rows_per_request = 512
    if long_req:
        # calibrate the rows per request on a first small sample (counted as warm-up)
        s0, _, _, _ = _oracle_sample(w, per_step, args.keep_user_queries, rows_per_request=8, seed=1)
        rows_per_request = int(max(4, min(512, 8 * per_step / max(s0, 1e-3))))
    for i in range(args.warmup):
        _oracle_sample(w, per_step / 4, args.keep_user_queries, rows_per_request=max(4, rows_per_request // 4),
                       seed=100 + i)
    tot_s, tot_pairs, desc = 0.0, 0, ""
    threads = 1
    for i in range(args.steps):
        s, pairs, desc, threads = _oracle_sample(w, per_step, args.keep_user_queries,
                                                 rows_per_request=rows_per_request, seed=1000 + i)
        tot_s += s
        tot_pairs += pairs
    flops = 4.0 * w.head_dim * w.num_heads * tot_pairs
    value = flops / tot_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, args.workload, "host cores"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"per step: {desc}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def run_compress(args):
    """--compress: history compression of the workload's K rows ([T, H*d]), HBM-bound."""
    import torch
    from generative_recommender_ranking_gb300 import binding as bd
    from generative_recommender_ranking_gb300 import build as bld
    bld.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = _workload(args.workload, 0, args.batch, args.history, args.heads, args.head_dim)
    segs = COMPRESS_SPECS[args.compress]
    hb, hl = [], []
    for b in range(w.batch):
        s0, e0 = int(w.offsets[b]), int(w.offsets[b + 1])
        idx = np.nonzero(w.types[s0:e0] == W.HIST)[0]
        hb.append(int(idx[0]) if len(idx) else 0)
        hl.append(len(idx))
    T = w.total_tokens
    raw = w.k.reshape(T, -1)
    x = (torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16) if raw.dtype == np.uint16
         else torch.from_numpy(raw)).to(dev)
    t = torch.from_numpy(w.t).to(dev)
    ty = torch.from_numpy(w.types).to(dev)
    out_off = bd.rec_attn_compress_lengths(w.offsets, hb, hl, segs)
    n = int(out_off[-1])
    x_out = torch.empty((n, x.shape[1]), dtype=x.dtype, device=dev)
    t_out = torch.empty(n, dtype=torch.int64, device=dev)
    ty_out = torch.empty(n, dtype=torch.int8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    call = lambda: bd.rec_attn_compress(w.offsets, hb, hl, segs, x, t, ty, x_out, t_out, ty_out, stream)
    for _ in range(max(args.warmup, 3)):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    elem = x.element_size()
    nbytes = (T + n) * x.shape[1] * elem + 9.0 * (T + n)
    gbs = nbytes / (ms * 1e-3) / 1e9
    pk = _peaks()
    print(json.dumps({
        "metric": "history compression GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "dtype": w.dtype,
        "data": "synthetic", "config": {"workload": args.workload, "rows_in": T, "rows_out": n,
                                        "width": int(x.shape[1]), "segments": segs,
                                        "l2": "flushed between timed steps (256 MiB write)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"],
                     "traffic": (_compress_traffic(args.workload, args.compress)
                                 if args.batch is None and args.history is None and args.heads is None
                                 and args.head_dim is None else None),
                     "kernel": "k_compress",
                     "peak_source": pk["source"], "algorithmic_bytes_per_launch": nbytes, "ms_per_launch": ms},
        "gpu_launches": args.steps}), flush=True)
    return 0


def run_serving(args):
    """--serving: per-request latency of scoring a request's candidates against its
    cached history (M-FALCON micro-batches; CADET's serving scenario): for each request,
    rec_attn_cache_create (rotated history K', V) then rec_attn_cache_score over the
    candidates in micro-batches of --micro-batch, timed with CUDA events; beside it the
    uncached path (one query-pruned plan over [history, candidates], keep = 0)."""
    import torch
    from generative_recommender_ranking_gb300 import binding as bd
    from generative_recommender_ranking_gb300 import build as bld
    bld.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = _workload(args.workload, 0, args.batch, args.history, args.heads, args.head_dim)
    params = bd.make_params(w.num_heads, w.head_dim, dtype=w.dtype, **w.mask, **w.rope)
    stream = torch.cuda.current_stream(dev)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        return (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16) if a.dtype == np.uint16
                else torch.from_numpy(a).to(dev))

    reqs = []
    for b in range(w.batch):
        s0, e0 = int(w.offsets[b]), int(w.offsets[b + 1])
        c = s0 + np.nonzero(w.types[s0:e0] == W.CAND)[0]
        h = np.arange(s0, c[0] if len(c) else e0)
        full = np.arange(s0, e0)
        reqs.append(dict(
            n_h=len(h), n_c=len(c),
            t_h=to_dev(w.t[h]), ty_h=to_dev(w.types[h]), k_h=to_dev(w.k[h]), v_h=to_dev(w.v[h]),
            t_c=to_dev(w.t[c]), q_c=to_dev(w.q[c]), k_c=to_dev(w.k[c]), v_c=to_dev(w.v[c]),
            off=np.array([0, len(full)]), off_d=to_dev(np.array([0, len(full)])), t=to_dev(w.t[full]),
            ty=to_dev(w.types[full]), q=to_dev(w.q[full]), k=to_dev(w.k[full]), v=to_dev(w.v[full])))
    n_c_max = max(r["n_c"] for r in reqs)
    bm = args.micro_batch if args.micro_batch > 0 else n_c_max
    out_c = torch.empty((n_c_max, w.num_heads, w.head_dim), dtype=reqs[0]["q_c"].dtype, device=dev)
    out_f = torch.empty((max(r["n_h"] + r["n_c"] for r in reqs), w.num_heads, w.head_dim),
                        dtype=reqs[0]["q"].dtype, device=dev)

    def cached(r):
        cache = bd.rec_attn_cache_create(params, [0, r["n_h"]], r["t_h"], r["ty_h"], r["k_h"], r["v_h"], bm, stream)
        for i0 in range(0, r["n_c"], bm):
            i1 = min(r["n_c"], i0 + bm)
            bd.rec_attn_cache_score(cache, [0, i1 - i0], r["t_c"][i0:], r["q_c"][i0:], r["k_c"][i0:],
                                    r["v_c"][i0:], out_c, None, stream)
        return cache

    def uncached(r):
        plan = bd.rec_attn_plan_query_pruned(params, 0, r["off"], r["off_d"], r["t"], r["ty"], stream)
        bd.rec_attn_fwd(plan, r["q"], r["k"], r["v"], out_f, None, stream)
        return plan

    def latencies(fn, free, n):
        for i in range(max(args.warmup, 3)):
            free(fn(reqs[i % len(reqs)]))
        torch.cuda.synchronize(dev)
        ms = []
        for i in range(n):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            h = fn(reqs[i % len(reqs)])
            b_.record(stream)
            b_.synchronize()
            ms.append(a_.elapsed_time(b_))
            free(h)
        return np.array(ms)

    n = max(args.steps, 50)
    lc = latencies(cached, bd.rec_attn_cache_free, n)
    lu = latencies(uncached, bd.rec_attn_free, n)
    # one scoring call against a cache made once per request and kept (a user whose
    # history is already cached): per micro-batch
    caches = [bd.rec_attn_cache_create(params, [0, r["n_h"]], r["t_h"], r["ty_h"], r["k_h"], r["v_h"], bm, stream)
              for r in reqs]

    def score_only(i):
        r = reqs[i % len(reqs)]
        i1 = min(r["n_c"], bm)
        bd.rec_attn_cache_score(caches[i % len(reqs)], [0, i1], r["t_c"], r["q_c"], r["k_c"], r["v_c"], out_c, None,
                                stream)

    for i in range(5):
        score_only(i)
    torch.cuda.synchronize(dev)
    ls = []
    for i in range(n):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        score_only(i)
        b_.record(stream)
        b_.synchronize()
        ls.append(a_.elapsed_time(b_))
    ls = np.array(ls)
    for c_ in caches:
        bd.rec_attn_cache_free(c_)
    cands = float(np.mean([r["n_c"] for r in reqs]))
    line = {
        "metric": "serving latency per request (cached history, candidate micro-batches)", "value": float(np.percentile(lc, 50)),
        "unit": "ms", "n_gpus": 1, "steps": n, "warmup": max(args.warmup, 3), "higher_is_better": False,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "requests": w.batch, "history_tokens": int(reqs[0]["n_h"]),
                   "candidates_per_request": int(cands), "micro_batch": bm, "heads": w.num_heads,
                   "head_dim": w.head_dim, "mask": w.mask},
        "cached": {"p50_ms": float(np.percentile(lc, 50)), "p99_ms": float(np.percentile(lc, 99)),
                   "mean_ms": float(lc.mean()), "candidates_per_s": cands / (lc.mean() * 1e-3),
                   "per_request": "rec_attn_cache_create + rec_attn_cache_score per micro-batch"},
        "score_call_cache_kept": {"p50_ms": float(np.percentile(ls, 50)), "p99_ms": float(np.percentile(ls, 99)),
                                  "candidates_per_call": int(min(bm, n_c_max)),
                                  "per_call": "rec_attn_cache_score against a cache made earlier"},
        "uncached": {"p50_ms": float(np.percentile(lu, 50)), "p99_ms": float(np.percentile(lu, 99)),
                     "mean_ms": float(lu.mean()),
                     "per_request": "rec_attn_plan_query_pruned(keep 0) + rec_attn_fwd over history + candidates"},
        "budget_context": "CADET reports a 50 ms p99 for scoring hundreds of candidates (other hardware, whole model)",
    }
    print(json.dumps(line), flush=True)
    return 0


def run_compress_fused(args):
    """--compress SPEC --fused-epilogue: one layer whose output feeds the next layer
    compressed.  Fused: plan + rec_attn_fwd_compress (the compression in the attention
    epilogue; O never reaches memory).  Unfused: plan + rec_attn_fwd + rec_attn_compress.
    Medians of CUDA-event times over --steps iterations (L2 flushed between them)."""
    import torch
    from generative_recommender_ranking_gb300 import binding as bd
    from generative_recommender_ranking_gb300 import build as bld
    bld.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = _workload(args.workload, 0, args.batch, args.history, args.heads, args.head_dim)
    segs = COMPRESS_SPECS[args.compress]
    hb, hl = [], []
    for b in range(w.batch):
        s0, e0 = int(w.offsets[b]), int(w.offsets[b + 1])
        idx = np.nonzero(w.types[s0:e0] == W.HIST)[0]
        hb.append(int(idx[0]) if len(idx) else 0)
        hl.append(len(idx))

    def to_dev(a):
        a = np.ascontiguousarray(a)
        return (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16) if a.dtype == np.uint16
                else torch.from_numpy(a).to(dev))

    q, k, v = to_dev(w.q), to_dev(w.k), to_dev(w.v)
    t, ty, off_d = to_dev(w.t), to_dev(w.types), to_dev(w.offsets)
    params = bd.make_params(w.num_heads, w.head_dim, dtype=w.dtype, **w.mask, **w.rope)
    out_off = bd.rec_attn_compress_lengths(w.offsets, hb, hl, segs)
    n = int(out_off[-1])
    T, H, d = w.total_tokens, w.num_heads, w.head_dim
    x_out = torch.empty((n, H, d), dtype=q.dtype, device=dev)
    t_out = torch.empty(n, dtype=torch.int64, device=dev)
    ty_out = torch.empty(n, dtype=torch.int8, device=dev)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def fused():
        p = bd.rec_attn_plan(params, w.offsets, off_d, t, ty, stream)
        bd.rec_attn_fwd_compress(p, q, k, v, hb, hl, segs, x_out, t_out, ty_out, stream)
        bd.rec_attn_free(p)

    def unfused():
        p = bd.rec_attn_plan(params, w.offsets, off_d, t, ty, stream)
        bd.rec_attn_fwd(p, q, k, v, o, None, stream)
        bd.rec_attn_compress(w.offsets, hb, hl, segs, o.view(T, H * d), t, ty, x_out.view(n, H * d), t_out, ty_out,
                             stream)
        bd.rec_attn_free(p)

    def med(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        for a_, b_ in evs:
            flush.zero_()
            a_.record(stream)
            fn()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a_.elapsed_time(b_) for a_, b_ in evs)

    tf, tu = med(fused), med(unfused)
    p = bd.rec_attn_plan(params, w.offsets, off_d, t, ty, stream)
    pairs = bd.rec_attn_visible_pairs(p)
    # the attention kernels alone (CUDA events the library records around them)
    bd.rec_attn_enable_timing(p)
    bd.rec_attn_fwd_compress(p, q, k, v, hb, hl, segs, x_out, t_out, ty_out, stream)
    attn_fused = bd.rec_attn_read_timings(p)[1]
    bd.rec_attn_fwd(p, q, k, v, o, None, stream)
    attn_plain = bd.rec_attn_read_timings(p)[1]
    bd.rec_attn_free(p)
    flops = 4.0 * d * H * pairs
    print(json.dumps({
        "metric": "attention layer with compressed output, ms per step (plan + forward + compression)",
        "value": tf, "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "higher_is_better": False, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "segments": segs, "rows_in": T, "rows_out": n, "heads": H,
                   "head_dim": d, "l2": "flushed between timed steps (256 MiB write)"},
        "fused_ms": tf, "unfused_ms": tu, "speedup": tu / tf,
        "attention_kernel_ms": {"with_compression_epilogue": attn_fused, "plain": attn_plain},
        "fused_tflops": flops / (tf * 1e-3) / 1e12,
        "bytes_saved_per_step": 2.0 * T * H * d * 2}), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    from generative_recommender_ranking_gb300 import binding as bd
    from generative_recommender_ranking_gb300 import build as bld
    from generative_recommender_ranking_gb300 import sharding

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    if rank == 0 or world == 1:
        bld.build()
    if world > 1:
        dist.barrier()

    w = _workload(args.workload, rank, args.batch, args.history, args.heads, args.head_dim)
    bf16 = w.dtype == "bf16"
    elem = 2 if bf16 else 4

    def host(a):
        t = torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a))
        return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

    hq, hk, hv = (host(a).pin_memory() for a in (w.q, w.k, w.v))
    ht = torch.from_numpy(np.ascontiguousarray(w.t)).pin_memory()
    hty = torch.from_numpy(np.ascontiguousarray(w.types)).pin_memory()
    hoff = torch.from_numpy(np.ascontiguousarray(w.offsets)).pin_memory()
    q, k, v = (x.to(dev) for x in (hq, hk, hv))
    t, ty, off_d = ht.to(dev), hty.to(dev), hoff.to(dev)
    out = torch.empty_like(q)
    off_h = np.ascontiguousarray(w.offsets)
    params = bd.make_params(w.num_heads, w.head_dim, dtype=w.dtype, **w.mask, **w.rope)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def mkplan(off_d_, t_, ty_, st=None):
        if args.keep_user_queries >= 0:
            return bd.rec_attn_plan_query_pruned(params, args.keep_user_queries, off_h, off_d_, t_, ty_, st)
        return bd.rec_attn_plan(params, off_h, off_d_, t_, ty_, st)

    # exact visible pairs (FLOP accounting) from the library's own counter
    plan = mkplan(off_d, t, ty)
    pairs = bd.rec_attn_visible_pairs(plan)
    cls = bd.rec_attn_tile_classes(plan)
    bd.rec_attn_free(plan)
    flops_fwd = 4.0 * w.head_dim * w.num_heads * pairs
    flops = flops_fwd * (3.5 if args.backward else 1.0)  # backward: 10 d per pair (2.5x forward)
    tokens = w.total_tokens
    if args.backward:
        lse_buf = torch.empty((tokens, w.num_heads), dtype=torch.float32, device=dev)
        gen = torch.Generator(device="cpu").manual_seed(77)
        dout = torch.randn(q.shape, generator=gen, dtype=torch.float32).to(q.dtype).to(dev)
        dq_, dk_, dv_ = (torch.empty_like(q) for _ in range(3))

    fused_dev = {}
    if args.fused:
        fi = W.fused_inputs(w)
        for name in ("q_norm_w", "k_norm_w", "q_gate", "k_gate", "out_gate"):
            a = getattr(fi, name)
            fused_dev[name] = (host(a) if a.dtype == np.uint16 else torch.from_numpy(a)).to(dev)
        fused_eps = fi.norm_eps

    def fwd(p, q_, k_, v_, out_=None, gates=None):
        out_ = out if out_ is None else out_
        gates = fused_dev if gates is None else gates
        if args.fused:
            bd.rec_attn_fwd_fused(p, q_, k_, v_, out_, None, stream, q_norm_weight=fused_dev["q_norm_w"],
                                  k_norm_weight=fused_dev["k_norm_w"], norm_eps=fused_eps,
                                  q_gate=gates["q_gate"], k_gate=gates["k_gate"],
                                  out_gate=gates["out_gate"])
        elif args.backward:
            bd.rec_attn_fwd(p, q_, k_, v_, out_, lse_buf, stream)
            if bwd_events is not None:
                bwd_events[-1][0].record(stream)
            bd.rec_attn_bwd(p, q_, k_, v_, out_, lse_buf, dout, dq_, dk_, dv_, stream)
            if bwd_events is not None:
                bwd_events[-1][1].record(stream)
        else:
            bd.rec_attn_fwd(p, q_, k_, v_, out_, None, stream)

    bwd_events = None  # per timed step: CUDA events around the backward call

    def step(timed=False):
        p = mkplan(off_d, t, ty, stream)
        if timed:
            bd.rec_attn_enable_timing(p)
            if args.backward:
                bwd_events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
        fwd(p, q, k, v)
        return p

    # grow the library's workspace pool to K live plans first (with the backward's
    # workspace, made on a plan's first backward call), so no timed step waits on a
    # driver allocation
    pre = [mkplan(off_d, t, ty, stream) for _ in range(args.steps)]
    if args.backward:
        for p_ in pre:
            fwd(p_, q, k, v)
    for p_ in pre:
        bd.rec_attn_free(p_)
    for _ in range(max(args.warmup, 3)):
        bd.rec_attn_free(step())
    torch.cuda.synchronize(dev)
    # the clock sampler starts here: warm-up continues, under the same load, until at
    # least args.soak_s seconds have passed, so the clocks sampled around the timed
    # region are those of a GPU that has been busy for a while
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    soak0 = time.perf_counter()
    n_soak = 0
    while time.perf_counter() - soak0 < args.soak_s:
        for _ in range(8):
            flush.zero_()
            bd.rec_attn_free(step())
            n_soak += 1
        torch.cuda.synchronize(dev)

    # ---- timed region: K steps, each bracketed by CUDA events on the launch stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    plans = []
    if args.backward:
        bwd_events = []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        p = step(timed=True)
        ev[i][1].record(stream)
        plans.append(p)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kt = [bd.rec_attn_read_timings(p) for p in plans]
    status = max(bd.rec_attn_device_status(p) for p in plans)
    for p in plans:
        bd.rec_attn_free(p)
    if status != bd.OK:
        raise RuntimeError(f"device status {status}: {bd.rec_attn_status_string(status)}")

    # ---- medians of args.median_iters iterations after 10 warm-ups: the forward alone
    # (one plan reused, as every layer of a model reuses it) and plan + forward
    def median_ms(fn, iters):
        for _ in range(10):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        torch.cuda.synchronize(dev)
        for a_, b_ in evs:
            flush.zero_()
            a_.record(stream)
            fn()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a_.elapsed_time(b_) for a_, b_ in evs)

    medians = None
    if args.median_iters > 0 and not args.backward:
        reused = mkplan(off_d, t, ty, stream)
        med_fwd = median_ms(lambda: fwd(reused, q, k, v), args.median_iters)
        bd.rec_attn_free(reused)
        med_step = median_ms(lambda: bd.rec_attn_free(step()), args.median_iters)
        medians = {"iterations": args.median_iters, "warmup": 10, "fwd_ms": med_fwd, "plan_fwd_ms": med_step,
                   "fwd_tflops": flops_fwd / (med_fwd * 1e-3) / 1e12,
                   "plan_fwd_tflops": flops_fwd / (med_step * 1e-3) / 1e12}
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = (f"sampled every 200 ms over {args.soak_s:.1f} s of warm-up steps ({n_soak}), the "
                            f"timed region and the median runs, back to back under load")
    total_ms = float(sum(step_ms))
    attn_ms = statistics.mean(x[1] for x in kt)
    bwd_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in bwd_events) if args.backward else 0.0
    bwd_events = None  # the end-to-end leg below records none
    rope_ms = statistics.mean(x[0] for x in kt)

    # ---- end to end through the C-ABI with host buffers: every step uploads its inputs
    # from pinned host memory and downloads its output.  Two device buffer sets: step i's
    # upload (copy stream) runs while step i-1 computes, its download (a second copy
    # stream) while step i+1 computes; the timed region spans the first upload to the last
    # download of the K steps.
    names = ["q", "k", "v", "t", "ty", "off"]
    host_in = {"q": hq, "k": hk, "v": hv, "t": ht, "ty": hty, "off": hoff}
    for n in ("q_gate", "k_gate", "out_gate"):  # fused: the per-token gates travel with Q/K/V
        if n in fused_dev:
            host_in[n] = fused_dev[n].cpu().pin_memory()
            names.append(n)
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = []
    for _ in range(2):
        sets.append({"in": {n: torch.empty(host_in[n].shape, dtype=host_in[n].dtype, device=dev) for n in names},
                     "out": torch.empty_like(out), "hout": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                     "up": torch.cuda.Event(), "done": torch.cuda.Event(), "down": torch.cuda.Event()})

    def e2e_steps(n_steps, ev=None):
        if ev is not None:
            ev[0].record(up_s)
        for i in range(n_steps):
            S = sets[i % 2]
            up_s.wait_event(S["down"])  # the set's previous output has been downloaded
            with torch.cuda.stream(up_s):
                for n in names:
                    S["in"][n].copy_(host_in[n], non_blocking=True)
            S["up"].record(up_s)
            stream.wait_event(S["up"])
            x = S["in"]
            p = mkplan(x["off"], x["t"], x["ty"], stream)
            fwd(p, x["q"], x["k"], x["v"], out_=S["out"], gates={n: x.get(n) for n in ("q_gate", "k_gate", "out_gate")})
            S["done"].record(stream)
            bd.rec_attn_free(p)
            down_s.wait_event(S["done"])
            with torch.cuda.stream(down_s):
                S["hout"].copy_(S["out"], non_blocking=True)
            S["down"].record(down_s)
        if ev is not None:
            ev[1].record(down_s)

    e2e_steps(2)  # untimed: the copy streams and the buffer sets warmed up
    torch.cuda.synchronize(dev)
    # E2E_RUNS runs of K steps, the median reported: on these hosts a host-device copy
    # now and then runs at a fraction of the link's rate (a 4.7 ms upload seen taking
    # 80 ms), which no schedule can hide; every run is listed with the line
    e2e_runs = []
    for _ in range(E2E_RUNS):
        e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        e2e_steps(args.steps, e2e_ev)
        torch.cuda.synchronize(dev)
        e2e_runs.append(e2e_ev[0].elapsed_time(e2e_ev[1]))
    e2e_ms = statistics.median(e2e_runs)
    h2d = sum(host_in[n].numel() * host_in[n].element_size() for n in names)
    d2h = out.numel() * out.element_size()

    # the host link alone (median of 5 copies each way, nothing else running): with the
    # copies overlapped, the e2e step cannot be shorter than the slower direction's copy
    def copy_ms(up: bool) -> float:
        S = sets[0]
        ts = []
        for _ in range(6):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_ = up_s if up else down_s
            a_.record(s_)
            with torch.cuda.stream(s_):
                if up:
                    for n in names:
                        S["in"][n].copy_(host_in[n], non_blocking=True)
                else:
                    S["hout"].copy_(S["out"], non_blocking=True)
            b_.record(s_)
            torch.cuda.synchronize(dev)
            ts.append(a_.elapsed_time(b_))
        return statistics.median(ts[1:])

    up_ms, down_ms = copy_ms(True), copy_ms(False)

    # slowest rank's times, total work of all ranks
    (total_ms, e2e_ms, attn_max), (all_flops, all_tokens) = sharding.aggregate(
        [total_ms, e2e_ms, attn_ms], [flops, float(tokens)], device=dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    pk = _peaks()
    ms_step = total_ms / args.steps
    value = all_flops * args.steps / (total_ms * 1e-3) / 1e12
    bytes_attn = (5.0 if args.fused else 4.0) * tokens * w.num_heads * w.head_dim * elem + 9.0 * tokens
    attn_tflops = flops_fwd / (attn_ms * 1e-3) / 1e12
    attn_gbs = bytes_attn / (attn_ms * 1e-3) / 1e9
    # full-size default batch only: the capture was taken on that launch
    traffic = (_traffic(args.workload + ("/fused" if args.fused else ""))
               if (args.batch is None and args.history is None and args.heads is None and args.head_dim is None
                   and world == 1) else None)
    hbm_bound = (flops_fwd / bytes_attn) < (pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9))
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": attn_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": attn_gbs / pk["hbm_gbs"], "traffic": traffic,
                "kernel": "k_attn_tc (masked softmax attention)", "peak_source": pk["source"],
                "algorithmic_bytes_per_launch": bytes_attn, "ms_per_launch": attn_ms}
    else:
        # the burst peak: the kernel runs at the maximum SM clock with no power-cap reason
        # in the sampled clocks; the fraction of the sustained (power-capped) figure is
        # given beside it
        roof = {"bound": "tensor", "achieved": attn_tflops, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": attn_tflops / pk["bf16_tflops"], "traffic": traffic,
                "kernel": "k_attn_tc (masked softmax attention)", "peak_source": pk["source"],
                "algorithmic_flops_per_launch": flops_fwd, "ms_per_launch": attn_ms,
                "peak_sustained": pk["bf16_tflops_sustained"],
                "frac_of_sustained": attn_tflops / pk["bf16_tflops_sustained"]}
    if args.backward:
        # the backward kernels dominate the step: bf16 runs on the tensor cores (dQ and
        # dK/dV modes of k_bwd_tc), fp32 on the CUDA cores
        bwd_tflops = 2.5 * flops_fwd / (bwd_ms * 1e-3) / 1e12
        fwd_part = {"achieved": attn_tflops, "unit": "TFLOP/s", "frac": attn_tflops / pk["bf16_tflops"],
                    "ms_per_launch": attn_ms}
        if bf16:
            roof = {"bound": "tensor", "achieved": bwd_tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": bwd_tflops / pk["bf16_tflops"], "traffic": None,
                    "kernel": "rec_attn_bwd: k_rope + k_bwd_rowc + k_bwd_tc<dQ> + k_bwd_tc<dK,dV> "
                              "(+ the new plan's k_bwd_schedule, k_bwd_colmask; tensor cores)",
                    "peak_source": pk["source"],
                    "algorithmic_flops_per_launch": 2.5 * flops_fwd, "ms_per_launch": bwd_ms,
                    "forward_attention": fwd_part}
        else:
            fp32_peak = FP32_FMA_PEAK_TFLOPS
            roof = {"bound": "alu", "achieved": bwd_tflops, "peak": fp32_peak, "unit": "TFLOP/s",
                    "frac": bwd_tflops / fp32_peak, "traffic": None,
                    "kernel": "rec_attn_bwd: k_rope + k_bwd_delta + k_bwd_dq + k_bwd_dkv (CUDA cores, fp32)",
                    "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 FLOP x 2070 MHz",
                    "algorithmic_flops_per_launch": 2.5 * flops_fwd, "ms_per_launch": bwd_ms,
                    "forward_attention": fwd_part}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "fp32",
        "data": "synthetic (seeded generators standing in for the pages' private logs)",
        "config": dict(_config(w, args.workload, f"dp{world} (requests sharded, no collective)"),
                       **({"fused": "QK-RMSNorm + Q/K sigmoid gates + output gate"} if args.fused else {}),
                       **({"keep_user_queries": args.keep_user_queries} if args.keep_user_queries >= 0 else {}),
                       **({"pass": "forward + backward (FLOPs 14 d per visible pair and head)"}
                          if args.backward else {})),
        "tokens_per_s": all_tokens * args.steps / (total_ms * 1e-3),
        "pct_of_bf16_peak": 100.0 * value / pk["bf16_tflops"],
        "visible_pairs_per_head": pairs,
        "tile_classes": {"skip": int((cls == 0).sum()), "partial": int((cls == 1).sum()),
                         "full": int((cls == 2).sum())},
        "kernel_ms": {"attention": attn_ms, "rope": rope_ms, "plan_and_overhead": ms_step - attn_ms - rope_ms},
        "fwd_only_tflops": flops_fwd / ((attn_ms + rope_ms) * 1e-3) / 1e12,
        **({"backward_ms": bwd_ms, "backward_tflops": 2.5 * flops_fwd / (bwd_ms * 1e-3) / 1e12}
           if args.backward else {}),
        "roofline": roof,
        "e2e": {"value": all_flops * args.steps / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps,
                "schedule": "every step uploads its inputs and downloads its output; uploads and downloads "
                            "on two copy streams overlap the neighbouring steps' compute (two buffer sets)",
                "runs_ms_per_step": [x / args.steps for x in e2e_runs],
                "statistic": f"median of {E2E_RUNS} runs of {args.steps} steps (this rank)",
                "link": {"h2d_gbs": h2d / (up_ms * 1e-3) / 1e9, "d2h_gbs": d2h / (down_ms * 1e-3) / 1e9,
                         "h2d_ms_per_step": up_ms, "d2h_ms_per_step": down_ms,
                         "bound_ms_per_step": max(ms_step, up_ms, down_ms),
                         "note": "pinned copies timed alone on this box; the overlapped step is bounded "
                                 "below by the slowest of compute, upload and download"}},
        # per step: k_plan (plus k_plan_tiles when requests average 32 tiles or more and
        # the planner splits them), k_build_masks, k_rope, k_attn_tc; the backward adds
        # k_rope, k_bwd_schedule, k_bwd_colmask (a new plan each step), k_bwd_rowc and the
        # two k_bwd_tc modes (the fp32 path: k_rope, k_bwd_delta, k_bwd_dq, k_bwd_dkv)
        "gpu_launches": (4 + _planner_split(w) + ((6 if bf16 else 4) if args.backward else 0)) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if medians is not None:
        line["median"] = medians
    if world == 1 and not args.no_cpu_baseline:
        secs, cpairs, desc, threads = _oracle_sample(w, args.cpu_budget, args.keep_user_queries)
        cval = 4.0 * w.head_dim * w.num_heads * cpairs / secs / 1e12
        line["cpu_baseline"] = {"value": cval, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"{desc} ({secs:.1f} s measured)",
                                "full_batch_s_extrapolated": secs * pairs / max(cpairs, 1)}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="tm20k_full", choices=W.NAMES + W.EXTRA_NAMES)
    ap.add_argument("--keep-user-queries", type=int, default=-1,
                    help="query pruning: compute every non-user query and the last N user queries of "
                         "each request (-1: all; 0: target attention)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's number of requests (small profiling cases)")
    ap.add_argument("--history", type=int, default=None,
                    help="tm20k workloads: history tokens per request (default 20000; context runs at 5000)")
    ap.add_argument("--heads", type=int, default=None, help="override the workload's number of heads")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="override the workload's head dimension (64 or 128 in bf16; 32 or 64 in fp32)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-s", type=float, default=2.0,
                    help="seconds of extra warm-up steps, with the clock sampler running, before the timed region")
    ap.add_argument("--median-iters", type=int, default=50,
                    help="iterations of the median runs (forward alone, plan + forward); 0 to skip")
    ap.add_argument("--compress", default=None, choices=sorted(COMPRESS_SPECS),
                    help="time history compression of the workload's key rows instead (HBM-bound)")
    ap.add_argument("--backward", action="store_true",
                    help="one step = plan + forward + backward (training); FLOPs 4d (forward) + 10d "
                         "(backward) per visible pair and head")
    ap.add_argument("--fused", action="store_true",
                    help="time rec_attn_fwd_fused with QK-RMSNorm, Q/K gates and the output gate on")
    ap.add_argument("--fused-epilogue", action="store_true",
                    help="with --compress: the compression fused into the attention epilogue against the "
                         "forward followed by the compression kernel")
    ap.add_argument("--serving", action="store_true",
                    help="per-request latency of candidate scoring against a cached history (use with "
                         "--workload cadet_serving)")
    ap.add_argument("--micro-batch", type=int, default=0,
                    help="--serving: candidates per scoring call (0: all of a request's candidates at once)")
    args = ap.parse_args(argv)
    if args.serving:
        return run_serving(args)
    if args.compress and args.fused_epilogue:
        return run_compress_fused(args)
    if args.compress:
        return run_compress(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
