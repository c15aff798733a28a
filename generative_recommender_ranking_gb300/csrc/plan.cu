// plan.cu -- planning kernels: per-tile type bounding boxes, (query tile, key tile)
// classification SKIP / PARTIAL / FULL, per-query-tile key-tile lists and a
// longest-first order of query tiles for the attention scheduler.
//
// The tile skipping follows the block-skipping idea of the CADET serving kernel
// (CADET review page, section on scoring hundreds of candidates in 50 ms) and SORT's
// "mask preload check" (SORT page, section 4.1): a key tile whose every pair is
// masked is never loaded, and a tile whose every pair is visible runs without
// per-element mask evaluation.
#include "rec_attn_internal.cuh"
#include "row_mask.cuh"

namespace recattn {

namespace {

// Three-valued outcome of a mask clause over two bounding boxes.  With
// NONE < SOME < ALL a conjunction is the minimum.
enum : int { kNone = 0, kSome = 1, kAll = 2 };

__device__ __forceinline__ int tv_and(int a, int b) { return a < b ? a : b; }

// p_j <= p_i
__device__ __forceinline__ int tv_causal(const TileBox& q, const TileBox& k) {
  return k.pmax <= q.pmin ? kAll : (k.pmin > q.pmax ? kNone : kSome);
}
// p_i - p_j < W
__device__ __forceinline__ int tv_window(const TileBox& q, const TileBox& k, int W) {
  return (q.pmax - k.pmin < W) ? kAll : ((q.pmin - k.pmax >= W) ? kNone : kSome);
}
// t_j <= t_i - delta, exact: x <= y - delta  <=>  (y >= MIN + delta) && x <= y - delta
__device__ __forceinline__ bool le_minus(long long x, long long y, long long delta) {
  return y >= (long long)(-0x7fffffffffffffffLL - 1) + delta && x <= y - delta;
}
__device__ __forceinline__ int tv_delay(const TileBox& q, const TileBox& k, long long delta) {
  if (le_minus(k.tmax, q.tmin, delta)) return kAll;
  if (!le_minus(k.tmin, q.tmax, delta)) return kNone;  // even the oldest key is too recent
  return kSome;
}
// t_j < t_i
__device__ __forceinline__ int tv_before(const TileBox& q, const TileBox& k) {
  return k.tmax < q.tmin ? kAll : (k.tmin >= q.tmax ? kNone : kSome);
}
// i == j (never ALL)
__device__ __forceinline__ int tv_diag(const TileBox& q, const TileBox& k) {
  return (k.pmax < q.pmin || k.pmin > q.pmax) ? kNone : kSome;
}

__device__ int tv_type_pair(const MaskP& m, int tq, int tk, const TileBox& q, const TileBox& k) {
  int v;
  const bool uq = is_user(tq), uk = is_user(tk);
  if (uq) {
    if (!uk) {
      v = kNone;
    } else if (m.bidir) {
      v = kAll;
    } else {
      v = tv_causal(q, k);
      if (m.window > 0 && tq != REC_ATTN_GLOBAL && tk != REC_ATTN_GLOBAL)
        v = tv_and(v, tv_window(q, k, m.window));
    }
  } else if (tq == REC_ATTN_RT) {
    v = uk ? kAll : (tk == REC_ATTN_RT ? tv_causal(q, k) : kNone);
  } else {
    v = uk ? kAll : (tk == REC_ATTN_RT ? tv_before(q, k) : tv_diag(q, k));
  }
  if (m.use_delay && !(tq == REC_ATTN_CAND && tk == REC_ATTN_CAND)) v = tv_and(v, tv_delay(q, k, m.delay));
  return v;
}

template <typename T>
__device__ __forceinline__ T warp_min(T v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    T w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w < v ? w : v;
  }
  return v;
}
template <typename T>
__device__ __forceinline__ T warp_max(T v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    T w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// hist[bin] += 1 for every active lane with one shared atomic per distinct bin of the
// warp (many lanes often share a bin); returns the counter's old value plus the lane's
// rank among the lanes with its bin.  Every lane of the warp calls it.
__device__ __forceinline__ int agg_inc(int* hist, int bin, bool active) {
  const unsigned grp = __match_any_sync(0xffffffffu, active ? bin : -1);
  const int lane = threadIdx.x & 31, leader = __ffs(grp) - 1;
  int base = 0;
  if (active && lane == leader) base = atomicAdd(&hist[bin], __popc(grp));
  base = __shfl_sync(0xffffffffu, base, leader);
  return base + __popc(grp & ((1u << lane) - 1u));
}

constexpr int kPlanThreads = 512;
constexpr int kCostBins = 4096;
constexpr int kStageTiles = 4096;
// shared scratch of the planner: the request's tile boxes while the pairs are
// classified, then (last block only) the cost histogram and per-tile costs
constexpr int kScratchBytes = 4 * (kCostBins + kStageTiles);
constexpr int kStageBoxTiles = kScratchBytes / (int)(kTypes * sizeof(TileBox));  // 256

// In-place exclusive scan of kCostBins counters by one block of kPlanThreads threads.
__device__ void block_exclusive_scan_bins(int* hist, int* part) {
  constexpr int per = kCostBins / kPlanThreads;
  int local = 0;
  for (int i = 0; i < per; ++i) local += hist[threadIdx.x * per + i];
  part[threadIdx.x] = local;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    const int v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = part[threadIdx.x] - local;
  for (int i = 0; i < per; ++i) {
    const int h = hist[threadIdx.x * per + i];
    hist[threadIdx.x * per + i] = run;
    run += h;
  }
  __syncthreads();
}

// The request holding tile g: the last b whose tiles start at or before g (an empty
// request shares its first tile index with the next one and is passed over).
__device__ __forceinline__ int request_of_tile(const ReqMeta* meta, int batch, long long g) {
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (meta[mid].tile_start <= g) lo = mid;
    else hi = mid;
  }
  return lo;
}

constexpr int kTileWarps = 8;   // k_plan_tiles: tiles per block, one warp each
constexpr int kSplitTiles = 32;  // mean tiles per request from which a request's tiles are split

// Phase 1 for tile tl of request m, by one warp: per-type bounding boxes, and the
// key-tile record the attention kernels build visibility bits from.
__device__ void tile_stats(const PlanDev& pd, const long long* t, const int8_t* ty, const ReqMeta& m, int tl,
                           int lane) {
  long long kt_t[4];
  int kt_y[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int pos = tl * kTile + u * 32 + lane;
    kt_t[u] = 0;
    kt_y[u] = -1;
    if (pos < m.len) {
      const long long tt = t[m.tok_start + pos];
      const int c = ty[m.tok_start + pos];
      if ((unsigned)c > 3u || tt >= kTimeLimit || tt <= -kTimeLimit) set_status(pd.status, REC_ATTN_ERR_DEVICE_INPUT);
      kt_t[u] = tt;
      kt_y[u] = (unsigned)c > 3u ? -1 : c;
    }
  }
  // next key's type and time, for the sortedness check of each type's run
  long long nx_t[4];
  int nx_y[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    nx_t[u] = __shfl_down_sync(0xffffffffu, kt_t[u], 1);
    nx_y[u] = __shfl_down_sync(0xffffffffu, kt_y[u], 1);
    const long long t0 = __shfl_sync(0xffffffffu, kt_t[u < 3 ? u + 1 : u], 0);
    const int y0 = __shfl_sync(0xffffffffu, kt_y[u < 3 ? u + 1 : u], 0);
    if (lane == 31) { nx_t[u] = t0; nx_y[u] = u < 3 ? y0 : -1; }
  }
  KeyTileRec* rec = pd.krec + (m.tile_start + tl);
#pragma unroll
  for (int u = 0; u < 4; ++u) rec->t[u * 32 + lane] = kt_t[u];
#pragma unroll
  for (int c = 0; c < kTypes; ++c) {
    int n = 0, pmn = 0x7fffffff, pmx = -1;
    long long tmn = 0x7fffffffffffffffLL, tmx = -0x7fffffffffffffffLL - 1;
    bool bad = false;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool mine = kt_y[u] == c;
      const unsigned bits = __ballot_sync(0xffffffffu, mine);
      if (lane == 0) rec->typebits[c][u] = bits;
      if (mine) {
        const int pos = tl * kTile + u * 32 + lane;
        n += 1;
        pmn = min(pmn, pos); pmx = max(pmx, pos);
        tmn = min(tmn, kt_t[u]); tmx = max(tmx, kt_t[u]);
        bad |= (nx_y[u] == c && nx_t[u] < kt_t[u]);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    const int a0 = warp_min(pmn), a1 = warp_max(pmx);
    const long long a2 = warp_min(tmn), a3 = warp_max(tmx);
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      TileBox bx;
      bx.cnt = n; bx.pmin = a0; bx.pmax = a1; bx.pad = 0; bx.tmin = a2; bx.tmax = a3;
      pd.boxes[(m.tile_start + tl) * kTypes + c] = bx;
      rec->run_lo[c] = n ? a0 - tl * kTile : 0;
      rec->run_n[c] = n;
      rec->sorted[c] = (n > 0 && a1 - a0 + 1 == n && !any_bad) ? 1 : 0;
      rec->pad[c] = 0;
    }
  }
}

// Phase 1 over the packed batch, one warp per tile (the planner's first kernel when a
// request's query tiles are split over several blocks).  Also zeroes the per-request
// costs those blocks add up.
__global__ void __launch_bounds__(32 * kTileWarps) k_plan_tiles(PlanDev pd, const long long* t, const int8_t* ty,
                                                               int batch, long long n_tiles) {
  for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < batch;
       r += (long long)gridDim.x * blockDim.x)
    pd.rcost[r] = 0;
  const long long g = (long long)blockIdx.x * kTileWarps + (threadIdx.x >> 5);
  if (g >= n_tiles) return;  // whole warps
  const ReqMeta m = pd.meta[request_of_tile(pd.meta, batch, g)];
  tile_stats(pd, t, ty, m, (int)(g - m.tile_start), threadIdx.x & 31);
}

// Phases 1 to 3 for one request (slices == 1), or phases 2 and 3 for one slice of it
// (phase 1 then ran in k_plan_tiles): block b * slices + sl takes the query tiles
// qt = sl, sl + slices, ... of request b, so few long requests still fill the GPU.
// Phase 4 in the last block to finish.
__global__ void __launch_bounds__(kPlanThreads) k_plan(MaskP mp, int heads, PlanDev pd,
                                                       const long long* offsets, const long long* t,
                                                       const int8_t* ty, int batch, int slices,
                                                       long long n_tiles) {
  __shared__ __align__(16) unsigned char s_scratch[kScratchBytes];
  const int b = (int)(blockIdx.x / slices), sl = (int)(blockIdx.x % slices);
  const ReqMeta m = pd.meta[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  // the device offsets must describe the same requests as the host copy
  if (sl == 0 && threadIdx.x == 0 && (offsets[b] != m.tok_start || offsets[b + 1] != m.tok_start + m.len))
    set_status(pd.status, REC_ATTN_ERR_DEVICE_INPUT);
  // this block's query tiles
  const int nrows = m.ntiles > sl ? (m.ntiles - sl + slices - 1) / slices : 0;
  if (slices == 1) {
    for (int tl = warp; tl < m.ntiles; tl += nwarps) tile_stats(pd, t, ty, m, tl, lane);
    __syncthreads();
  }

  // Query pruning: the position of the first kept user token, i.e. the keep_user-th
  // user token (GLOBAL or HIST) counted from the end of the request (0: every query).
  __shared__ int s_keep;
  if (threadIdx.x == 0) {
    int pos = 0;
    if (mp.keep_user >= 0) {
      pos = m.len;  // no user token kept unless found below
      int need = mp.keep_user;
      for (int tl = m.ntiles - 1; tl >= 0 && need > 0; --tl) {
        const TileBox* bx = pd.boxes + (m.tile_start + tl) * kTypes;
        const int nu = bx[REC_ATTN_GLOBAL].cnt + bx[REC_ATTN_HIST].cnt;
        if (nu < need) {
          need -= nu;
          if (nu > 0) pos = tl * kTile;  // every user token of the tile is kept
          continue;
        }
        // the need-th user token from the tile's end
        const KeyTileRec* rec = pd.krec + (m.tile_start + tl);
        for (int c = kTile - 1; c >= 0; --c) {
          const int w = c >> 5, bit = c & 31;
          const bool u = ((rec->typebits[REC_ATTN_GLOBAL][w] | rec->typebits[REC_ATTN_HIST][w]) >> bit) & 1u;
          if (u && --need == 0) { pos = tl * kTile + c; break; }
        }
        need = 0;
      }
    }
    s_keep = pos;
    if (sl == 0) pd.qkeep[b] = pos;
  }

  // Phase 2: class of every (query tile, key tile) pair of the block's query tiles, with
  // the request's boxes staged in shared memory when they fit.
  const long long npairs = (long long)nrows * m.ntiles;
  const bool staged_boxes = m.ntiles <= kStageBoxTiles;
  TileBox* s_box = reinterpret_cast<TileBox*>(s_scratch);
  if (staged_boxes)
    for (int i = threadIdx.x; i < m.ntiles * kTypes; i += blockDim.x) s_box[i] = pd.boxes[m.tile_start * kTypes + i];
  __syncthreads();
  const TileBox* boxes = staged_boxes ? s_box : pd.boxes + m.tile_start * kTypes;
  for (long long idx = threadIdx.x; idx < npairs; idx += blockDim.x) {
    const int qt = sl + (int)(idx / m.ntiles) * slices, kt = (int)(idx % m.ntiles);
    const TileBox* qb = boxes + qt * kTypes;
    const TileBox* kb = boxes + kt * kTypes;
    int lo = kAll, hi = kNone;
    for (int a = 0; a < kTypes; ++a) {
      const TileBox q = qb[a];
      if (!q.cnt) continue;
      for (int c = 0; c < kTypes; ++c) {
        const TileBox k = kb[c];
        if (!k.cnt) continue;
        const int v = tv_type_pair(mp, a, c, q, k);
        lo = min(lo, v); hi = max(hi, v);
      }
    }
    const bool k_full = (kt + 1) * kTile <= m.len;
    uint8_t cl;
    if (hi == kNone) cl = REC_ATTN_TILE_SKIP;
    else if (lo == kAll && k_full) cl = REC_ATTN_TILE_FULL;
    else cl = REC_ATTN_TILE_PARTIAL;
    pd.cls[m.cls_start + (long long)qt * m.ntiles + kt] = cl;
  }
  __syncthreads();

  // Phase 3: compact each query tile's non-SKIP key tiles (one warp per query tile).
  __shared__ int s_rcost;
  if (threadIdx.x == 0) s_rcost = 0;
  __syncthreads();
  for (int ri = warp; ri < nrows; ri += nwarps) {
    const int qt = sl + ri * slices;
    // a query tile whose every token is a user token before the first kept one
    // computes nothing: no key list, no cost, the kernels skip it
    const TileBox* qbx = pd.boxes + (m.tile_start + qt) * kTypes;
    const bool pruned = min(m.len, (qt + 1) * kTile) <= s_keep && qbx[REC_ATTN_RT].cnt == 0 &&
                        qbx[REC_ATTN_CAND].cnt == 0;
    if (pruned) {
      if (lane == 0) {
        const long long g = m.tile_start + qt;
        pd.kcount[g] = -1;
        pd.qcost[g] = 0;
        pd.qreq[g] = b;
      }
      // its PARTIAL pairs still appear in the backward's per-key-tile lists: no table slot
      const long long rb = m.cls_start + (long long)qt * m.ntiles;
      for (int kt = lane; kt < m.ntiles; kt += 32)
        if (pd.cls[rb + kt] == REC_ATTN_TILE_PARTIAL) pd.pslot[rb + kt] = -1;
      continue;
    }
    const long long rb = m.cls_start + (long long)qt * m.ntiles;  // the query tile's row of pairs
    const uint8_t* row = pd.cls + rb;
    uint32_t* out = pd.klist + rb;
    int n = 0, nfull = 0;
    for (int k0 = 0; k0 < m.ntiles; k0 += 32) {
      const int kt = k0 + lane;
      const uint32_t c = kt < m.ntiles ? row[kt] : 0u;
      const unsigned bal = __ballot_sync(0xffffffffu, c != 0);
      // PARTIAL pairs take the next mask-table slots (while there are any)
      const unsigned pb = __ballot_sync(0xffffffffu, c == REC_ATTN_TILE_PARTIAL);
      int s0 = 0;
      if (lane == 0 && pb) s0 = atomicAdd(&pd.counters[7], __popc(pb));
      s0 = __shfl_sync(0xffffffffu, s0, 0);
      if (c) {
        const int j = n + __popc(bal & ((1u << lane) - 1u));
        out[j] = (uint32_t)kt | (c << 24);
        int slot = -1;
        if (c == REC_ATTN_TILE_PARTIAL) {
          const int s = s0 + __popc(pb & ((1u << lane) - 1u));
          if (s < pd.mcap) {
            slot = s;
            pd.minfo[s] = make_int2((int)(m.tile_start + qt), kt);
          }
          pd.pslot[rb + kt] = slot;
        }
        pd.kslot[rb + j] = slot;
      }
      n += __popc(bal);
      nfull += __popc(__ballot_sync(0xffffffffu, c == REC_ATTN_TILE_FULL));
    }
    if (lane == 0) {
      const long long g = m.tile_start + qt;
      pd.kcount[g] = n;
      const int cost = 2 * nfull + 3 * (n - nfull) + 1;  // a PARTIAL tile costs ~1.5 FULL ones
      pd.qcost[g] = cost;
      pd.qreq[g] = b;
      atomicAdd(&s_rcost, cost);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (slices == 1) pd.rcost[b] = s_rcost;
    else if (s_rcost) atomicAdd(pd.rcost + b, s_rcost);
  }

  // Phase 4: the last block to finish writes the work-item order.  The order only
  // affects load balance and cache reuse, never results.
  //  - heavy query tiles (cost above 16x the mean, e.g. a candidate tile that reads a
  //    whole 20K history next to window-only tiles) go first, most expensive first;
  //  - then the rest, request by request (most expensive first), inside a request
  //    head by head, inside a head from the last query tile to the first, so the
  //    items running at the same time share K'/V tiles in L2.
  __shared__ int s_ticket;
  int* s_hist = reinterpret_cast<int*>(s_scratch);  // [kCostBins] (the boxes are no longer read)
  int* s_qc = s_hist + kCostBins;                    // [kStageTiles] per-tile costs (n_tiles <= kStageTiles)
  __shared__ int s_part[kPlanThreads];
  __shared__ unsigned long long s_sum;
  __shared__ int s_max, s_nheavy;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_ticket = atomicAdd(&pd.counters[0], 1);
  __syncthreads();
  if (s_ticket != (int)gridDim.x - 1) return;
  __threadfence();
  const int B = batch;
  const bool staged = n_tiles <= kStageTiles;
  if (threadIdx.x == 0) { s_sum = 0; s_max = 1; s_nheavy = 0; }
  for (int i = threadIdx.x; i < kCostBins; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  {
    unsigned long long part = 0;
    for (long long q = threadIdx.x; q < n_tiles; q += blockDim.x) {
      const int c = __ldcg(pd.qcost + q);
      if (staged) s_qc[q] = c;
      part += (unsigned long long)c;
    }
    int rmax = 1;
    for (int r = threadIdx.x; r < B; r += blockDim.x) rmax = max(rmax, __ldcg(pd.rcost + r));
    // one shared atomic per warp (512 contending ones took microseconds)
#pragma unroll
    for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    rmax = warp_max(rmax);
    if ((threadIdx.x & 31) == 0) {
      atomicAdd(&s_sum, part);
      atomicMax(&s_max, rmax);
    }
  }
  __syncthreads();
  const long long total = (long long)s_sum;
  auto qc = [&](long long q) { return staged ? s_qc[q] : __ldcg(pd.qcost + q); };
  // heavy: qcost * n_tiles > 16 * total
  auto heavy = [&](long long q) { return (long long)qc(q) * n_tiles > 16 * total; };
  // heavy query tiles, counting-sorted by cost (descending) into the front of `items`
  for (long long q = threadIdx.x; q < n_tiles; q += blockDim.x)
    if (heavy(q)) {
      atomicAdd(&s_hist[kCostBins - 1 - min(qc(q), kCostBins - 1)], 1);
      atomicAdd(&s_nheavy, 1);
    }
  __syncthreads();
  const long long heavy_items = (long long)s_nheavy * heads;
  if (heavy_items > 0) {
    block_exclusive_scan_bins(s_hist, s_part);
    for (long long q = threadIdx.x; q < n_tiles; q += blockDim.x)
      if (heavy(q)) {
        const int pos = atomicAdd(&s_hist[kCostBins - 1 - min(qc(q), kCostBins - 1)], 1);
        for (int h = 0; h < heads; ++h) pd.items[(long long)pos * heads + h] = (int)(q * heads + h);
      }
    __syncthreads();
    for (int i = threadIdx.x; i < kCostBins; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();
  }
  // requests by cost, descending
  const long long mx = s_max;
  // (whole warps in both loops: requests of equal cost share a bin)
  for (int r0 = threadIdx.x & ~31; r0 < B; r0 += blockDim.x) {
    const int r = r0 + (threadIdx.x & 31);
    const int key = r < B ? (int)((long long)__ldcg(pd.rcost + r) * (kCostBins - 1) / mx) : 0;
    agg_inc(s_hist, kCostBins - 1 - key, r < B);
  }
  __syncthreads();
  block_exclusive_scan_bins(s_hist, s_part);
  for (int r0 = threadIdx.x & ~31; r0 < B; r0 += blockDim.x) {
    const int r = r0 + (threadIdx.x & 31);
    const int key = r < B ? (int)((long long)__ldcg(pd.rcost + r) * (kCostBins - 1) / mx) : 0;
    const int pos = agg_inc(s_hist, kCostBins - 1 - key, r < B);
    if (r < B) pd.rorder[pos] = r;
  }
  __syncthreads();
  // light items per request (in rorder order) -> first light item of each request
  long long carry = heavy_items;
  for (int base = 0; base < B; base += blockDim.x) {
    const int k = base + threadIdx.x;
    int v = 0;
    if (k < B) {
      const ReqMeta rm = pd.meta[__ldcg(pd.rorder + k)];
      v = rm.ntiles;
      if (heavy_items > 0)
        for (int qt = 0; qt < rm.ntiles; ++qt) v -= heavy(rm.tile_start + qt) ? 1 : 0;
      v *= heads;
    }
    s_part[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
      const int add = threadIdx.x >= off ? s_part[threadIdx.x - off] : 0;
      __syncthreads();
      s_part[threadIdx.x] += add;
      __syncthreads();
    }
    if (k < B) pd.roff[k] = (int)(carry + s_part[threadIdx.x] - v);
    const int chunk_total = s_part[kPlanThreads - 1];
    __syncthreads();
    carry += chunk_total;
  }
  if (threadIdx.x == 0) pd.roff[B] = (int)carry;
  __syncthreads();
  // each (request, head): its light query tiles, last to first
  const long long n_kh = (long long)B * heads;
  if (slices == 1) {  // short requests: one thread per (request, head)
    for (long long kh = threadIdx.x; kh < n_kh; kh += blockDim.x) {
      const int k = (int)(kh / heads), h = (int)(kh % heads);
      const ReqMeta rm = pd.meta[__ldcg(pd.rorder + k)];
      const int r0 = __ldcg(pd.roff + k), nl = (__ldcg(pd.roff + k + 1) - r0) / heads;
      long long w = r0 + (long long)h * nl;
      for (int qt = rm.ntiles - 1; qt >= 0; --qt)
        if (heavy_items == 0 || !heavy(rm.tile_start + qt)) pd.items[w++] = (int)((rm.tile_start + qt) * heads + h);
    }
    return;
  }
  // long requests: a warp takes 32 of them; each lane looks up one (its loads all in
  // flight together), then the warp writes them one after the other, lane i taking the
  // i-th tile of each group of 32 counted from the end
  for (long long base = (long long)warp * 32; base < n_kh; base += (long long)nwarps * 32) {
    long long my_ts = 0, my_w = 0;
    int my_nt = 0, my_h = 0;
    if (base + lane < n_kh) {
      const int k = (int)((base + lane) / heads);
      my_h = (int)((base + lane) % heads);
      const ReqMeta rm = pd.meta[__ldcg(pd.rorder + k)];
      const int r0 = __ldcg(pd.roff + k), nl = (__ldcg(pd.roff + k + 1) - r0) / heads;
      my_ts = rm.tile_start;
      my_nt = rm.ntiles;
      my_w = r0 + (long long)my_h * nl;
    }
    const int cnt = (int)min(32LL, n_kh - base);
    for (int i = 0; i < cnt; ++i) {
      const long long ts = __shfl_sync(0xffffffffu, my_ts, i);
      const int nt = __shfl_sync(0xffffffffu, my_nt, i), h = __shfl_sync(0xffffffffu, my_h, i);
      long long w = __shfl_sync(0xffffffffu, my_w, i);
      for (int top = nt - 1; top >= 0; top -= 32) {
        const int qt = top - lane;
        const bool light = qt >= 0 && (heavy_items == 0 || !heavy(ts + qt));
        const unsigned bl = __ballot_sync(0xffffffffu, light);
        if (light) pd.items[w + __popc(bl & ((1u << lane) - 1u))] = (int)((ts + qt) * heads + h);
        w += __popc(bl);
      }
    }
  }
}

// The mask table: per slot (a PARTIAL pair), each of the query tile's 128 rows builds its
// visibility bits over the key tile exactly as the attention kernels would (row time and
// type from the query tile's record, key times and types from the key tile's record,
// which is staged in shared memory).  Slots are visited with a grid stride.
__global__ void __launch_bounds__(kTile) k_build_masks(MaskP mp, PlanDev pd) {
  __shared__ KeyTileRec s_rec;
  const int used = min(__ldcg(pd.counters + 7), pd.mcap);
  const int r = threadIdx.x;
  for (int s = blockIdx.x; s < used; s += gridDim.x) {
    const int2 info = pd.minfo[s];
    const long long g = info.x;
    const int kt = info.y;
    const ReqMeta m = pd.meta[pd.qreq[g]];
    const int qt = (int)(g - m.tile_start);
    __syncthreads();  // the previous slot's readers of s_rec are done
    const uint4* src = reinterpret_cast<const uint4*>(pd.krec + m.tile_start + kt);
    for (int i = r; i < (int)(sizeof(KeyTileRec) / 16); i += blockDim.x) reinterpret_cast<uint4*>(&s_rec)[i] = src[i];
    __syncthreads();
    const KeyTileRec* qr = pd.krec + g;
    const long long ti = qr->t[r];
    int tyi = -1;
#pragma unroll
    for (int c = 0; c < kTypes; ++c)
      if ((qr->typebits[c][r >> 5] >> (r & 31)) & 1u) tyi = c;
    const int pi = qt * kTile + r;
    RowMask rm;
    row_mask_setup(mp, pi < m.len, pi, ti, tyi, rm);
    uint32_t vm[4];
    build_mask(rm, &s_rec, kt * kTile, vm);
    reinterpret_cast<uint4*>(pd.mtab)[(long long)s * kTile + r] = make_uint4(vm[0], vm[1], vm[2], vm[3]);
  }
}

// Visible-pair counter: one block per query tile, one thread per query row.
__global__ void __launch_bounds__(kTile) k_count_pairs(MaskP mp, PlanDev pd, const long long* t,
                                                       const int8_t* ty) {
  const long long g = blockIdx.x;
  const int b = pd.qreq[g];
  const ReqMeta m = pd.meta[b];
  const int qt = (int)(g - m.tile_start);
  const int r = threadIdx.x, pi = qt * kTile + r;
  __shared__ long long s_t[kTile];
  __shared__ int s_ty[kTile];
  __shared__ unsigned long long s_sum;
  if (r == 0) s_sum = 0;
  __syncthreads();
  long long ti = 0;
  int tyi = -1;
  if (pi < m.len) { ti = t[m.tok_start + pi]; tyi = ty[m.tok_start + pi]; }
  const bool row_ok = pi < m.len && query_kept(tyi, pi, pd.qkeep[b]);
  bool thr_ok; long long thr;
  delay_bound(ti, mp.delay, thr_ok, thr);
  unsigned long long cnt = 0;
  const int n = pd.kcount[g];
  const uint32_t* list = pd.klist + m.cls_start + (long long)qt * m.ntiles;
  for (int j = 0; j < n; ++j) {
    const uint32_t e = list[j];
    const int kt = (int)(e & 0xffffffu), cl = (int)(e >> 24);
    __syncthreads();
    const int pj = kt * kTile + r;
    s_t[r] = pj < m.len ? t[m.tok_start + pj] : 0;
    s_ty[r] = pj < m.len ? (int)ty[m.tok_start + pj] : -1;
    __syncthreads();
    if (!row_ok) continue;
    if (cl == REC_ATTN_TILE_FULL) { cnt += kTile; continue; }
    for (int c = 0; c < kTile; ++c)
      cnt += vis_pred(mp, pi, ti, tyi, thr_ok, thr, kt * kTile + c, s_t[c], s_ty[c]) ? 1u : 0u;
  }
  atomicAdd(&s_sum, cnt);
  __syncthreads();
  if (r == 0) atomicAdd(pd.pairs, s_sum);
}

}  // namespace

cudaError_t launch_plan(const MaskP& mp, int heads, const PlanDev& pd, const long long* offsets_dev,
                        const long long* t, const int8_t* ty, int batch, long long n_tiles,
                        cudaEvent_t prologue_ok, cudaStream_t st) {
  if (batch <= 0) return prologue_ok ? cudaEventRecord(prologue_ok, st) : cudaSuccess;
  // One block per request while requests are short: the planner then runs beside the
  // RoPE prologue and ends first.  Long requests (the pair classification grows with
  // the square of a request's tiles) are split over enough blocks for two per SM, with
  // phase 1 in a kernel of its own before them.
  long long slices = 1;
  const long long mean_tiles = (n_tiles + batch - 1) / batch;
  if (mean_tiles >= kSplitTiles) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    slices = (2LL * sms + batch - 1) / batch;
    if (slices > mean_tiles) slices = mean_tiles;
  }
  if (slices > 1) {
    const long long tile_blocks = (n_tiles + kTileWarps - 1) / kTileWarps;
    k_plan_tiles<<<(unsigned)tile_blocks, 32 * kTileWarps, 0, st>>>(pd, t, ty, batch, n_tiles);
  } else {
    slices = 1;
  }
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && prologue_ok) e = cudaEventRecord(prologue_ok, st);
  if (e != cudaSuccess) return e;
  k_plan<<<(unsigned)(batch * slices), kPlanThreads, 0, st>>>(mp, heads, pd, offsets_dev, t, ty, batch,
                                                              (int)slices, n_tiles);
  return cudaGetLastError();
}

cudaError_t launch_build_masks(const MaskP& mp, const PlanDev& pd, int num_sms, cudaStream_t st) {
  if (pd.mcap <= 0) return cudaSuccess;
  // up to 32 blocks of 128 threads per SM, most with one slot (blocks past the slots in
  // use return at once): the table is on the way to the attention kernel when the
  // planner runs beside a short prologue (8 per SM: SORT step 0.797 ms, 32: 0.791)
  const int grid = pd.mcap < 32 * num_sms ? pd.mcap : 32 * num_sms;
  k_build_masks<<<grid, kTile, 0, st>>>(mp, pd);
  return cudaGetLastError();
}

cudaError_t launch_count_pairs(const MaskP& mp, const PlanDev& pd, const long long* t,
                               const int8_t* ty, long long n_tiles, cudaStream_t st) {
  if (n_tiles <= 0) return cudaSuccess;
  k_count_pairs<<<(unsigned)n_tiles, kTile, 0, st>>>(mp, pd, t, ty);
  return cudaGetLastError();
}

}  // namespace recattn
