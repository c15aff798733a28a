// attn_tc.cu -- bf16 masked softmax attention on the sm_103a tensor cores.
//
// Softmax(QK^T/sqrt(d) + M) V (TM20K review page, section 2.1; LazFormer review page,
// section 2.3, Eq. 19-21) for the plan's (query tile, head) work items, skipping the
// key tiles the plan classified SKIP (block skipping of the CADET serving kernel;
// SORT section 4.1).  Rows that see no key are written as zeros.
//
// One persistent CTA per SM runs two independent item streams, so the tensor core
// works on one stream while the other stream's softmax runs.  12 warps:
//   warp 0, 1     TMA producers (stream 0, 1): claim items from a global counter in
//                 the planner's order (heaviest items first, then request by request,
//                 head by head), publish item descriptors and per-stage tile
//                 info in shared memory, load Q', K', V (and, for PARTIAL tiles, the
//                 key-tile record) with TMA / bulk copies into per-stream rings;
//   warp 2, 3     MMA issuers (stream 0, 1).  d = 64: S = Q'K'^T over a whole 128-key
//                 tile (N = 128), issued as soon as the softmax has read the previous
//                 S; P has TMEM columns of its own and O += P V is issued per 64-key
//                 half.  d = 128: each tile is two 64-key chunks with S double-buffered
//                 and P written over the first columns of its chunk's S;
//   warps 4..7    softmax of stream 0, warps 8..11 softmax of stream 1: one query row
//                 per thread (TMEM lane quadrant = warp % 4).  PARTIAL tiles build the
//                 row's 128-bit visibility mask from position ranges, per-type key
//                 bitmaps and, for time clauses, a binary search over time-sorted
//                 runs; FULL tiles skip the mask.  Online softmax in the exp2 domain
//                 with a lazily updated reference maximum; O rescaled in TMEM only when
//                 the maximum grows by more than 2^8, and only then does the softmax
//                 wait for the PV that precedes it.  P rounded to bf16; the row sum l
//                 is the fp32 sum of the unrounded exponentials.  Row times and types
//                 come from the query tile's planner record, bulk-copied next to Q.
// Every wait on an mbarrier is bounded (REC_ATTN_ERR_TIMEOUT in the status word).
#include <climits>

#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "ptx_sm103.cuh"
#include "row_mask.cuh"
#include "wait.cuh"

namespace recattn {

namespace {

constexpr int kStreams = 2;
constexpr int kSlab = kTile * 128;           // 128 rows x 128 B: one 64-column swizzle slab
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;          // keep the reference max until it is exceeded by 2^8
constexpr float kLazySum = 256.f;            // LAZY: a chunk whose exponentials sum below this keeps the reference
constexpr int kRecBytes = (int)sizeof(KeyTileRec);
constexpr int kMaskBytes = kTile * 16;  // a PARTIAL tile's 128 rows of visibility bits (mask table)
constexpr int kStageRec = kMaskBytes > kRecBytes ? kMaskBytes : kRecBytes;  // per K/V stage: one or the other
constexpr int kChunk = 64;                   // keys per S chunk (a 128-key tile is two chunks)

template <int D>
struct Cfg;
// QB: Q buffers per stream, NS: K/V stages per stream, WIDE: S over the whole 128-key
// tile with P in TMEM columns of its own (else two 64-key chunks, P over S).
template <>
struct Cfg<64> {
  static constexpr int QB = 2, NS = 2;
  static constexpr bool WIDE = true;
};
template <>
struct Cfg<128> {
  static constexpr int QB = 1, NS = 1;
  static constexpr bool WIDE = false;
};
// per stream one producer warp and one MMA-issuer warp, then two softmax warpgroups
constexpr int kRoleWarps = 2 * kStreams;
constexpr int kThreads = 32 * (kRoleWarps + 8);

// TMEM columns of one stream (lane base included by the caller).
//   WIDE:    [stream] S 128 | P 64 (bf16 pairs) | O D      -> 2 x 256 for D = 64
//   chunked: S [stream][2 chunks][64], then O [stream][D]   -> 256 + 2 x 128 for D = 128
struct TmemMap {
  uint32_t s, p, o;
};
template <int D>
__device__ __forceinline__ TmemMap tmem_map(uint32_t base, int s) {
  TmemMap m;
  if (Cfg<D>::WIDE) {
    m.s = base + (uint32_t)(s * (kTile + kTile / 2 + D));
    m.p = m.s + kTile;
    m.o = m.p + kTile / 2;
  } else {
    m.s = base + (uint32_t)(s * kTile);
    m.p = 0;
    m.o = base + 2u * kTile + (uint32_t)(s * D);
  }
  return m;
}
static_assert(kStreams * (kTile + kTile / 2 + 64) <= (int)kTmemCols, "WIDE TMEM map");
static_assert(2 * kTile + kStreams * 128 <= (int)kTmemCols, "chunked TMEM map");

struct ItemDesc {
  long long tok0;  // first token of the query tile (global index)
  int pos0;        // request-local position of the tile's first row
  int rows;        // valid rows in the tile
  int h;
  int n;           // non-SKIP key tiles; -1: every query of the tile is pruned
  int req;         // the item's request; -1: the stream is done
  int keep;        // first kept user position of the request (query pruning)
};
static_assert(sizeof(ItemDesc) == 32, "");

struct StageInfo {
  int kt;
  int cls;
  int tab;  // PARTIAL: 1 = the stage holds the tile's rows of the mask table, 0 = the key record
  int pad;
};

template <int D>
struct Layout {
  static constexpr int QB = Cfg<D>::QB, NS = Cfg<D>::NS;
  static constexpr int kQBytes = kTile * D * 2;
  static constexpr int kKVBytes = kTile * D * 2;
  static constexpr int kQ = 0;                                   // [stream][QB]
  static constexpr int kK = kQ + kStreams * QB * kQBytes;        // [stream][NS]
  static constexpr int kV = kK + kStreams * NS * kKVBytes;       // [stream][NS]
  static constexpr int kRec = kV + kStreams * NS * kKVBytes;      // [stream][NS] KeyTileRec or mask rows
  static constexpr int kQRec = kRec + kStreams * NS * kStageRec;  // [stream][QB] KeyTileRec of the query tile
  static constexpr int kInfo = kQRec + kStreams * QB * kRecBytes; // [stream][NS] StageInfo
  static constexpr int kItems = (kInfo + kStreams * NS * (int)sizeof(StageInfo) + 15) & ~15;  // [stream][2] ItemDesc
  static constexpr int kBars = (kItems + kStreams * 2 * 32 + 7) & ~7;
  static constexpr int kBarsPerStream = 2 + 2 + 2 * QB + 4 * NS + 9;
  static constexpr int kTotal = kBars + kStreams * kBarsPerStream * 8 + 16;
  static constexpr int kDynamic = kTotal + 1024;  // slack to align the base to 1024 B
};

// mbarriers of one stream
struct SBars {
  // k_free[st]: the softmax has seen S of the stage's tile complete (so K was read)
  // and has read the stage's tile info and key record; v_empty[st]: the tile's last
  // PV completed.  K and V of a stage are refilled independently.
  uint64_t *item_full, *item_empty, *q_full, *q_empty, *k_full, *v_full, *k_free, *v_empty;
  // s_full, p_full, pv_done: [2] each.  Chunked: indexed by the stream's chunk count
  // mod 2.  WIDE: s_full[0] only (one S buffer), s_free when the softmax has read S,
  // p_full / pv_done indexed by the 64-key half of the tile.
  uint64_t *s_full, *s_free, *p_full, *pv_done, *o_ready, *mma_done;
  template <int D>
  __device__ void bind(uint64_t* b) {
    constexpr int QB = Cfg<D>::QB, NS = Cfg<D>::NS;
    item_full = b; item_empty = b + 2; q_full = b + 4; q_empty = q_full + QB;
    k_full = q_empty + QB; v_full = k_full + NS; k_free = v_full + NS; v_empty = k_free + NS;
    s_full = v_empty + NS; s_free = s_full + 2; p_full = s_free + 1; pv_done = p_full + 2;
    o_ready = pv_done + 2;
    mma_done = o_ready + 1;
  }
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
  return bounded_wait(bar, parity, abort_flag, status, kWaitNs);
}
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > kWaitNs / 4) return;
}
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int* status) {
  const bool ok = wait_bar(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Packed fp32 pairs for the fma.rn.f32x2 instruction.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// max(a, b, c) in one instruction (NaN operands are ignored, as with fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------------------------------------------ producer
template <int D>
__device__ void run_producer(const AttnArgs& a, const void* tq, const void* tk, const void* tv, uint8_t* sm,
                             int s, const SBars& B, volatile int* abort_flag) {
  using L = Layout<D>;
  constexpr int QB = L::QB, NS = L::NS;
  ItemDesc* items = reinterpret_cast<ItemDesc*>(sm + L::kItems) + s * 2;
  StageInfo* info = reinterpret_cast<StageInfo*>(sm + L::kInfo) + s * NS;
  uint8_t* qbuf = sm + L::kQ + s * QB * L::kQBytes;
  uint8_t* kbuf = sm + L::kK + s * NS * L::kKVBytes;
  uint8_t* vbuf = sm + L::kV + s * NS * L::kKVBytes;
  uint8_t* rbuf = sm + L::kRec + s * NS * kStageRec;
  uint8_t* qrbuf = sm + L::kQRec + s * QB * kRecBytes;
  uint32_t it_cnt = 0, q_it = 0, kv_it = 0;
  bool q_used[QB], k_used[NS], v_used[NS];
  uint32_t q_ph[QB], k_ph[NS], v_ph[NS];
  for (int i = 0; i < QB; ++i) { q_used[i] = false; q_ph[i] = 0; }
  for (int i = 0; i < NS; ++i) { k_used[i] = v_used[i] = false; k_ph[i] = v_ph[i] = 0; }
  for (;;) {
    const long long w = atomicAdd(a.counters + 1, 1);
    const int slot = (int)(it_cnt & 1);
    if (!wait_bar(B.item_empty + slot, ((it_cnt >> 1) & 1) ^ 1, abort_flag, a.status)) break;
    ++it_cnt;
    ItemDesc* d = items + slot;
    if (w >= a.n_items) {
      d->req = -1;
      ptx::mbar_arrive(B.item_full + slot);
      break;
    }
    const WorkItem it = decode_item(a, w, true);
    d->tok0 = it.m.tok_start + (long long)it.qt * kTile;
    d->pos0 = it.qt * kTile;
    d->rows = min(kTile, it.m.len - it.qt * kTile);
    d->h = it.h;
    d->n = it.n;
    d->keep = it.keep;
    d->req = it.b;
    ptx::mbar_arrive(B.item_full + slot);
    if (it.n <= 0) continue;
    const int qb = (int)(q_it % QB);
    if (!wait_bar(B.q_empty + qb, ((q_it / QB) & 1) ^ 1, abort_flag, a.status)) break;
    ptx::mbar_arrive_expect_tx(B.q_full + qb, L::kQBytes + kRecBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      ptx::tma_load_2d(qbuf + qb * L::kQBytes + c * kSlab, tq, it.h * D + c * 64, (int)d->tok0, B.q_full + qb);
    // the query tile's times and type bitmaps (its rows' metadata for the softmax)
    ptx::bulk_load(qrbuf + qb * kRecBytes, a.krec + it.m.tile_start + it.qt, kRecBytes, B.q_full + qb);
    q_used[qb] = true; q_ph[qb] = (q_it / QB) & 1;
    ++q_it;
    for (int j = 0; j < it.n; ++j) {
      const uint32_t e = it.list[j];
      const int slot = it.slots[j];
      const int kt = (int)(e & 0xffffffu), cl = (int)(e >> 24);
      const int st = (int)(kv_it % NS);
      const uint32_t ph = (kv_it / NS) & 1;
      if (!wait_bar(B.k_free + st, ph ^ 1, abort_flag, a.status)) goto drain;
      info[st].kt = kt;
      info[st].cls = cl;
      const bool partial = cl != REC_ATTN_TILE_FULL;
      const int y = (int)(it.m.tok_start + (long long)kt * kTile);
      const bool tab = partial && slot >= 0;
      info[st].tab = tab ? 1 : 0;
      ptx::mbar_arrive_expect_tx(B.k_full + st, L::kKVBytes + (partial ? (tab ? kMaskBytes : kRecBytes) : 0));
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        ptx::tma_load_2d(kbuf + st * L::kKVBytes + c * kSlab, tk, it.h * D + c * 64, y, B.k_full + st);
      if (tab) ptx::bulk_load(rbuf + st * kStageRec, a.mtab + (long long)slot * (kMaskBytes / 4), kMaskBytes, B.k_full + st);
      else if (partial) ptx::bulk_load(rbuf + st * kStageRec, a.krec + it.m.tile_start + kt, kRecBytes, B.k_full + st);
      k_used[st] = true; k_ph[st] = ph;
      if (!wait_bar(B.v_empty + st, ph ^ 1, abort_flag, a.status)) goto drain;
      ptx::mbar_arrive_expect_tx(B.v_full + st, L::kKVBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        ptx::tma_load_2d(vbuf + st * L::kKVBytes + c * kSlab, tv, it.h * D + c * 64, y, B.v_full + st);
      v_used[st] = true; v_ph[st] = ph;
      ++kv_it;
    }
  }
drain:
  // every load issued must land before the CTA exits (only waits after an abort)
  for (int i = 0; i < QB; ++i)
    if (q_used[i]) drain_bar(B.q_full + i, q_ph[i]);
  for (int i = 0; i < NS; ++i) {
    if (k_used[i]) drain_bar(B.k_full + i, k_ph[i]);
    if (v_used[i]) drain_bar(B.v_full + i, v_ph[i]);
  }
}

// ------------------------------------------------------------------ MMA issuer
// Per stream, one thread issues every MMA; tiles are counted across the stream's items.
//
// WIDE (d = 64): S(t) = Q' K'(t)^T over the whole 128-key tile (N = 128) into the
// stream's single S buffer.  S(t+1) is issued as soon as the softmax has read S(t)
// into registers (s_free), so it runs while the softmax computes exponentials.  P(t)
// has its own 64 TMEM columns, one 32-column half per 64-key chunk; O += P_c(t) V_c(t)
// is issued per chunk once that half of P is written (p_full[c]).
//
// Chunked (d = 128, where a separate P does not fit next to O): each tile is two
// 64-key chunks; chunk g of the stream has its S in buffer g % 2 and its P overwrites
// the first 32 columns of that buffer.  Issue order: S(0), S(1), then for every chunk
// g: PV(g) once P(g) is ready, then S(g+2) into the buffer PV(g) has just read (the
// tensor core runs one thread's MMAs in order).
template <int D>
__device__ void run_mma(const AttnArgs& a, uint8_t* sm, int s, const SBars& B, uint32_t tmem,
                        volatile int* abort_flag) {
  using L = Layout<D>;
  constexpr int QB = L::QB, NS = L::NS;
  constexpr bool WIDE = Cfg<D>::WIDE;
  constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kTile, WIDE ? kTile : kChunk, false, false);
  constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(kTile, D, false, true);
  const ItemDesc* items = reinterpret_cast<const ItemDesc*>(sm + L::kItems) + s * 2;
  const uint32_t q_addr = ptx::smem_u32(sm + L::kQ + s * QB * L::kQBytes);
  const uint32_t k_addr = ptx::smem_u32(sm + L::kK + s * NS * L::kKVBytes);
  const uint32_t v_addr = ptx::smem_u32(sm + L::kV + s * NS * L::kKVBytes);
  const TmemMap tm = tmem_map<D>(tmem, s);
  uint32_t it_cnt = 0, q_it = 0, kv_it = 0, p_it = 0, s_ch = 0;
  for (;;) {
    const int slot = (int)(it_cnt & 1);
    if (!wait_bar(B.item_full + slot, (it_cnt >> 1) & 1, abort_flag, a.status)) break;
    ++it_cnt;
    const bool end = items[slot].req < 0;
    const int n = items[slot].n;
    ptx::mbar_arrive(B.item_empty + slot);
    if (end) break;
    if (n <= 0) continue;
    const int qb = (int)(q_it % QB);
    if (!wait_bar(B.q_full + qb, (q_it / QB) & 1, abort_flag, a.status)) break;
    ++q_it;
    ptx::tc_fence_after();
    const uint32_t qa = q_addr + qb * L::kQBytes;
    if constexpr (WIDE) {
      // S(j) of this item; s_ch counts the stream's S tiles
      auto issue_s = [&](int j) -> bool {
        const int st = (int)((kv_it + j) % NS);
        if (s_ch > 0 && !wait_bar(B.s_free, (s_ch - 1) & 1, abort_flag, a.status)) return false;
        if (!wait_bar(B.k_full + st, ((kv_it + j) / NS) & 1, abort_flag, a.status)) return false;
        ptx::tc_fence_after();
        const uint32_t kb = k_addr + st * L::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
          ptx::umma_f16(tm.s, ptx::smem_desc_sw128(qa + off, 16, 1024), ptx::smem_desc_sw128(kb + off, 16, 1024),
                        idesc_s, kk > 0 ? 1u : 0u);
        }
        ptx::umma_commit(B.s_full);
        ++s_ch;
        if (j == n - 1) ptx::umma_commit(B.q_empty + qb);  // last S of the item issued
        return true;
      };
      if (!issue_s(0)) goto out;
      for (int j = 0; j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) goto out;
        const int st = (int)((kv_it + j) % NS);
        const uint32_t vb = v_addr + st * L::kKVBytes;
        const uint32_t pc = p_it++;  // the stream's PV tile count
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          if (!wait_bar(B.p_full + c, pc & 1, abort_flag, a.status)) goto out;
          ptx::tc_fence_after();
          if (c == 0) {
            if (!wait_bar(B.v_full + st, ((kv_it + j) / NS) & 1, abort_flag, a.status)) goto out;
            ptx::tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < kChunk / 16; ++kk)
            ptx::umma_f16_ts(tm.o, tm.p + c * (kChunk / 2) + kk * 8,
                             ptx::smem_desc_sw128(vb + (c * kChunk + kk * 16) * 128, kSlab, 1024), idesc_o,
                             (j > 0 || c > 0 || kk > 0) ? 1u : 0u);
          ptx::umma_commit(B.pv_done + c);
        }
        ptx::umma_commit(B.v_empty + st);
      }
    } else {
      const int nch = 2 * n;
      // S(g) = Q' K'(g)^T for chunk g of this item, into buffer s_ch % 2
      auto issue_s = [&](int g) -> bool {
        const int j = g >> 1, c = g & 1;
        const int st = (int)((kv_it + j) % NS);
        if (c == 0) {
          if (!wait_bar(B.k_full + st, ((kv_it + j) / NS) & 1, abort_flag, a.status)) return false;
          ptx::tc_fence_after();
        }
        const uint32_t kb = k_addr + st * L::kKVBytes + c * (kChunk * 128);
        const uint32_t d_tmem = tm.s + (s_ch & 1) * kChunk;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
          ptx::umma_f16(d_tmem, ptx::smem_desc_sw128(qa + off, 16, 1024), ptx::smem_desc_sw128(kb + off, 16, 1024),
                        idesc_s, kk > 0 ? 1u : 0u);
        }
        ptx::umma_commit(B.s_full + (s_ch & 1));
        ++s_ch;
        if (g == nch - 1) ptx::umma_commit(B.q_empty + qb);  // last S of the item issued
        return true;
      };
      const uint32_t ch0 = s_ch;  // global chunk index of this item's chunk 0
      if (!issue_s(0) || !issue_s(1)) goto out;
      for (int g = 0; g < nch; ++g) {
        const int j = g >> 1, c = g & 1;
        const int st = (int)((kv_it + j) % NS);
        const uint32_t pc = p_it++;  // the stream's chunk count
        if (!wait_bar(B.p_full + (pc & 1), (pc >> 1) & 1, abort_flag, a.status)) goto out;
        ptx::tc_fence_after();
        if (c == 0) {
          if (!wait_bar(B.v_full + st, ((kv_it + j) / NS) & 1, abort_flag, a.status)) goto out;
          ptx::tc_fence_after();
        }
        // O += P(g) V(g): P from TMEM, V rows of this chunk (both 64-column slabs)
        const uint32_t vb = v_addr + st * L::kKVBytes;
        const uint32_t pa = tm.s + ((ch0 + g) & 1) * kChunk;
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
          ptx::umma_f16_ts(tm.o, pa + kk * 8,
                           ptx::smem_desc_sw128(vb + c * (kChunk * 128) + kk * 16 * 128, kSlab, 1024), idesc_o,
                           (g > 0 || kk > 0) ? 1u : 0u);
        ptx::umma_commit(B.pv_done + (pc & 1));
        if (c == 1) ptx::umma_commit(B.v_empty + st);
        if (NS >= 2) {
          if (g + 2 < nch && !issue_s(g + 2)) goto out;
        } else if (c == 1) {
          // one K/V stage: the next tile's K can only land after this tile's last PV,
          // so both of its S chunks are issued here
          if (g + 1 < nch && !issue_s(g + 1)) goto out;
          if (g + 2 < nch && !issue_s(g + 2)) goto out;
        }
      }
    }
    ptx::umma_commit(B.o_ready);
    kv_it += n;
  }
out:
  // all issued MMAs must complete before TMEM is released
  ptx::umma_commit(B.mma_done);
  drain_bar(B.mma_done, 0);
}

// ------------------------------------------------------------------ softmax
// The exponentials of one 64-key chunk against the reference m (log2 domain): P packed
// to bf16 pairs and the sum rs of the unrounded exponentials.
__device__ __forceinline__ void exp_chunk(const float (&x)[kChunk], float sl2, float m, uint32_t (&pk)[kChunk / 2],
                                          float& rs) {
  const unsigned long long sl2x2 = pack2(sl2, sl2), negm2 = pack2(-m, -m);
  unsigned long long acc0 = 0ull, acc1 = 0ull;  // packed partial sums (+0.0f pairs)
#pragma unroll
  for (int e = 0; e < kChunk / 2; ++e) {
    float y0, y1;
    unpack2(ffma2(pack2(x[2 * e], x[2 * e + 1]), sl2x2, negm2), y0, y1);
    const float e0 = ex2(y0), e1 = ex2(y1);
    const __nv_bfloat162 pb = __floats2bfloat162_rn(e0, e1);
    pk[e] = *reinterpret_cast<const uint32_t*>(&pb);
    if (e & 1) acc1 = fadd2(acc1, pack2(e0, e1));
    else acc0 = fadd2(acc0, pack2(e0, e1));
  }
  float r0, r1, r2, r3;
  unpack2(acc0, r0, r1);
  unpack2(acc1, r2, r3);
  rs = (r0 + r1) + (r2 + r3);
}

// One 64-key chunk of a row: masked scores, lazy reference-max update, P = 2^(x*sl2 - m)
// in bf16 pairs, the sum rs of the exponentials, and the factor corr (needed when resc)
// by which O and l must be scaled before P is added.  The reference m_ref moves only when
// the chunk's maximum exceeds it by 2^kRescaleLog2, so P stays below 2^8.
//
// LAZY (rows of many key tiles, where the maximum rarely moves): with a finite reference
// the exponentials are formed against it at once, and the chunk's maximum is only taken
// when one of them could be large, which their sum bounds (every term is at most the
// sum): below kLazySum the chunk is done with no rescale; otherwise (and for a row's
// first visible chunk) the maximum becomes the reference and the chunk is formed again.
// This trades the maximum's instructions on most chunks for more live registers.
template <bool LAZY>
__device__ __forceinline__ void softmax_chunk(const uint32_t (&sr)[kChunk], bool partial, uint32_t w0, uint32_t w1,
                                              float sl2, float& m_ref, uint32_t (&pk)[kChunk / 2], float& corr,
                                              bool& resc, float& rs) {
  float x[kChunk];
#pragma unroll
  for (int e = 0; e < kChunk; ++e) x[e] = __uint_as_float(sr[e]);
  if (partial) {
#pragma unroll
    for (int e = 0; e < kChunk; ++e)
      if (!(((e < 32 ? w0 : w1) >> (e & 31)) & 1u)) x[e] = -INFINITY;
  }
  if constexpr (LAZY) {
    corr = 1.f;
    resc = false;
    if (m_ref != -INFINITY) {
      exp_chunk(x, sl2, m_ref, pk, rs);
      if (rs < kLazySum) return;
    }
  }
  // row maximum as a depth-4 tree of three-input maxima (21 + 7 + 3 + 1)
  static_assert(kChunk == 64, "the max tree covers 64 scores");
  float m1[22], m2[8];
#pragma unroll
  for (int i = 0; i < 21; ++i) m1[i] = fmax3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  m1[21] = x[63];
#pragma unroll
  for (int i = 0; i < 7; ++i) m2[i] = fmax3(m1[3 * i], m1[3 * i + 1], m1[3 * i + 2]);
  m2[7] = m1[21];
  const float mx = fmax3(fmax3(m2[0], m2[1], m2[2]), fmax3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
  const float m_tile = mx * sl2;  // -inf stays -inf (sl2 > 0)
  // LAZY: a sum at or above kLazySum means some term exceeded 2^2, so the maximum moves
  const float m_new = LAZY ? (m_tile > m_ref ? m_tile : m_ref) : ((m_tile > m_ref + kRescaleLog2) ? m_tile : m_ref);
  const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
  // O (and l) need scaling only when a finite running max moved; while it is -inf
  // every P so far was exactly 0, so O and l are 0
  resc = m_new != m_ref && m_ref != -INFINITY;
  corr = resc ? ex2(m_ref - m_use) : 1.f;
  exp_chunk(x, sl2, m_use, pk, rs);
  m_ref = m_new;
}

template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tm_o, float corr) {
#pragma unroll
  for (int half = 0; half < D / 64; ++half) {
    uint32_t o[64];
    ptx::tmem_ld64(tm_o + half * 64, o);
#pragma unroll
    for (int e = 0; e < 64; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
    ptx::tmem_st64(tm_o + half * 64, o);
  }
}

// Compression epilogue: 64 output columns (block cb) of this row's O go to its group's
// output row.  The rows of a 32-row warp block that share a group are summed across
// lanes (segmented by the group's last lane); a group inside the block is written
// once, in bf16, by its first lane; a group that straddles a block boundary (groups
// are at most 32 rows) leaves the block's fp32 partial in the fix-up buffer, part 0
// from the lower block and part 1 from the upper, summed by k_cmp_fixup.
template <int D>
__device__ __forceinline__ void cmp_store(const AttnArgs& a, const CmpReq& cr, int h, int pi, bool row_ok,
                                          int lane, float (&v)[64], int cb) {
  const CmpArgs& c = a.cmp;
  int glo = pi, ghi = pi + 1;
  long long orow = -1;
  if (row_ok) orow = cmp_group_of(c, cr, pi, glo, ghi);
  const int r0 = pi - lane;  // the warp block's first request-local row (a multiple of 32)
  // the lanes of this row's group inside the block (groups are runs of consecutive rows)
  const int first = max(glo, r0) - r0, last = min(ghi, r0 + 32) - 1 - r0;
  for (int off = 1; off < c.span; off <<= 1) {
#pragma unroll
    for (int e = 0; e < 64; ++e) {
      const float u = __shfl_down_sync(0xffffffffu, v[e], off);
      if (lane + off <= last) v[e] += u;
    }
  }
  if (!row_ok || lane != first) return;
  const int H = a.heads;
  if (glo >= r0 && ghi <= r0 + 32) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(c.x_out) + (orow * H + h) * D + cb * 64;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 pb = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
        wv[e] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      reinterpret_cast<uint4*>(dst)[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  } else {
    const bool upper = glo < r0;  // this block holds the group's later rows
    const long long k = cr.fix_start + (upper ? r0 : r0 + 32) / 32;
    float* dst = c.fix + ((k * 2 + (upper ? 1 : 0)) * H + h) * D + cb * 64;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

// GATE: the attention output gate is applied in the epilogue (a separate
// instantiation, so the plain epilogue carries none of its code).  CMP: the output is
// the history compression of O (cmp_store) instead of O.  LAZY: softmax_chunk's lazy
// maximum, for plans whose items run over many key tiles.
template <int D, bool GATE, bool CMP, bool LAZY>
__device__ void run_softmax(const AttnArgs& a, uint8_t* sm, int s, const SBars& B, uint32_t tmem,
                            volatile int* abort_flag) {
  using L = Layout<D>;
  constexpr int NS = L::NS;
  constexpr bool WIDE = Cfg<D>::WIDE;
  const ItemDesc* items = reinterpret_cast<const ItemDesc*>(sm + L::kItems) + s * 2;
  const StageInfo* info = reinterpret_cast<const StageInfo*>(sm + L::kInfo) + s * NS;
  const uint8_t* recs = sm + L::kRec + s * NS * kStageRec;  // per stage: key record or mask rows
  const KeyTileRec* qrecs = reinterpret_cast<const KeyTileRec*>(sm + L::kQRec) + s * L::QB;
  const int lane = threadIdx.x & 31;
  const int quad = (threadIdx.x >> 5) & 3;  // TMEM lanes this warp may access
  const int row = quad * 32 + lane;
  const TmemMap tm = tmem_map<D>(tmem + ((uint32_t)(quad * 32) << 16), s);
  const float sl2 = a.scale * 1.4426950408889634f;  // scale * log2(e)
  const int H = a.heads;
  const bool wide = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;  // O's 64-column pieces 32-byte aligned
  // ch: the stream's S chunk count (chunked) or S tile count (WIDE)
  uint32_t it_cnt = 0, kv_it = 0, ch = 0, o_it = 0, q_it = 0;
  for (;;) {
    const int slot = (int)(it_cnt & 1);
    if (!wait_bar_warp(B.item_full + slot, (it_cnt >> 1) & 1, abort_flag, a.status)) return;
    ++it_cnt;
    const ItemDesc d = items[slot];
    ptx::mbar_arrive(B.item_empty + slot);
    if (d.req < 0) return;
    const bool row_ok = row < d.rows;
    const int pi = d.pos0 + row;
    const long long tok = d.tok0 + row;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + (tok * H + d.h) * D;
    if (d.n <= 0) {  // no visible key tile: zero rows; -1: a tile of pruned queries
      if constexpr (CMP) {  // every row is computed (no pruning): zeros into the groups
        const CmpReq cr = a.cmp.req[d.req];
#pragma unroll 1
        for (int cb = 0; cb < D / 64; ++cb) {
          float v[64];
#pragma unroll
          for (int e = 0; e < 64; ++e) v[e] = 0.f;
          cmp_store<D>(a, cr, d.h, pi, row_ok, lane, v, cb);
        }
      } else if (d.n == 0 && row_ok && query_kept(a.ty[tok], pi, d.keep)) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
        if (a.lse) a.lse[tok * H + d.h] = -INFINITY;
      }
      continue;
    }
    // this row's time and type, from the query tile's record next to Q
    const int qb = (int)(q_it % L::QB);
    if (!wait_bar_warp(B.q_full + qb, (q_it / L::QB) & 1, abort_flag, a.status)) return;
    ++q_it;
    const KeyTileRec* qr = qrecs + qb;
    const long long ti = qr->t[row];
    int tyi = -1;
#pragma unroll
    for (int c = 0; c < kTypes; ++c)
      if ((qr->typebits[c][row >> 5] >> (row & 31)) & 1u) tyi = c;
    ptx::mbar_arrive(B.q_empty + qb);  // the Q buffer and its record may be refilled
    const bool out_ok = row_ok && query_kept(tyi, pi, d.keep);  // pruned rows are computed, not written
    // GATE: the row's gate (D bf16, whole 128-byte lines) is prefetched into L2 while the
    // item runs and read in the epilogue, so no registers hold it through the tiles
    if constexpr (GATE) {
      if (out_ok) {
        const char* g0 = reinterpret_cast<const char*>(static_cast<const __nv_bfloat16*>(a.out_gate) +
                                                       (tok * H + d.h) * D);
#pragma unroll
        for (int c = 0; c < D * 2 / 128; ++c) asm volatile("prefetch.global.L2 [%0];" ::"l"(g0 + 128 * c));
      }
    }
    RowMask rm;
    row_mask_setup(a.mask, row_ok, pi, ti, tyi, rm);
    float m_ref = -INFINITY, l = 0.f;
    bool p1_pending = false;
    for (int j = 0; j < d.n; ++j) {
      const int st = (int)(kv_it % NS);
      const uint32_t kph = (kv_it / NS) & 1;
      ++kv_it;
      // the stage's tile info and key record (written by the producer / bulk copy)
      if (!wait_bar_warp(B.k_full + st, kph, abort_flag, a.status)) return;
      const StageInfo inf = info[st];
      const bool partial = inf.cls != REC_ATTN_TILE_FULL;
      uint32_t vm[4] = {~0u, ~0u, ~0u, ~0u};
      if (partial) {
        if (inf.tab) {
          const uint4 w = reinterpret_cast<const uint4*>(recs + st * kStageRec)[row];
          vm[0] = w.x; vm[1] = w.y; vm[2] = w.z; vm[3] = w.w;
        } else {
          build_mask(rm, reinterpret_cast<const KeyTileRec*>(recs + st * kStageRec), inf.kt * kTile, vm);
        }
      }
      if constexpr (WIDE) {
        const uint32_t t = ch++;
        if (!wait_bar_warp(B.s_full, t & 1, abort_flag, a.status)) return;
        ptx::mbar_arrive(B.k_free + st);  // S(t) has read K; info and record were read above
        ptx::tc_fence_after();
        uint32_t sr[kChunk], pk[kChunk / 2];
        float corr, rs;
        bool resc;
        ptx::tmem_ld64_async(tm.s, sr);
        ptx::tmem_wait_ld(sr);
        if (p1_pending) {  // publish the previous tile's P half 1, stored while this S loaded
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(B.p_full + 1);
          p1_pending = false;
        }
        softmax_chunk<LAZY>(sr, partial, vm[0], vm[1], sl2, m_ref, pk, corr, resc, rs);
        l = l * corr + rs;
        // P half c may be overwritten once PV_c(t-1) has read it; O may be rescaled
        // once every earlier PV has landed.  Each pv_done[c] completes once per tile
        // and PV_c(t) needs P half c of tile t, so every parity wait here is exact.
        if (t > 0 && !wait_bar_warp(B.pv_done + 0, (t - 1) & 1, abort_flag, a.status)) return;
        if (__any_sync(0xffffffffu, resc)) {
          if (!wait_bar_warp(B.pv_done + 1, (t - 1) & 1, abort_flag, a.status)) return;
          ptx::tc_fence_after();
          rescale_o<D>(tm.o, corr);
        }
        ptx::tc_fence_after();
        ptx::tmem_st32_async(tm.p, pk);
        ptx::tmem_ld64_async(tm.s + kChunk, sr);  // the second half loads while P half 0 stores
        ptx::tmem_wait_ld(sr);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(B.p_full + 0);
        ptx::mbar_arrive(B.s_free);  // S(t) is in registers: S(t+1) may overwrite it
        softmax_chunk<LAZY>(sr, partial, vm[2], vm[3], sl2, m_ref, pk, corr, resc, rs);
        l = l * corr + rs;
        if (t > 0 && !wait_bar_warp(B.pv_done + 1, (t - 1) & 1, abort_flag, a.status)) return;
        if (__any_sync(0xffffffffu, resc)) {
          if (!wait_bar_warp(B.pv_done + 0, t & 1, abort_flag, a.status)) return;
          ptx::tc_fence_after();
          rescale_o<D>(tm.o, corr);
        }
        ptx::tc_fence_after();
        ptx::tmem_st32_async(tm.p + kChunk / 2, pk);
        p1_pending = true;  // published after the next S load, or before the epilogue
      } else {
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const uint32_t buf = ch & 1;
          if (!wait_bar_warp(B.s_full + buf, (ch >> 1) & 1, abort_flag, a.status)) return;
          if (c == 1) ptx::mbar_arrive(B.k_free + st);  // both S chunks have read K
          ptx::tc_fence_after();
          uint32_t sr[kChunk], pk[kChunk / 2];
          float corr, rs;
          bool resc;
          ptx::tmem_ld64(tm.s + buf * kChunk, sr);
          softmax_chunk<LAZY>(sr, partial, c ? vm[2] : vm[0], c ? vm[3] : vm[1], sl2, m_ref, pk, corr, resc, rs);
          l = l * corr + rs;
          // O may only be rescaled once PV(ch-1) has landed.  The two pv_done barriers
          // alternate by chunk, and PV(ch+1) cannot start before P(ch+1) exists, so the
          // barrier of chunk ch-1 is at most at that chunk's phase: the parity wait is
          // exact although most chunks never wait on it.
          if (__any_sync(0xffffffffu, resc)) {
            if (!wait_bar_warp(B.pv_done + ((ch - 1) & 1), ((ch - 1) >> 1) & 1, abort_flag, a.status)) return;
            ptx::tc_fence_after();
            rescale_o<D>(tm.o, corr);
          }
          ptx::tmem_st32(tm.s + buf * kChunk, pk);  // P over the first 32 columns of S
          ptx::tc_fence_before();
          ptx::mbar_arrive(B.p_full + (ch & 1));
          ++ch;
        }
      }
    }
    if (p1_pending) {
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(B.p_full + 1);
    }
    // epilogue: O / l (times sigmoid of the output gate)
    if (!wait_bar_warp(B.o_ready, o_it & 1, abort_flag, a.status)) return;
    ++o_it;
    ptx::tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int half = 0; half < D / 64; ++half) {
      uint32_t o[64];
      ptx::tmem_ld64(tm.o + half * 64, o);
      if constexpr (CMP) {
        float v[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) v[e] = __uint_as_float(o[e]) * inv;
        cmp_store<D>(a, a.cmp.req[d.req], d.h, pi, row_ok, lane, v, half);
      } else if (out_ok) {
        // two 16-byte chunks (16 columns) at a time: one 32-byte store when O is 32-byte
        // aligned (whole sectors; a warp's rows lie H * d * 2 bytes apart), else two
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) {
          uint32_t wv[8];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int c = 2 * c2 + h2;
            float sc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) sc[e] = inv;
            if constexpr (GATE) {
              const uint4 gv = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.out_gate) +
                                                              (tok * H + d.h) * D + half * 64)[c];
              const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
                sc[2 * e] *= sigmoidf_fast(gf.x);
                sc[2 * e + 1] *= sigmoidf_fast(gf.y);
              }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 pb = __floats2bfloat162_rn(__uint_as_float(o[c * 8 + 2 * e]) * sc[2 * e],
                                                              __uint_as_float(o[c * 8 + 2 * e + 1]) * sc[2 * e + 1]);
              wv[4 * h2 + e] = *reinterpret_cast<const uint32_t*>(&pb);
            }
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + half * 64) + 2 * c2;
          if (wide) {
            ptx::st_global_v8(dst, wv[0], wv[1], wv[2], wv[3], wv[4], wv[5], wv[6], wv[7]);
          } else {
            dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
          }
        }
      }
    }
    if (!CMP && out_ok && a.lse) {
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      a.lse[tok * H + d.h] = l > 0.f ? (m_use + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    ptx::tc_fence_before();  // O reads ordered before the next item's PV(0)
  }
}

template <int D, bool GATE, bool CMP, bool LAZY>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using L = Layout<D>;
  constexpr int QB = L::QB, NS = L::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kStreams * L::kBarsPerStream);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kStreams * L::kBarsPerStream) + 1;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreams; ++s) {
      SBars B;
      B.bind<D>(bars + s * L::kBarsPerStream);
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(B.item_full + i, 1);
        ptx::mbar_init(B.item_empty + i, 1 + 128);
      }
      for (int i = 0; i < QB; ++i) {
        ptx::mbar_init(B.q_full + i, 1);
        ptx::mbar_init(B.q_empty + i, 1 + 128);  // last S MMA done + every softmax thread read its row
      }
      for (int i = 0; i < NS; ++i) {
        ptx::mbar_init(B.k_full + i, 1);
        ptx::mbar_init(B.v_full + i, 1);
        ptx::mbar_init(B.k_free + i, 128);
        ptx::mbar_init(B.v_empty + i, 1);
      }
      ptx::mbar_init(B.s_full, 1);
      ptx::mbar_init(B.s_full + 1, 1);
      ptx::mbar_init(B.s_free, 128);
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(B.p_full + i, 128);
        ptx::mbar_init(B.pv_done + i, 1);
      }
      ptx::mbar_init(B.o_ready, 1);
      ptx::mbar_init(B.mma_done, 1);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kRoleWarps) {
    const int s = warp & 1;
    SBars B;
    B.bind<D>(bars + s * L::kBarsPerStream);
    if ((threadIdx.x & 31) == 0) {
      if (warp < 2) run_producer<D>(a, &tm_q, &tm_k, &tm_v, sm, s, B, abort_flag);
      else run_mma<D>(a, sm, s, B, tmem, abort_flag);
    }
  } else {
    const int s = (warp - kRoleWarps) >> 2;
    SBars B;
    B.bind<D>(bars + s * L::kBarsPerStream);
    run_softmax<D, GATE, CMP, LAZY>(a, sm, s, B, tmem, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  // the last CTA to leave resets the item counter for the next launch
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.counters + 2, 1) == (int)gridDim.x - 1) {
      atomicExch(a.counters + 1, 0);
      atomicExch(a.counters + 2, 0);
    }
  }
}

template <int D, bool GATE, bool CMP, bool LAZY>
cudaError_t launch_t(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                     int grid, cudaStream_t st) {
  using L = Layout<D>;
  static_assert(L::kDynamic <= 227 * 1024, "shared memory budget");
  cudaError_t e =
      cudaFuncSetAttribute(k_attn_tc<D, GATE, CMP, LAZY>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamic);
  if (e != cudaSuccess) return e;
  k_attn_tc<D, GATE, CMP, LAZY><<<grid, kThreads, L::kDynamic, st>>>(q, k, v, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, int grid,
                   cudaStream_t st) {
  if (a.cmp.req) return launch_t<D, false, true, false>(a, q, k, v, grid, st);
  if (a.out_gate) return launch_t<D, true, false, false>(a, q, k, v, grid, st);
  if constexpr (Cfg<D>::WIDE) {
    if (a.long_items) return launch_t<D, false, false, true>(a, q, k, v, grid, st);
  }
  return launch_t<D, false, false, false>(a, q, k, v, grid, st);
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           int head_dim, int grid, cudaStream_t st) {
  if (a.n_items <= 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch<64>(a, q, k, v, grid, st);
    case 128: return launch<128>(a, q, k, v, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace recattn
