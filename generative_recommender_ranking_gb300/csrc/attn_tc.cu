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
//   warp 2, 3     MMA issuers (stream 0, 1): each 128-key tile is two 64-key chunks;
//                 S(g) = Q'K'(g)^T goes to TMEM buffer g % 2 of the stream, so S(g+1)
//                 is computed while the softmax works on chunk g; O += P(g) V(g) reads
//                 P straight from TMEM (P overwrites the first 32 columns of S(g));
//   warps 4..7    softmax of stream 0, warps 8..11 softmax of stream 1: one query row
//                 per thread (TMEM lane quadrant = warp % 4).  PARTIAL tiles build the
//                 row's 128-bit visibility mask from position ranges, per-type key
//                 bitmaps and, for time clauses, a binary search over time-sorted
//                 runs; FULL tiles skip the mask.  Online softmax in the exp2 domain
//                 with a lazily updated reference maximum; O rescaled in TMEM only when
//                 the maximum grows by more than 2^8; P rounded to bf16.  The row sum l
//                 is the sum of exactly those rounded P values (for d = 64 the PV MMA
//                 computes it: a block of bf16 ones is appended to V as 16 extra output
//                 columns), so every output row is an exact convex combination of the
//                 value rows it saw.  Row times and types come from the query tile's
//                 planner record, bulk-copied next to Q.
// Every wait on an mbarrier is bounded (REC_ATTN_ERR_TIMEOUT in the status word).
#include <climits>

#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "ptx_sm103.cuh"

namespace recattn {

namespace {

constexpr int kStreams = 2;
constexpr int kThreads = 384;
constexpr int kSlab = kTile * 128;           // 128 rows x 128 B: one 64-column swizzle slab
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;          // keep the reference max until it is exceeded by 2^8
constexpr int kRecBytes = (int)sizeof(KeyTileRec);
constexpr int kChunk = 64;                   // keys per S chunk (a 128-key tile is two chunks)

template <int D>
struct Cfg;
// QB: Q buffers per stream, NS: K/V stages per stream, SUM: the PV MMA also sums P
// (a block of ones appended to V as 16 extra output columns), OC: TMEM columns of O.
template <>
struct Cfg<64> {
  static constexpr int QB = 2, NS = 2;
  static constexpr bool SUM = true;
  static constexpr int OC = 64 + 16;
};
template <>
struct Cfg<128> {
  static constexpr int QB = 1, NS = 1;
  static constexpr bool SUM = false;
  static constexpr int OC = 128;
};

struct ItemDesc {
  long long tok0;  // first token of the query tile (global index)
  int pos0;        // request-local position of the tile's first row
  int rows;        // valid rows in the tile
  int h;
  int n;           // non-SKIP key tiles
  int end;         // 1: the stream is done
  int pad;
};
static_assert(sizeof(ItemDesc) == 32, "");

struct StageInfo {
  int kt;
  int cls;
};

template <int D>
struct Layout {
  static constexpr int QB = Cfg<D>::QB, NS = Cfg<D>::NS;
  static constexpr int kQBytes = kTile * D * 2;
  static constexpr int kKVBytes = kTile * D * 2;
  static constexpr int kQ = 0;                                   // [stream][QB]
  static constexpr int kK = kQ + kStreams * QB * kQBytes;        // [stream][NS]
  static constexpr int kV = kK + kStreams * NS * kKVBytes;       // [stream][NS]
  static constexpr int kOnes = kV + kStreams * NS * kKVBytes;    // 128 x 64 bf16 ones (SUM only)
  static constexpr int kRec = kOnes + (Cfg<D>::SUM ? kSlab : 0);  // [stream][NS] KeyTileRec
  static constexpr int kQRec = kRec + kStreams * NS * kRecBytes;  // [stream][QB] KeyTileRec of the query tile
  static constexpr int kInfo = kQRec + kStreams * QB * kRecBytes; // [stream][NS] StageInfo
  static constexpr int kItems = (kInfo + kStreams * NS * 8 + 15) & ~15;  // [stream][2] ItemDesc
  static constexpr int kBars = (kItems + kStreams * 2 * 32 + 7) & ~7;
  static constexpr int kBarsPerStream = 2 + 2 + 2 * QB + 3 * NS + 6;
  static constexpr int kTotal = kBars + kStreams * kBarsPerStream * 8 + 16;
  static constexpr int kDynamic = kTotal + 1024;  // slack to align the base to 1024 B
};

// mbarriers of one stream
struct SBars {
  uint64_t *item_full, *item_empty, *q_full, *q_empty, *k_full, *v_full, *kv_empty;
  uint64_t *s_full, *p_full, *pv_done, *o_ready, *mma_done;  // s_full: [2], one per S buffer
  template <int D>
  __device__ void bind(uint64_t* b) {
    constexpr int QB = Cfg<D>::QB, NS = Cfg<D>::NS;
    item_full = b; item_empty = b + 2; q_full = b + 4; q_empty = q_full + QB;
    k_full = q_empty + QB; v_full = k_full + NS; kv_empty = v_full + NS;
    s_full = kv_empty + NS; p_full = s_full + 2; pv_done = p_full + 1; o_ready = pv_done + 1;
    mma_done = o_ready + 1;
  }
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > kWaitNs) {
      *abort_flag = 1;
      set_status(status, REC_ATTN_ERR_TIMEOUT);
      return false;
    }
  }
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

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bits lo..hi (inclusive, tile-local key indices) of a 128-bit mask.
__device__ __forceinline__ void range_bits(int lo, int hi, uint32_t (&r)[4]) {
  lo = max(lo, 0);
  hi = min(hi, kTile - 1);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int a = max(lo - 32 * w, 0), b = min(hi - 32 * w, 31);
    r[w] = (a > b) ? 0u : ((0xffffffffu >> (31 - b)) & (0xffffffffu << a));
  }
}

// A query row's visibility, per key type, as a position interval [plo, phi]
// (request-local; empty when plo > phi) and an optional time bound t_j <= thr.
struct RowMask {
  int plo[kTypes], phi[kTypes];
  long long thr[kTypes];
  int timed[kTypes];
};

// The predicate of include/rec_attn.h, split per key type into the interval and time
// clauses it reduces to for a fixed query row.
__device__ __forceinline__ void row_mask_setup(const MaskP& m, bool row_ok, int pi, long long ti, int tyi,
                                               RowMask& r) {
  bool dok; long long dthr;
  delay_bound(ti, m.delay, dok, dthr);
  const bool valid = row_ok && (unsigned)tyi <= 3u;
#pragma unroll
  for (int c = 0; c < kTypes; ++c) {
    int lo = INT_MIN / 2, hi = INT_MAX / 2;
    bool vis = valid, timed = false;
    long long thr = LLONG_MAX;
    const bool uq = is_user(tyi), uk = is_user(c);
    if (uq) {
      if (!uk) {
        vis = false;
      } else if (!m.bidir) {
        hi = pi;
        if (m.window > 0 && tyi != REC_ATTN_GLOBAL && c != REC_ATTN_GLOBAL) lo = pi - m.window + 1;
      }
    } else if (tyi == REC_ATTN_RT) {
      if (!uk) {
        if (c == REC_ATTN_RT) hi = pi;
        else vis = false;
      }
    } else {  // candidate query
      if (!uk) {
        if (c == REC_ATTN_RT) {  // real-time events strictly before the candidate
          timed = true;
          if (ti == LLONG_MIN) vis = false;
          else thr = ti - 1;
        } else {                 // itself only
          lo = pi; hi = pi;
        }
      }
    }
    if (m.use_delay && !(tyi == REC_ATTN_CAND && c == REC_ATTN_CAND)) {
      if (!dok) vis = false;
      timed = true;
      thr = min(thr, dthr);
    }
    r.plo[c] = vis ? lo : 1;
    r.phi[c] = vis ? hi : 0;
    r.thr[c] = thr;
    r.timed[c] = timed ? 1 : 0;
  }
}

// 128-bit visibility mask of one row against a PARTIAL key tile starting at
// request-local position k0.
__device__ __forceinline__ void build_mask(const RowMask& rm, const KeyTileRec* rec, int k0, uint32_t (&vm)[4]) {
  vm[0] = vm[1] = vm[2] = vm[3] = 0u;
#pragma unroll
  for (int c = 0; c < kTypes; ++c) {
    // the record comes from the planner; its run is still clamped to the tile so no
    // value in it can index outside the record
    const int rl = min(max(rec->run_lo[c], 0), kTile - 1);
    const int n = min(max(rec->run_n[c], 0), kTile - rl);
    const int lo = rm.plo[c] - k0, hi = rm.phi[c] - k0;
    if (n == 0 || lo > hi || hi < 0 || lo >= kTile) continue;
    uint32_t r[4];
    range_bits(lo, hi, r);
#pragma unroll
    for (int w = 0; w < 4; ++w) r[w] &= rec->typebits[c][w];
    if (rm.timed[c]) {
      const long long thr = rm.thr[c];
      if (rec->sorted[c]) {
        // keys of this type form a run with non-decreasing times: count t_j <= thr
        int first = 0, len = n;
        while (len > 0) {
          const int half = len >> 1;
          if (rec->t[rl + first + half] <= thr) { first += half + 1; len -= half + 1; }
          else len = half;
        }
        uint32_t tr[4];
        range_bits(rl, rl + first - 1, tr);
#pragma unroll
        for (int w = 0; w < 4; ++w) r[w] &= tr[w];
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t bits = 0;
#pragma unroll 8
          for (int b = 0; b < 32; ++b) bits |= (rec->t[w * 32 + b] <= thr ? 1u : 0u) << b;
          r[w] &= bits;
        }
      }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) vm[w] |= r[w];
  }
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
  uint8_t* rbuf = sm + L::kRec + s * NS * kRecBytes;
  uint8_t* qrbuf = sm + L::kQRec + s * QB * kRecBytes;
  uint32_t it_cnt = 0, q_it = 0, kv_it = 0;
  bool q_used[QB], st_used[NS];
  uint32_t q_ph[QB], st_ph[NS];
  for (int i = 0; i < QB; ++i) { q_used[i] = false; q_ph[i] = 0; }
  for (int i = 0; i < NS; ++i) { st_used[i] = false; st_ph[i] = 0; }
  for (;;) {
    const long long w = atomicAdd(a.counters + 1, 1);
    const int slot = (int)(it_cnt & 1);
    if (!wait_bar(B.item_empty + slot, ((it_cnt >> 1) & 1) ^ 1, abort_flag, a.status)) break;
    ++it_cnt;
    ItemDesc* d = items + slot;
    if (w >= a.n_items) {
      d->end = 1;
      ptx::mbar_arrive(B.item_full + slot);
      break;
    }
    const WorkItem it = decode_item(a, w, true);
    d->tok0 = it.m.tok_start + (long long)it.qt * kTile;
    d->pos0 = it.qt * kTile;
    d->rows = min(kTile, it.m.len - it.qt * kTile);
    d->h = it.h;
    d->n = it.n;
    d->end = 0;
    ptx::mbar_arrive(B.item_full + slot);
    if (it.n == 0) continue;
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
      const int kt = (int)(e & 0xffffffu), cl = (int)(e >> 24);
      const int st = (int)(kv_it % NS);
      const uint32_t ph = (kv_it / NS) & 1;
      if (!wait_bar(B.kv_empty + st, ph ^ 1, abort_flag, a.status)) goto drain;
      info[st].kt = kt;
      info[st].cls = cl;
      const bool partial = cl != REC_ATTN_TILE_FULL;
      const int y = (int)(it.m.tok_start + (long long)kt * kTile);
      ptx::mbar_arrive_expect_tx(B.k_full + st, L::kKVBytes + (partial ? kRecBytes : 0));
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        ptx::tma_load_2d(kbuf + st * L::kKVBytes + c * kSlab, tk, it.h * D + c * 64, y, B.k_full + st);
      if (partial) ptx::bulk_load(rbuf + st * kRecBytes, a.krec + it.m.tile_start + kt, kRecBytes, B.k_full + st);
      ptx::mbar_arrive_expect_tx(B.v_full + st, L::kKVBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        ptx::tma_load_2d(vbuf + st * L::kKVBytes + c * kSlab, tv, it.h * D + c * 64, y, B.v_full + st);
      st_used[st] = true; st_ph[st] = ph;
      ++kv_it;
    }
  }
drain:
  // every load issued must land before the CTA exits (only waits after an abort)
  for (int i = 0; i < QB; ++i)
    if (q_used[i]) drain_bar(B.q_full + i, q_ph[i]);
  for (int i = 0; i < NS; ++i)
    if (st_used[i]) { drain_bar(B.k_full + i, st_ph[i]); drain_bar(B.v_full + i, st_ph[i]); }
}

// ------------------------------------------------------------------ MMA issuer
// Per stream, each 128-key tile is processed as two 64-key chunks.  Chunk g of the
// stream (counted across items) has its S in TMEM buffer g % 2; its P overwrites the
// first 32 columns of that buffer.  Issue order: S(0), S(1), then for every chunk g:
// PV(g) once P(g) is ready, then S(g+2) into the buffer PV(g) has just read.  So while
// the softmax works on chunk g, S(g+1) is already computed.
template <int D>
__device__ void run_mma(const AttnArgs& a, uint8_t* sm, int s, const SBars& B, uint32_t tmem,
                        volatile int* abort_flag) {
  using L = Layout<D>;
  constexpr int QB = L::QB, NS = L::NS;
  constexpr int OC = Cfg<D>::OC;
  constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kTile, kChunk, false, false);
  constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(kTile, OC, false, true);
  const ItemDesc* items = reinterpret_cast<const ItemDesc*>(sm + L::kItems) + s * 2;
  const uint32_t q_addr = ptx::smem_u32(sm + L::kQ + s * QB * L::kQBytes);
  const uint32_t k_addr = ptx::smem_u32(sm + L::kK + s * NS * L::kKVBytes);
  const uint32_t v_addr = ptx::smem_u32(sm + L::kV + s * NS * L::kKVBytes);
  const uint32_t tm_s = tmem + (uint32_t)(s * kTile);
  const uint32_t tm_o = tmem + 2u * kTile + (uint32_t)(s * OC);
  const uint32_t ones_addr = ptx::smem_u32(sm + L::kOnes);
  uint32_t it_cnt = 0, q_it = 0, kv_it = 0, p_it = 0, s_ch = 0;
  for (;;) {
    const int slot = (int)(it_cnt & 1);
    if (!wait_bar(B.item_full + slot, (it_cnt >> 1) & 1, abort_flag, a.status)) break;
    ++it_cnt;
    const int end = items[slot].end, n = items[slot].n;
    ptx::mbar_arrive(B.item_empty + slot);
    if (end) break;
    if (n == 0) continue;
    const int qb = (int)(q_it % QB);
    if (!wait_bar(B.q_full + qb, (q_it / QB) & 1, abort_flag, a.status)) break;
    ++q_it;
    ptx::tc_fence_after();
    const uint32_t qa = q_addr + qb * L::kQBytes;
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
      const uint32_t d_tmem = tm_s + (s_ch & 1) * kChunk;
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
      if (!wait_bar(B.p_full, p_it & 1, abort_flag, a.status)) goto out;
      ++p_it;
      ptx::tc_fence_after();
      if (c == 0) {
        if (!wait_bar(B.v_full + st, ((kv_it + j) / NS) & 1, abort_flag, a.status)) goto out;
        ptx::tc_fence_after();
      }
      // O += P(g) V(g): P from TMEM, V rows of this chunk; the second 64-column block
      // of B is the next V slab (D = 128) or the block of ones whose first 16 output
      // columns give the row sum of P (D = 64)
      const uint32_t vb = v_addr + st * L::kKVBytes;
      const uint32_t lbo = Cfg<D>::SUM ? ones_addr - vb : (uint32_t)kSlab;
      const uint32_t pa = tm_s + ((ch0 + g) & 1) * kChunk;
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk)
        ptx::umma_f16_ts(tm_o, pa + kk * 8,
                         ptx::smem_desc_sw128(vb + c * (kChunk * 128) + kk * 16 * 128, lbo, 1024), idesc_o,
                         (g > 0 || kk > 0) ? 1u : 0u);
      ptx::umma_commit(B.pv_done);
      if (c == 1) ptx::umma_commit(B.kv_empty + st);
      if (NS >= 2) {
        if (g + 2 < nch && !issue_s(g + 2)) goto out;
      } else if (c == 1) {
        // one K/V stage: the next tile's K can only land after this tile's last PV,
        // so both of its S chunks are issued here
        if (g + 1 < nch && !issue_s(g + 1)) goto out;
        if (g + 2 < nch && !issue_s(g + 2)) goto out;
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
template <int D>
__device__ void run_softmax(const AttnArgs& a, uint8_t* sm, int s, const SBars& B, uint32_t tmem,
                            volatile int* abort_flag) {
  using L = Layout<D>;
  constexpr int NS = L::NS;
  const ItemDesc* items = reinterpret_cast<const ItemDesc*>(sm + L::kItems) + s * 2;
  const StageInfo* info = reinterpret_cast<const StageInfo*>(sm + L::kInfo) + s * NS;
  const KeyTileRec* recs = reinterpret_cast<const KeyTileRec*>(sm + L::kRec) + s * NS;
  const KeyTileRec* qrecs = reinterpret_cast<const KeyTileRec*>(sm + L::kQRec) + s * L::QB;
  constexpr int OC = Cfg<D>::OC;
  const int lane = threadIdx.x & 31;
  const int quad = (threadIdx.x >> 5) & 3;  // TMEM lanes this warp may access
  const int row = quad * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tm_s = tmem + lane_off + (uint32_t)(s * kTile);
  const uint32_t tm_o = tmem + lane_off + 2u * kTile + (uint32_t)(s * OC);
  const float sl2 = a.scale * 1.4426950408889634f;  // scale * log2(e)
  const int H = a.heads;
  uint32_t it_cnt = 0, kv_it = 0, ch = 0, o_it = 0, q_it = 0;
  for (;;) {
    const int slot = (int)(it_cnt & 1);
    if (!wait_bar_warp(B.item_full + slot, (it_cnt >> 1) & 1, abort_flag, a.status)) return;
    ++it_cnt;
    const ItemDesc d = items[slot];
    ptx::mbar_arrive(B.item_empty + slot);
    if (d.end) return;
    const bool row_ok = row < d.rows;
    const int pi = d.pos0 + row;
    const long long tok = d.tok0 + row;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + (tok * H + d.h) * D;
    if (d.n == 0) {
      if (row_ok) {
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
    RowMask rm;
    row_mask_setup(a.mask, row_ok, pi, ti, tyi, rm);
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < d.n; ++j) {
      const int st = (int)(kv_it % NS);
      const uint32_t kph = (kv_it / NS) & 1;
      ++kv_it;
      // the stage's tile info and key record (written by the producer / bulk copy)
      if (!wait_bar_warp(B.k_full + st, kph, abort_flag, a.status)) return;
      const StageInfo inf = info[st];
      const bool partial = inf.cls != REC_ATTN_TILE_FULL;
      uint32_t vm[4] = {~0u, ~0u, ~0u, ~0u};
      if (partial) build_mask(rm, recs + st, inf.kt * kTile, vm);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const uint32_t buf = ch & 1;
        if (!wait_bar_warp(B.s_full + buf, (ch >> 1) & 1, abort_flag, a.status)) return;
        ptx::tc_fence_after();
        uint32_t sr[kChunk];
        ptx::tmem_ld64(tm_s + buf * kChunk, sr);
        float x[kChunk];
#pragma unroll
        for (int e = 0; e < kChunk; ++e) x[e] = __uint_as_float(sr[e]);
        if (partial) {
          const uint32_t w0 = c ? vm[2] : vm[0], w1 = c ? vm[3] : vm[1];
#pragma unroll
          for (int e = 0; e < kChunk; ++e)
            if (!(((e < 32 ? w0 : w1) >> (e & 31)) & 1u)) x[e] = -INFINITY;
        }
        float mx = x[0];
#pragma unroll
        for (int e = 1; e < kChunk; ++e) mx = fmaxf(mx, x[e]);
        const float m_tile = mx * sl2;  // -inf stays -inf (sl2 > 0)
        const float m_new = (m_tile > m_ref + kRescaleLog2) ? m_tile : m_ref;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float corr = ex2(m_ref - m_use);  // 0 when m_ref = -inf, 1 when unchanged
        uint32_t pk[kChunk / 2];
        float rs = 0.f;
        const unsigned long long sl2x2 = pack2(sl2, sl2), negm2 = pack2(-m_use, -m_use);
#pragma unroll
        for (int e = 0; e < kChunk / 2; ++e) {
          float y0, y1;
          unpack2(ffma2(pack2(x[2 * e], x[2 * e + 1]), sl2x2, negm2), y0, y1);
          const __nv_bfloat162 pb = __floats2bfloat162_rn(ex2(y0), ex2(y1));
          if (!Cfg<D>::SUM) rs += __low2float(pb) + __high2float(pb);
          pk[e] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        if (!Cfg<D>::SUM) l = l * corr + rs;
        // Every PV completion is waited for in order (one phase per chunk, so the
        // parity wait is exact); O may only be rescaled once PV(ch-1) has landed, and
        // PV(ch-1) was issued as soon as P(ch-1) was ready, so this rarely waits.
        if (ch > 0) {
          if (!wait_bar_warp(B.pv_done, (ch - 1) & 1, abort_flag, a.status)) return;
          ptx::tc_fence_after();
        }
        if ((j > 0 || c > 0) && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
          for (int half = 0; half < D / 64; ++half) {
            uint32_t o[64];
            ptx::tmem_ld64(tm_o + half * 64, o);
#pragma unroll
            for (int e = 0; e < 64; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            ptx::tmem_st64(tm_o + half * 64, o);
          }
          if (Cfg<D>::SUM) {  // the row-sum columns
            uint32_t o[16];
            ptx::tmem_ld16(tm_o + D, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            ptx::tmem_st16(tm_o + D, o);
          }
        }
        ptx::tmem_st32(tm_s + buf * kChunk, pk);  // P over the first 32 columns of S
        ptx::tc_fence_before();
        ptx::mbar_arrive(B.p_full);
        m_ref = m_new;
        ++ch;
      }
    }
    // epilogue: O / l
    if (!wait_bar_warp(B.o_ready, o_it & 1, abort_flag, a.status)) return;
    ++o_it;
    ptx::tc_fence_after();
    if (Cfg<D>::SUM) {
      uint32_t o[16];
      ptx::tmem_ld16(tm_o + D, o);
      l = __uint_as_float(o[0]);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int half = 0; half < D / 64; ++half) {
      uint32_t o[64];
      ptx::tmem_ld64(tm_o + half * 64, o);
      if (row_ok) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 pb = __floats2bfloat162_rn(__uint_as_float(o[c * 8 + 2 * e]) * inv,
                                                            __uint_as_float(o[c * 8 + 2 * e + 1]) * inv);
            wv[e] = *reinterpret_cast<const uint32_t*>(&pb);
          }
          reinterpret_cast<uint4*>(orow + half * 64)[c] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
    if (row_ok && a.lse) {
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      a.lse[tok * H + d.h] = l > 0.f ? (m_use + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    ptx::tc_fence_before();  // O reads ordered before the next item's PV(0)
  }
}

template <int D>
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
        ptx::mbar_init(B.kv_empty + i, 1);
      }
      ptx::mbar_init(B.s_full, 1);
      ptx::mbar_init(B.s_full + 1, 1);
      ptx::mbar_init(B.p_full, 128);
      ptx::mbar_init(B.pv_done, 1);
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
  if (Cfg<D>::SUM) {  // bf16 ones, read by the PV MMA as extra B columns
    uint4* ones = reinterpret_cast<uint4*>(sm + L::kOnes);
    for (int i = threadIdx.x; i < kSlab / 16; i += blockDim.x)
      ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    const int s = warp & 1;
    SBars B;
    B.bind<D>(bars + s * L::kBarsPerStream);
    if ((threadIdx.x & 31) == 0) {
      if (warp < 2) run_producer<D>(a, &tm_q, &tm_k, &tm_v, sm, s, B, abort_flag);
      else run_mma<D>(a, sm, s, B, tmem, abort_flag);
    }
  } else {
    const int s = (warp - 4) >> 2;
    SBars B;
    B.bind<D>(bars + s * L::kBarsPerStream);
    run_softmax<D>(a, sm, s, B, tmem, abort_flag);
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

template <int D>
cudaError_t launch(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, int grid,
                   cudaStream_t st) {
  using L = Layout<D>;
  static_assert(L::kDynamic <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(k_attn_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamic);
  if (e != cudaSuccess) return e;
  k_attn_tc<D><<<grid, kThreads, L::kDynamic, st>>>(q, k, v, a);
  return cudaGetLastError();
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
