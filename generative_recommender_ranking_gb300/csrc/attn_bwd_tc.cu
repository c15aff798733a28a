// attn_bwd_tc.cu -- backward pass of the masked time-RoPE attention on the sm_103a
// tensor cores (bf16 inputs and gradients, fp32 accumulation, head_dim 64 or 128).
//
// Gradients of O = Softmax(QK^T/sqrt(d) + M) V (TM20K review page, section 2.1;
// LazFormer review page, Eq. 19-21) through the time-RoPE (CADET review page, time
// encoding).  With P rebuilt from the forward's log-sum-exp, P_ij = exp(s_ij - lse_i)
// on visible pairs, D_i = <dO_i, O_i> and dS_ij = P_ij (dP_ij - D_i):
//   mode DQ:   dQ'_i = scale sum_j dS_ij K'_j
//   mode DKV:  dV_j = sum_i P_ij dO_i,  dK'_j = scale sum_i dS_ij Q'_i
// and dQ = R(t_i)^T dQ', dK = R(t_j)^T dK' (the rotation is orthogonal).
//
// Both modes share one persistent kernel shape: at head_dim 64 two CTAs per SM (256
// TMEM columns each), at 128 one (512 columns: the accumulators are twice as wide), and
// six warps -- warp 0 loads with TMA, one thread of warp 1 issues every MMA,
// warps 2..5 are the compute warpgroup (one TMEM lane, i.e. one tile row, per
// thread).  The producer claims the planner's (tile, head) items from a global counter
// and publishes each item's descriptor in shared memory for the other roles; mode DKV
// visits key tiles in the mirrored order of the query tiles, so under causal masks
// both modes start with their heaviest items.  Per item the resident operand pair
// stays in shared memory (DQ: Q', dO; DKV: K', V) and the streamed pair (DQ: K', V of
// the query tile's non-SKIP key tiles; DKV: Q', dO of the query tiles whose class
// against the key tile is not SKIP) runs through a two-stage ring.  A streamed tile
// is two 64-wide steps:
//   DQ   S = Q' K'_h^T and dP = dO V_h^T (N = 64); the compute warps write dS (bf16)
//        over the first columns of S; dQ += dS K'_h with dS read from TMEM.  S is
//        double-buffered, so the next step's S runs during this step's compute.
//   DKV  S^T = K' Q'_h^T and dP^T = V dO_h^T; the compute warps write P^T and dS^T
//        (bf16) over them; dV += P^T dO_h and dK += dS^T Q'_h.
// TMEM columns:  DQ   S[0] 0..63 | S[1] 64..127 | dP 128..191 | dQ 192..192+d
//                DKV  S^T 0..63 | dP^T 64..127 | dV 128..128+d | dK 128+d..128+2d
// The accumulators stay in TMEM across an item's tiles; the epilogue scales, undoes
// the rotation and writes bf16 rows.  Everything a compute thread needs besides TMEM
// comes through shared memory with the tiles: the planner's records of the item's tile
// and the streamed tiles (times, type bitmaps) and the rows' constants -lse * log2(e)
// and -D, stored for row pairs as {-lse2(2k), -lse2(2k+1), -D(2k), -D(2k+1)} so that a
// pair of query columns takes one f32x2 operation (k_bwd_rowc, tile-padded so that a
// bulk copy moves a tile's 128 rows), and the item descriptors (k_bwd_schedule, once
// per plan) come from the producer.  PARTIAL tiles take the forward's per-row
// visibility bits (row_mask.cuh), built from the key tile's planner record; in DKV
// each thread first acts as a row of the query tile, builds that row's bits against
// the item's key tile, and the warps transpose the bits into per-key columns with
// shuffles.  PARTIAL pairs with a slot in the plan's mask table skip both: DQ reads the
// table's rows, DKV its columns (transposed once per plan by k_bwd_colmask), bulk-copied
// with the streamed tile.  FULL tiles skip the mask.  The MMAs of one thread run in issue order, so
// an MMA that overwrites TMEM columns an earlier MMA reads needs no wait.  Every
// mbarrier wait is bounded (REC_ATTN_ERR_TIMEOUT in the status word).
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "launchers.cuh"
#include "ptx_sm103.cuh"
#include "row_mask.cuh"
#include "wait.cuh"

namespace recattn {

namespace {

constexpr int kStep = 64;                   // keys (DQ) or queries (DKV) per MMA step
constexpr int kSlab = kTile * 128;          // 128 rows x 64 bf16 columns, 128-byte swizzled
constexpr int kNS = 2;                      // stages of the streamed ring
// Per head dimension: a [128][D] bf16 tile is D / 64 slabs; TMEM columns of the
// accumulators (DQ: S[0] 0..63 | S[1] 64..127 | dP 128..191 | dQ 192..; DKV: S^T 0..63 |
// dP^T 64..127 | dV 128.. | dK 128 + D..); d = 64 runs two CTAs per SM, d = 128 one.
template <int D>
struct BCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr uint32_t kCols = D == 64 ? 256 : 512;
  static constexpr int kBlocksPerSM = D == 64 ? 2 : 1;
  static constexpr uint32_t kDQ = 192, kDV = 128, kDK = 128 + D;
};
constexpr int kRecB = (int)sizeof(KeyTileRec);
constexpr int kMaskB = kTile * 16;  // a PARTIAL pair's 128 rows (or columns) of the mask table
constexpr int kStageRecB = kMaskB > kRecB ? kMaskB : kRecB;  // per streamed stage: one or the other
constexpr int kThreadsB = 192;
constexpr uint64_t kWaitNsB = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;

// mbarriers
enum : int {
  kResFull = 0,
  kResEmpty,
  kStrFull,
  kStrEmpty = kStrFull + kNS,
  kSyFull = kStrEmpty + kNS,  // the step's two score MMAs completed
  kXReady,                    // [2, by step parity] the compute warps wrote the step's bf16 operands
                              // (in mode DQ the next step's scores go out before this step's
                              // operands are consumed, so the compute warps may finish a whole step
                              // ahead of the issuer's wait; with one barrier per parity a barrier
                              // cannot complete twice before its wait)
  kDpFree = kXReady + 2,      // DQ: the compute warps loaded the step's dP
  kAccFull,                   // the item's last accumulating MMA completed
  kAccEmpty,                  // the compute warps read the accumulators
  kGroup,                     // DKV: barrier of the 128 compute threads
  kItemFull,                  // [2] the producer published an item descriptor
  kItemEmpty = kItemFull + 2, // [2] the MMA issuer and the compute warps copied it
  kMmaDone = kItemEmpty + 2,
  kNumBars
};

// The ready barrier of step `step` (a stream-wide step count) and its wait parity.
__host__ __device__ constexpr int xready(uint32_t step) { return kXReady + (int)(step & 1u); }
__host__ __device__ constexpr uint32_t xready_parity(uint32_t step) { return (step >> 1) & 1u; }

// Byte offsets from the 1024-aligned base of dynamic shared memory.
constexpr int kRowB = kTile * 8;  // {-lse2, -D} of a tile's rows, paired (row_neg_lse2 / row_neg_d)
template <int D>
struct BL {
  static constexpr int kTileBytes = BCfg<D>::kTileBytes;
  static constexpr int kRes = 0;                             // [2] resident tiles
  static constexpr int kStr = kRes + 2 * kTileBytes;         // [kNS][2] streamed tiles
  static constexpr int kSRec = kStr + 2 * kNS * kTileBytes;  // [kNS] records of the streamed tiles
  static constexpr int kSRow = kSRec + kNS * kStageRecB;     // DKV: [kNS] row constants of the query tiles
  static constexpr int kRRec = kSRow + kNS * kRowB;          // record of the item's tile
  static constexpr int kRRow = kRRec + kRecB;                // DQ: row constants of the query tile
  static constexpr int kCol = kRRow + kRowB;                 // DKV: [2][128 keys] 128 query bits
  static constexpr int kItems = kCol + 2 * kTile * 16;       // [2] published item descriptors
  static constexpr int kBarsOff = kItems + 2 * 64;
  static constexpr int kTotal = kBarsOff + kNumBars * 8 + 16;  // + abort flag and TMEM slot
  static constexpr int kDynamic = kTotal + 1024;               // slack to align the base
};
static_assert(BL<64>::kSRec % 16 == 0 && BL<64>::kSRow % 16 == 0 && BL<64>::kRRec % 16 == 0 &&
                  BL<64>::kRRow % 16 == 0 && BL<64>::kCol % 16 == 0 && BL<128>::kSRec % 16 == 0 &&
                  BL<128>::kSRow % 16 == 0 && BL<128>::kRRec % 16 == 0 && BL<128>::kRRow % 16 == 0 &&
                  BL<128>::kCol % 16 == 0,
              "bulk-copy alignment");
static_assert(BL<64>::kBarsOff % 8 == 0 && BL<128>::kBarsOff % 8 == 0, "mbarrier alignment");
static_assert(2 * (BL<64>::kDynamic + 1024) <= 228 * 1024, "two CTAs per SM at d = 64");
static_assert(BL<128>::kDynamic <= 227 * 1024, "one CTA per SM at d = 128");

__device__ __forceinline__ bool bw_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
  return bounded_wait(bar, parity, abort_flag, status, kWaitNsB);
}
__device__ __forceinline__ bool bw_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             int* status) {
  const bool ok = bw_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void bw_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > kWaitNsB / 4) return;
}

// A published item: its descriptor (as three 16-byte words) and the end flag.
struct ItemSlot {
  uint4 d[3];
  int end;
  int pad[3];
};
static_assert(sizeof(ItemSlot) == 64, "");

__device__ __forceinline__ BwdItemDesc unpack_desc(const uint4 (&nx)[3]) {
  BwdItemDesc d;
  d.tok_start = (long long)(((unsigned long long)nx[0].y << 32) | nx[0].x);
  d.t_ref = (long long)(((unsigned long long)nx[0].w << 32) | nx[0].z);
  d.list = (long long)(((unsigned long long)nx[1].y << 32) | nx[1].x);
  d.len = (int)nx[1].z;
  d.tile = (int)nx[1].w;
  d.tile_start = (int)nx[2].x;
  d.h = (int)nx[2].y;
  d.n = (int)nx[2].z;
  d.pad = 0;
  return d;
}

// Consumer side of the item slots: the next item's descriptor, or false at the end
// (or after an abort).  warp_arrive: the compute warps arrive once per warp.
template <int D>
__device__ __forceinline__ bool next_item(uint8_t* sm, uint64_t* bars, uint32_t& it_cnt, bool warp_arrive,
                                          BwdItemDesc& d, volatile int* abort_flag, int* status) {
  const int slot = (int)(it_cnt & 1);
  const uint32_t ph = (it_cnt >> 1) & 1;
  ++it_cnt;
  const bool ok = warp_arrive ? bw_wait_warp(bars + kItemFull + slot, ph, abort_flag, status)
                              : bw_wait(bars + kItemFull + slot, ph, abort_flag, status);
  if (!ok) return false;
  const ItemSlot* is = reinterpret_cast<const ItemSlot*>(sm + BL<D>::kItems) + slot;
  const uint4 nx[3] = {is->d[0], is->d[1], is->d[2]};
  const int end = is->end;
  if (warp_arrive) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bars + kItemEmpty + slot);
  } else {
    ptx::mbar_arrive(bars + kItemEmpty + slot);
  }
  if (end) return false;
  d = unpack_desc(nx);
  return true;
}

// The streamed tiles of an item, in order: request-local tile index, class and
// mask-table slot (-1: none).
struct Cursor {
  const uint32_t* list;
  const int* slots;
  int r;
  __device__ __forceinline__ void init(const uint32_t* base, const int* slot_base, const BwdItemDesc& d) {
    list = base + d.list;
    slots = slot_base + d.list;
    r = 0;
  }
  __device__ __forceinline__ void next(int& tile, int& cls, int& slot) {
    const uint32_t e = list[r];
    slot = slots[r];
    ++r;
    tile = (int)(e & 0xffffffu);
    cls = (int)(e >> 24);
  }
};

// ------------------------------------------------------------------ producer
// maps: resident pair res[0], res[1]; streamed pair str[0], str[1].
//   DQ:  resident Q', dO + the query tile's record and row constants; streamed K', V
//        (+ the key tile's record when the tile is PARTIAL).
//   DKV: resident K', V + the key tile's record; streamed Q', dO + the query tile's
//        record and row constants.
template <int D, bool DKV>
__device__ void bwd_producer(const BwdArgs& a, const void* const (&res)[2], const void* const (&str)[2],
                             uint8_t* sm, uint64_t* bars, volatile int* abort_flag) {
  const uint32_t* lists = DKV ? a.qlist : a.klist;
  uint32_t it_n = 0, s_it = 0, it_cnt = 0;
  bool res_used = false, str_used[kNS];
  uint32_t res_ph = 0, str_ph[kNS];
  for (int i = 0; i < kNS; ++i) { str_used[i] = false; str_ph[i] = 0; }
  const uint4* descs = reinterpret_cast<const uint4*>(a.desc + (DKV ? a.n_items : 0));
  using L = BL<D>;
  constexpr int kTileBytes = L::kTileBytes;
  ItemSlot* slots = reinterpret_cast<ItemSlot*>(sm + L::kItems);
  int* counter = a.counters + (DKV ? 5 : 3);
  for (;;) {
    const long long w = atomicAdd(counter, 1);
    const int slot = (int)(it_cnt & 1);
    if (!bw_wait(bars + kItemEmpty + slot, ((it_cnt >> 1) & 1) ^ 1, abort_flag, a.status)) goto drain;
    ++it_cnt;
    if (w >= a.n_items) {
      slots[slot].end = 1;
      ptx::mbar_arrive(bars + kItemFull + slot);
      break;
    }
    uint4 nx[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) nx[k] = descs[3 * w + k];
#pragma unroll
    for (int k = 0; k < 3; ++k) slots[slot].d[k] = nx[k];
    slots[slot].end = 0;
    ptx::mbar_arrive(bars + kItemFull + slot);  // release: the slot's contents reach the waiters
    const BwdItemDesc d = unpack_desc(nx);
    if (d.n <= 0) continue;

    if (!bw_wait(bars + kResEmpty, (it_n & 1) ^ 1, abort_flag, a.status)) goto drain;
    {
      const int x = d.h * D;
      const long long g = (long long)d.tile_start + d.tile;
      const float2* rows_h = a.rowc + (long long)d.h * a.n_tiles * kTile;  // head h's row constants
      ptx::mbar_arrive_expect_tx(bars + kResFull, 2 * kTileBytes + kRecB + (DKV ? 0 : kRowB));
      const int y = (int)(d.tok_start + (long long)d.tile * kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        ptx::tma_load_2d(sm + L::kRes + c * kSlab, res[0], x + 64 * c, y, bars + kResFull);
        ptx::tma_load_2d(sm + L::kRes + kTileBytes + c * kSlab, res[1], x + 64 * c, y, bars + kResFull);
      }
      ptx::bulk_load(sm + L::kRRec, a.krec + g, kRecB, bars + kResFull);
      if (!DKV) ptx::bulk_load(sm + L::kRRow, rows_h + g * kTile, kRowB, bars + kResFull);
      res_used = true;
      res_ph = it_n & 1;
      ++it_n;
      Cursor cur;
      cur.init(lists, DKV ? a.qslot : a.kslot, d);
      for (int j = 0; j < d.n; ++j) {
        int tile, cls, tslot;
        cur.next(tile, cls, tslot);
        const int st = (int)(s_it % kNS);
        const uint32_t ph = (s_it / kNS) & 1;
        if (!bw_wait(bars + kStrEmpty + st, ph ^ 1, abort_flag, a.status)) goto drain;
        const long long gs = (long long)d.tile_start + tile;
        // PARTIAL tiles with a mask-table slot: the tile's rows (DQ) or columns (DKV) of the
        // table; otherwise DQ reads the key record on PARTIAL tiles, DKV the query record
        const bool tab = cls != REC_ATTN_TILE_FULL && tslot >= 0;
        const bool rec = !tab && (DKV || cls != REC_ATTN_TILE_FULL);
        const int ys = (int)(d.tok_start + (long long)tile * kTile);
        ptx::mbar_arrive_expect_tx(bars + kStrFull + st,
                                   2 * kTileBytes + (tab ? kMaskB : rec ? kRecB : 0) + (DKV ? kRowB : 0));
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          ptx::tma_load_2d(sm + L::kStr + (2 * st) * kTileBytes + c * kSlab, str[0], x + 64 * c, ys,
                           bars + kStrFull + st);
          ptx::tma_load_2d(sm + L::kStr + (2 * st + 1) * kTileBytes + c * kSlab, str[1], x + 64 * c, ys,
                           bars + kStrFull + st);
        }
        if (tab)
          ptx::bulk_load(sm + L::kSRec + st * kStageRecB, (DKV ? a.ctab : a.mtab) + (long long)tslot * (kMaskB / 4),
                         kMaskB, bars + kStrFull + st);
        else if (rec)
          ptx::bulk_load(sm + L::kSRec + st * kStageRecB, a.krec + gs, kRecB, bars + kStrFull + st);
        if (DKV) ptx::bulk_load(sm + L::kSRow + st * kRowB, rows_h + gs * kTile, kRowB, bars + kStrFull + st);
        str_used[st] = true;
        str_ph[st] = ph;
        ++s_it;
      }
    }
  }
drain:
  // every copy issued must land before the CTA exits (only waits after an abort)
  if (res_used) bw_drain(bars + kResFull, res_ph);
  for (int i = 0; i < kNS; ++i)
    if (str_used[i]) bw_drain(bars + kStrFull + i, str_ph[i]);
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return ptx::smem_desc_sw128(addr, 16, 1024); }
// MN-major operand: 64-column blocks of N one slab apart
__device__ __forceinline__ uint64_t mndesc(uint32_t addr) { return ptx::smem_desc_sw128(addr, kSlab, 1024); }

// Scores over K = D (both operands K-major, the K steps of 16 columns four per slab;
// B = 64 rows of a tile): N = 64.
template <int D>
__device__ __forceinline__ void mma_scores(uint32_t d, uint32_t a_addr, uint32_t b_addr) {
  constexpr uint32_t id = ptx::idesc_bf16_f32(kTile, kStep, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
    ptx::umma_f16(d, kdesc(a_addr + off), kdesc(b_addr + off), id, kk > 0);
  }
}
// D (+)= A B with A (128 x 64, bf16) in TMEM and B = 64 rows of a tile as the K
// dimension (MN-major: the tile's D columns are N).
template <int D>
__device__ __forceinline__ void mma_acc(uint32_t d, uint32_t a_tmem, uint32_t b_rows, bool accumulate) {
  constexpr uint32_t id = ptx::idesc_bf16_f32(kTile, D, false, true);
#pragma unroll
  for (int kk = 0; kk < kStep / 16; ++kk)
    ptx::umma_f16_ts(d, a_tmem + kk * 8, mndesc(b_rows + kk * 16 * 128), id, (accumulate || kk > 0) ? 1u : 0u);
}

template <int D, bool DKV>
__device__ void bwd_mma(const BwdArgs& a, uint8_t* sm, uint64_t* bars, uint32_t tmem, volatile int* abort_flag) {
  using L = BL<D>;
  using C = BCfg<D>;
  constexpr int kTileBytes = L::kTileBytes;
  const uint32_t res0 = ptx::smem_u32(sm + L::kRes), res1 = res0 + kTileBytes;
  const uint32_t str = ptx::smem_u32(sm + L::kStr);
  constexpr uint32_t kHalfBytes = kStep * 128;  // 64 rows of a tile
  uint32_t it_n = 0, s_it = 0, step = 0, it_cnt = 0;
  BwdItemDesc it;
  while (next_item<D>(sm, bars, it_cnt, false, it, abort_flag, a.status)) {
    if (it.n <= 0) continue;
    if (!bw_wait(bars + kResFull, it_n & 1, abort_flag, a.status)) goto out;
    ptx::tc_fence_after();
    {
      const uint32_t ii = it_n++;
      const int nsteps = 2 * it.n;
      const uint32_t step0 = step;
      // the streamed stage of local step ls; waits for it on the tile's first step
      auto stage_of = [&](int ls, bool wait_full, int& st) -> bool {
        const uint32_t sj = s_it + (uint32_t)(ls >> 1);
        st = (int)(sj % kNS);
        if (wait_full && (ls & 1) == 0) {
          if (!bw_wait(bars + kStrFull + st, (sj / kNS) & 1, abort_flag, a.status)) return false;
          ptx::tc_fence_after();
        }
        return true;
      };
      // the first accumulating MMA of an item overwrites the accumulators: the compute
      // warps must have read the previous item's
      auto acc_free = [&]() -> bool {
        if (ii == 0) return true;
        if (!bw_wait(bars + kAccEmpty, (ii - 1) & 1, abort_flag, a.status)) return false;
        ptx::tc_fence_after();
        return true;
      };
      if constexpr (!DKV) {
        // S(ls) = Q' K'_h^T into S buffer (step0 + ls) % 2, dP(ls) = dO V_h^T.  dP(ls + 1)
        // goes out as soon as the compute warps have loaded dP(ls), so both scores of
        // the next step are ready when this step's compute ends.
        auto issue_scores = [&](int ls) -> bool {
          int st;
          if (!stage_of(ls, true, st)) return false;
          const uint32_t half = (uint32_t)(ls & 1) * kHalfBytes;
          mma_scores<D>(tmem + ((step0 + ls) & 1) * kStep, res0, str + (2 * st) * kTileBytes + half);
          mma_scores<D>(tmem + 128, res1, str + (2 * st + 1) * kTileBytes + half);
          ptx::umma_commit(bars + kSyFull);
          if (ls == nsteps - 1) ptx::umma_commit(bars + kResEmpty);  // Q' and dO read for the last time
          return true;
        };
        if (!issue_scores(0)) goto out;
        for (int ls = 0; ls < nsteps; ++ls) {
          int st;
          stage_of(ls, false, st);
          if (ls + 1 < nsteps) {
            if (!bw_wait(bars + kDpFree, (step0 + ls) & 1, abort_flag, a.status)) goto out;
            ptx::tc_fence_after();
            if (!issue_scores(ls + 1)) goto out;
          }
          if (!bw_wait(bars + xready(step0 + ls), xready_parity(step0 + ls), abort_flag, a.status)) goto out;
          ptx::tc_fence_after();
          if (ls == 0 && !acc_free()) goto out;
          const uint32_t kb = str + (2 * st) * kTileBytes + (ls & 1) * kHalfBytes;
          mma_acc<D>(tmem + C::kDQ, tmem + ((step0 + ls) & 1) * kStep, kb, ls > 0);  // dQ += dS K'_h
          if (ls & 1) ptx::umma_commit(bars + kStrEmpty + st);
        }
      } else {
        // S^T = K' Q'_h^T and dP^T = V dO_h^T
        auto issue_scores = [&](int ls) -> bool {
          int st;
          if (!stage_of(ls, true, st)) return false;
          mma_scores<D>(tmem + 0, res0, str + (2 * st) * kTileBytes + (ls & 1) * kHalfBytes);
          mma_scores<D>(tmem + 64, res1, str + (2 * st + 1) * kTileBytes + (ls & 1) * kHalfBytes);
          ptx::umma_commit(bars + kSyFull);
          if (ls == nsteps - 1) ptx::umma_commit(bars + kResEmpty);  // K' and V read for the last time
          return true;
        };
        if (!issue_scores(0)) goto out;
        for (int ls = 0; ls < nsteps; ++ls) {
          int st;
          stage_of(ls, false, st);
          if (!bw_wait(bars + xready(step0 + ls), xready_parity(step0 + ls), abort_flag, a.status)) goto out;
          ptx::tc_fence_after();
          if (ls == 0 && !acc_free()) goto out;
          const uint32_t qb = str + (2 * st) * kTileBytes + (ls & 1) * kHalfBytes;
          const uint32_t ob = str + (2 * st + 1) * kTileBytes + (ls & 1) * kHalfBytes;
          mma_acc<D>(tmem + C::kDV, tmem + 0, ob, ls > 0);   // dV += P^T dO_h
          mma_acc<D>(tmem + C::kDK, tmem + 64, qb, ls > 0);  // dK += dS^T Q'_h
          if (ls & 1) ptx::umma_commit(bars + kStrEmpty + st);
          if (ls + 1 < nsteps && !issue_scores(ls + 1)) goto out;
        }
      }
      step += (uint32_t)nsteps;
      s_it += (uint32_t)it.n;
      ptx::umma_commit(bars + kAccFull);
    }
  }
out:
  // all issued MMAs must complete before TMEM is released
  ptx::umma_commit(bars + kMmaDone);
  bw_drain(bars + kMmaDone, 0);
}

// ------------------------------------------------------------------ compute warps
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// fp32 pairs for the f32x2 instructions (one instruction for two columns)
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f2add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// The row-constant table of one tile (128 rows): rows 2k and 2k+1 share 16 bytes,
// {-lse2(2k), -lse2(2k+1), -D(2k), -D(2k+1)}, with lse2 = lse * log2(e).
__device__ __forceinline__ float row_neg_lse2(const float* tab, int r) { return tab[(r >> 1) * 4 + (r & 1)]; }
__device__ __forceinline__ float row_neg_d(const float* tab, int r) { return tab[(r >> 1) * 4 + 2 + (r & 1)]; }

// 32 words (64 bf16, one 128-byte row piece) to global memory: 32-byte stores when the
// gradient buffers are 32-byte aligned (each store then fills whole sectors; the rows of
// a warp lie H * d * 2 bytes apart), else 16-byte stores.
__device__ __forceinline__ void st_words(void* dst, const uint32_t (&w)[32], bool wide) {
  if (wide) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      ptx::st_global_v8(static_cast<char*>(dst) + 32 * c, w[8 * c], w[8 * c + 1], w[8 * c + 2], w[8 * c + 3],
                        w[8 * c + 4], w[8 * c + 5], w[8 * c + 6], w[8 * c + 7]);
  } else {
    uint4* d4 = static_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  }
}

// One output row: x * scale, then (rotate) R(dt)^T over adjacent pairs, as bf16.  The
// angles (at most a few tens of radians) take the hardware sine and cosine: their
// error, about 1e-5 rad here, is far below the bf16 rounding of the result.
// (64 columns of a row at dst; omega: their 32 rotation pairs)
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const uint32_t (&acc)[64], float scale, bool rotate,
                                         float dt, const float* omega, bool wide) {
  uint32_t w[32];
#pragma unroll
  for (int p = 0; p < 32; ++p) {
    float u = __uint_as_float(acc[2 * p]) * scale, v = __uint_as_float(acc[2 * p + 1]) * scale;
    if (rotate) {
      float sn, cs;
      __sincosf(dt * omega[p], &sn, &cs);
      const float u2 = u * cs + v * sn;
      v = -u * sn + v * cs;
      u = u2;
    }
    w[p] = bf16x2(u, v);
  }
  st_words(dst, w, wide);
}

template <int D>
__device__ __forceinline__ void zero_row(__nv_bfloat16* dst) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
}

// A row's time and type from a tile record (type -1 past the request end).
__device__ __forceinline__ void rec_row(const KeyTileRec* rec, int row, long long& t, int& ty) {
  t = rec->t[row];
  ty = -1;
#pragma unroll
  for (int c = 0; c < kTypes; ++c)
    if ((rec->typebits[c][row >> 5] >> (row & 31)) & 1u) ty = c;
}

// DQ: thread = query row of the item's tile.
template <int D>
__device__ void bwd_compute_dq(const BwdArgs& a, uint8_t* sm, uint64_t* bars, uint32_t tmem,
                               volatile int* abort_flag) {
  using BL = recattn::BL<D>;
  const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3, row = quad * 32 + lane;
  const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
  const float sl2 = a.scale * kLog2e;
  const uint8_t* sstage = sm + BL::kSRec;  // per stage: key record or mask-table rows
  const KeyTileRec* rrec = reinterpret_cast<const KeyTileRec*>(sm + BL::kRRec);
  const float* rrow = reinterpret_cast<const float*>(sm + BL::kRRow);
  const int H = a.heads;
  const unsigned long long sl2x2 = f2pack(sl2, sl2);
  const bool wide = (reinterpret_cast<uintptr_t>(a.dq) & 31) == 0;  // row pieces 32-byte aligned
  uint32_t it_n = 0, s_it = 0, step = 0, it_cnt = 0;
  BwdItemDesc it;
  while (next_item<D>(sm, bars, it_cnt, true, it, abort_flag, a.status)) {
    const int pi = it.tile * kTile + row;
    const bool row_ok = pi < it.len;
    const long long tok = it.tok_start + pi, grow = tok * H + it.h;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + grow * D;
    if (it.n <= 0) {  // no visible key tile
      if (row_ok) zero_row<D>(dst);
      continue;
    }
    // the row's time, type and constants, loaded with Q'
    if (!bw_wait_warp(bars + kResFull, it_n & 1, abort_flag, a.status)) return;
    long long ti;
    int tyi;
    rec_row(rrec, row, ti, tyi);
    const float nl = row_neg_lse2(rrow, row), nd = row_neg_d(rrow, row);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bars + kResEmpty);
    // a row that sees no key contributes nothing: its P is exp2(s - inf) = 0, so FULL
    // tiles need no mask for it
    const bool live = row_ok && nl != INFINITY;
    const unsigned long long nl2 = f2pack(live ? nl : -INFINITY, live ? nl : -INFINITY), nd2 = f2pack(nd, nd);
    RowMask rm;
    row_mask_setup(a.mask, live, pi, ti, tyi, rm);
    Cursor cur;
    cur.init(a.klist, a.kslot, it);
    for (int j = 0; j < it.n; ++j) {
      int kt, cls, tslot;
      cur.next(kt, cls, tslot);
      const int st = (int)(s_it % kNS);
      const uint32_t ph = (s_it / kNS) & 1;
      ++s_it;
      const uint32_t f = live ? ~0u : 0u;
      uint32_t vm[4] = {f, f, f, f};
      if (cls != REC_ATTN_TILE_FULL) {
        if (!bw_wait_warp(bars + kStrFull + st, ph, abort_flag, a.status)) return;
        if (tslot >= 0) {  // the row's words of the mask table (zero for rows that see no key)
          const uint4 w = reinterpret_cast<const uint4*>(sstage + st * kStageRecB)[row];
          vm[0] = w.x; vm[1] = w.y; vm[2] = w.z; vm[3] = w.w;
        } else {
          build_mask(rm, reinterpret_cast<const KeyTileRec*>(sstage + st * kStageRecB), kt * kTile, vm);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + kStrEmpty + st);  // the stage's record was read
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh, ++step) {
        if (!bw_wait_warp(bars + kSyFull, step & 1, abort_flag, a.status)) return;
        ptx::tc_fence_after();
        const uint32_t sb = tl + (step & 1) * kStep;
        const uint32_t wb[2] = {hh ? vm[2] : vm[0], hh ? vm[3] : vm[1]};  // this step's 64 keys
        // dP of both chunks and S of the first, then dP's columns go back to the MMA issuer
        uint32_t d[64], sr[32], pk[16];
        ptx::tmem_ld32x2_async(tl + 128, tl + 160, d);
        ptx::tmem_ld32_async(sb, sr);
        ptx::tmem_wait_ld(d);
        ptx::tmem_wait_ld32(sr);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + kDpFree);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (c == 1) {
            ptx::tmem_ld32_async(sb + 32, sr);
            ptx::tmem_wait_ld32(sr);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float y0, y1;
            f2unpack(f2fma(f2pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), sl2x2, nl2), y0, y1);
            float p0 = ex2(y0), p1 = ex2(y1);
            if (cls != REC_ATTN_TILE_FULL) {
              p0 = ((wb[c] >> (2 * e)) & 1u) ? p0 : 0.f;
              p1 = ((wb[c] >> (2 * e + 1)) & 1u) ? p1 : 0.f;
            }
            float g0, g1;
            f2unpack(f2mul(f2pack(p0, p1), f2add(f2pack(__uint_as_float(d[32 * c + 2 * e]),
                                                        __uint_as_float(d[32 * c + 2 * e + 1])), nd2)), g0, g1);
            pk[e] = bf16x2(g0, g1);
          }
          ptx::tmem_st16_async(sb + 16 * c, pk);  // dS over S columns already read
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + xready(step));
      }
    }
    if (!bw_wait_warp(bars + kAccFull, it_n & 1, abort_flag, a.status)) return;
    ++it_n;
    ptx::tc_fence_after();
    if constexpr (D == 64) {
      uint32_t acc[64];
      ptx::tmem_ld64(tl + BCfg<D>::kDQ, acc);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + kAccEmpty);
      if (row_ok) store_row(dst, acc, a.scale, a.rotate != 0, (float)(ti - it.t_ref), a.omega, wide);
    } else {
#pragma unroll 1
      for (int hc = 0; hc < D / 64; ++hc) {
        uint32_t acc[64];
        ptx::tmem_ld64(tl + BCfg<D>::kDQ + 64 * hc, acc);
        if (hc == D / 64 - 1) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bars + kAccEmpty);
        }
        if (row_ok)
          store_row(dst + 64 * hc, acc, a.scale, a.rotate != 0, (float)(ti - it.t_ref), a.omega + 32 * hc, wide);
      }
    }
  }
}

// Transpose of the 32 x 32 bit matrix held one row per lane: afterwards lane b holds
// bit l = bit b of lane l's input.  Five rounds swap the off-diagonal blocks of width
// 16, 8, 4, 2 and 1 between lanes l and l ^ j.
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint32_t m = j == 16 ? 0x0000ffffu : j == 8 ? 0x00ff00ffu : j == 4 ? 0x0f0f0f0fu : j == 2 ? 0x33333333u : 0x55555555u;
    const uint32_t p = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) ? ((x & ~m) | ((p & ~m) >> j)) : ((x & m) | ((p & m) << j));
  }
  return x;
}

// The 128 compute threads meet (bounded); `n` counts the uses of the barrier.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& n, volatile int* abort_flag, int* status) {
  ptx::mbar_arrive(bar);
  return bw_wait_warp(bar, (n++) & 1, abort_flag, status);
}

// DKV: thread = key row of the item's tile (and, while the masks are built, a row of
// the query tile).  The column bits of the next query tile are built while the tensor
// core runs the second half of the current one (two buffers of column bits).
template <int D>
__device__ void bwd_compute_dkv(const BwdArgs& a, uint8_t* sm, uint64_t* bars, uint32_t tmem,
                                volatile int* abort_flag) {
  using BL = recattn::BL<D>;
  const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3, row = quad * 32 + lane;
  const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
  const float sl2 = a.scale * kLog2e;
  const KeyTileRec* rrec = reinterpret_cast<const KeyTileRec*>(sm + BL::kRRec);
  const uint8_t* sstage = sm + BL::kSRec;  // per stage: query record or mask-table columns
  const float* srow = reinterpret_cast<const float*>(sm + BL::kSRow);
  const unsigned long long sl2x2 = f2pack(sl2, sl2);
  const bool wide = ((reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) & 31) == 0;
  uint32_t* colS = reinterpret_cast<uint32_t*>(sm + BL::kCol);
  const int H = a.heads;
  uint32_t it_n = 0, s_it = 0, step = 0, grp = 0, cbuf = 0, it_cnt = 0;
  BwdItemDesc it;
  while (next_item<D>(sm, bars, it_cnt, true, it, abort_flag, a.status)) {
    const int pj = it.tile * kTile + row;
    const bool key_ok = pj < it.len;
    const long long growk = (it.tok_start + pj) * H + it.h;
    __nv_bfloat16* dkr = static_cast<__nv_bfloat16*>(a.dk) + growk * D;
    __nv_bfloat16* dvr = static_cast<__nv_bfloat16*>(a.dv) + growk * D;
    if (it.n <= 0) {  // no query sees this key tile
      if (key_ok) { zero_row<D>(dkr); zero_row<D>(dvr); }
      continue;
    }
    if (!bw_wait_warp(bars + kResFull, it_n & 1, abort_flag, a.status)) return;  // the key tile's record
    const long long tj = rrec->t[row];
    Cursor cur;
    cur.init(a.qlist, a.qslot, it);
    // Column bits of the item's j-th query tile (stage st) into buffer `buf`: the key's
    // words of the mask table's columns when the pair has a slot; otherwise, as query
    // row `row` of the tile, this thread builds the row's bits over the key tile and
    // each warp transposes its 32 rows into per-key words.
    auto prepare = [&](int j, int qt, int cls, int tslot, int st, uint32_t ph, uint32_t buf) -> bool {
      if (!bw_wait_warp(bars + kStrFull + st, ph, abort_flag, a.status)) return false;
      // after the item's last read of the key tile's record, its buffer may be refilled
      auto release_rec = [&]() {
        if (j == it.n - 1) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bars + kResEmpty);
        }
      };
      if (cls == REC_ATTN_TILE_FULL) {  // the steps of a FULL tile apply no mask
        release_rec();
        return true;
      }
      if (tslot >= 0) {
        reinterpret_cast<uint4*>(colS + buf * (kTile * 4))[row] =
            reinterpret_cast<const uint4*>(sstage + st * kStageRecB)[row];
        release_rec();
        return true;
      }
      const int qi = qt * kTile + row;
      long long tq;
      int tyq;
      rec_row(reinterpret_cast<const KeyTileRec*>(sstage + st * kStageRecB), row, tq, tyq);
      const bool live = qi < it.len && row_neg_lse2(srow + st * 2 * kTile, row) != INFINITY;
      const uint32_t f = live ? ~0u : 0u;
      uint32_t vm[4] = {f, f, f, f};
      RowMask rm;
      row_mask_setup(a.mask, live, qi, tq, tyq, rm);
      build_mask(rm, rrec, it.tile * kTile, vm);
      release_rec();
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) colS[buf * (kTile * 4) + (32 * wd + lane) * 4 + quad] = transpose32(vm[wd], lane);
      return true;
    };
    int qt, cls, tslot;
    cur.next(qt, cls, tslot);
    int scls = cls;  // the class of the query tile the steps run on
    int st = (int)(s_it % kNS);
    if (!prepare(0, qt, cls, tslot, st, (s_it / kNS) & 1, cbuf)) return;
    ++s_it;
    for (int j = 0; j < it.n; ++j) {
      // every thread's words of this tile are written, and every thread has read the
      // other buffer's (a tile ago), which prepare() overwrites next
      if (!group_sync(bars + kGroup, grp, abort_flag, a.status)) return;
      const uint4 cm = reinterpret_cast<const uint4*>(colS)[cbuf * kTile + row];
      const float* rows = srow + st * 2 * kTile;
      int nqt = 0, ncls = 0, nslot = -1, nst = 0;
      uint32_t nph = 0;
      if (j + 1 < it.n) {
        cur.next(nqt, ncls, nslot);
        nst = (int)(s_it % kNS);
        nph = (s_it / kNS) & 1;
        ++s_it;
      }
      // one 64-query step: P^T and dS^T over the scores' TMEM columns
      auto do_step = [&](int hh) -> bool {
        if (!bw_wait_warp(bars + kSyFull, step & 1, abort_flag, a.status)) return false;
        ++step;
        ptx::tc_fence_after();
        const uint32_t wb[2] = {hh ? cm.z : cm.x, hh ? cm.w : cm.y};  // this step's 64 queries
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t r[64], pk[16];
          ptx::tmem_ld32x2_async(tl + 32 * c, tl + 64 + 32 * c, r);
          // {-lse2, -D} of the chunk's 32 queries, a pair per 16-byte load (broadcast)
          const float4* q4 = reinterpret_cast<const float4*>(rows + (hh * kStep + c * 32) * 2);
          const uint32_t bits = wb[c];
          ptx::tmem_wait_ld(r);
          float p[32];
#pragma unroll
          for (int g = 0; g < 16; ++g) {
            const float4 k2 = q4[g];
            float x0, x1;
            f2unpack(f2fma(f2pack(__uint_as_float(r[2 * g]), __uint_as_float(r[2 * g + 1])), sl2x2,
                           f2pack(k2.x, k2.y)), x0, x1);
            x0 = ex2(x0);
            x1 = ex2(x1);
            if (scls != REC_ATTN_TILE_FULL) {  // FULL: queries past the request end have -lse2 = -inf
              x0 = ((bits >> (2 * g)) & 1u) ? x0 : 0.f;
              x1 = ((bits >> (2 * g + 1)) & 1u) ? x1 : 0.f;
            }
            p[2 * g] = x0;
            p[2 * g + 1] = x1;
            pk[g] = bf16x2(x0, x1);
          }
          ptx::tmem_st16_async(tl + 16 * c, pk);  // P^T over S^T columns already read
#pragma unroll
          for (int g = 0; g < 16; ++g) {
            const float4 k2 = q4[g];
            float g0, g1;
            f2unpack(f2mul(f2pack(p[2 * g], p[2 * g + 1]),
                           f2add(f2pack(__uint_as_float(r[32 + 2 * g]), __uint_as_float(r[32 + 2 * g + 1])),
                                 f2pack(k2.z, k2.w))), g0, g1);
            pk[g] = bf16x2(g0, g1);
          }
          ptx::tmem_st16_async(tl + 64 + 16 * c, pk);  // dS^T over dP^T columns already read
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + xready(step - 1));  // step was counted on at the wait
        return true;
      };
      if (!do_step(0)) return;
      if (j + 1 < it.n && !prepare(j + 1, nqt, ncls, nslot, nst, nph, cbuf ^ 1u)) return;
      if (!do_step(1)) return;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + kStrEmpty + st);  // the stage's record and constants were read
      st = nst;
      scls = ncls;
      cbuf ^= 1u;
    }
    if (!bw_wait_warp(bars + kAccFull, it_n & 1, abort_flag, a.status)) return;
    ++it_n;
    ptx::tc_fence_after();
    // 64 columns at a time: dV packed and stored, then dK scaled, rotated back and stored
#pragma unroll 1
    for (int hc = 0; hc < D / 64; ++hc) {
      uint32_t acc[64], wv[32];
      ptx::tmem_ld64(tl + BCfg<D>::kDV + 64 * hc, acc);  // dV, packed before dK is read
#pragma unroll
      for (int p = 0; p < 32; ++p) wv[p] = bf16x2(__uint_as_float(acc[2 * p]), __uint_as_float(acc[2 * p + 1]));
      ptx::tmem_ld64(tl + BCfg<D>::kDK + 64 * hc, acc);
      if (hc == D / 64 - 1) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + kAccEmpty);
      }
      if (key_ok) {
        st_words(dvr + 64 * hc, wv, wide);
        store_row(dkr + 64 * hc, acc, a.scale, a.rotate != 0, (float)(tj - it.t_ref), a.omega + 32 * hc, wide);
      }
    }
  }
}

// ------------------------------------------------------------------ row constants
// Block = (tile g, head h): D_i = <dO_i, O_i> for the tile's 128 rows, eight threads per
// row (16 bytes of dO and O each, coalesced), written negated with -lse * log2(e) into
// the tile-padded table, rows paired (row_neg_lse2 / row_neg_d).  lse2 is -inf for rows
// that see no key and +inf for rows past the request end and pruned rows, so that
// every P of the latter is exp2(s - inf) = 0 whatever mask bits they have.
template <int D>
__global__ void __launch_bounds__(256) k_bwd_rowc(BwdArgs a) {
  constexpr int kLanes = D / 8;  // 16-byte chunks of a row, one per thread
  const long long g = blockIdx.x;
  const int h = blockIdx.y, H = a.heads;
  const int b = a.qreq[g];
  const ReqMeta m = a.meta[b];
  const int tile = (int)(g - m.tile_start);
  const int sub = threadIdx.x & (kLanes - 1);
  float* out = reinterpret_cast<float*>(a.rowc + ((long long)h * a.n_tiles + g) * kTile);
  const int keep = a.qkeep[b];
#pragma unroll 1
  for (int r = threadIdx.x / kLanes; r < kTile; r += 256 / kLanes) {
    const int p = tile * kTile + r;
    const bool in = p < m.len;
    // a pruned query (a query-pruned plan) has no output, so no gradient flows from it;
    // its forward lse and O were never written
    const bool ok = in && query_kept(a.ty[m.tok_start + p], p, keep);
    const long long row = (m.tok_start + p) * H + h;
    float acc = 0.f;
    if (ok) {
      const uint4 x = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) + row * D)[sub];
      const uint4 y = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.out) + row * D)[sub];
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[i]));
        const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[i]));
        acc = fmaf(fx.x, fy.x, fmaf(fx.y, fy.y, acc));
      }
    }
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (sub == 0) {
      const float l = ok ? a.lse[row] : INFINITY;
      out[(r >> 1) * 4 + (r & 1)] = -(l == -INFINITY ? -INFINITY : l * kLog2e);
      out[(r >> 1) * 4 + 2 + (r & 1)] = -acc;
    }
  }
}

// ------------------------------------------------------------------ schedule
// Threads [0, n_tiles): the transposed tile lists -- for key tile g, the query tiles
// of its request whose class against it is not SKIP, in order.  Threads
// [n_tiles, n_tiles + n_items): the descriptors of item w for both modes (DKV: the
// mirrored key tile of the item's query tile).
__global__ void __launch_bounds__(128) k_bwd_schedule(BwdSchedArgs s) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < s.n_tiles) {
    const ReqMeta m = s.meta[s.qreq[i]];
    const int kt = (int)(i - m.tile_start);
    uint32_t* out = s.qlist + m.cls_start + (long long)kt * m.ntiles;
    int* out_slot = s.qslot + m.cls_start + (long long)kt * m.ntiles;
    int n = 0;
    for (int qt = 0; qt < m.ntiles; ++qt) {
      const long long pair = m.cls_start + (long long)qt * m.ntiles + kt;
      const int c = s.cls[pair];
      if (c == REC_ATTN_TILE_SKIP) continue;
      out[n] = (uint32_t)qt | ((uint32_t)c << 24);
      const int p = c == REC_ATTN_TILE_PARTIAL ? s.pslot[pair] : -1;
      out_slot[n] = (p >= 0 && p < s.mcap) ? p : -1;  // a slot always indexes the table
      ++n;
    }
    return;
  }
  const long long w = i - s.n_tiles;
  if (w >= s.n_items) return;
  const long long e = s.items[w];
  const long long g = e / s.heads;
  const ReqMeta m = s.meta[s.qreq[g]];
  const int qt = (int)(g - m.tile_start), kt = m.ntiles - 1 - qt;
  BwdItemDesc d;
  d.tok_start = m.tok_start;
  d.t_ref = s.t[m.tok_start];
  d.len = m.len;
  d.tile_start = (int)m.tile_start;
  d.h = (int)(e % s.heads);
  d.pad = 0;
  d.list = m.cls_start + (long long)qt * m.ntiles;
  d.tile = qt;
  d.n = max(s.kcount[g], 0);
  s.desc[w] = d;
  const uint8_t* col = s.cls + m.cls_start + kt;
  int n = 0;
  for (int r = 0; r < m.ntiles; ++r) n += col[(long long)r * m.ntiles] != REC_ATTN_TILE_SKIP;
  d.list = m.cls_start + (long long)kt * m.ntiles;
  d.tile = kt;
  d.n = n;
  s.desc[s.n_items + w] = d;
}

// The mask table's columns (once per plan): per slot, each warp transposes its 32 query
// rows' words into per-key words, so key j of the tile finds the 128 query bits of its
// column as four words.
__global__ void __launch_bounds__(kTile) k_bwd_colmask(BwdSchedArgs s) {
  const int used = min(__ldcg(s.counters + 7), s.mcap);
  const int r = threadIdx.x, lane = r & 31, quad = r >> 5;
  for (int slot = blockIdx.x; slot < used; slot += gridDim.x) {
    const uint4 w = reinterpret_cast<const uint4*>(s.mtab)[(long long)slot * kTile + r];
    const uint32_t vm[4] = {w.x, w.y, w.z, w.w};
    uint32_t* out = s.ctab + (long long)slot * kTile * 4;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) out[(32 * wd + lane) * 4 + quad] = transpose32(vm[wd], lane);
  }
}

// ------------------------------------------------------------------ kernel
// maps: Q', K', V, dO, each a [T][H*64] bf16 view with 64 x 128 boxes.
template <int D, bool DKV>
__global__ void __launch_bounds__(kThreadsB, BCfg<D>::kBlocksPerSM)
    k_bwd_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using BL = recattn::BL<D>;
  constexpr uint32_t kCols = BCfg<D>::kCols;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BL::kBarsOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars) + 1;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bars + kResFull, 1);
    ptx::mbar_init(bars + kResEmpty, 1 + 4);  // MMAs done + the compute warps read the record
    for (int i = 0; i < kNS; ++i) {
      ptx::mbar_init(bars + kStrFull + i, 1);
      ptx::mbar_init(bars + kStrEmpty + i, 1 + 4);  // MMAs done + the compute warps read the record
    }
    ptx::mbar_init(bars + kSyFull, 1);
    for (int i = 0; i < 2; ++i) ptx::mbar_init(bars + kXReady + i, 4);
    ptx::mbar_init(bars + kDpFree, 4);
    ptx::mbar_init(bars + kAccFull, 1);
    ptx::mbar_init(bars + kAccEmpty, 4);
    ptx::mbar_init(bars + kGroup, 128);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bars + kItemFull + i, 1);
      ptx::mbar_init(bars + kItemEmpty + i, 1 + 4);  // the MMA issuer and the four compute warps
    }
    ptx::mbar_init(bars + kMmaDone, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) {
      const void* const res[2] = {DKV ? (const void*)&tm_k : (const void*)&tm_q,
                                  DKV ? (const void*)&tm_v : (const void*)&tm_do};
      const void* const str[2] = {DKV ? (const void*)&tm_q : (const void*)&tm_k,
                                  DKV ? (const void*)&tm_do : (const void*)&tm_v};
      bwd_producer<D, DKV>(a, res, str, sm, bars, abort_flag);
    }
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) bwd_mma<D, DKV>(a, sm, bars, tmem, abort_flag);
  } else {
    if constexpr (DKV) bwd_compute_dkv<D>(a, sm, bars, tmem, abort_flag);
    else bwd_compute_dq<D>(a, sm, bars, tmem, abort_flag);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kCols);
  }
  // the last CTA to leave resets the item counter for the next launch
  if (threadIdx.x == 0) {
    int* counter = a.counters + (DKV ? 5 : 3);
    __threadfence();
    if (atomicAdd(counter + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(counter, 0);
      atomicExch(counter + 1, 0);
    }
  }
}

template <int D, bool DKV>
cudaError_t launch_mode(const CUtensorMap (&maps)[4], const BwdArgs& a, int grid, cudaStream_t st) {
  cudaError_t e =
      cudaFuncSetAttribute(k_bwd_tc<D, DKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, BL<D>::kDynamic);
  if (e != cudaSuccess) return e;
  k_bwd_tc<D, DKV><<<grid, kThreadsB, BL<D>::kDynamic, st>>>(maps[0], maps[1], maps[2], maps[3], a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap (&maps)[4], int num_sms, cudaStream_t st) {
  k_bwd_rowc<D><<<dim3((unsigned)a.n_tiles, (unsigned)a.heads), 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long cap = (long long)BCfg<D>::kBlocksPerSM * num_sms;
  const int grid = (int)(a.n_items < cap ? a.n_items : cap);
  e = launch_mode<D, false>(maps, a, grid, st);
  if (e != cudaSuccess) return e;
  return launch_mode<D, true>(maps, a, grid, st);
}

}  // namespace

cudaError_t launch_bwd_schedule(const BwdSchedArgs& s, int num_sms, cudaStream_t st) {
  const long long n = s.n_tiles + s.n_items;
  if (n <= 0) return cudaSuccess;
  k_bwd_schedule<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || s.mcap <= 0) return e;
  k_bwd_colmask<<<s.mcap < 8 * num_sms ? s.mcap : 8 * num_sms, kTile, 0, st>>>(s);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_tc(const BwdArgs& a, const CUtensorMap (&maps)[4], int head_dim, int num_sms,
                               cudaStream_t st) {
  if (a.n_items <= 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch_bwd_d<64>(a, maps, num_sms, st);
    case 128: return launch_bwd_d<128>(a, maps, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace recattn
