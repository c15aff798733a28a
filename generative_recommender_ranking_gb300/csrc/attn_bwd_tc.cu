// attn_bwd_tc.cu -- backward pass of the masked time-RoPE attention on the sm_103a
// tensor cores (bf16 inputs and gradients, fp32 accumulation, head_dim 64).
//
// Gradients of O = Softmax(QK^T/sqrt(d) + M) V (TM20K review page, section 2.1;
// LazFormer review page, Eq. 19-21) through the time-RoPE (CADET review page, time
// encoding).  With P rebuilt from the forward's log-sum-exp, P_ij = exp(s_ij - lse_i)
// on visible pairs, D_i = <dO_i, O_i> and dS_ij = P_ij (dP_ij - D_i):
//   mode DQ:   dQ'_i = scale sum_j dS_ij K'_j
//   mode DKV:  dV_j = sum_i P_ij dO_i,  dK'_j = scale sum_i dS_ij Q'_i
// and dQ = R(t_i)^T dQ', dK = R(t_j)^T dK' (the rotation is orthogonal).
//
// Both modes share one persistent kernel shape: two CTAs per SM (256 TMEM columns
// each) and six warps -- warp 0 loads with TMA, one thread of warp 1 issues every MMA,
// warps 2..5 are the compute warpgroup (one TMEM lane, i.e. one tile row, per
// thread).  CTAs walk the planner's (tile, head) items with a static stride; mode DKV
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
// TMEM columns:  DQ   S[0] 0..63 | S[1] 64..127 | dP 128..191 | dQ 192..255
//                DKV  S^T 0..63 | dP^T 64..127 | dV 128..191 | dK 192..255
// The accumulators stay in TMEM across an item's tiles; the epilogue scales, undoes
// the rotation and writes bf16 rows.  PARTIAL tiles take the forward's per-row
// visibility bits (row_mask.cuh), built from the key tile's planner record; in DKV
// each thread first acts as a row of the query tile, builds that row's bits against
// the item's key tile, and the warps transpose the bits into per-key columns with
// ballots.  FULL tiles skip the mask.  The MMAs of one thread run in issue order, so
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

constexpr int kD = 64;
constexpr int kStep = 64;                   // keys (DQ) or queries (DKV) per MMA step
constexpr int kTileBytes = kTile * kD * 2;  // one [128][64] bf16 tile, 128-byte swizzled
constexpr int kNS = 2;                      // stages of the streamed ring
constexpr int kRecB = (int)sizeof(KeyTileRec);
constexpr int kThreadsB = 192;
constexpr uint32_t kCols = 256;
constexpr uint64_t kWaitNsB = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;

// mbarriers
enum : int {
  kResFull = 0,
  kResEmpty,
  kStrFull,
  kStrEmpty = kStrFull + kNS,
  kSyFull = kStrEmpty + kNS,  // the step's two score MMAs completed
  kXReady,                    // the compute warps wrote the step's bf16 operands
  kAccFull,                   // the item's last accumulating MMA completed
  kAccEmpty,                  // the compute warps read the accumulators
  kGroup,                     // DKV: barrier of the 128 compute threads
  kMmaDone,
  kNumBars
};

// Byte offsets from the 1024-aligned base of dynamic shared memory.
struct BL {
  static constexpr int kRes = 0;                             // [2] resident tiles
  static constexpr int kStr = kRes + 2 * kTileBytes;         // [kNS][2] streamed tiles
  static constexpr int kSRec = kStr + 2 * kNS * kTileBytes;  // DQ: [kNS] streamed key-tile records
  static constexpr int kRRec = kSRec + kNS * kRecB;          // DKV: the item's key-tile record
  static constexpr int kCol = kRRec + kRecB;                 // DKV: [128 keys] 128 query bits
  static constexpr int kLse = kCol + kTile * 16;             // DKV: [128] lse * log2(e) of the query tile
  static constexpr int kDlt = kLse + kTile * 4;              // DKV: [128] D of the query tile
  static constexpr int kBarsOff = kDlt + kTile * 4;
  static constexpr int kTotal = kBarsOff + kNumBars * 8 + 16;  // + abort flag and TMEM slot
  static constexpr int kDynamic = kTotal + 1024;               // slack to align the base
};
static_assert(BL::kSRec % 16 == 0 && BL::kRRec % 16 == 0 && BL::kCol % 16 == 0, "bulk-copy alignment");
static_assert(BL::kBarsOff % 8 == 0, "mbarrier alignment");
static_assert(2 * (BL::kDynamic + 1024) <= 228 * 1024, "two CTAs per SM");

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

// One work item: the tile whose rows this CTA owns (DQ: query tile, DKV: key tile)
// and its streamed tiles.
struct BItem {
  ReqMeta m;
  int h;
  int tile;  // request-local
  int n;     // streamed (non-SKIP) tiles
};

template <bool DKV>
__device__ __forceinline__ BItem decode_bitem(const BwdArgs& a, long long w) {
  BItem it;
  const long long e = a.items[w];
  const long long g = e / a.heads;
  it.h = (int)(e % a.heads);
  it.m = a.meta[a.qreq[g]];
  const int qt = (int)(g - it.m.tile_start);
  if constexpr (!DKV) {
    it.tile = qt;
    it.n = max(a.kcount[g], 0);
  } else {
    it.tile = it.m.ntiles - 1 - qt;
    const uint8_t* col = a.cls + it.m.cls_start + it.tile;
    int n = 0;
    for (int r = 0; r < it.m.ntiles; ++r) n += col[(long long)r * it.m.ntiles] != REC_ATTN_TILE_SKIP;
    it.n = n;
  }
  return it;
}

// The streamed tiles of an item in order: request-local tile index and class.
template <bool DKV>
struct Cursor {
  const uint32_t* list;  // DQ: the query tile's key-tile list
  const uint8_t* col;    // DKV: column `tile` of the request's class matrix
  int ntiles, r;
  __device__ __forceinline__ void init(const BwdArgs& a, const BItem& it) {
    ntiles = it.m.ntiles;
    r = 0;
    if constexpr (!DKV) list = a.klist + it.m.cls_start + (long long)it.tile * it.m.ntiles;
    else col = a.cls + it.m.cls_start + it.tile;
  }
  __device__ __forceinline__ void next(int& tile, int& cls) {
    if constexpr (!DKV) {
      const uint32_t e = list[r++];
      tile = (int)(e & 0xffffffu);
      cls = (int)(e >> 24);
    } else {
      while (r < ntiles - 1 && col[(long long)r * ntiles] == REC_ATTN_TILE_SKIP) ++r;
      tile = r;
      cls = col[(long long)r * ntiles];
      ++r;
    }
  }
};

// ------------------------------------------------------------------ producer
// maps: resident pair res[0], res[1]; streamed pair str[0], str[1].
template <bool DKV>
__device__ void bwd_producer(const BwdArgs& a, const void* const (&res)[2], const void* const (&str)[2],
                             uint8_t* sm, uint64_t* bars, volatile int* abort_flag) {
  uint32_t it_n = 0, s_it = 0;
  bool res_used = false, str_used[kNS];
  uint32_t res_ph = 0, str_ph[kNS];
  for (int i = 0; i < kNS; ++i) { str_used[i] = false; str_ph[i] = 0; }
  for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
    const BItem it = decode_bitem<DKV>(a, w);
    if (it.n <= 0) continue;
    if (!bw_wait(bars + kResEmpty, (it_n & 1) ^ 1, abort_flag, a.status)) goto drain;
    {
      const int x = it.h * kD;
      const int y = (int)(it.m.tok_start + (long long)it.tile * kTile);
      ptx::mbar_arrive_expect_tx(bars + kResFull, 2 * kTileBytes + (DKV ? kRecB : 0));
      ptx::tma_load_2d(sm + BL::kRes, res[0], x, y, bars + kResFull);
      ptx::tma_load_2d(sm + BL::kRes + kTileBytes, res[1], x, y, bars + kResFull);
      if (DKV) ptx::bulk_load(sm + BL::kRRec, a.krec + it.m.tile_start + it.tile, kRecB, bars + kResFull);
      res_used = true;
      res_ph = it_n & 1;
      ++it_n;
      Cursor<DKV> cur;
      cur.init(a, it);
      for (int j = 0; j < it.n; ++j) {
        int tile, cls;
        cur.next(tile, cls);
        const int st = (int)(s_it % kNS);
        const uint32_t ph = (s_it / kNS) & 1;
        if (!bw_wait(bars + kStrEmpty + st, ph ^ 1, abort_flag, a.status)) goto drain;
        const bool rec = !DKV && cls != REC_ATTN_TILE_FULL;  // DQ masks PARTIAL tiles with the key record
        const int ys = (int)(it.m.tok_start + (long long)tile * kTile);
        ptx::mbar_arrive_expect_tx(bars + kStrFull + st, 2 * kTileBytes + (rec ? kRecB : 0));
        ptx::tma_load_2d(sm + BL::kStr + (2 * st) * kTileBytes, str[0], x, ys, bars + kStrFull + st);
        ptx::tma_load_2d(sm + BL::kStr + (2 * st + 1) * kTileBytes, str[1], x, ys, bars + kStrFull + st);
        if (rec)
          ptx::bulk_load(sm + BL::kSRec + st * kRecB, a.krec + it.m.tile_start + tile, kRecB, bars + kStrFull + st);
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
__device__ __forceinline__ uint64_t mndesc(uint32_t addr) { return ptx::smem_desc_sw128(addr, kTileBytes, 1024); }

// D = A B^T over K = 64 (both operands K-major, B = 64 rows of a tile): N = 64.
__device__ __forceinline__ void mma_scores(uint32_t d, uint32_t a_addr, uint32_t b_addr) {
  constexpr uint32_t id = ptx::idesc_bf16_f32(kTile, kStep, false, false);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) ptx::umma_f16(d, kdesc(a_addr + kk * 32), kdesc(b_addr + kk * 32), id, kk > 0);
}
// D (+)= A B with A (128 x 64, bf16) in TMEM and B = 64 rows of a tile as the K
// dimension (MN-major: the tile's 64 columns are N).
__device__ __forceinline__ void mma_acc(uint32_t d, uint32_t a_tmem, uint32_t b_rows, bool accumulate) {
  constexpr uint32_t id = ptx::idesc_bf16_f32(kTile, kD, false, true);
#pragma unroll
  for (int kk = 0; kk < kStep / 16; ++kk)
    ptx::umma_f16_ts(d, a_tmem + kk * 8, mndesc(b_rows + kk * 16 * 128), id, (accumulate || kk > 0) ? 1u : 0u);
}

template <bool DKV>
__device__ void bwd_mma(const BwdArgs& a, uint8_t* sm, uint64_t* bars, uint32_t tmem, volatile int* abort_flag) {
  const uint32_t res0 = ptx::smem_u32(sm + BL::kRes), res1 = res0 + kTileBytes;
  const uint32_t str = ptx::smem_u32(sm + BL::kStr);
  constexpr uint32_t kHalfBytes = kStep * 128;  // 64 rows of a tile
  uint32_t it_n = 0, s_it = 0, step = 0;
  for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
    const BItem it = decode_bitem<DKV>(a, w);
    if (it.n <= 0) continue;
    if (!bw_wait(bars + kResFull, it_n & 1, abort_flag, a.status)) goto out;
    if (it_n > 0 && !bw_wait(bars + kAccEmpty, (it_n - 1) & 1, abort_flag, a.status)) goto out;
    ptx::tc_fence_after();
    ++it_n;
    {
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
      if constexpr (!DKV) {
        // S(ls) = Q' K'_h^T into S buffer (step0 + ls) % 2
        auto issue_s = [&](int ls) -> bool {
          int st;
          if (!stage_of(ls, true, st)) return false;
          mma_scores(tmem + ((step0 + ls) & 1) * kStep, res0,
                     str + (2 * st) * kTileBytes + (ls & 1) * kHalfBytes);
          return true;
        };
        if (!issue_s(0)) goto out;
        for (int ls = 0; ls < nsteps; ++ls) {
          int st;
          stage_of(ls, false, st);
          const uint32_t kb = str + (2 * st) * kTileBytes + (ls & 1) * kHalfBytes;
          const uint32_t vb = str + (2 * st + 1) * kTileBytes + (ls & 1) * kHalfBytes;
          mma_scores(tmem + 128, res1, vb);  // dP = dO V_h^T
          ptx::umma_commit(bars + kSyFull);
          if (ls + 1 < nsteps && !issue_s(ls + 1)) goto out;
          if (!bw_wait(bars + kXReady, (step0 + ls) & 1, abort_flag, a.status)) goto out;
          ptx::tc_fence_after();
          mma_acc(tmem + 192, tmem + ((step0 + ls) & 1) * kStep, kb, ls > 0);  // dQ += dS K'_h
          if (ls & 1) ptx::umma_commit(bars + kStrEmpty + st);
        }
      } else {
        // S^T = K' Q'_h^T and dP^T = V dO_h^T
        auto issue_scores = [&](int ls) -> bool {
          int st;
          if (!stage_of(ls, true, st)) return false;
          mma_scores(tmem + 0, res0, str + (2 * st) * kTileBytes + (ls & 1) * kHalfBytes);
          mma_scores(tmem + 64, res1, str + (2 * st + 1) * kTileBytes + (ls & 1) * kHalfBytes);
          ptx::umma_commit(bars + kSyFull);
          return true;
        };
        if (!issue_scores(0)) goto out;
        for (int ls = 0; ls < nsteps; ++ls) {
          int st;
          stage_of(ls, false, st);
          if (!bw_wait(bars + kXReady, (step0 + ls) & 1, abort_flag, a.status)) goto out;
          ptx::tc_fence_after();
          const uint32_t qb = str + (2 * st) * kTileBytes + (ls & 1) * kHalfBytes;
          const uint32_t ob = str + (2 * st + 1) * kTileBytes + (ls & 1) * kHalfBytes;
          mma_acc(tmem + 128, tmem + 0, ob, ls > 0);   // dV += P^T dO_h
          mma_acc(tmem + 192, tmem + 64, qb, ls > 0);  // dK += dS^T Q'_h
          if (ls & 1) ptx::umma_commit(bars + kStrEmpty + st);
          if (ls + 1 < nsteps && !issue_scores(ls + 1)) goto out;
        }
      }
      step += (uint32_t)nsteps;
      s_it += (uint32_t)it.n;
      ptx::umma_commit(bars + kAccFull);
      ptx::umma_commit(bars + kResEmpty);
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

// One output row: x * scale, then (rotate) R(dt)^T over adjacent pairs, as bf16.
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const uint32_t (&acc)[64], float scale, bool rotate,
                                         float dt, const float* omega) {
  uint32_t w[32];
#pragma unroll
  for (int p = 0; p < 32; ++p) {
    float u = __uint_as_float(acc[2 * p]) * scale, v = __uint_as_float(acc[2 * p + 1]) * scale;
    if (rotate) {
      float sn, cs;
      sincosf(dt * omega[p], &sn, &cs);
      const float u2 = u * cs + v * sn;
      v = -u * sn + v * cs;
      u = u2;
    }
    w[p] = bf16x2(u, v);
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < 8; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* dst) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
}

// The bf16 operands of one 32-column chunk.  DQ: dS from S (s) and dP (d) with the
// row's constants; bits = the chunk's visibility bits.
__device__ __forceinline__ void ds_chunk(const uint32_t (&r)[64], uint32_t bits, float sl2, float lse2, float dlt,
                                         uint32_t (&pk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float p0 = ex2(fmaf(__uint_as_float(r[2 * e]), sl2, -lse2));
    float p1 = ex2(fmaf(__uint_as_float(r[2 * e + 1]), sl2, -lse2));
    p0 = ((bits >> (2 * e)) & 1u) ? p0 : 0.f;
    p1 = ((bits >> (2 * e + 1)) & 1u) ? p1 : 0.f;
    pk[e] = bf16x2(p0 * (__uint_as_float(r[32 + 2 * e]) - dlt), p1 * (__uint_as_float(r[32 + 2 * e + 1]) - dlt));
  }
}

// DQ: thread = query row of the item's tile.
__device__ void bwd_compute_dq(const BwdArgs& a, uint8_t* sm, uint64_t* bars, uint32_t tmem,
                               volatile int* abort_flag) {
  const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3, row = quad * 32 + lane;
  const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
  const float sl2 = a.scale * kLog2e;
  const KeyTileRec* srec = reinterpret_cast<const KeyTileRec*>(sm + BL::kSRec);
  const int H = a.heads;
  uint32_t it_n = 0, s_it = 0, step = 0;
  for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
    const BItem it = decode_bitem<false>(a, w);
    const int pi = it.tile * kTile + row;
    const bool row_ok = pi < it.m.len;
    const long long tok = it.m.tok_start + pi, grow = tok * H + it.h;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + grow * kD;
    if (it.n <= 0) {  // no visible key tile
      if (row_ok) zero_row(dst);
      continue;
    }
    long long ti = 0;
    int tyi = -1;
    float lse2 = 0.f, dlt = 0.f;
    bool live = false;  // a row that sees no key (lse = -inf) contributes nothing
    if (row_ok) {
      ti = a.t[tok];
      tyi = a.ty[tok];
      const float l = a.lse[grow];
      dlt = a.delta[grow];
      live = l != -INFINITY;
      lse2 = live ? l * kLog2e : 0.f;
    }
    RowMask rm;
    row_mask_setup(a.mask, live, pi, ti, tyi, rm);
    Cursor<false> cur;
    cur.init(a, it);
    for (int j = 0; j < it.n; ++j) {
      int kt, cls;
      cur.next(kt, cls);
      const int st = (int)(s_it % kNS);
      const uint32_t ph = (s_it / kNS) & 1;
      ++s_it;
      const uint32_t f = live ? ~0u : 0u;
      uint32_t vm[4] = {f, f, f, f};
      if (cls != REC_ATTN_TILE_FULL) {
        if (!bw_wait_warp(bars + kStrFull + st, ph, abort_flag, a.status)) return;
        build_mask(rm, srec + st, kt * kTile, vm);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + kStrEmpty + st);  // the stage's record was read
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh, ++step) {
        if (!bw_wait_warp(bars + kSyFull, step & 1, abort_flag, a.status)) return;
        ptx::tc_fence_after();
        const uint32_t sb = tl + (step & 1) * kStep;
        const uint32_t wb[2] = {hh ? vm[2] : vm[0], hh ? vm[3] : vm[1]};  // this step's 64 keys
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[64], pk[16];
          ptx::tmem_ld32x2_async(sb + 32 * c, tl + 128 + 32 * c, r);
          ptx::tmem_wait_ld(r);
          ds_chunk(r, wb[c], sl2, lse2, dlt, pk);
          ptx::tmem_st16_async(sb + 16 * c, pk);  // over S columns already read
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + kXReady);
      }
    }
    if (!bw_wait_warp(bars + kAccFull, it_n & 1, abort_flag, a.status)) return;
    ++it_n;
    ptx::tc_fence_after();
    uint32_t acc[64];
    ptx::tmem_ld64(tl + 192, acc);
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bars + kAccEmpty);
    if (row_ok) store_row(dst, acc, a.scale, a.rotate != 0, (float)(ti - a.t[it.m.tok_start]), a.omega);
  }
}

// The 128 compute threads meet (bounded); `n` counts the uses of the barrier.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& n, volatile int* abort_flag, int* status) {
  ptx::mbar_arrive(bar);
  return bw_wait_warp(bar, (n++) & 1, abort_flag, status);
}

// DKV: thread = key row of the item's tile (and, while the masks are built, a row of
// the query tile).
__device__ void bwd_compute_dkv(const BwdArgs& a, uint8_t* sm, uint64_t* bars, uint32_t tmem,
                                volatile int* abort_flag) {
  const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3, row = quad * 32 + lane;
  const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
  const float sl2 = a.scale * kLog2e;
  const KeyTileRec* rrec = reinterpret_cast<const KeyTileRec*>(sm + BL::kRRec);
  uint32_t* colS = reinterpret_cast<uint32_t*>(sm + BL::kCol);
  float* lseS = reinterpret_cast<float*>(sm + BL::kLse);
  float* dltS = reinterpret_cast<float*>(sm + BL::kDlt);
  const int H = a.heads;
  uint32_t it_n = 0, step = 0, grp = 0;
  for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
    const BItem it = decode_bitem<true>(a, w);
    const int pj = it.tile * kTile + row;
    const bool key_ok = pj < it.m.len;
    const long long tokk = it.m.tok_start + pj, growk = tokk * H + it.h;
    __nv_bfloat16* dkr = static_cast<__nv_bfloat16*>(a.dk) + growk * kD;
    __nv_bfloat16* dvr = static_cast<__nv_bfloat16*>(a.dv) + growk * kD;
    if (it.n <= 0) {  // no query sees this key tile
      if (key_ok) { zero_row(dkr); zero_row(dvr); }
      continue;
    }
    const long long tj = key_ok ? a.t[tokk] : 0;
    if (!bw_wait_warp(bars + kResFull, it_n & 1, abort_flag, a.status)) return;  // the key tile's record
    Cursor<true> cur;
    cur.init(a, it);
    for (int j = 0; j < it.n; ++j) {
      int qt, cls;
      cur.next(qt, cls);
      // as query row `row` of query tile qt: its visibility bits over the key tile
      const int qi = qt * kTile + row;
      const bool q_ok = qi < it.m.len;
      const long long tokq = it.m.tok_start + qi, growq = tokq * H + it.h;
      long long tq = 0;
      int tyq = -1;
      float lq = -INFINITY, dq = 0.f;
      if (q_ok) {
        tq = a.t[tokq];
        tyq = a.ty[tokq];
        lq = a.lse[growq];
        dq = a.delta[growq];
      }
      const bool live = q_ok && lq != -INFINITY;
      const uint32_t f = live ? ~0u : 0u;
      uint32_t vm[4] = {f, f, f, f};
      if (cls != REC_ATTN_TILE_FULL) {
        RowMask rm;
        row_mask_setup(a.mask, live, qi, tq, tyq, rm);
        build_mask(rm, rrec, it.tile * kTile, vm);
      }
      if (j == it.n - 1) {  // the key tile's record is not read again in this item
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + kResEmpty);
      }
      // lane b keeps the bits of key 32 w + b over this warp's 32 queries
      uint32_t colw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int wd = 0; wd < 4; ++wd)
#pragma unroll
        for (int b = 0; b < 32; ++b) {
          const uint32_t bal = __ballot_sync(0xffffffffu, (vm[wd] >> b) & 1u);
          colw[wd] = lane == b ? bal : colw[wd];
        }
      if (!group_sync(bars + kGroup, grp, abort_flag, a.status)) return;  // last tile's readers are done
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) colS[(32 * wd + lane) * 4 + quad] = colw[wd];
      lseS[row] = live ? lq * kLog2e : 0.f;
      dltS[row] = dq;
      if (!group_sync(bars + kGroup, grp, abort_flag, a.status)) return;
      const uint4 cm = reinterpret_cast<const uint4*>(colS)[row];
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh, ++step) {
        if (!bw_wait_warp(bars + kSyFull, step & 1, abort_flag, a.status)) return;
        ptx::tc_fence_after();
        const uint32_t wb[2] = {hh ? cm.z : cm.x, hh ? cm.w : cm.y};  // this step's 64 queries
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[64], pp[16], pd[16];
          ptx::tmem_ld32x2_async(tl + 32 * c, tl + 64 + 32 * c, r);
          const float4* l4 = reinterpret_cast<const float4*>(lseS + hh * kStep + c * 32);
          const float4* d4 = reinterpret_cast<const float4*>(dltS + hh * kStep + c * 32);
          const uint32_t bits = wb[c];
          ptx::tmem_wait_ld(r);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float4 lv = l4[g], dv = d4[g];
            const float lsv[4] = {lv.x, lv.y, lv.z, lv.w}, dsv[4] = {dv.x, dv.y, dv.z, dv.w};
            float p[4], s[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int e = 4 * g + u;
              const float x = ex2(fmaf(__uint_as_float(r[e]), sl2, -lsv[u]));
              p[u] = ((bits >> e) & 1u) ? x : 0.f;
              s[u] = p[u] * (__uint_as_float(r[32 + e]) - dsv[u]);
            }
            pp[2 * g] = bf16x2(p[0], p[1]);
            pp[2 * g + 1] = bf16x2(p[2], p[3]);
            pd[2 * g] = bf16x2(s[0], s[1]);
            pd[2 * g + 1] = bf16x2(s[2], s[3]);
          }
          ptx::tmem_st16_async(tl + 16 * c, pp);       // P^T over S^T columns already read
          ptx::tmem_st16_async(tl + 64 + 16 * c, pd);  // dS^T over dP^T columns already read
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + kXReady);
      }
    }
    if (!bw_wait_warp(bars + kAccFull, it_n & 1, abort_flag, a.status)) return;
    ++it_n;
    ptx::tc_fence_after();
    uint32_t acc[64];
    ptx::tmem_ld64(tl + 128, acc);
    if (key_ok) store_row(dvr, acc, 1.f, false, 0.f, a.omega);
    ptx::tmem_ld64(tl + 192, acc);
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bars + kAccEmpty);
    if (key_ok) store_row(dkr, acc, a.scale, a.rotate != 0, (float)(tj - a.t[it.m.tok_start]), a.omega);
  }
}

// ------------------------------------------------------------------ kernel
// maps: Q', K', V, dO, each a [T][H*64] bf16 view with 64 x 128 boxes.
template <bool DKV>
__global__ void __launch_bounds__(kThreadsB, 2)
    k_bwd_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BL::kBarsOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars) + 1;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bars + kResFull, 1);
    ptx::mbar_init(bars + kResEmpty, DKV ? 1 + 4 : 1);  // DKV: the compute warps read the key record
    for (int i = 0; i < kNS; ++i) {
      ptx::mbar_init(bars + kStrFull + i, 1);
      ptx::mbar_init(bars + kStrEmpty + i, DKV ? 1 : 1 + 4);  // DQ: the compute warps read the key record
    }
    ptx::mbar_init(bars + kSyFull, 1);
    ptx::mbar_init(bars + kXReady, 4);
    ptx::mbar_init(bars + kAccFull, 1);
    ptx::mbar_init(bars + kAccEmpty, 4);
    ptx::mbar_init(bars + kGroup, 128);
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
      bwd_producer<DKV>(a, res, str, sm, bars, abort_flag);
    }
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) bwd_mma<DKV>(a, sm, bars, tmem, abort_flag);
  } else {
    if constexpr (DKV) bwd_compute_dkv(a, sm, bars, tmem, abort_flag);
    else bwd_compute_dq(a, sm, bars, tmem, abort_flag);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kCols);
  }
}

template <bool DKV>
cudaError_t launch_mode(const CUtensorMap (&maps)[4], const BwdArgs& a, int grid, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(k_bwd_tc<DKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, BL::kDynamic);
  if (e != cudaSuccess) return e;
  k_bwd_tc<DKV><<<grid, kThreadsB, BL::kDynamic, st>>>(maps[0], maps[1], maps[2], maps[3], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const BwdArgs& a, const CUtensorMap (&maps)[4], int num_sms, cudaStream_t st) {
  if (a.n_items <= 0) return cudaSuccess;
  const long long cap = 2LL * num_sms;  // two CTAs per SM
  const int grid = (int)(a.n_items < cap ? a.n_items : cap);
  cudaError_t e = launch_mode<false>(maps, a, grid, st);
  if (e != cudaSuccess) return e;
  return launch_mode<true>(maps, a, grid, st);
}

}  // namespace recattn
