// row_mask.cuh -- a query row's visibility bits against one key tile, built from the
// planner's key-tile record instead of per-element predicate calls (shared by the
// forward and backward tensor-core kernels).
#pragma once

#include <climits>

#include "rec_attn_internal.cuh"

namespace recattn {

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

}  // namespace recattn
