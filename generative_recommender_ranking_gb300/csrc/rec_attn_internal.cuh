// rec_attn_internal.cuh -- structures and device helpers shared by the CUDA sources
// of the GB300 masked time-RoPE attention library (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "rec_attn.h"

namespace recattn {

constexpr int kTile = REC_ATTN_TILE;  // tokens per query / key tile
constexpr int kTypes = 4;             // GLOBAL, HIST, RT, CAND
constexpr int kMaxPairs = 64;         // head_dim <= 128
constexpr long long kTimeLimit = (1LL << 62);

// One request of the packed batch.
struct ReqMeta {
  long long tok_start;   // first token (global index)
  int len;               // tokens in the request
  int ntiles;            // ceil(len / kTile)
  long long tile_start;  // first tile (global tile index)
  long long cls_start;   // first entry of the request's ntiles x ntiles class matrix
};

// Bounding box of one token type inside one tile (positions are request-local).
struct TileBox {
  int cnt, pmin, pmax, pad;
  long long tmin, tmax;
};

// Per key tile, what the attention kernel needs to build a row's visibility bits
// without per-element predicate calls (filled by the planner, copied into shared
// memory next to the K tile for PARTIAL tiles).
struct KeyTileRec {
  uint32_t typebits[kTypes][4];  // bit c of word c/32: key c of the tile has this type
  int run_lo[kTypes];            // first key (tile-local) of the type
  int run_n[kTypes];             // keys of the type in the tile
  int sorted[kTypes];            // 1: the type's keys are contiguous with non-decreasing times
  int pad[kTypes];
  long long t[kTile];            // key timestamps (0 past the request end)
};
static_assert(sizeof(KeyTileRec) == 1152, "record must stay a multiple of 16 bytes");

// Mask parameters as the kernels see them.
struct MaskP {
  int use_delay;
  int window;
  int bidir;
  int keep_user;  // query pruning: user queries kept per request, counted from the end; < 0: all
  long long delay;
};

// Device workspace owned by a plan.
struct PlanDev {
  ReqMeta* meta;        // [B]
  TileBox* boxes;       // [NT][4]
  KeyTileRec* krec;     // [NT]
  uint8_t* cls;         // [NC]
  uint32_t* klist;      // [NC]: per query tile, the non-SKIP key tiles (kt | class << 24)
  int* kcount;          // [NT]: entries in each query tile's list
  int* qcost;           // [NT]: scheduling cost of each query tile
  int* qreq;            // [NT]: request of each query tile
  int* items;           // [NT*H]: work items (query tile * H + head) in execution order
  int* rcost;           // [B]: scheduling cost of each request
  int* rorder;          // [B]: requests, most expensive first
  int* roff;            // [B+1]: first item of each request in `items` (in rorder order)
  int* qkeep;           // [B]: query pruning: user tokens before this position compute nothing
  int* treq;            // [NT]: request of each tile (uploaded with the request table)
  int* counters;        // [8]: plan ticket, attention item counter and exit ticket, backward
                        // item counters and exit tickets, mask-table slot counter
  int* status;          // [1]: first device error (rec_attn_status)
  unsigned long long* pairs;  // [1]: visible-pair counter
  // Mask table: the 128 rows' visibility bits of PARTIAL tile pairs, built once per plan
  // (the masks do not depend on the head), for up to mcap pairs; the others build their
  // bits in the kernels.
  int* kslot;           // [NC], aligned with klist: table slot of the entry, -1 if none
  int* pslot;           // [NC], class-matrix order: table slot of the pair, -1 if none
  int2* minfo;          // [mcap]: (global query tile, key tile) of each slot
  uint32_t* mtab;       // [mcap][128 rows][4 words]
  int mcap;
};

// History compression: one request of the batch, and the kernel arguments.
constexpr int kMaxSegments = 8;
struct CompressReq {
  long long in_start, len;         // input rows of the request
  long long hist_begin, hist_len;  // request-local history range
  long long out_start, out_len;    // output rows of the request
};
struct CompressArgs {
  const CompressReq* req;
  int batch;
  int n_seg;
  long long rows_out;
  long long seg_len[kMaxSegments];  // recency segments from the newest (< 0: the rest)
  int seg_group[kMaxSegments];
  long long width;                  // elements per row
  const void* x;
  const long long* t;
  const int8_t* ty;
  void* x_out;
  long long* t_out;
  int8_t* ty_out;
};

// Record a device-side error; the first error wins.
__device__ __forceinline__ void set_status(int* st, int code) { atomicCAS(st, 0, code); }

__device__ __forceinline__ bool is_user(int ty) { return ty == REC_ATTN_GLOBAL || ty == REC_ATTN_HIST; }

// Whether a query row is computed under query pruning: every non-user token, and the
// user tokens at or after the request's first kept user position.
__device__ __forceinline__ bool query_kept(int ty, int pos, int keep_pos) {
  return !is_user(ty) || pos >= keep_pos;
}

// vis(i, j) for two tokens of one request.  `thr_ok`/`thr` encode the exact delay
// bound of the query (t_i - delta): thr_ok is false when t_i - delta lies below the
// int64 range, in which case no key is old enough.  Types outside 0..3 see nothing.
__device__ __forceinline__ bool vis_pred(const MaskP& m, int pi, long long ti, int tyi,
                                         bool thr_ok, long long thr, int pj, long long tj,
                                         int tyj) {
  if ((unsigned)tyi > 3u || (unsigned)tyj > 3u) return false;
  bool v;
  const bool ui = is_user(tyi), uj = is_user(tyj);
  if (ui) {
    if (!uj) {
      v = false;
    } else if (m.bidir) {
      v = true;
    } else {
      v = pj <= pi;
      if (m.window > 0 && tyi != REC_ATTN_GLOBAL && tyj != REC_ATTN_GLOBAL)
        v = v && (pi - pj < m.window);
    }
  } else if (tyi == REC_ATTN_RT) {
    v = uj || (tyj == REC_ATTN_RT && pj <= pi);
  } else {  // candidate
    v = uj || (tyj == REC_ATTN_RT ? (tj < ti) : (pi == pj));
  }
  if (m.use_delay && !(tyi == REC_ATTN_CAND && tyj == REC_ATTN_CAND && pi == pj))
    v = v && thr_ok && (tj <= thr);
  return v;
}

// Query-side delay bound t_i - delta, exact (see vis_pred).
__device__ __forceinline__ void delay_bound(long long ti, long long delta, bool& ok,
                                            long long& thr) {
  ok = ti >= (long long)(-0x7fffffffffffffffLL - 1) + delta;
  thr = ok ? ti - delta : 0;
}

}  // namespace recattn
