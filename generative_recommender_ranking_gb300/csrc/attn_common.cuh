// attn_common.cuh -- arguments shared by the attention kernels.
#pragma once

#include "rec_attn_internal.cuh"

namespace recattn {

// History compression fused into the attention epilogue: per request, where its rows
// go (rows before the history copied, history rows summed in groups, rows after it
// copied) and where its 32-row blocks keep the partial sums of groups that straddle
// two blocks.
struct CmpReq {
  long long out_start;  // first output row of the request
  long long fix_start;  // first 32-row block boundary of the request in the fix-up buffer
  int hist_begin, hist_len, n_groups, pad;
};
struct CmpArgs {
  const CmpReq* req;    // [B]
  void* x_out;          // [rows_out][H][d]
  float* fix;           // [boundaries][2 parts][H][d] fp32
  int n_seg;
  int span;             // largest group (<= 32)
  long long seg_len[kMaxSegments];  // recency segments from the newest (< 0: the rest)
  int seg_group[kMaxSegments];
};

// Output row (global) of request-local row pi and the request-local rows [glo, ghi) of
// its group: the inverse of the compression's grouping (recency segments counted from
// the newest row, the oldest group of a segment partial, groups in time order).
__host__ __device__ __forceinline__ long long cmp_group_of(const CmpArgs& c, const CmpReq& r, int pi, int& glo, int& ghi) {
  if (pi < r.hist_begin) { glo = pi; ghi = pi + 1; return r.out_start + pi; }
  if (pi >= r.hist_begin + r.hist_len) {
    glo = pi; ghi = pi + 1;
    return r.out_start + pi - r.hist_len + r.n_groups;
  }
  // 32-bit arithmetic: requests are shorter than 2^31 rows
  const int Lh = r.hist_len;
  const int rank_i = Lh - 1 - (pi - r.hist_begin);  // 0: the newest history row
  int rank = 0, newer_groups = 0;
  for (int u = 0; u < c.n_seg && rank < Lh; ++u) {
    const int room = Lh - rank;
    const int m = (c.seg_len[u] < 0 || c.seg_len[u] > room) ? room : (int)c.seg_len[u];
    const int g = c.seg_group[u];
    if (rank_i < rank + m) {
      const int q = (rank_i - rank) / g;  // 0: the segment's newest group
      const int r0 = rank + q * g;
      const int r1 = rank + ((q + 1) * g < m ? (q + 1) * g : m);
      glo = r.hist_begin + Lh - r1;
      ghi = r.hist_begin + Lh - r0;
      const int from_newest = newer_groups + q;  // groups between it and the newest row
      return r.out_start + r.hist_begin + (r.n_groups - 1 - from_newest);
    }
    newer_groups += (m + g - 1) / g;
    rank += m;
  }
  glo = pi; ghi = pi + 1;  // unreachable: the segments cover the history
  return r.out_start + pi;
}

struct AttnArgs {
  const ReqMeta* meta;
  const int* qreq;
  const int* kcount;
  const uint32_t* klist;
  const int* items;  // work items (query tile * H + head), execution order
  const long long* t;
  const int8_t* ty;
  const void* q;     // rotated (or raw when RoPE is off) queries [T][H][d]
  const void* k;     // rotated keys
  const void* v;
  void* out;
  const void* out_gate;  // optional [T][H][d] in the I/O dtype: O <- O * sigmoid(out_gate)
  float* lse;        // optional [T][H]
  int* status;
  int* counters;     // [1]: dynamic item counter, [2]: exit ticket (both reset at kernel end)
  const KeyTileRec* krec;
  const int* qkeep;  // [B] first kept user position of each request (query pruning)
  const int* kslot;       // per key-tile list entry: mask-table slot (-1: build the bits)
  const uint32_t* mtab;   // mask table: [slot][128 rows][4 words]
  long long n_items; // query tiles x heads
  int heads;
  float scale;       // softmax scale (natural-log domain)
  MaskP mask;
  CmpArgs cmp;       // compression epilogue (kernels instantiated with it only)
  int long_items;    // 1: the items run over many key tiles (the softmax's lazy maximum pays)
};

// Arguments of the time-RoPE prologue.
struct RopeArgs {
  const ReqMeta* meta;
  const int* tile_req;     // [NT] request of each tile (uploaded with the request table)
  int batch;               // requests in meta (the prologue needs nothing the planner writes)
  const long long* t;
  const int8_t* ty;        // token types (read only when skip_user_q)
  int skip_user_q;         // 1: no Q' for GLOBAL / HIST tokens (a plan where no user token queries)
  const void* q;
  const void* k;
  void* qr;                // rotated outputs, same layout [T][H][d]
  void* kr;
  int heads, head_dim;
  float omega[kMaxPairs];  // rad per second, pair i
};

// Serving with a cached history (M-FALCON): one region of a request's rows in the
// cache's combined layout, filled by k_rope_slots from packed source rows.  The
// first `len` destination rows take source rows src_start.. (rotated keys and
// queries, copied values, times, types); rows len..cap-1 are padding (zeros, the
// time of the last source row or the reference, the constant type).
struct SlotReq {
  long long src_start;  // first source row
  long long dst_start;  // first destination row
  long long ref_row;    // row holding the request's rotation reference time
  int ref_dst;          // 1: ref_row indexes the destination times, 0: the source times
  int len;              // source rows
  int cap;              // destination rows (len <= cap)
  int pad;
};
static_assert(sizeof(SlotReq) == 40, "");

struct SlotArgs {
  const SlotReq* req;
  const int* chunk_req;    // per 128-row chunk of the regions: its request
  const int* chunk_row0;   // and its first row within the region
  const long long* t_src;  // [source rows]
  const int8_t* ty_src;    // [source rows], or null: every written row takes ty_const
  int ty_const;
  const void* q_src;       // [source][H][d] or null (no queries)
  const void* k_src;
  const void* v_src;
  void* q_dst;             // [destination][H][d]
  void* k_dst;
  void* v_dst;
  long long* t_dst;
  int8_t* ty_dst;
  // gather direction (k_slots_gather): out rows of the source layout from the destination layout
  const void* o_comb;      // [destination][H][d]
  const float* lse_comb;   // [destination][H] or null
  void* o_out;             // [source][H][d]
  float* lse_out;          // [source][H] or null
  int heads, head_dim;
  float omega[kMaxPairs];  // rad per second, pair i (all zero: no rotation)
};

// One backward work item as the tensor-core kernels read it (one 48-byte record per
// item and mode, written once per plan by k_bwd_schedule).
struct BwdItemDesc {
  long long tok_start;  // first token of the item's request (global)
  long long t_ref;      // its time: the rotation's reference
  long long list;       // offset of the item's streamed-tile list (kt or qt | class << 24)
  int len;              // request length
  int tile;             // request-local tile whose rows the item owns
  int tile_start;       // global index of the request's first tile
  int h;
  int n;                // streamed tiles
  int pad;
};
static_assert(sizeof(BwdItemDesc) == 48, "three 16-byte loads");

// Arguments of the backward kernels.
struct BwdArgs {
  const ReqMeta* meta;
  int batch;
  const int* items;        // work items (query tile * H + head), the planner's execution order
  const int* qreq;         // request of each tile
  const KeyTileRec* krec;  // per tile: type bitmaps and times (tensor-core kernels' masks)
  long long n_items;       // tiles x heads
  int* status;             // device status word (first error wins)
  int* counters;           // [3], [4]: dQ item counter and exit ticket; [5], [6]: dK/dV (reset at kernel end)
  long long n_tiles;
  // tensor-core path (bf16): per-plan schedule and per-call row constants
  const BwdItemDesc* desc;  // [2][n_items]: dQ items, then dK/dV items (mirrored key tiles)
  const uint32_t* qlist;    // per key tile: query tiles with a non-SKIP class (qt | class << 24)
  float2* rowc;             // [H][n_tiles][128 rows]: -lse * log2(e) and -D, rows paired as
                            // {-lse2(2k), -lse2(2k+1), -D(2k), -D(2k+1)} (lse2 -inf: the row sees
                            // no key; +inf: past the request end or pruned)
  const int* kslot;         // per key-tile list entry: mask-table slot (-1: build the bits)
  const uint32_t* mtab;     // mask table, rows: [slot][128 query rows][4 words over the keys]
  const int* qslot;         // per query-tile list entry (qlist): mask-table slot, -1 if none
  const uint32_t* ctab;     // mask table, columns: [slot][128 keys][4 words over the queries]
  const int* kcount;       // per query tile: entries in its key-tile list
  const int* qkeep;        // [B] query pruning: user tokens before this position compute nothing
  const uint32_t* klist;   // per query tile: non-SKIP key tiles (kt | class << 24)
  const uint8_t* cls;      // per request: ntiles x ntiles class matrix
  const long long* t;
  const int8_t* ty;
  const void* q;           // rotated queries Q' (or raw without the RoPE) [T][H][d]
  const void* k;           // rotated keys K'
  const void* v;
  const void* out;         // forward output O
  const void* dout;        // upstream gradient dO (with out: the row constants <dO, O>)
  const void* dout_attn;   // the gradient that reaches the attention (dO, or dO * sigmoid(output gate))
  const float* lse;        // forward log-sum-exp [T][H]
  float* delta;            // workspace [T][H]: <dO, O> per row
  void* dq;                // outputs [T][H][d] (w.r.t. the unrotated Q, K)
  void* dk;
  void* dv;
  long long rows;          // T * H
  int heads;
  float scale;
  int rotate;              // 1: undo the time-RoPE on dQ', dK'
  MaskP mask;
  float omega[kMaxPairs];  // rad per second, pair i
};

// Arguments of the backward schedule kernel (run once per plan).
struct BwdSchedArgs {
  const ReqMeta* meta;
  const int* qreq;
  const int* items;
  const int* kcount;
  const uint8_t* cls;
  const long long* t;
  long long n_tiles, n_items;
  int heads;
  BwdItemDesc* desc;
  uint32_t* qlist;
  const int* pslot;         // per (query tile, key tile): mask-table slot, -1 if none
  int* qslot;               // written: per qlist entry, the pair's slot
  const int* counters;      // [7]: mask-table slots handed out
  const uint32_t* mtab;
  uint32_t* ctab;           // written: the table's columns
  int mcap;
};

// Fused steps of the prologue, applied before the rotation: QK-RMSNorm
// (x / sqrt(mean(x^2) + eps) * w[h]) and then the sigmoid gate x * sigmoid(g).
struct FusedArgs {
  const float* q_norm_w;  // [H][d] or null
  const float* k_norm_w;
  float eps;
  const void* q_gate;     // [T][H][d] in the I/O dtype, or null
  const void* k_gate;
};

// Backward through the output gate O = A * sigmoid(c): dA = dO * sigmoid(c) and
// dc = dO * O * (1 - sigmoid(c)), elementwise over n values.
struct GateArgs {
  long long n;
  const void* dout;
  const void* out;
  const void* gate;
  void* dout_attn;
  void* dgate;
};

// Backward through the QK-RMSNorm and the sigmoid gate of one side (Q or K): per
// (token, head) row a (the input), the gain w[h] and the gate c (either may be null) and
// dg, the gradient of the gated, normalised row: da, dc and the gain gradient dw
// (fp32 [H][d], zeroed by the caller, accumulated).
struct NormGateArgs {
  long long rows;  // tokens
  int heads, head_dim;
  float eps;
  const void* a;
  const float* w;
  const void* gate;
  const void* dg;
  void* da;
  void* dgate;
  float* dw;
};

// sigmoid(x) = (1 + tanh(x / 2)) / 2, one hardware tanh (relative error about 2^-11,
// below the bf16 rounding that follows) and one FMA.
__device__ __forceinline__ float sigmoidf_fast(float x) {
  float th;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * x));
  return fmaf(0.5f, th, 0.5f);
}

// The gates' sigmoid per I/O type: bf16 paths take the hardware tanh (its error is
// below the bf16 rounding that follows), fp32 paths one exponential.
template <typename E>
__device__ __forceinline__ float sigmoid_io(float x) {
  if constexpr (sizeof(E) == 2) return sigmoidf_fast(x);
  else return 1.f / (1.f + __expf(-x));
}

// One work item: (query tile, head).
struct WorkItem {
  ReqMeta m;
  int qt;            // query tile index inside the request
  int h;
  int n;             // non-SKIP key tiles; -1: every row of the tile is pruned
  int keep;          // first kept user position of the request (query pruning)
  int b;             // request
  const uint32_t* list;
  const int* slots;  // mask-table slots of the list's entries
};

__device__ __forceinline__ WorkItem decode_item(const AttnArgs& a, long long w, bool ordered) {
  WorkItem it;
  const long long e = ordered ? (long long)a.items[w] : w;
  const long long qg = e / a.heads;
  it.h = (int)(e % a.heads);
  const int b = a.qreq[qg];
  it.m = a.meta[b];
  it.qt = (int)(qg - it.m.tile_start);
  it.n = a.kcount[qg];
  it.keep = a.qkeep[b];
  it.b = b;
  it.list = a.klist + it.m.cls_start + (long long)it.qt * it.m.ntiles;
  it.slots = a.kslot + it.m.cls_start + (long long)it.qt * it.m.ntiles;
  return it;
}

}  // namespace recattn
