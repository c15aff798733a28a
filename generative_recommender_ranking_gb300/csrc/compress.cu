// compress.cu -- history compression: sums of groups of consecutive history tokens,
// the group size set per recency segment.
//
// LazFormer review page, Eq. 16-18 (keep the most recent tokens, sum the older ones
// in groups, the last group over its actual range) and Table 6; TM20K review page,
// PATM (position segments with merge factors) and LPTM (adjacent history pairs
// summed, targets never merged).  Segment i (0 = newest) covers the next seg_len[i]
// history tokens going back in time (all the rest when negative) in groups of
// seg_group[i]; the oldest group of a segment is the partial one.  Output rows keep
// time order: the tokens before the history, the merged groups (oldest first, the
// latest member time, type HIST), then the tokens after it.
//
// One warp per output row; each lane sums its 16-byte columns over the group's rows in
// fp32 and rounds once.  HBM-bound: every input row is read once, every output row
// written once.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "launchers.cuh"
#include "rec_attn_internal.cuh"

namespace recattn {

namespace {

template <typename E>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static __device__ __forceinline__ void add(const void* p, float (&acc)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  }
  static __device__ __forceinline__ void store(void* p, const float (&acc)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Vec<float> {
  static __device__ __forceinline__ void add(const void* p, float (&acc)[8]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
  }
  static __device__ __forceinline__ void store(void* p, const float (&acc)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
};

// Input history rows [lo, hi) (0 = oldest) of output group j (0 = oldest) of a history
// of Lh tokens.
__device__ __forceinline__ void group_range(const CompressArgs& a, long long Lh, long long j, long long& lo,
                                            long long& hi) {
  long long start[kMaxSegments], m[kMaxSegments], ng[kMaxSegments];
  int used = 0;
  long long rank = 0;
  for (int i = 0; i < a.n_seg && rank < Lh; ++i) {
    const long long room = Lh - rank;
    const long long mi = (a.seg_len[i] < 0 || a.seg_len[i] > room) ? room : a.seg_len[i];
    start[used] = rank;
    m[used] = mi;
    ng[used] = (mi + a.seg_group[i] - 1) / a.seg_group[i];
    ++used;
    rank += mi;
  }
  lo = hi = 0;
  for (int u = used - 1; u >= 0; --u) {  // the oldest segment first
    if (j < ng[u]) {
      const long long q = ng[u] - 1 - j;  // q = 0: the segment's newest group
      const long long g = a.seg_group[u];
      const long long r0 = start[u] + q * g;
      const long long r1 = start[u] + ((q + 1) * g < m[u] ? (q + 1) * g : m[u]);
      lo = Lh - r1;
      hi = Lh - r0;
      return;
    }
    j -= ng[u];
  }
}

template <typename E>
__global__ void __launch_bounds__(256) k_compress(CompressArgs a) {
  using V = Vec<E>;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows_out) return;
  // the request of this output row
  int lo_b = 0, hi_b = a.batch;
  while (hi_b - lo_b > 1) {
    const int mid = (lo_b + hi_b) >> 1;
    if (a.req[mid].out_start <= row) lo_b = mid;
    else hi_b = mid;
  }
  const CompressReq r = a.req[lo_b];
  const long long p = row - r.out_start;
  const long long n_groups = r.out_len - (r.len - r.hist_len);
  long long src_lo, src_hi;
  bool merged = false;
  if (p < r.hist_begin) {
    src_lo = r.in_start + p;
  } else if (p >= r.hist_begin + n_groups) {
    src_lo = r.in_start + p - n_groups + r.hist_len;
  } else {
    long long glo, ghi;
    group_range(a, r.hist_len, p - r.hist_begin, glo, ghi);
    src_lo = r.in_start + r.hist_begin + glo;
    src_hi = r.in_start + r.hist_begin + ghi;
    merged = true;
  }
  if (!merged) src_hi = src_lo + 1;
  const long long row_bytes = a.width * (long long)sizeof(E);
  const int vecs = (int)(row_bytes / 16);
  const char* x = static_cast<const char*>(a.x);
  char* y = static_cast<char*>(a.x_out);
  for (int c = lane; a.x && c < vecs; c += 32) {  // (no rows: times and types only)
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (long long s = src_lo; s < src_hi; ++s) V::add(x + s * row_bytes + c * 16, acc);
    V::store(y + row * row_bytes + c * 16, acc);
  }
  if (lane == 0) {
    long long tmax = a.t[src_lo];
    for (long long s = src_lo + 1; s < src_hi; ++s) tmax = max(tmax, a.t[s]);
    a.t_out[row] = tmax;
    a.ty_out[row] = merged ? (int8_t)REC_ATTN_HIST : a.ty[src_lo];
  }
}

// The history groups of the fused compression epilogue that straddle a 32-row block
// boundary: one block per boundary (request-local rows 32k - 1 and 32k); when one group
// holds both rows, its two fp32 partials are summed and rounded once.
__global__ void __launch_bounds__(256) k_cmp_fixup(CmpArgs c, int batch, const int* req_len, long long n_fix,
                                                   int heads, int head_dim) {
  const long long f = blockIdx.x;
  if (f >= n_fix) return;
  int lo_b = 0, hi_b = batch;
  while (hi_b - lo_b > 1) {
    const int mid = (lo_b + hi_b) >> 1;
    if (c.req[mid].fix_start <= f) lo_b = mid;
    else hi_b = mid;
  }
  const CmpReq r = c.req[lo_b];
  const long long k = f - r.fix_start;
  const long long R = 32 * k;
  if (k < 1 || R >= req_len[lo_b]) return;
  int glo, ghi;
  const long long orow = cmp_group_of(c, r, (int)(R - 1), glo, ghi);
  if (ghi <= R) return;  // no group crosses this boundary
  const int n = heads * head_dim;
  const float* p0 = c.fix + (f * 2) * n;
  const float* p1 = p0 + n;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(c.x_out) + orow * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = __float2bfloat16_rn(p0[i] + p1[i]);
}

}  // namespace

cudaError_t launch_cmp_fixup(const CmpArgs& c, int batch, const int* req_len, long long n_fix, int heads,
                             int head_dim, cudaStream_t st) {
  if (n_fix <= 0) return cudaSuccess;
  k_cmp_fixup<<<(unsigned)n_fix, 256, 0, st>>>(c, batch, req_len, n_fix, heads, head_dim);
  return cudaGetLastError();
}

cudaError_t launch_compress(const CompressArgs& a, int dtype, cudaStream_t st) {
  if (a.rows_out <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((a.rows_out + 7) / 8);  // 8 warps per block
  if (dtype == REC_ATTN_BF16) k_compress<__nv_bfloat16><<<blocks, 256, 0, st>>>(a);
  else k_compress<float><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace recattn
