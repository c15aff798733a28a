// rope.cu -- time-RoPE prologue: Q' = RoPE(Q, t), K' = RoPE(K, t) for every token.
//
// CADET review page, section on time encoding and self-gating: component pair i of
// a query or key turns by alpha_i(t) = t * phi_min / dt_max * base^(2i/d).  Scores
// depend only on t_i - t_j, so each request is rotated relative to its first token:
// dt = t - t_ref is formed exactly in int64 and only then converted to fp32, which
// keeps Unix-scale timestamps (~1.7e9 s) from losing precision in the angle.  The
// per-pair angular speed omega_i is computed on the host in fp64 and rounded once.
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace recattn {

namespace {

template <typename E>
struct Pair;
template <>
struct Pair<__nv_bfloat16> {
  using V = __nv_bfloat162;
  static __device__ __forceinline__ float2 load(const V* p) { return __bfloat1622float2(*p); }
  static __device__ __forceinline__ void store(V* p, float a, float b) { *p = __floats2bfloat162_rn(a, b); }
};
template <>
struct Pair<float> {
  using V = float2;
  static __device__ __forceinline__ float2 load(const V* p) { return *p; }
  static __device__ __forceinline__ void store(V* p, float a, float b) { *p = make_float2(a, b); }
};

// One block per global tile; threads walk (token, pair) and loop over heads so each
// angle's sin/cos is computed once per token and pair.
template <typename E>
__global__ void __launch_bounds__(256) k_rope(RopeArgs a) {
  using P = Pair<E>;
  using V = typename P::V;
  const long long g = blockIdx.x;
  const ReqMeta m = a.meta[a.qreq[g]];
  const int tl = (int)(g - m.tile_start);
  const long long t_ref = a.t[m.tok_start];
  const int half = a.head_dim >> 1;
  const V* q = reinterpret_cast<const V*>(a.q);
  const V* k = reinterpret_cast<const V*>(a.k);
  V* qr = reinterpret_cast<V*>(a.qr);
  V* kr = reinterpret_cast<V*>(a.kr);
  for (int idx = threadIdx.x; idx < kTile * half; idx += blockDim.x) {
    const int r = idx / half, i = idx - r * half;
    const int pos = tl * kTile + r;
    if (pos >= m.len) break;
    const long long tok = m.tok_start + pos;
    const long long dt = a.t[tok] - t_ref;
    float s, c;
    sincosf((float)dt * a.omega[i], &s, &c);
    for (int h = 0; h < a.heads; ++h) {
      const long long e = (tok * a.heads + h) * half + i;
      const float2 x = P::load(q + e);
      P::store(qr + e, x.x * c - x.y * s, x.x * s + x.y * c);
      const float2 y = P::load(k + e);
      P::store(kr + e, y.x * c - y.y * s, y.x * s + y.y * c);
    }
  }
}

}  // namespace

cudaError_t launch_rope(const RopeArgs& a, int dtype, long long n_tiles, cudaStream_t st) {
  if (n_tiles <= 0) return cudaSuccess;
  if (dtype == REC_ATTN_BF16) k_rope<__nv_bfloat16><<<(unsigned)n_tiles, 256, 0, st>>>(a);
  else k_rope<float><<<(unsigned)n_tiles, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace recattn
