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

// 16 bytes of a head row: 8 bf16 or 4 fp32 values, i.e. 4 or 2 rotation pairs.
template <typename E>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kPairs = 4;
  static __device__ __forceinline__ void load(const void* p, float (&x)[8]) {
    unpack(*reinterpret_cast<const uint4*>(p), x);
  }
  // the 16 raw bytes of a chunk, as values
  static __device__ __forceinline__ void unpack(const uint4 v, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(void* p, const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Chunk<float> {
  static constexpr int kPairs = 2;
  static __device__ __forceinline__ void load(const void* p, float (&x)[8]) {
    unpack(*reinterpret_cast<const uint4*>(p), x);
  }
  static __device__ __forceinline__ void unpack(const uint4 v, float (&x)[8]) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y); x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ void store(void* p, const float (&x)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};

// One (token, chunk) unit of the prologue: K' and, when WQ, Q' for every head.  The
// first four heads' 16-byte loads go out before the angle math (they do not depend on
// the time), later heads four at a time, all kept raw until used.
template <typename E, bool WQ>
__device__ __forceinline__ void rope_rows(const RopeArgs& a, const char* __restrict__ q, const char* __restrict__ k,
                                          char* __restrict__ qr, char* __restrict__ kr, long long head_bytes,
                                          long long tok, long long row0, int c, long long t_ref) {
  using C = Chunk<E>;
  constexpr int kPairs = C::kPairs;
  uint4 rq[4], rk[4];  // raw 16-byte chunks of four heads
  auto load4 = [&](int h0) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (h0 + u < a.heads) {
        if constexpr (WQ) rq[u] = *reinterpret_cast<const uint4*>(q + row0 + (h0 + u) * head_bytes);
        rk[u] = *reinterpret_cast<const uint4*>(k + row0 + (h0 + u) * head_bytes);
      }
  };
  load4(0);
  const float dt = (float)(a.t[tok] - t_ref);  // exact int64 difference, then fp32
  float sn[kPairs], cs[kPairs];
#pragma unroll
  for (int p = 0; p < kPairs; ++p) sincosf(dt * a.omega[c * kPairs + p], &sn[p], &cs[p]);
  for (int h0 = 0; h0 < a.heads; h0 += 4) {
    if (h0 > 0) load4(h0);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (h0 + u >= a.heads) break;
      float y[8];
      C::unpack(rk[u], y);
      if constexpr (WQ) {
        float x[8];
        C::unpack(rq[u], x);
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          const float x0 = x[2 * p], x1 = x[2 * p + 1];
          x[2 * p] = x0 * cs[p] - x1 * sn[p];
          x[2 * p + 1] = x0 * sn[p] + x1 * cs[p];
        }
        C::store(qr + row0 + (h0 + u) * head_bytes, x);
      }
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        const float y0 = y[2 * p], y1 = y[2 * p + 1];
        y[2 * p] = y0 * cs[p] - y1 * sn[p];
        y[2 * p + 1] = y0 * sn[p] + y1 * cs[p];
      }
      C::store(kr + row0 + (h0 + u) * head_bytes, y);
    }
  }
}

// Thread work unit: one token and one 16-byte chunk of its head rows, for every head,
// so each angle's sin/cos is computed once per token.  A block covers 256 / chunks
// tokens of one tile (chunks = 16-byte chunks per head row, 8 or 16), so a tile takes
// chunks / 2 blocks and each thread one unit (`rope_rows`).
template <typename E>
__global__ void __launch_bounds__(256, 4) k_rope(RopeArgs a) {
  using C = Chunk<E>;
  constexpr int kPairs = C::kPairs;
  const int chunks = a.head_dim / (2 * kPairs);
  const int tpb = (int)blockDim.x / chunks;  // tokens per block
  const int bpt = kTile / tpb;               // blocks per tile
  const long long g = blockIdx.x / bpt;
  const ReqMeta m = a.meta[a.tile_req[g]];
  const int tl = (int)(g - m.tile_start);
  const int rows = min(kTile, m.len - tl * kTile);
  const int r = (int)(blockIdx.x % bpt) * tpb + (int)threadIdx.x / chunks;
  const int c = (int)threadIdx.x % chunks;
  if (r >= rows) return;
  const char* __restrict__ q = static_cast<const char*>(a.q);
  const char* __restrict__ k = static_cast<const char*>(a.k);
  char* __restrict__ qr = static_cast<char*>(a.qr);
  char* __restrict__ kr = static_cast<char*>(a.kr);
  const long long head_bytes = (long long)a.head_dim * (long long)sizeof(E);
  const long long tok = m.tok_start + tl * kTile + r;
  const long long row0 = tok * a.heads * head_bytes + (long long)c * 16;
  const long long t_ref = a.t[m.tok_start];
  // a plan in which no user token queries never reads their Q' rows (their query tiles
  // are skipped or their rows are computed and not written), so they are not rotated
  if (a.skip_user_q && is_user(a.ty[tok])) rope_rows<E, false>(a, q, k, qr, kr, head_bytes, tok, row0, c, t_ref);
  else rope_rows<E, true>(a, q, k, qr, kr, head_bytes, tok, row0, c, t_ref);
}

// Sum of v over the `group` consecutive lanes that hold one head row (group is a
// power of two dividing 32 and every lane of the warp takes part).
__device__ __forceinline__ float group_sum(float v, int group) {
  for (int off = group >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// x <- x / sqrt(mean over the head row of x^2 + eps) * w, then x <- x * sigmoid(g):
// the fused QK-RMSNorm and sigmoid gate of one 16-byte chunk of a head row (g holds
// the chunk's gate pre-activations when `gated`).
template <typename E>
__device__ __forceinline__ void norm_gate(float (&x)[8], bool act, const float* w, float eps, bool gated,
                                          const float (&g)[8], int e0, int chunks, int d) {
  constexpr int kElems = 2 * Chunk<E>::kPairs;
  if (w) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < kElems; ++e) ss = fmaf(x[e], x[e], ss);
    ss = group_sum(ss, chunks);
    const float r = rsqrtf(ss / (float)d + eps);
    if (act) {
#pragma unroll
      for (int e = 0; e < kElems; ++e) x[e] *= r * w[e0 + e];
    }
  }
  if (gated) {
#pragma unroll
    for (int e = 0; e < kElems; ++e) x[e] *= sigmoid_io<E>(g[e]);
  }
}

// The prologue with the fused steps: per (token, head) row, QK-RMSNorm and the
// sigmoid gate on Q and K, then the rotation (omega all zero: none).  Every lane of
// a warp runs every iteration (inactive lanes carry zeros), so the row sums can use
// warp shuffles over the lanes of one row.
template <typename E>
__global__ void __launch_bounds__(256, 3) k_rope_fused(RopeArgs a, FusedArgs f) {
  using C = Chunk<E>;
  constexpr int kPairs = C::kPairs;
  // one (token, chunk) unit per thread, 256 / chunks tokens of one tile per block (as in
  // k_rope); a block's warps hold whole head rows, so every lane runs the row sums
  const int chunks = a.head_dim / (2 * kPairs);
  const int tpb = (int)blockDim.x / chunks;  // tokens per block
  const int bpt = kTile / tpb;               // blocks per tile
  const long long g = blockIdx.x / bpt;
  const ReqMeta m = a.meta[a.tile_req[g]];
  const int tl = (int)(g - m.tile_start);
  const int rows = min(kTile, m.len - tl * kTile);
  const long long head_bytes = (long long)a.head_dim * (long long)sizeof(E);
  {
    const int rr = (int)(blockIdx.x % bpt) * tpb + (int)threadIdx.x / chunks;
    const bool act = rr < rows;  // inactive lanes carry zeros through the row sums
    const int r = act ? rr : 0, c = (int)threadIdx.x % chunks;
    const long long tok = m.tok_start + tl * kTile + r;
    const long long row0 = tok * a.heads * head_bytes + (long long)c * 16;
    const bool qg = f.q_gate != nullptr, kg = f.k_gate != nullptr;
    // two heads at a time: their q, k and gate chunks (up to eight 16-byte loads) in flight
    // together, kept raw until used; the first two heads' loads go out before the angles
    uint4 rq[2], rk[2], rgq[2], rgk[2];
    auto load2 = [&](int h0) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        rq[u] = rk[u] = rgq[u] = rgk[u] = make_uint4(0u, 0u, 0u, 0u);
        if (act && h0 + u < a.heads) {
          const long long off = row0 + (h0 + u) * head_bytes;
          rq[u] = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.q) + off);
          rk[u] = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.k) + off);
          if (qg) rgq[u] = *reinterpret_cast<const uint4*>(static_cast<const char*>(f.q_gate) + off);
          if (kg) rgk[u] = *reinterpret_cast<const uint4*>(static_cast<const char*>(f.k_gate) + off);
        }
      }
    };
    load2(0);
    const float dt = act ? (float)(a.t[tok] - a.t[m.tok_start]) : 0.f;
    float sn[kPairs], cs[kPairs];
#pragma unroll
    for (int p = 0; p < kPairs; ++p) sincosf(dt * a.omega[c * kPairs + p], &sn[p], &cs[p]);
    for (int h0 = 0; h0 < a.heads; h0 += 2) {
      if (h0 > 0) load2(h0);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (h0 + u >= a.heads) break;  // uniform across the block
        const int h = h0 + u;
        const long long off = row0 + h * head_bytes;
        float x[8], y[8], gx[8], gy[8];
        C::unpack(rq[u], x);
        C::unpack(rk[u], y);
        C::unpack(rgq[u], gx);
        C::unpack(rgk[u], gy);
        const int e0 = h * a.head_dim + c * 2 * kPairs;
        norm_gate<E>(x, act, f.q_norm_w, f.eps, qg, gx, e0, chunks, a.head_dim);
        norm_gate<E>(y, act, f.k_norm_w, f.eps, kg, gy, e0, chunks, a.head_dim);
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
          const float x0 = x[2 * p], x1 = x[2 * p + 1], y0 = y[2 * p], y1 = y[2 * p + 1];
          x[2 * p] = x0 * cs[p] - x1 * sn[p];
          x[2 * p + 1] = x0 * sn[p] + x1 * cs[p];
          y[2 * p] = y0 * cs[p] - y1 * sn[p];
          y[2 * p + 1] = y0 * sn[p] + y1 * cs[p];
        }
        if (act) {
          C::store(static_cast<char*>(a.qr) + off, x);
          C::store(static_cast<char*>(a.kr) + off, y);
        }
      }
    }
  }
}

// Rows of one 128-row chunk of a region into the cache's combined layout (serving
// with a cached history): rotated K (and Q), copied V, times and types; padding rows
// past the region's source rows get zeros.  One (row, 16-byte chunk) unit per thread
// over every head, 256 / chunks rows per block as in k_rope.
template <typename E>
__global__ void __launch_bounds__(256, 4) k_rope_slots(SlotArgs a) {
  using C = Chunk<E>;
  constexpr int kPairs = C::kPairs;
  const int chunks = a.head_dim / (2 * kPairs);
  const int tpb = (int)blockDim.x / chunks;
  const int bpt = kTile / tpb;
  const long long g = blockIdx.x / bpt;
  const SlotReq rq = a.req[a.chunk_req[g]];
  const int row = a.chunk_row0[g] + (int)(blockIdx.x % bpt) * tpb + (int)threadIdx.x / chunks;
  const int c = (int)threadIdx.x % chunks;
  if (row >= rq.cap) return;
  const long long head_bytes = (long long)a.head_dim * (long long)sizeof(E);
  const long long dst = rq.dst_start + row;
  const long long d0 = dst * a.heads * head_bytes + (long long)c * 16;
  if (row >= rq.len) {  // padding
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int h = 0; h < a.heads; ++h) {
      *reinterpret_cast<uint4*>(static_cast<char*>(a.k_dst) + d0 + h * head_bytes) = z;
      *reinterpret_cast<uint4*>(static_cast<char*>(a.v_dst) + d0 + h * head_bytes) = z;
      if (a.q_dst) *reinterpret_cast<uint4*>(static_cast<char*>(a.q_dst) + d0 + h * head_bytes) = z;
    }
    if (c == 0) {
      const long long t_ref = rq.ref_dst ? a.t_dst[rq.ref_row] : a.t_src[rq.ref_row];
      a.t_dst[dst] = rq.len > 0 ? a.t_src[rq.src_start + rq.len - 1] : t_ref;
      a.ty_dst[dst] = (int8_t)a.ty_const;
    }
    return;
  }
  const long long src = rq.src_start + row;
  const long long s0 = src * a.heads * head_bytes + (long long)c * 16;
  const long long t_ref = rq.ref_dst ? a.t_dst[rq.ref_row] : a.t_src[rq.ref_row];
  const long long ts = a.t_src[src];
  const float dt = (float)(ts - t_ref);  // exact int64 difference, then fp32
  float sn[kPairs], cs[kPairs];
#pragma unroll
  for (int p = 0; p < kPairs; ++p) sincosf(dt * a.omega[c * kPairs + p], &sn[p], &cs[p]);
  for (int h = 0; h < a.heads; ++h) {
    const long long so = s0 + h * head_bytes, dof = d0 + h * head_bytes;
    const uint4 rk = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.k_src) + so);
    const uint4 rv = *reinterpret_cast<const uint4*>(static_cast<const char*>(a.v_src) + so);
    float y[8];
    C::unpack(rk, y);
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      const float y0 = y[2 * p], y1 = y[2 * p + 1];
      y[2 * p] = y0 * cs[p] - y1 * sn[p];
      y[2 * p + 1] = y0 * sn[p] + y1 * cs[p];
    }
    C::store(static_cast<char*>(a.k_dst) + dof, y);
    *reinterpret_cast<uint4*>(static_cast<char*>(a.v_dst) + dof) = rv;
    if (a.q_src) {
      float x[8];
      C::load(static_cast<const char*>(a.q_src) + so, x);
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        const float x0 = x[2 * p], x1 = x[2 * p + 1];
        x[2 * p] = x0 * cs[p] - x1 * sn[p];
        x[2 * p + 1] = x0 * sn[p] + x1 * cs[p];
      }
      C::store(static_cast<char*>(a.q_dst) + dof, x);
    }
  }
  if (c == 0) {
    a.t_dst[dst] = ts;
    a.ty_dst[dst] = a.ty_src ? a.ty_src[src] : (int8_t)a.ty_const;
  }
}

// The outputs of a region's source rows back from the combined layout (16 bytes per
// thread; the lse of a row by its first chunk's thread).
__global__ void __launch_bounds__(256) k_slots_gather(SlotArgs a, int elem) {
  const int chunks = a.head_dim * elem / 16;
  const int tpb = (int)blockDim.x / chunks;
  const int bpt = kTile / tpb;
  const long long g = blockIdx.x / bpt;
  const SlotReq rq = a.req[a.chunk_req[g]];
  const int row = a.chunk_row0[g] + (int)(blockIdx.x % bpt) * tpb + (int)threadIdx.x / chunks;
  const int c = (int)threadIdx.x % chunks;
  if (row >= rq.len) return;
  const long long head_bytes = (long long)a.head_dim * elem;
  const long long src = rq.src_start + row, dst = rq.dst_start + row;
  for (int h = 0; h < a.heads; ++h)
    *reinterpret_cast<uint4*>(static_cast<char*>(a.o_out) + (src * a.heads + h) * head_bytes + c * 16) =
        *reinterpret_cast<const uint4*>(static_cast<const char*>(a.o_comb) + (dst * a.heads + h) * head_bytes +
                                        c * 16);
  if (a.lse_out && c == 0)
    for (int h = 0; h < a.heads; ++h) a.lse_out[src * a.heads + h] = a.lse_comb[dst * a.heads + h];
}

}  // namespace

cudaError_t launch_rope_slots(const SlotArgs& a, int dtype, long long n_chunks, cudaStream_t st) {
  if (n_chunks <= 0) return cudaSuccess;
  const int chunks = a.head_dim * (dtype == REC_ATTN_BF16 ? 2 : 4) / 16;
  const unsigned blocks = (unsigned)(n_chunks * (chunks / 2));
  if (dtype == REC_ATTN_BF16) k_rope_slots<__nv_bfloat16><<<blocks, 256, 0, st>>>(a);
  else k_rope_slots<float><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_slots_gather(const SlotArgs& a, int dtype, long long n_chunks, cudaStream_t st) {
  if (n_chunks <= 0) return cudaSuccess;
  const int elem = dtype == REC_ATTN_BF16 ? 2 : 4;
  const int chunks = a.head_dim * elem / 16;
  const unsigned blocks = (unsigned)(n_chunks * (chunks / 2));
  k_slots_gather<<<blocks, 256, 0, st>>>(a, elem);
  return cudaGetLastError();
}

cudaError_t launch_rope_fused(const RopeArgs& a, const FusedArgs& f, int dtype, long long n_tiles, cudaStream_t st) {
  if (n_tiles <= 0) return cudaSuccess;
  const int chunks = a.head_dim * (dtype == REC_ATTN_BF16 ? 2 : 4) / 16;
  const unsigned blocks = (unsigned)(n_tiles * (chunks / 2));  // 256 / chunks tokens per block
  if (dtype == REC_ATTN_BF16) k_rope_fused<__nv_bfloat16><<<blocks, 256, 0, st>>>(a, f);
  else k_rope_fused<float><<<blocks, 256, 0, st>>>(a, f);
  return cudaGetLastError();
}

cudaError_t launch_rope(const RopeArgs& a, int dtype, long long n_tiles, cudaStream_t st) {
  if (n_tiles <= 0) return cudaSuccess;
  // 256 threads = 256 / chunks tokens per block, chunks / 2 blocks per tile
  const int chunks = a.head_dim * (dtype == REC_ATTN_BF16 ? 2 : 4) / 16;
  const unsigned blocks = (unsigned)(n_tiles * (chunks / 2));
  if (dtype == REC_ATTN_BF16) k_rope<__nv_bfloat16><<<blocks, 256, 0, st>>>(a);
  else k_rope<float><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace recattn
