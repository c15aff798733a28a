// attn_bwd.cu -- backward pass of the masked time-RoPE softmax attention on the CUDA
// cores (fp32 inputs, head_dim 32 or 64), and the row term D of both backward paths
// (the bf16 path runs on the tensor cores: attn_bwd_tc.cu).
//
// Gradients of O = Softmax(QK^T/sqrt(d) + M) V (TM20K review page, section 2.1;
// LazFormer review page, Eq. 19-21) through the time-RoPE (CADET review page, time
// encoding): with P the forward probabilities, rebuilt from the forward's
// log-sum-exp as P_ij = exp(s_ij - lse_i) on visible pairs,
//   dV_j = sum_i P_ij dO_i,  dP_ij = <dO_i, V_j>,  D_i = <dO_i, O_i>,
//   dS_ij = P_ij (dP_ij - D_i),  dQ'_i = scale sum_j dS_ij K'_j,  dK'_j = scale sum_i dS_ij Q'_i,
// and dQ = R(t_i)^T dQ', dK = R(t_j)^T dK' (the rotation is orthogonal).
//
// Three kernels walk the planner's tile lists, so SKIP tiles cost nothing here either:
//   k_bwd_delta  D_i per (token, head), fp32 or bf16 rows;
//   k_bwd_dq     one block per (query tile, head), d/32 threads per query row, over the
//                query tile's non-SKIP key tiles (K', V and key metadata staged in
//                shared memory);
//   k_bwd_dkv    one block per (key tile, head), d/32 threads per key row, over the
//                query tiles whose class against this key tile is not SKIP (Q', dO,
//                lse, D and query metadata staged in shared memory).
// FULL tiles skip the per-pair mask predicate.  Rows with no visible key (lse = -inf)
// contribute nothing.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "launchers.cuh"

namespace recattn {

namespace {

template <typename E>
__device__ __forceinline__ float ld_elem(const void* base, long long i);
template <>
__device__ __forceinline__ float ld_elem<float>(const void* base, long long i) {
  return static_cast<const float*>(base)[i];
}
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const void* base, long long i) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}
template <typename E>
__device__ __forceinline__ void st_elem(void* base, long long i, float x);
template <>
__device__ __forceinline__ void st_elem<float>(void* base, long long i, float x) {
  static_cast<float*>(base)[i] = x;
}

// Each row (query or key) is handled by kSplit = D / 32 neighbouring threads; part p
// of a row holds its 32 contiguous dims [32 p, 32 p + 32), so a thread reads its share
// of a staged row with 16-byte shared-memory loads (all threads of a part read the same
// address: a broadcast), a rotation pair never straddles two threads, and dot products
// need log2(kSplit) shuffles.
template <int D>
struct Split {
  static constexpr int kSplit = D / 32;
  static constexpr int kThreads = kTile * kSplit;
};

template <int S>
__device__ __forceinline__ float part_sum(float v) {
#pragma unroll
  for (int o = 1; o < S; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// y <- R(t)^T y over adjacent pairs (the inverse of the prologue's rotation), on the
// 32 dims [32 part, 32 part + 32) this thread holds: pairs 16 part .. 16 part + 15.
__device__ __forceinline__ void rotate_back(float (&y)[32], int part, float dt, const float* omega) {
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    float sn, cs;
    sincosf(dt * omega[16 * part + p], &sn, &cs);
    const float u = y[2 * p], w = y[2 * p + 1];
    y[2 * p] = u * cs + w * sn;
    y[2 * p + 1] = -u * sn + w * cs;
  }
}

// 32 contiguous floats of a staged shared-memory row, as eight 16-byte loads.
__device__ __forceinline__ void lds32(const float* p, float (&x)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = reinterpret_cast<const float4*>(p)[i];
    x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
}

// The request of global tile g (binary search over the request table).
__device__ __forceinline__ int tile_request(const ReqMeta* meta, int batch, long long g) {
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (meta[mid].tile_start <= g) lo = mid;
    else hi = mid;
  }
  return lo;
}

template <typename E, int D>
__global__ void __launch_bounds__(128) k_bwd_delta(BwdArgs a) {
  const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (token, head) row
  if (r >= a.rows) return;
  float acc = 0.f;
#pragma unroll 8
  for (int e = 0; e < D; ++e) acc = fmaf(ld_elem<E>(a.dout, r * D + e), ld_elem<E>(a.out, r * D + e), acc);
  a.delta[r] = acc;
}

template <int D>
struct BwdSmem {
  // K', V (dQ kernel) or Q' * scale, dO (dK/dV kernel); rows padded to keep 16-byte alignment
  __align__(16) float a[kTile][D + 4];
  __align__(16) float b[kTile][D + 4];
  long long t[kTile];
  int ty[kTile];
  float lse[kTile], dlt[kTile];
};

// dQ: block = (query tile g, head h); kSplit threads per query row.
template <typename E, int D>
__global__ void __launch_bounds__(Split<D>::kThreads) k_bwd_dq(BwdArgs a) {
  constexpr int S = Split<D>::kSplit;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
  const long long g = blockIdx.x;
  const int h = blockIdx.y, H = a.heads;
  const int b = tile_request(a.meta, a.batch, g);
  const ReqMeta m = a.meta[b];
  const int qt = (int)(g - m.tile_start), r = threadIdx.x / S, part = threadIdx.x % S, pi = qt * kTile + r;
  const bool row_ok = pi < m.len;
  const long long tok = m.tok_start + pi, row = tok * H + h;
  float q[32], go[32], acc[32];
  long long ti = 0;
  int tyi = -1;
  float lse = -INFINITY, dlt = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) { q[e] = 0.f; go[e] = 0.f; acc[e] = 0.f; }
  if (row_ok) {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      q[e] = ld_elem<E>(a.q, row * D + 32 * part + e) * a.scale;
      go[e] = ld_elem<E>(a.dout_attn, row * D + 32 * part + e);
    }
    ti = a.t[tok];
    tyi = a.ty[tok];
    if (query_kept(tyi, pi, a.qkeep[b])) {  // a pruned query has no output: no gradient
      lse = a.lse[row];
      dlt = a.delta[row];
    }
  }
  const bool live = row_ok && lse != -INFINITY;
  bool thr_ok; long long thr;
  delay_bound(ti, a.mask.delay, thr_ok, thr);
  const int n = a.kcount[g];
  const uint32_t* list = a.klist + m.cls_start + (long long)qt * m.ntiles;
  for (int j = 0; j < n; ++j) {
    const uint32_t ent = list[j];
    const int kt = (int)(ent & 0xffffffu), cl = (int)(ent >> 24);
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * D; idx += blockDim.x) {
      const int c = idx / D, e = idx - c * D;
      const int pj = kt * kTile + c;
      const bool ok = pj < m.len;
      const long long src = ((m.tok_start + pj) * H + h) * D + e;
      sm.a[c][e] = ok ? ld_elem<E>(a.k, src) : 0.f;
      sm.b[c][e] = ok ? ld_elem<E>(a.v, src) : 0.f;
    }
    for (int c = threadIdx.x; c < kTile; c += blockDim.x) {
      const int pj = kt * kTile + c;
      const bool ok = pj < m.len;
      sm.t[c] = ok ? a.t[m.tok_start + pj] : 0;
      sm.ty[c] = ok ? (int)a.ty[m.tok_start + pj] : -1;
    }
    __syncthreads();
    // every part of a row takes the same branches, so the shuffles below see whole pairs
    for (int c = 0; c < kTile; ++c) {
      bool vis = live;
      if (vis && cl != REC_ATTN_TILE_FULL)
        vis = vis_pred(a.mask, pi, ti, tyi, thr_ok, thr, kt * kTile + c, sm.t[c], sm.ty[c]);
      float kc[32], vc[32];
      lds32(&sm.a[c][32 * part], kc);
      lds32(&sm.b[c][32 * part], vc);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        s = fmaf(q[e], kc[e], s);
        dp = fmaf(go[e], vc[e], dp);
      }
      s = part_sum<S>(s);
      dp = part_sum<S>(dp);
      const float ds = vis ? __expf(s - lse) * (dp - dlt) * a.scale : 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] = fmaf(ds, kc[e], acc[e]);
    }
  }
  if (!row_ok) return;
  if (a.rotate) rotate_back(acc, part, (float)(ti - a.t[m.tok_start]), a.omega);
#pragma unroll
  for (int e = 0; e < 32; ++e) st_elem<E>(a.dq, row * D + 32 * part + e, acc[e]);
}

// dK, dV: block = (key tile g, head h); kSplit threads per key row.
template <typename E, int D>
__global__ void __launch_bounds__(Split<D>::kThreads) k_bwd_dkv(BwdArgs a) {
  constexpr int S = Split<D>::kSplit;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
  const long long g = blockIdx.x;
  const int h = blockIdx.y, H = a.heads;
  const int b = tile_request(a.meta, a.batch, g);
  const ReqMeta m = a.meta[b];
  const int kt = (int)(g - m.tile_start), r = threadIdx.x / S, part = threadIdx.x % S, pj = kt * kTile + r;
  const bool row_ok = pj < m.len;
  const long long tok = m.tok_start + pj, row = tok * H + h;
  float k[32], v[32], dk[32], dv[32];
  long long tj = 0;
  int tyj = -1;
#pragma unroll
  for (int e = 0; e < 32; ++e) { k[e] = 0.f; v[e] = 0.f; dk[e] = 0.f; dv[e] = 0.f; }
  if (row_ok) {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      k[e] = ld_elem<E>(a.k, row * D + 32 * part + e);
      v[e] = ld_elem<E>(a.v, row * D + 32 * part + e);
    }
    tj = a.t[tok];
    tyj = a.ty[tok];
  }
  const uint8_t* col = a.cls + m.cls_start + kt;  // column kt of the request's class matrix
  for (int qt = 0; qt < m.ntiles; ++qt) {
    const int cl = col[(long long)qt * m.ntiles];
    if (cl == REC_ATTN_TILE_SKIP) continue;
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * D; idx += blockDim.x) {
      const int c = idx / D, e = idx - c * D;
      const int pi = qt * kTile + c;
      const bool ok = pi < m.len;
      const long long src = ((m.tok_start + pi) * H + h) * D + e;
      sm.a[c][e] = ok ? ld_elem<E>(a.q, src) * a.scale : 0.f;
      sm.b[c][e] = ok ? ld_elem<E>(a.dout_attn, src) : 0.f;
    }
    for (int c = threadIdx.x; c < kTile; c += blockDim.x) {
      const int pi = qt * kTile + c;
      const bool ok = pi < m.len;
      const long long qrow = (m.tok_start + pi) * H + h;
      sm.t[c] = ok ? a.t[m.tok_start + pi] : 0;
      sm.ty[c] = ok ? (int)a.ty[m.tok_start + pi] : -1;
      const bool kept = ok && query_kept(sm.ty[c], pi, a.qkeep[b]);  // pruned queries give no gradient
      sm.lse[c] = kept ? a.lse[qrow] : -INFINITY;
      sm.dlt[c] = kept ? a.delta[qrow] : 0.f;
    }
    __syncthreads();
    for (int c = 0; c < kTile; ++c) {
      const float lse = sm.lse[c];
      bool vis = row_ok && lse != -INFINITY;  // a query that sees no key contributes nothing
      if (vis && cl != REC_ATTN_TILE_FULL) {
        bool thr_ok; long long thr;
        delay_bound(sm.t[c], a.mask.delay, thr_ok, thr);
        vis = vis_pred(a.mask, qt * kTile + c, sm.t[c], sm.ty[c], thr_ok, thr, pj, tj, tyj);
      }
      float qc[32], gc[32];
      lds32(&sm.a[c][32 * part], qc);
      lds32(&sm.b[c][32 * part], gc);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        s = fmaf(qc[e], k[e], s);
        dp = fmaf(gc[e], v[e], dp);
      }
      s = part_sum<S>(s);
      dp = part_sum<S>(dp);
      const float p = vis ? __expf(s - lse) : 0.f;
      const float ds = p * (dp - sm.dlt[c]);  // sm.a already carries the scale
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        dv[e] = fmaf(p, gc[e], dv[e]);
        dk[e] = fmaf(ds, qc[e], dk[e]);
      }
    }
  }
  if (!row_ok) return;
  if (a.rotate) rotate_back(dk, part, (float)(tj - a.t[m.tok_start]), a.omega);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    st_elem<E>(a.dk, row * D + 32 * part + e, dk[e]);
    st_elem<E>(a.dv, row * D + 32 * part + e, dv[e]);
  }
}

template <typename E, int D>
cudaError_t launch_delta_t(const BwdArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  k_bwd_delta<E, D><<<(unsigned)((a.rows + 127) / 128), 128, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename E, int D>
cudaError_t launch_bwd_t(const BwdArgs& a, long long n_tiles, cudaStream_t st) {
  if (n_tiles <= 0) return cudaSuccess;
  const dim3 grid((unsigned)n_tiles, (unsigned)a.heads);
  const int smem = (int)sizeof(BwdSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(k_bwd_dq<E, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_bwd_dkv<E, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k_bwd_dq<E, D><<<grid, Split<D>::kThreads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_bwd_dkv<E, D><<<grid, Split<D>::kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_delta(const BwdArgs& a, int dtype, int head_dim, cudaStream_t st) {
  if (dtype == REC_ATTN_BF16) {
    if (head_dim == 64) return launch_delta_t<__nv_bfloat16, 64>(a, st);
  } else {
    if (head_dim == 32) return launch_delta_t<float, 32>(a, st);
    if (head_dim == 64) return launch_delta_t<float, 64>(a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_bwd_simt(const BwdArgs& a, int head_dim, long long n_tiles, cudaStream_t st) {
  if (head_dim == 32) return launch_bwd_t<float, 32>(a, n_tiles, st);
  if (head_dim == 64) return launch_bwd_t<float, 64>(a, n_tiles, st);
  return cudaErrorInvalidValue;
}

}  // namespace recattn
