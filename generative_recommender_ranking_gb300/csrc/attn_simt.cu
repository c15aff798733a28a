// attn_simt.cu -- fp32 masked softmax attention on the CUDA cores (fp32 inputs and
// outputs; tensor-core TF32 would not hold 1e-4 against the fp64 reference).
//
// Softmax(QK^T/sqrt(d) + M) V (TM20K review page, section 2.1; LazFormer review
// page, Eq. 19-21) over the plan's non-SKIP key tiles: one block per (query tile,
// head), one thread per query row, an exact online softmax in fp32 with expf.
// PARTIAL tiles evaluate the mask per element; FULL tiles skip it.
#include "attn_common.cuh"

namespace recattn {

namespace {

template <int D>
__global__ void __launch_bounds__(kTile) k_attn_simt(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  long long* s_t = reinterpret_cast<long long*>(smem);
  int* s_ty = reinterpret_cast<int*>(s_t + kTile);
  float (*s_k)[D + 1] = reinterpret_cast<float (*)[D + 1]>(s_ty + kTile);
  float (*s_v)[D] = reinterpret_cast<float (*)[D]>(&s_k[kTile][0]);
  const WorkItem it = decode_item(a, blockIdx.x, false);
  if (it.n < 0) return;  // every query of the tile is pruned
  const int r = threadIdx.x, pi = it.qt * kTile + r;
  const bool row_ok = pi < it.m.len;
  const long long tok = it.m.tok_start + pi;
  const int H = a.heads;
  const float* Q = static_cast<const float*>(a.q);
  const float* K = static_cast<const float*>(a.k);
  const float* Vv = static_cast<const float*>(a.v);
  float q[D], o[D];
  long long ti = 0;
  int tyi = -1;
#pragma unroll
  for (int e = 0; e < D; ++e) { q[e] = 0.f; o[e] = 0.f; }
  if (row_ok) {
    const float* src = Q + (tok * H + it.h) * D;
#pragma unroll
    for (int e = 0; e < D; ++e) q[e] = src[e] * a.scale;
    ti = a.t[tok];
    tyi = a.ty[tok];
  }
  bool thr_ok; long long thr;
  delay_bound(ti, a.mask.delay, thr_ok, thr);
  float mrun = -INFINITY, l = 0.f;
  for (int j = 0; j < it.n; ++j) {
    const uint32_t ent = it.list[j];
    const int kt = (int)(ent & 0xffffffu), cl = (int)(ent >> 24);
    __syncthreads();
    // stage the key tile: K', V rows and key metadata
    for (int idx = r; idx < kTile * D; idx += kTile) {
      const int c = idx / D, e = idx - c * D;
      const int pj = kt * kTile + c;
      const bool ok = pj < it.m.len;
      const long long src = ((it.m.tok_start + pj) * H + it.h) * D + e;
      s_k[c][e] = ok ? K[src] : 0.f;
      s_v[c][e] = ok ? Vv[src] : 0.f;
    }
    {
      const int pj = kt * kTile + r;
      const bool ok = pj < it.m.len;
      s_t[r] = ok ? a.t[it.m.tok_start + pj] : 0;
      s_ty[r] = ok ? (int)a.ty[it.m.tok_start + pj] : -1;
    }
    __syncthreads();
    if (!row_ok) continue;
    for (int c = 0; c < kTile; ++c) {
      if (cl != REC_ATTN_TILE_FULL &&
          !vis_pred(a.mask, pi, ti, tyi, thr_ok, thr, kt * kTile + c, s_t[c], s_ty[c]))
        continue;
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) s = fmaf(q[e], s_k[c][e], s);
      if (s > mrun) {
        const float corr = expf(mrun - s);
        l *= corr;
#pragma unroll
        for (int e = 0; e < D; ++e) o[e] *= corr;
        mrun = s;
      }
      const float p = expf(s - mrun);
      l += p;
#pragma unroll
      for (int e = 0; e < D; ++e) o[e] = fmaf(p, s_v[c][e], o[e]);
    }
  }
  if (!row_ok || !query_kept(tyi, pi, it.keep)) return;
  float* dst = static_cast<float*>(a.out) + (tok * H + it.h) * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (a.out_gate) {  // the attention output gate, O * sigmoid(g)
    const float* g = static_cast<const float*>(a.out_gate) + (tok * H + it.h) * D;
#pragma unroll
    for (int e = 0; e < D; ++e) dst[e] = o[e] * inv * sigmoid_io<float>(g[e]);
  } else {
#pragma unroll
    for (int e = 0; e < D; ++e) dst[e] = o[e] * inv;
  }
  if (a.lse) a.lse[tok * H + it.h] = l > 0.f ? mrun + logf(l) : -INFINITY;
}

template <int D>
cudaError_t launch(const AttnArgs& a, unsigned grid, cudaStream_t st) {
  const size_t smem = kTile * (sizeof(long long) + sizeof(int)) + kTile * (2 * D + 1) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_attn_simt<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_attn_simt<D><<<grid, kTile, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a, int head_dim, cudaStream_t st) {
  if (a.n_items <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)a.n_items;
  switch (head_dim) {
    case 32: return launch<32>(a, grid, st);
    case 64: return launch<64>(a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace recattn
