// bwd_fused.cu -- backward through the fused steps of rec_attn_fwd_fused, around the
// attention backward: the output gate before it, QK-RMSNorm and the Q/K sigmoid gates
// after it.
//
// Forward (SORT review page, section 3.3.2 "Attention Gate & QK Norm"; TM20K review
// page, QK Norm; CADET review page, self-gating): per head row a of Q or K,
// n = a / r * w with r = sqrt(mean(a^2) + eps), g = n * sigmoid(c), then the time-RoPE;
// the attention output A is gated, O = A * sigmoid(c_o).  The chain rule gives
//   dA = dO * sigmoid(c_o),  dc_o = dO * A * sigmoid'(c_o) = dO * O * (1 - sigmoid(c_o)),
//   dn = dg * sigmoid(c),    dc = dg * n * sigmoid(c) (1 - sigmoid(c)),
//   da = w * dn / r - a * sum(dn * w * a) / (d r^3),  dw = sum over tokens of dn * a / r,
// where dg is the attention backward's gradient of the rotated-back Q or K.  The
// sigmoid is the forward's (bf16: one hardware tanh; fp32: one exponential).
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "launchers.cuh"

namespace recattn {

namespace {

template <typename E>
__device__ __forceinline__ float ld(const void* p, long long i) {
  if constexpr (sizeof(E) == 2) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  else return static_cast<const float*>(p)[i];
}
template <typename E>
__device__ __forceinline__ void st(void* p, long long i, float x) {
  if constexpr (sizeof(E) == 2) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else static_cast<float*>(p)[i] = x;
}
template <typename E>
__device__ __forceinline__ float sig(float x) {
  return sigmoid_io<E>(x);  // the forward's
}

template <typename E>
__global__ void __launch_bounds__(256) k_bwd_gate(GateArgs a) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < a.n; i += (long long)gridDim.x * blockDim.x) {
    const float go = ld<E>(a.dout, i), o = ld<E>(a.out, i), s = sig<E>(ld<E>(a.gate, i));
    st<E>(a.dout_attn, i, go * s);
    st<E>(a.dgate, i, go * o * (1.f - s));
  }
}

// Block = 8 warps over 16 tokens each of one head (blockIdx.y); a lane holds d / 32
// elements of a row.  The gain gradient is summed per lane over the warp's tokens,
// then over the block's warps in shared memory, then added to dw once per block.
constexpr int kRowsPerWarp = 16;

template <typename E, int EPL>
__global__ void __launch_bounds__(256) k_bwd_norm_gate(NormGateArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y, H = a.heads, d = a.head_dim;
  __shared__ float s_dw[8][128];
  float dwp[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) dwp[i] = 0.f;
  const long long r0 = ((long long)blockIdx.x * 8 + warp) * kRowsPerWarp;
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const long long tok = r0 + rr;
    if (tok >= a.rows) break;  // uniform across the warp
    const long long base = (tok * H + h) * d;
    float av[EPL], dn[EPL], nv[EPL], sg[EPL];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      av[i] = ld<E>(a.a, base + e);
      ss = fmaf(av[i], av[i], ss);
    }
    float r = 1.f;
    if (a.w) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      r = sqrtf(ss / (float)d + a.eps);
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      const float w = a.w ? a.w[h * d + e] : 1.f;
      nv[i] = a.w ? av[i] / r * w : av[i];
      sg[i] = a.gate ? sig<E>(ld<E>(a.gate, base + e)) : 1.f;
      const float dg = ld<E>(a.dg, base + e);
      dn[i] = dg * sg[i];
      if (a.gate) st<E>(a.dgate, base + e, dg * nv[i] * sg[i] * (1.f - sg[i]));
      dot = fmaf(dn[i] * w, av[i], dot);
    }
    if (a.w) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    const float c3 = dot / ((float)d * r * r * r);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      if (a.w) {
        const float w = a.w[h * d + e];
        st<E>(a.da, base + e, w * dn[i] / r - av[i] * c3);
        dwp[i] = fmaf(dn[i], av[i] / r, dwp[i]);
      } else {
        st<E>(a.da, base + e, dn[i]);
      }
    }
  }
  if (!a.w) return;
#pragma unroll
  for (int i = 0; i < EPL; ++i) s_dw[warp][lane * EPL + i] = dwp[i];
  __syncthreads();
  for (int e = threadIdx.x; e < d; e += blockDim.x) {
    float sum = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) sum += s_dw[w8][e];
    atomicAdd(a.dw + h * d + e, sum);
  }
}

template <typename E>
cudaError_t launch_norm_gate_t(const NormGateArgs& a, cudaStream_t st) {
  const dim3 grid((unsigned)((a.rows + 8 * kRowsPerWarp - 1) / (8 * kRowsPerWarp)), (unsigned)a.heads);
  switch (a.head_dim) {
    case 32: k_bwd_norm_gate<E, 1><<<grid, 256, 0, st>>>(a); break;
    case 64: k_bwd_norm_gate<E, 2><<<grid, 256, 0, st>>>(a); break;
    case 128: k_bwd_norm_gate<E, 4><<<grid, 256, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_gate(const GateArgs& a, int dtype, cudaStream_t st) {
  if (a.n <= 0) return cudaSuccess;
  const long long blocks = (a.n + 255) / 256;
  const unsigned grid = (unsigned)(blocks < 65536 ? blocks : 65536);
  if (dtype == REC_ATTN_BF16) k_bwd_gate<__nv_bfloat16><<<grid, 256, 0, st>>>(a);
  else k_bwd_gate<float><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_norm_gate(const NormGateArgs& a, int dtype, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  return dtype == REC_ATTN_BF16 ? launch_norm_gate_t<__nv_bfloat16>(a, st) : launch_norm_gate_t<float>(a, st);
}

}  // namespace recattn
