// attn_tc.cu -- bf16 masked softmax attention on the sm_103a tensor cores.
//
// Softmax(QK^T/sqrt(d) + M) V (TM20K review page, section 2.1; LazFormer review page,
// section 2.3, Eq. 19-21) for the plan's (query tile, head) work items, skipping the
// key tiles the plan classified SKIP (block skipping of the CADET serving kernel;
// SORT section 4.1).  Rows that see no key are written as zeros.
//
// One persistent CTA per SM, 6 warps with fixed roles:
//   warp 0      TMA producer: Q' tile once per item, K'/V tiles into an NS-stage ring;
//   warp 1      MMA issuer: S = Q'K'^T into one of two TMEM S buffers (tcgen05.mma,
//               kind::f16, fp32 accumulate), then O += P V into the TMEM O buffer;
//   warps 2..5  softmax: one query row per thread (TMEM lane quadrant = warp % 4).
//               tcgen05.ld of the S row, per-element mask on PARTIAL tiles, online
//               softmax in the exp2 domain, P rounded to bf16 into shared memory in the
//               128-byte-swizzled K-major layout the PV MMA reads, O rescaled in TMEM
//               when the running maximum grows, O / l in the epilogue.
// The row sum l is accumulated from the bf16-rounded P values the PV MMA consumes, so
// every output row is an exact convex combination of the value rows it saw.
// Every wait on an mbarrier is bounded (REC_ATTN_ERR_TIMEOUT in the status word).
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "ptx_sm103.cuh"

namespace recattn {

namespace {

constexpr int kThreads = 192;
constexpr int kSlab = kTile * 128;        // 128 rows x 128 B: one 64-column swizzle slab
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256;

template <int D, int NS>
struct Layout {
  static constexpr int kQBytes = kTile * D * 2;
  static constexpr int kKVBytes = kTile * D * 2;
  static constexpr int kPBytes = kTile * kTile * 2;
  static constexpr int kMetaWarp = kTile * 8 + kTile;  // int64 times + int8 types
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + NS * kKVBytes;
  static constexpr int kP = kV + NS * kKVBytes;
  static constexpr int kMeta = kP + kPBytes;
  static constexpr int kBars = (kMeta + 4 * kMetaWarp + 7) & ~7;
  static constexpr int kNumBars = 2 + 3 * NS + 2 + 1 + 1 + 1;
  static constexpr int kTotal = kBars + kNumBars * 8 + 16;
  static constexpr int kDynamic = kTotal + 1024;  // slack to align the base to 1024 B
};

template <int NS>
struct Bars {
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* k_full;
  uint64_t* v_full;
  uint64_t* kv_empty;
  uint64_t* s_full;  // [2]
  uint64_t* p_full;
  uint64_t* pv_done;
  uint64_t* mma_done;
  volatile int* abort_flag;
  uint32_t* tmem_slot;
  __device__ Bars(uint8_t* base) {
    uint64_t* b = reinterpret_cast<uint64_t*>(base);
    q_full = b; q_empty = b + 1; k_full = b + 2; v_full = k_full + NS; kv_empty = v_full + NS;
    s_full = kv_empty + NS; p_full = s_full + 2; pv_done = p_full + 1; mma_done = pv_done + 1;
    abort_flag = reinterpret_cast<volatile int*>(mma_done + 1);
    tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1) + 1;
  }
};

// Bounded wait; on timeout raises the CTA abort flag and records the status.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > kWaitNs) {
      *abort_flag = 1;
      set_status(status, REC_ATTN_ERR_TIMEOUT);
      return false;
    }
  }
}
// Bounded wait used only while shutting down after an abort.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > kWaitNs / 4) return;
}
// Warp-uniform wait: every lane waits, then the warp agrees on the outcome.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int* status) {
  const bool ok = wait_bar(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ producer
template <int D, int NS>
__device__ void run_producer(const AttnArgs& a, const void* tq, const void* tk, const void* tv,
                             uint8_t* sm, const Bars<NS>& B) {
  using L = Layout<D, NS>;
  uint32_t q_it = 0, kv_it = 0;
  uint32_t stage_phase[NS];
  bool stage_used[NS];
  for (int s = 0; s < NS; ++s) { stage_phase[s] = 0; stage_used[s] = false; }
  bool q_used = false;
  uint32_t q_phase = 0;
  ptx::prefetch_tensormap(tq);
  ptx::prefetch_tensormap(tk);
  ptx::prefetch_tensormap(tv);
  for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
    const WorkItem it = decode_item(a, w, true);
    if (it.n == 0) continue;
    if (!wait_bar(B.q_empty, (q_it & 1) ^ 1, B.abort_flag, a.status)) goto drain;
    ptx::mbar_arrive_expect_tx(B.q_full, L::kQBytes);
    {
      const int y = (int)(it.m.tok_start + (long long)it.qt * kTile);
#pragma unroll
      for (int s = 0; s < D / 64; ++s) ptx::tma_load_2d(sm + L::kQ + s * kSlab, tq, it.h * D + s * 64, y, B.q_full);
    }
    q_used = true; q_phase = q_it & 1; ++q_it;
    for (int j = 0; j < it.n; ++j) {
      const int kt = (int)(it.list[j] & 0xffffffu);
      const int st = (int)(kv_it % NS);
      const uint32_t ph = (kv_it / NS) & 1;
      if (!wait_bar(B.kv_empty + st, ph ^ 1, B.abort_flag, a.status)) goto drain;
      const int y = (int)(it.m.tok_start + (long long)kt * kTile);
      ptx::mbar_arrive_expect_tx(B.k_full + st, L::kKVBytes);
#pragma unroll
      for (int s = 0; s < D / 64; ++s)
        ptx::tma_load_2d(sm + L::kK + st * L::kKVBytes + s * kSlab, tk, it.h * D + s * 64, y, B.k_full + st);
      ptx::mbar_arrive_expect_tx(B.v_full + st, L::kKVBytes);
#pragma unroll
      for (int s = 0; s < D / 64; ++s)
        ptx::tma_load_2d(sm + L::kV + st * L::kKVBytes + s * kSlab, tv, it.h * D + s * 64, y, B.v_full + st);
      stage_used[st] = true; stage_phase[st] = ph;
      ++kv_it;
    }
  }
drain:
  // Every load issued must land before the CTA exits (only waits after an abort).
  if (q_used) drain_bar(B.q_full, q_phase);
  for (int s = 0; s < NS; ++s)
    if (stage_used[s]) { drain_bar(B.k_full + s, stage_phase[s]); drain_bar(B.v_full + s, stage_phase[s]); }
}

// ------------------------------------------------------------------ MMA issuer
template <int D, int NS>
__device__ void run_mma(const AttnArgs& a, uint8_t* sm, const Bars<NS>& B, uint32_t tmem) {
  using L = Layout<D, NS>;
  constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kTile, kTile, false, false);
  constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(kTile, D, false, true);
  const uint32_t q_addr = ptx::smem_u32(sm + L::kQ);
  const uint32_t k_addr = ptx::smem_u32(sm + L::kK);
  const uint32_t v_addr = ptx::smem_u32(sm + L::kV);
  const uint32_t p_addr = ptx::smem_u32(sm + L::kP);
  uint32_t q_it = 0, kv_it = 0, s_it = 0, p_it = 0;
  for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
    const WorkItem it = decode_item(a, w, true);
    if (it.n == 0) continue;
    if (!wait_bar(B.q_full, q_it & 1, B.abort_flag, a.status)) goto out;
    ++q_it;
    ptx::tc_fence_after();
    for (int j = -1; j < it.n; ++j) {
      // S(j + 1) = Q' K'(j + 1)^T into S buffer (s_it & 1)
      if (j + 1 < it.n) {
        const int st = (int)((kv_it + j + 1) % NS);
        const uint32_t ph = ((kv_it + j + 1) / NS) & 1;
        if (!wait_bar(B.k_full + st, ph, B.abort_flag, a.status)) goto out;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + ((s_it & 1) ? kTmemS1 : kTmemS0);
        const uint32_t kb = k_addr + st * L::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
          ptx::umma_f16(d_tmem, ptx::smem_desc_sw128(q_addr + off, 16, 1024),
                        ptx::smem_desc_sw128(kb + off, 16, 1024), idesc_s, kk > 0);
        }
        ptx::umma_commit(B.s_full + (s_it & 1));
        ++s_it;
        if (j + 2 == it.n) ptx::umma_commit(B.q_empty);  // last S of the item issued
      }
      if (j < 0) continue;
      // O += P(j) V(j)
      if (!wait_bar(B.p_full, p_it & 1, B.abort_flag, a.status)) goto out;
      ++p_it;
      ptx::tc_fence_after();
      const int st = (int)((kv_it + j) % NS);
      const uint32_t ph = ((kv_it + j) / NS) & 1;
      if (!wait_bar(B.v_full + st, ph, B.abort_flag, a.status)) goto out;
      ptx::tc_fence_after();
      const uint32_t vb = v_addr + st * L::kKVBytes;
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint32_t pa = p_addr + (kk >> 2) * kSlab + (kk & 3) * 32;
        const uint32_t va = vb + kk * 16 * 128;  // 16 keys per step, 128 B per key row
        ptx::umma_f16(tmem + kTmemO, ptx::smem_desc_sw128(pa, 16, 1024), ptx::smem_desc_sw128(va, kSlab, 1024),
                      idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
      }
      ptx::umma_commit(B.pv_done);
      ptx::umma_commit(B.kv_empty + st);
    }
    kv_it += it.n;
  }
out:
  // All issued MMAs must complete before TMEM is released.
  ptx::umma_commit(B.mma_done);
  drain_bar(B.mma_done, 0);
}

// ------------------------------------------------------------------ softmax
template <int D, int NS>
__device__ void run_softmax(const AttnArgs& a, uint8_t* sm, const Bars<NS>& B, uint32_t tmem, int sw) {
  using L = Layout<D, NS>;
  const int lane = threadIdx.x & 31;
  const int quad = (threadIdx.x >> 5) & 3;  // TMEM lanes this warp may access
  const int row = quad * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  long long* kmt = reinterpret_cast<long long*>(sm + L::kMeta + sw * L::kMetaWarp);
  int8_t* kmy = reinterpret_cast<int8_t*>(kmt + kTile);
  uint8_t* prow = sm + L::kP + row * 128;
  const float sl2 = a.scale * 1.4426950408889634f;  // scale * log2(e)
  const int H = a.heads;
  uint32_t s_it = 0, pv_it = 0;
  for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
    const WorkItem it = decode_item(a, w, true);
    const int pi = it.qt * kTile + row;
    const bool row_ok = pi < it.m.len;
    const long long tok = it.m.tok_start + pi;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + (tok * H + it.h) * D;
    if (it.n == 0) {
      if (row_ok) {
        uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
        if (a.lse) a.lse[tok * H + it.h] = -INFINITY;
      }
      continue;
    }
    long long ti = 0;
    int tyi = -1;
    if (row_ok) { ti = a.t[tok]; tyi = a.ty[tok]; }
    bool thr_ok; long long thr;
    delay_bound(ti, a.mask.delay, thr_ok, thr);
    float m_run = -INFINITY, l = 0.f;
    for (int j = 0; j < it.n; ++j) {
      const uint32_t ent = it.list[j];
      const int kt = (int)(ent & 0xffffffu);
      const bool partial = (ent >> 24) != REC_ATTN_TILE_FULL;
      if (partial) {  // key metadata of this tile, staged per warp
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kTile / 32; ++u) {
          const int c = lane + 32 * u, pj = kt * kTile + c;
          const bool ok = pj < it.m.len;
          kmt[c] = ok ? a.t[it.m.tok_start + pj] : 0;
          kmy[c] = ok ? a.ty[it.m.tok_start + pj] : (int8_t)-1;
        }
        __syncwarp();
      }
      if (!wait_bar_warp(B.s_full + (s_it & 1), (s_it >> 1) & 1, B.abort_flag, a.status)) return;
      ptx::tc_fence_after();
      uint32_t sr[kTile];
      ptx::tmem_ld128(tmem + lane_off + ((s_it & 1) ? kTmemS1 : kTmemS0), sr);
      ++s_it;
      float s[kTile];
#pragma unroll
      for (int c = 0; c < kTile; ++c) s[c] = __uint_as_float(sr[c]);
      if (partial) {
        uint32_t vm[kTile / 32];
#pragma unroll
        for (int w4 = 0; w4 < kTile / 32; ++w4) {
          uint32_t bits = 0;
#pragma unroll 4
          for (int b = 0; b < 32; ++b) {
            const int c = w4 * 32 + b;
            const bool v = vis_pred(a.mask, pi, ti, tyi, thr_ok, thr, kt * kTile + c, kmt[c], kmy[c]);
            bits |= (v ? 1u : 0u) << b;
          }
          vm[w4] = row_ok ? bits : 0u;
        }
#pragma unroll
        for (int c = 0; c < kTile; ++c)
          if (!((vm[c >> 5] >> (c & 31)) & 1u)) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kTile; ++c) mx = fmaxf(mx, s[c]);
      const float m_tile = mx * sl2;  // -inf stays -inf (sl2 > 0)
      const float m_new = fmaxf(m_run, m_tile);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = ex2(m_run - m_use);
      uint32_t pk[kTile / 2];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kTile / 2; ++c) {
        const float p0 = ex2(fmaf(s[2 * c], sl2, -m_use));
        const float p1 = ex2(fmaf(s[2 * c + 1], sl2, -m_use));
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        rs += __low2float(pb) + __high2float(pb);
        pk[c] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      l = l * corr + rs;
      if (j > 0) {
        // PV(j-1) must be done before P is overwritten and before O is rescaled.
        if (!wait_bar_warp(B.pv_done, pv_it & 1, B.abort_flag, a.status)) return;
        ++pv_it;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
          for (int half = 0; half < D / 64; ++half) {
            uint32_t o[64];
            const uint32_t ta = tmem + lane_off + kTmemO + half * 64;
            ptx::tmem_ld64(ta, o);
#pragma unroll
            for (int e = 0; e < 64; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            ptx::tmem_st64(ta, o);
          }
        }
      }
      // P row -> shared memory, K-major with the 128-byte swizzle (16-byte chunk
      // index XOR row % 8), two 64-key slabs.
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        const int slab = c16 >> 3, cc = c16 & 7;
        uint4 v4 = make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
        *reinterpret_cast<uint4*>(prow + slab * kSlab + ((cc ^ (row & 7)) << 4)) = v4;
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(B.p_full);
      m_run = m_new;
    }
    // epilogue: O / l
    if (!wait_bar_warp(B.pv_done, pv_it & 1, B.abort_flag, a.status)) return;
    ++pv_it;
    ptx::tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int half = 0; half < D / 64; ++half) {
      uint32_t o[64];
      ptx::tmem_ld64(tmem + lane_off + kTmemO + half * 64, o);
      if (row_ok) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 pb = __floats2bfloat162_rn(__uint_as_float(o[c * 8 + 2 * e]) * inv,
                                                            __uint_as_float(o[c * 8 + 2 * e + 1]) * inv);
            wv[e] = *reinterpret_cast<const uint32_t*>(&pb);
          }
          reinterpret_cast<uint4*>(orow + half * 64)[c] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
    if (row_ok && a.lse) {
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      a.lse[tok * H + it.h] = l > 0.f ? (m_use + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    ptx::tc_fence_before();
  }
}

template <int D, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using L = Layout<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars<NS> B(sm + L::kBars);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(B.q_full, 1);
    ptx::mbar_init(B.q_empty, 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(B.k_full + s, 1);
      ptx::mbar_init(B.v_full + s, 1);
      ptx::mbar_init(B.kv_empty + s, 1);
    }
    ptx::mbar_init(B.s_full, 1);
    ptx::mbar_init(B.s_full + 1, 1);
    ptx::mbar_init(B.p_full, 128);
    ptx::mbar_init(B.pv_done, 1);
    ptx::mbar_init(B.mma_done, 1);
    *B.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(B.tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *B.tmem_slot;

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) run_producer<D, NS>(a, &tm_q, &tm_k, &tm_v, sm, B);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) run_mma<D, NS>(a, sm, B, tmem);
  } else {
    run_softmax<D, NS>(a, sm, B, tmem, warp - 2);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int NS>
cudaError_t launch(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                   int grid, cudaStream_t st) {
  using L = Layout<D, NS>;
  cudaError_t e = cudaFuncSetAttribute(k_attn_tc<D, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamic);
  if (e != cudaSuccess) return e;
  k_attn_tc<D, NS><<<grid, kThreads, L::kDynamic, st>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           int head_dim, int grid, cudaStream_t st) {
  if (a.n_items <= 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch<64, 3>(a, q, k, v, grid, st);
    case 128: return launch<128, 2>(a, q, k, v, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace recattn
