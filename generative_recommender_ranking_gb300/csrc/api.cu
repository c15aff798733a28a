// api.cu -- host side of the C-ABI declared in include/rec_attn.h: argument
// validation (always before any CUDA call, so bad arguments never launch work),
// plan ownership, stream-ordered workspace from a library-owned memory pool, TMA
// descriptor encoding and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <vector>

#include "launchers.cuh"
#include "rec_attn.h"
#include "workspace.cuh"

#define REC_ATTN_API extern "C" __attribute__((visibility("default")))

using namespace recattn;

struct rec_attn_plan_s {
  rec_attn_params p;
  int device = 0;
  int num_sms = 0;
  int32_t batch = 0;
  long long T = 0, NT = 0, NC = 0;
  cudaStream_t stream = nullptr;  // stream of the last use
  void* ws = nullptr;
  size_t ws_bytes = 0;
  PlanDev pd{};
  std::vector<int> req_tiles;  // host copy: tiles of each request (argument checks)
  std::vector<int64_t> offsets_host;  // host copy of the request offsets [B+1]
  void* qrot = nullptr;
  void* krot = nullptr;
  void* qk_extra = nullptr;  // Q'/K' buffers of a plan without the RoPE, made on the first fused call
  // workspace of the backward pass, made on its first call: fp32 path D [T][H];
  // bf16 path the item descriptors, transposed tile lists (built once) and row constants
  void* bwd_ws = nullptr;
  bool bwd_sched = false;
  const long long* t = nullptr;
  const int8_t* ty = nullptr;
  MaskP mask{};
  float omega[kMaxPairs] = {};
  // cached TMA descriptors for the last (q', k', v) pointers
  const void* map_src[3] = {nullptr, nullptr, nullptr};
  CUtensorMap maps[3];
  // Planning runs on a library side stream (after the caller's stream has produced the
  // offsets, times and types: ev_in), so the RoPE prologue of rec_attn_fwd, on the
  // caller's stream, overlaps the planning kernels.  The prologue waits for the
  // request-table upload and, when long requests are split, the planner's first kernel
  // (ev_meta); the attention kernel waits for the planner (ev_plan).
  cudaStream_t side = nullptr;
  cudaEvent_t ev_in = nullptr, ev_meta = nullptr, ev_plan = nullptr;
  // optional kernel timing: events around the RoPE prologue and the attention kernel
  bool timing = false;
  bool timed = false;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
};

namespace recattn {

// Parameter checks and tensor maps shared with the no-allocation entry point.
rec_attn_status check_params(const rec_attn_params* p) {
  if (!p) return REC_ATTN_ERR_INVALID_ARG;
  if (p->abi_version != REC_ATTN_ABI_VERSION) return REC_ATTN_ERR_INVALID_ARG;
  if (p->num_heads < 1 || p->head_dim < 2 || (p->head_dim & 1)) return REC_ATTN_ERR_INVALID_ARG;
  if (p->dtype != REC_ATTN_BF16 && p->dtype != REC_ATTN_FP32) return REC_ATTN_ERR_INVALID_ARG;
  if ((p->use_delay != 0 && p->use_delay != 1) || (p->use_rope != 0 && p->use_rope != 1) ||
      (p->hist_bidirectional != 0 && p->hist_bidirectional != 1))
    return REC_ATTN_ERR_INVALID_ARG;
  if (p->delay_s < 0 || p->delay_s > (1LL << 62) || p->window < 0) return REC_ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale >= 0.f)) return REC_ATTN_ERR_INVALID_ARG;
  if (p->use_rope) {
    if (!(std::isfinite(p->phi_min) && std::isfinite(p->dt_max_s) && std::isfinite(p->rope_base)))
      return REC_ATTN_ERR_INVALID_ARG;
    if (p->dt_max_s <= 0.0 || p->rope_base <= 0.0) return REC_ATTN_ERR_INVALID_ARG;
  }
  if (p->dtype == REC_ATTN_BF16 && p->head_dim != 64 && p->head_dim != 128) return REC_ATTN_ERR_UNSUPPORTED;
  if (p->dtype == REC_ATTN_FP32 && p->head_dim != 32 && p->head_dim != 64) return REC_ATTN_ERR_UNSUPPORTED;
  // TMA rows of the [T][H*d] bf16 view must stay below 2^32 elements per dimension
  if ((long long)p->num_heads * p->head_dim > (1LL << 20)) return REC_ATTN_ERR_UNSUPPORTED;
  return REC_ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D map over a [T][H*d] bf16 tensor; box = 64 columns x 128 rows, 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* base, long long T, long long cols) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)T};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Long items: rows without a window over requests of at least 32 tiles on average
// (4096 tokens), where a row's running maximum rarely moves from one key tile to the
// next, so the softmax takes its lazy maximum; shorter items keep the plain one (the
// lazy one holds more registers: measured 2% faster at 40 tiles a request, even at 20,
// and 1.5 to 19% slower on the short-item workloads).
int long_items(const rec_attn_params& p, int batch, long long n_tiles) {
  return (p.window == 0 && batch > 0 && n_tiles >= 32LL * batch) ? 1 : 0;
}

}  // namespace recattn

namespace {

std::mutex g_pool_mu;
std::map<int, cudaMemPool_t> g_pools;
std::map<int, cudaStream_t> g_side;

// Library-owned non-blocking stream per device for the RoPE prologue.
cudaError_t side_stream_for(int device, cudaStream_t* out) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  auto it = g_side.find(device);
  if (it != g_side.end()) { *out = it->second; return cudaSuccess; }
  cudaStream_t st;
  cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
  if (e != cudaSuccess) return e;
  g_side[device] = st;
  *out = st;
  return cudaSuccess;
}

rec_attn_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return REC_ATTN_OK;
  if (e == cudaErrorMemoryAllocation) return REC_ATTN_ERR_OOM;
  return REC_ATTN_ERR_CUDA;
}

// Library-owned pool per device; it keeps freed blocks so repeated plan/free cycles
// do not return to the driver.
cudaError_t pool_for(int device, cudaMemPool_t* out) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  auto it = g_pools.find(device);
  if (it != g_pools.end()) { *out = it->second; return cudaSuccess; }
  cudaMemPoolProps props;
  std::memset(&props, 0, sizeof props);
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = device;
  cudaMemPool_t pool;
  cudaError_t e = cudaMemPoolCreate(&pool, &props);
  if (e != cudaSuccess) return e;
  uint64_t keep = ~0ull;
  e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  if (e != cudaSuccess) return e;
  g_pools[device] = pool;
  *out = pool;
  return cudaSuccess;
}

// Closes the attention kernel's timing window: events 0..1 bracket the RoPE
// prologue, events 2..3 the attention kernel.
rec_attn_status finish_timing(rec_attn_plan_s* plan, cudaStream_t st, cudaError_t launch_err) {
  if (launch_err != cudaSuccess) return from_cuda(launch_err);
  if (!plan->timing) return REC_ATTN_OK;
  cudaError_t e = cudaEventRecord(plan->ev[3], st);
  if (e != cudaSuccess) return from_cuda(e);
  plan->timed = true;
  return REC_ATTN_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

REC_ATTN_API const char* rec_attn_status_string(rec_attn_status s) {
  switch (s) {
    case REC_ATTN_OK: return "ok";
    case REC_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case REC_ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case REC_ATTN_ERR_CUDA: return "CUDA runtime error";
    case REC_ATTN_ERR_OOM: return "out of device memory";
    case REC_ATTN_ERR_TIMEOUT: return "device wait timed out";
    case REC_ATTN_ERR_DEVICE_INPUT: return "device input out of range (token type, timestamp or offsets)";
  }
  return "unknown status";
}

namespace {

rec_attn_status plan_impl(const rec_attn_params* params, int32_t keep_user_queries, int32_t batch,
                          const int64_t* offsets_host, const int64_t* offsets_dev, const int64_t* timestamps_dev,
                          const int8_t* types_dev, void* stream, rec_attn_plan_t** plan_out) {
  if (!plan_out) return REC_ATTN_ERR_INVALID_ARG;
  *plan_out = nullptr;
  rec_attn_status st = check_params(params);
  if (st != REC_ATTN_OK) return st;
  if (batch < 0 || (batch > 0 && !offsets_host)) return REC_ATTN_ERR_INVALID_ARG;
  std::vector<ReqMeta> meta((size_t)batch);
  long long NT = 0, NC = 0, T = 0;
  if (batch > 0) {
    if (offsets_host[0] != 0) return REC_ATTN_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b) {
      const long long len = offsets_host[b + 1] - offsets_host[b];
      if (len < 0) return REC_ATTN_ERR_INVALID_ARG;
      if (len > REC_ATTN_MAX_REQUEST_LEN) return REC_ATTN_ERR_UNSUPPORTED;
      ReqMeta& m = meta[b];
      m.tok_start = offsets_host[b];
      m.len = (int)len;
      m.ntiles = (int)((len + kTile - 1) / kTile);
      m.tile_start = NT;
      m.cls_start = NC;
      NT += m.ntiles;
      NC += (long long)m.ntiles * m.ntiles;
    }
    T = offsets_host[batch];
    if (T >= (1LL << 31) || NT * params->num_heads >= (1LL << 31)) return REC_ATTN_ERR_UNSUPPORTED;
    if (!offsets_dev || (T > 0 && (!timestamps_dev || !types_dev))) return REC_ATTN_ERR_INVALID_ARG;
  }

  rec_attn_plan_s* plan = new (std::nothrow) rec_attn_plan_s();
  if (!plan) return REC_ATTN_ERR_OOM;
  plan->p = *params;
  if (plan->p.softmax_scale == 0.f) plan->p.softmax_scale = 1.f / std::sqrt((float)params->head_dim);
  plan->batch = batch;
  plan->T = T; plan->NT = NT; plan->NC = NC;
  try {
    plan->req_tiles.resize((size_t)batch);
    plan->offsets_host.assign(offsets_host ? offsets_host : nullptr, offsets_host ? offsets_host + batch + 1 : nullptr);
  } catch (...) {
    delete plan;
    return REC_ATTN_ERR_OOM;
  }
  for (int32_t b = 0; b < batch; ++b) plan->req_tiles[b] = meta[b].ntiles;
  plan->stream = static_cast<cudaStream_t>(stream);
  plan->t = reinterpret_cast<const long long*>(timestamps_dev);
  plan->ty = types_dev;
  plan->mask.use_delay = params->use_delay;
  plan->mask.keep_user = keep_user_queries < 0 ? -1 : keep_user_queries;
  plan->mask.delay = params->use_delay ? params->delay_s : 0;
  plan->mask.window = params->window;
  plan->mask.bidir = params->hist_bidirectional;
  if (params->use_rope)
    for (int i = 0; i < params->head_dim / 2 && i < kMaxPairs; ++i)
      plan->omega[i] = (float)(params->phi_min / params->dt_max_s *
                               std::pow(params->rope_base, 2.0 * i / (double)params->head_dim));

  cudaError_t e = cudaGetDevice(&plan->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&plan->num_sms, cudaDevAttrMultiProcessorCount, plan->device);
  if (e != cudaSuccess) { delete plan; return from_cuda(e); }

  // workspace layout
  const size_t elem = params->dtype == REC_ATTN_BF16 ? 2 : 4;
  const size_t qk_bytes = (size_t)T * params->num_heads * params->head_dim * elem;
  const WsLayout lay = ws_layout(batch, NT, NC, params->num_heads, params->use_rope ? qk_bytes : 0,
                                 mask_capacity(NT, NC));
  plan->ws_bytes = lay.total;

  cudaMemPool_t pool;
  e = pool_for(plan->device, &pool);
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&plan->ws, plan->ws_bytes, pool, plan->stream);
  if (e != cudaSuccess) { delete plan; return from_cuda(e); }
  char* w = static_cast<char*>(plan->ws);
  plan->pd = ws_bind(w, lay);
  PlanDev& pd = plan->pd;
  plan->qrot = params->use_rope ? w + lay.rq : nullptr;
  plan->krot = params->use_rope ? w + lay.rk : nullptr;

  for (cudaEvent_t* ev : {&plan->ev_in, &plan->ev_meta, &plan->ev_plan})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e == cudaSuccess) e = side_stream_for(plan->device, &plan->side);
  // the side stream starts after the caller's stream reaches this point (inputs ready,
  // workspace allocated)
  if (e == cudaSuccess) e = cudaEventRecord(plan->ev_in, plan->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->side, plan->ev_in, 0);
  if (e != cudaSuccess) {
    cudaFreeAsync(plan->ws, plan->stream);
    for (cudaEvent_t ev : {plan->ev_in, plan->ev_meta, plan->ev_plan})
      if (ev) cudaEventDestroy(ev);
    delete plan;
    return from_cuda(e);
  }
  {
    // the zeroed header (counters, status word), the request table and the request of
    // every tile (so the prologue needs no search), laid out as in the workspace and
    // uploaded in one copy (a pageable copy: staged before the call returns)
    std::vector<char> up(lay.tr - lay.hdr + sizeof(int) * (size_t)NT, 0);
    if (batch > 0) std::memcpy(up.data() + (lay.meta - lay.hdr), meta.data(), sizeof(ReqMeta) * (size_t)batch);
    int* treq = reinterpret_cast<int*>(up.data() + (lay.tr - lay.hdr));
    for (int32_t b = 0; b < batch; ++b)
      for (int i = 0; i < meta[b].ntiles; ++i) treq[meta[b].tile_start + i] = b;
    e = cudaMemcpyAsync(w + lay.hdr, up.data(), up.size(), cudaMemcpyHostToDevice, plan->side);
  }
  if (e == cudaSuccess)
    e = launch_plan(plan->mask, params->num_heads, pd, reinterpret_cast<const long long*>(offsets_dev), plan->t,
                    plan->ty, batch, NT, plan->ev_meta, plan->side);
  if (e == cudaSuccess) e = launch_build_masks(plan->mask, pd, plan->num_sms, plan->side);
  if (e == cudaSuccess) e = cudaEventRecord(plan->ev_plan, plan->side);
  if (e != cudaSuccess) {
    cudaStreamWaitEvent(plan->stream, plan->ev_plan, 0);
    cudaFreeAsync(plan->ws, plan->stream);
    for (cudaEvent_t ev : {plan->ev_in, plan->ev_meta, plan->ev_plan}) cudaEventDestroy(ev);
    delete plan;
    return from_cuda(e);
  }
  *plan_out = plan;
  return REC_ATTN_OK;
}

}  // namespace

REC_ATTN_API rec_attn_status rec_attn_plan(const rec_attn_params* params, int32_t batch,
                                           const int64_t* offsets_host, const int64_t* offsets_dev,
                                           const int64_t* timestamps_dev, const int8_t* types_dev, void* stream,
                                           rec_attn_plan_t** plan_out) {
  return plan_impl(params, -1, batch, offsets_host, offsets_dev, timestamps_dev, types_dev, stream, plan_out);
}

REC_ATTN_API rec_attn_status rec_attn_plan_query_pruned(const rec_attn_params* params, int32_t keep_user_queries,
                                                        int32_t batch, const int64_t* offsets_host,
                                                        const int64_t* offsets_dev, const int64_t* timestamps_dev,
                                                        const int8_t* types_dev, void* stream,
                                                        rec_attn_plan_t** plan_out) {
  if (plan_out) *plan_out = nullptr;
  if (keep_user_queries < -1) return REC_ATTN_ERR_INVALID_ARG;
  return plan_impl(params, keep_user_queries, batch, offsets_host, offsets_dev, timestamps_dev, types_dev, stream,
                   plan_out);
}

REC_ATTN_API int64_t rec_attn_query_keep(int64_t hist_len, int64_t n_min, int32_t layer, int32_t n_layers) {
  if (hist_len < 0 || n_min < 0 || n_layers < 1 || layer < 1 || layer > n_layers) return -1;
  if (n_layers == 1) return hist_len;
  // N_l = min(Lh, max(N_min, Round[Lh - (l - 1) / (L - 1) * (Lh - N_min)])), exact in
  // integers: Round[x / q] with x = Lh (L-1) - (l-1)(Lh - N_min), q = L - 1, half away from 0
  const long long q = n_layers - 1;
  const long long x = hist_len * q - (long long)(layer - 1) * (hist_len - n_min);
  const long long r = x >= 0 ? (2 * x + q) / (2 * q) : -((-2 * x + q) / (2 * q));
  return std::min<long long>(hist_len, std::max<long long>(n_min, r));
}

namespace {

// The forward of rec_attn_fwd and rec_attn_fwd_fused (f == nullptr: no fused step).
// cmp: the history compression epilogue (the output goes to cmp->x_out, checked by the
// caller; out and lse are then unused).
rec_attn_status fwd_impl(rec_attn_plan_t* plan, const void* q, const void* k, const void* v,
                         const rec_attn_fused* f, void* out, float* lse, void* stream,
                         const CmpArgs* cmp = nullptr) {
  if (!plan) return REC_ATTN_ERR_INVALID_ARG;
  const rec_attn_params& p = plan->p;
  const long long T = plan->T;
  if (T > 0 && cmp) {
    if (!q || !k || !v) return REC_ATTN_ERR_INVALID_ARG;
    const void* ptrs[3] = {q, k, v};
    for (const void* x : ptrs)
      if (reinterpret_cast<uintptr_t>(x) & 15u) return REC_ATTN_ERR_INVALID_ARG;
  } else if (T > 0) {
    if (!q || !k || !v || !out) return REC_ATTN_ERR_INVALID_ARG;
    const void* ptrs[4] = {q, k, v, out};
    for (const void* x : ptrs)
      if (reinterpret_cast<uintptr_t>(x) & 15u) return REC_ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return REC_ATTN_ERR_INVALID_ARG;
    const size_t elem = p.dtype == REC_ATTN_BF16 ? 2 : 4;
    const size_t bytes = (size_t)T * p.num_heads * p.head_dim * elem;
    if (overlaps(out, bytes, q, bytes) || overlaps(out, bytes, k, bytes) || overlaps(out, bytes, v, bytes))
      return REC_ATTN_ERR_INVALID_ARG;
    if (lse && (overlaps(lse, (size_t)T * p.num_heads * 4, out, bytes)))
      return REC_ATTN_ERR_INVALID_ARG;
    if (f) {
      if (!(f->norm_eps >= 0.f) || !std::isfinite(f->norm_eps)) return REC_ATTN_ERR_INVALID_ARG;
      const void* gates[3] = {f->q_gate, f->k_gate, f->out_gate};
      for (const void* g : gates)
        if (reinterpret_cast<uintptr_t>(g) & 15u) return REC_ATTN_ERR_INVALID_ARG;
      if (overlaps(out, bytes, f->out_gate, f->out_gate ? bytes : 0)) return REC_ATTN_ERR_INVALID_ARG;
      const float* ws[2] = {f->q_norm_weight, f->k_norm_weight};
      for (const float* w : ws)
        if (reinterpret_cast<uintptr_t>(w) & 3u) return REC_ATTN_ERR_INVALID_ARG;
    }
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (dev != plan->device) return REC_ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  plan->stream = st;
  if (T == 0) return REC_ATTN_OK;

  const void* qs = q;
  const void* ks = k;
  const bool fuse_qk = f && (f->q_norm_weight || f->k_norm_weight || f->q_gate || f->k_gate);
  if (fuse_qk) {
    // fused QK-RMSNorm / gates, then the rotation (if the plan has one), into Q'/K'
    if (!plan->qrot) {
      if (!plan->qk_extra) {
        const size_t elem = p.dtype == REC_ATTN_BF16 ? 2 : 4;
        const size_t qk_bytes = ((size_t)T * p.num_heads * p.head_dim * elem + 255) & ~(size_t)255;
        cudaMemPool_t pool;
        e = pool_for(plan->device, &pool);
        if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&plan->qk_extra, 2 * qk_bytes, pool, st);
        if (e != cudaSuccess) { plan->qk_extra = nullptr; return from_cuda(e); }
        plan->krot = static_cast<char*>(plan->qk_extra) + qk_bytes;
      }
      plan->qrot = plan->qk_extra;
    }
    e = cudaStreamWaitEvent(st, plan->ev_meta, 0);
    if (e == cudaSuccess && plan->timing) {
      plan->timed = false;
      e = cudaEventRecord(plan->ev[0], st);
    }
    if (e != cudaSuccess) return from_cuda(e);
    RopeArgs ra;
    ra.meta = plan->pd.meta; ra.tile_req = plan->pd.treq; ra.batch = plan->batch; ra.t = plan->t;
    ra.ty = plan->ty; ra.skip_user_q = 0;
    ra.q = q; ra.k = k; ra.qr = plan->qrot; ra.kr = plan->krot;
    ra.heads = p.num_heads; ra.head_dim = p.head_dim;
    std::memcpy(ra.omega, plan->omega, sizeof ra.omega);  // all zero without the RoPE
    FusedArgs fa;
    fa.q_norm_w = f->q_norm_weight; fa.k_norm_w = f->k_norm_weight; fa.eps = f->norm_eps;
    fa.q_gate = f->q_gate; fa.k_gate = f->k_gate;
    e = launch_rope_fused(ra, fa, p.dtype, plan->NT, st);
    if (e == cudaSuccess && plan->timing) e = cudaEventRecord(plan->ev[1], st);
    if (e != cudaSuccess) return from_cuda(e);
    qs = plan->qrot; ks = plan->krot;
  } else if (p.use_rope) {
    e = cudaStreamWaitEvent(st, plan->ev_meta, 0);  // the request table (not the planner)
    if (e == cudaSuccess && plan->timing) {
      plan->timed = false;
      e = cudaEventRecord(plan->ev[0], st);
    }
    if (e != cudaSuccess) return from_cuda(e);
    RopeArgs ra;
    ra.meta = plan->pd.meta; ra.tile_req = plan->pd.treq; ra.batch = plan->batch; ra.t = plan->t;
    ra.ty = plan->ty; ra.skip_user_q = 0;
    ra.q = q; ra.k = k; ra.qr = plan->qrot; ra.kr = plan->krot;
    ra.heads = p.num_heads; ra.head_dim = p.head_dim;
    std::memcpy(ra.omega, plan->omega, sizeof ra.omega);
    ra.skip_user_q = plan->mask.keep_user == 0 ? 1 : 0;  // target attention: no user token queries
    e = launch_rope(ra, p.dtype, plan->NT, st);
    if (e == cudaSuccess && plan->timing) e = cudaEventRecord(plan->ev[1], st);
    if (e != cudaSuccess) return from_cuda(e);
    qs = plan->qrot; ks = plan->krot;
  } else if (plan->timing) {
    plan->timed = false;
    e = cudaEventRecord(plan->ev[0], st);
    if (e == cudaSuccess) e = cudaEventRecord(plan->ev[1], st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  e = cudaStreamWaitEvent(st, plan->ev_plan, 0);
  if (e != cudaSuccess) return from_cuda(e);
  if (plan->timing) {
    e = cudaEventRecord(plan->ev[2], st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  AttnArgs a{};
  a.meta = plan->pd.meta; a.qreq = plan->pd.qreq; a.kcount = plan->pd.kcount; a.klist = plan->pd.klist;
  a.items = plan->pd.items; a.t = plan->t; a.ty = plan->ty;
  a.counters = plan->pd.counters; a.krec = plan->pd.krec; a.qkeep = plan->pd.qkeep;
  a.kslot = plan->pd.kslot; a.mtab = plan->pd.mtab;
  a.q = qs; a.k = ks; a.v = v; a.out = out; a.lse = lse; a.status = plan->pd.status;
  a.out_gate = f ? f->out_gate : nullptr;
  a.n_items = plan->NT * p.num_heads; a.heads = p.num_heads; a.scale = p.softmax_scale; a.mask = plan->mask;
  if (cmp) a.cmp = *cmp;
  a.long_items = long_items(p, plan->batch, plan->NT);
  if (p.dtype == REC_ATTN_FP32) {
    e = launch_attn_simt(a, p.head_dim, st);
    return finish_timing(plan, st, e);
  }
  const void* srcs[3] = {qs, ks, v};
  const long long cols = (long long)p.num_heads * p.head_dim;
  for (int i = 0; i < 3; ++i) {
    if (plan->map_src[i] != srcs[i]) {
      if (!encode_map(&plan->maps[i], srcs[i], T, cols)) { plan->map_src[i] = nullptr; return REC_ATTN_ERR_CUDA; }
      plan->map_src[i] = srcs[i];
    }
  }
  const long long items = a.n_items;
  const int grid = (int)(items < plan->num_sms ? items : plan->num_sms);
  e = launch_attn_tc(a, plan->maps[0], plan->maps[1], plan->maps[2], p.head_dim, grid, st);
  return finish_timing(plan, st, e);
}

}  // namespace

REC_ATTN_API rec_attn_status rec_attn_fwd(rec_attn_plan_t* plan, const void* q, const void* k, const void* v,
                                          void* out, float* lse, void* stream) {
  return fwd_impl(plan, q, k, v, nullptr, out, lse, stream);
}

REC_ATTN_API rec_attn_status rec_attn_fwd_fused(rec_attn_plan_t* plan, const void* q, const void* k,
                                                const void* v, const rec_attn_fused* fused, void* out,
                                                float* lse, void* stream) {
  if (!fused) return REC_ATTN_ERR_INVALID_ARG;
  return fwd_impl(plan, q, k, v, fused, out, lse, stream);
}

namespace {

// The backward of rec_attn_bwd and rec_attn_bwd_fused.  fa: the fused Q/K steps to
// recompute Q' and K' with (nullptr: the time-RoPE alone); dout_attn: the gradient that
// reaches the attention itself (dout, or dout * sigmoid(output gate)), while the row
// constants D = <dout, out> use dout and out as given.
rec_attn_status bwd_impl(rec_attn_plan_t* plan, const void* q, const void* k, const void* v, const void* out,
                         const float* lse, const void* dout, const void* dout_attn, void* dq, void* dk, void* dv,
                         void* stream, const FusedArgs* fa) {
  if (!plan) return REC_ATTN_ERR_INVALID_ARG;
  const rec_attn_params& p = plan->p;
  const long long T = plan->T;
  const bool dim_ok = p.dtype == REC_ATTN_BF16 ? (p.head_dim == 64 || p.head_dim == 128)
                                               : (p.head_dim == 32 || p.head_dim == 64);
  if (!dim_ok) return REC_ATTN_ERR_UNSUPPORTED;
  if (T > 0) {
    const void* ptrs[8] = {q, k, v, out, dout, dq, dk, dv};
    for (const void* x : ptrs)
      if (!x || (reinterpret_cast<uintptr_t>(x) & 15u)) return REC_ATTN_ERR_INVALID_ARG;
    if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return REC_ATTN_ERR_INVALID_ARG;
    const size_t elem = p.dtype == REC_ATTN_BF16 ? 2 : 4;
    const size_t bytes = (size_t)T * p.num_heads * p.head_dim * elem;
    const void* ins[6] = {q, k, v, out, dout, lse};
    const size_t in_bytes[6] = {bytes, bytes, bytes, bytes, bytes, (size_t)T * p.num_heads * 4};
    void* outs[3] = {dq, dk, dv};
    for (int o = 0; o < 3; ++o) {
      for (int i = 0; i < 6; ++i)
        if (overlaps(outs[o], bytes, ins[i], in_bytes[i])) return REC_ATTN_ERR_INVALID_ARG;
      for (int o2 = o + 1; o2 < 3; ++o2)
        if (overlaps(outs[o], bytes, outs[o2], bytes)) return REC_ATTN_ERR_INVALID_ARG;
    }
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (dev != plan->device) return REC_ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  plan->stream = st;
  if (T == 0) return REC_ATTN_OK;
  const bool tc = p.dtype == REC_ATTN_BF16;
  const long long n_items = plan->NT * p.num_heads;
  // bf16 workspace: descriptors [2][n_items] | row constants [H][NT][128] | lists [NC] |
  // their mask-table slots [NC] | the mask table's columns [mcap][128][4]
  const size_t off_rowc = (size_t)2 * n_items * sizeof(BwdItemDesc);
  const size_t off_ql = off_rowc + (size_t)plan->NT * p.num_heads * kTile * sizeof(float2);
  const size_t off_qs = off_ql + (((size_t)plan->NC * sizeof(uint32_t) + 15) & ~(size_t)15);
  const size_t off_ct = off_qs + (((size_t)plan->NC * sizeof(int) + 15) & ~(size_t)15);
  const size_t ws_bytes = tc ? off_ct + (size_t)plan->pd.mcap * kTile * 16 : (size_t)T * p.num_heads * sizeof(float);
  if (!plan->bwd_ws) {
    cudaMemPool_t pool;
    e = pool_for(plan->device, &pool);
    if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&plan->bwd_ws, ws_bytes, pool, st);
    if (e != cudaSuccess) { plan->bwd_ws = nullptr; return from_cuda(e); }
  }
  char* bws = static_cast<char*>(plan->bwd_ws);
  const void* qs = q;
  const void* ks = k;
  if (fa) {  // the fused steps and the rotation again, into the plan's Q'/K' buffers
    if (!plan->qrot) {
      if (!plan->qk_extra) {
        const size_t elem = p.dtype == REC_ATTN_BF16 ? 2 : 4;
        const size_t qk_bytes = ((size_t)T * p.num_heads * p.head_dim * elem + 255) & ~(size_t)255;
        cudaMemPool_t pool;
        e = pool_for(plan->device, &pool);
        if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&plan->qk_extra, 2 * qk_bytes, pool, st);
        if (e != cudaSuccess) { plan->qk_extra = nullptr; return from_cuda(e); }
        plan->krot = static_cast<char*>(plan->qk_extra) + qk_bytes;
      }
      plan->qrot = plan->qk_extra;
    }
    e = cudaStreamWaitEvent(st, plan->ev_meta, 0);
    if (e != cudaSuccess) return from_cuda(e);
    RopeArgs ra;
    ra.meta = plan->pd.meta; ra.tile_req = plan->pd.treq; ra.batch = plan->batch; ra.t = plan->t;
    ra.ty = plan->ty; ra.skip_user_q = 0;
    ra.q = q; ra.k = k; ra.qr = plan->qrot; ra.kr = plan->krot;
    ra.heads = p.num_heads; ra.head_dim = p.head_dim;
    std::memcpy(ra.omega, plan->omega, sizeof ra.omega);  // all zero without the RoPE
    e = launch_rope_fused(ra, *fa, p.dtype, plan->NT, st);
    if (e != cudaSuccess) return from_cuda(e);
    qs = plan->qrot; ks = plan->krot;
  } else if (p.use_rope) {  // Q' and K' again, into the plan's workspace
    e = cudaStreamWaitEvent(st, plan->ev_meta, 0);
    if (e != cudaSuccess) return from_cuda(e);
    RopeArgs ra;
    ra.meta = plan->pd.meta; ra.tile_req = plan->pd.treq; ra.batch = plan->batch; ra.t = plan->t;
    ra.ty = plan->ty; ra.skip_user_q = 0;
    ra.q = q; ra.k = k; ra.qr = plan->qrot; ra.kr = plan->krot;
    ra.heads = p.num_heads; ra.head_dim = p.head_dim;
    std::memcpy(ra.omega, plan->omega, sizeof ra.omega);
    e = launch_rope(ra, p.dtype, plan->NT, st);
    if (e != cudaSuccess) return from_cuda(e);
    qs = plan->qrot; ks = plan->krot;
  }
  e = cudaStreamWaitEvent(st, plan->ev_plan, 0);
  if (e != cudaSuccess) return from_cuda(e);
  BwdArgs a;
  a.meta = plan->pd.meta; a.batch = plan->batch; a.kcount = plan->pd.kcount; a.klist = plan->pd.klist;
  a.qkeep = plan->pd.qkeep;
  a.items = plan->pd.items; a.qreq = plan->pd.qreq; a.krec = plan->pd.krec;
  a.n_items = plan->NT * p.num_heads;
  a.status = plan->pd.status;
  a.counters = plan->pd.counters;
  a.cls = plan->pd.cls; a.t = plan->t; a.ty = plan->ty;
  a.q = qs; a.k = ks; a.v = v; a.out = out; a.dout = dout; a.dout_attn = dout_attn; a.lse = lse;
  a.delta = tc ? nullptr : reinterpret_cast<float*>(bws);
  a.n_tiles = plan->NT;
  a.desc = tc ? reinterpret_cast<const BwdItemDesc*>(bws) : nullptr;
  a.rowc = tc ? reinterpret_cast<float2*>(bws + off_rowc) : nullptr;
  a.qlist = tc ? reinterpret_cast<const uint32_t*>(bws + off_ql) : nullptr;
  a.kslot = plan->pd.kslot; a.mtab = plan->pd.mtab;
  a.qslot = tc ? reinterpret_cast<const int*>(bws + off_qs) : nullptr;
  a.ctab = tc ? reinterpret_cast<const uint32_t*>(bws + off_ct) : nullptr;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.rows = T * p.num_heads; a.heads = p.num_heads; a.scale = p.softmax_scale;
  a.rotate = p.use_rope; a.mask = plan->mask;
  std::memcpy(a.omega, plan->omega, sizeof a.omega);
  if (!tc) {
    e = launch_bwd_delta(a, p.dtype, p.head_dim, st);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(launch_attn_bwd_simt(a, p.head_dim, plan->NT, st));
  }
  if (!plan->bwd_sched) {  // the plan's masks never change: its backward schedule is built once
    BwdSchedArgs sa;
    sa.meta = plan->pd.meta; sa.qreq = plan->pd.qreq; sa.items = plan->pd.items; sa.kcount = plan->pd.kcount;
    sa.cls = plan->pd.cls; sa.t = plan->t; sa.n_tiles = plan->NT; sa.n_items = n_items; sa.heads = p.num_heads;
    sa.desc = reinterpret_cast<BwdItemDesc*>(bws);
    sa.qlist = reinterpret_cast<uint32_t*>(bws + off_ql);
    sa.pslot = plan->pd.pslot; sa.qslot = reinterpret_cast<int*>(bws + off_qs);
    sa.counters = plan->pd.counters; sa.mtab = plan->pd.mtab;
    sa.ctab = reinterpret_cast<uint32_t*>(bws + off_ct); sa.mcap = plan->pd.mcap;
    e = launch_bwd_schedule(sa, plan->num_sms, st);
    if (e != cudaSuccess) return from_cuda(e);
    plan->bwd_sched = true;
  }
  CUtensorMap maps[4];  // Q', K', V, the attention's dO
  const void* srcs[4] = {qs, ks, v, dout_attn};
  const long long cols = (long long)p.num_heads * p.head_dim;
  for (int i = 0; i < 4; ++i)
    if (!encode_map(&maps[i], srcs[i], T, cols)) return REC_ATTN_ERR_CUDA;
  return from_cuda(launch_attn_bwd_tc(a, maps, p.head_dim, plan->num_sms, st));
}

}  // namespace

REC_ATTN_API rec_attn_status rec_attn_bwd(rec_attn_plan_t* plan, const void* q, const void* k, const void* v,
                                          const void* out, const float* lse, const void* dout, void* dq,
                                          void* dk, void* dv, void* stream) {
  return bwd_impl(plan, q, k, v, out, lse, dout, dout, dq, dk, dv, stream, nullptr);
}

REC_ATTN_API rec_attn_status rec_attn_bwd_fused(rec_attn_plan_t* plan, const void* q, const void* k, const void* v,
                                                const rec_attn_fused* fused, const void* out, const float* lse,
                                                const void* dout, void* dq, void* dk, void* dv,
                                                const rec_attn_fused_grads* grads, void* stream) {
  if (!plan || !fused || !grads) return REC_ATTN_ERR_INVALID_ARG;
  const rec_attn_params& p = plan->p;
  const long long T = plan->T;
  if (!(fused->norm_eps >= 0.f) || !std::isfinite(fused->norm_eps)) return REC_ATTN_ERR_INVALID_ARG;
  const bool qside = fused->q_norm_weight || fused->q_gate, kside = fused->k_norm_weight || fused->k_gate;
  // a gradient for every step that is on
  if ((fused->q_gate && !grads->dq_gate) || (fused->k_gate && !grads->dk_gate) ||
      (fused->out_gate && !grads->dout_gate) || (fused->q_norm_weight && !grads->dq_norm_weight) ||
      (fused->k_norm_weight && !grads->dk_norm_weight))
    return REC_ATTN_ERR_INVALID_ARG;
  const size_t elem = p.dtype == REC_ATTN_BF16 ? 2 : 4;
  const size_t bytes = (size_t)T * p.num_heads * p.head_dim * elem;
  if (T > 0) {
    const void* al16[6] = {fused->q_gate, fused->k_gate, fused->out_gate, grads->dq_gate, grads->dk_gate,
                           grads->dout_gate};
    for (const void* x : al16)
      if (reinterpret_cast<uintptr_t>(x) & 15u) return REC_ATTN_ERR_INVALID_ARG;
    const void* al4[4] = {fused->q_norm_weight, fused->k_norm_weight, grads->dq_norm_weight, grads->dk_norm_weight};
    for (const void* x : al4)
      if (reinterpret_cast<uintptr_t>(x) & 3u) return REC_ATTN_ERR_INVALID_ARG;
    void* gouts[3] = {grads->dq_gate, grads->dk_gate, grads->dout_gate};
    const void* gins[8] = {q, k, v, out, dout, fused->q_gate, fused->k_gate, fused->out_gate};
    for (void* g : gouts)
      for (const void* x : gins)
        if (g && x && overlaps(g, bytes, x, bytes)) return REC_ATTN_ERR_INVALID_ARG;
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (dev != plan->device) return REC_ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) return bwd_impl(plan, q, k, v, out, lse, dout, dout, dq, dk, dv, stream, nullptr);
  // scratch: the attention's dO (with an output gate) and the gradients of the gated,
  // normalised Q and K (with a Q- or K-side step)
  const size_t rows = ws_up(bytes);
  char* scratch = nullptr;
  const size_t n_scr = (fused->out_gate ? 1 : 0) + (qside ? 1 : 0) + (kside ? 1 : 0);
  if (n_scr) {
    cudaMemPool_t pool;
    e = pool_for(plan->device, &pool);
    if (e == cudaSuccess) e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch), n_scr * rows, pool, st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  char* next = scratch;
  void* dout_attn = fused->out_gate ? next : const_cast<void*>(dout);
  if (fused->out_gate) next += rows;
  void* dgq = qside ? next : dq;
  if (qside) next += rows;
  void* dgk = kside ? next : dk;
  GateArgs ga{};
  ga.n = (long long)T * p.num_heads * p.head_dim;
  ga.dout = dout; ga.out = out; ga.gate = fused->out_gate; ga.dout_attn = dout_attn; ga.dgate = grads->dout_gate;
  if (fused->out_gate) e = launch_bwd_gate(ga, p.dtype, st);
  FusedArgs fa;
  fa.q_norm_w = fused->q_norm_weight; fa.k_norm_w = fused->k_norm_weight; fa.eps = fused->norm_eps;
  fa.q_gate = fused->q_gate; fa.k_gate = fused->k_gate;
  rec_attn_status s = REC_ATTN_OK;
  if (e == cudaSuccess) s = bwd_impl(plan, q, k, v, out, lse, dout, dout_attn, dgq, dgk, dv, stream, &fa);
  for (int side = 0; side < 2 && e == cudaSuccess && s == REC_ATTN_OK; ++side) {
    if (!(side == 0 ? qside : kside)) continue;
    NormGateArgs na{};
    na.rows = T; na.heads = p.num_heads; na.head_dim = p.head_dim; na.eps = fused->norm_eps;
    na.a = side == 0 ? q : k;
    na.w = side == 0 ? fused->q_norm_weight : fused->k_norm_weight;
    na.gate = side == 0 ? fused->q_gate : fused->k_gate;
    na.dg = side == 0 ? dgq : dgk;
    na.da = side == 0 ? dq : dk;
    na.dgate = side == 0 ? grads->dq_gate : grads->dk_gate;
    na.dw = side == 0 ? grads->dq_norm_weight : grads->dk_norm_weight;
    if (na.dw) e = cudaMemsetAsync(na.dw, 0, sizeof(float) * (size_t)p.num_heads * p.head_dim, st);
    if (e == cudaSuccess) e = launch_bwd_norm_gate(na, p.dtype, st);
  }
  if (scratch) {
    const cudaError_t ef = cudaFreeAsync(scratch, st);
    if (e == cudaSuccess) e = ef;
  }
  if (s != REC_ATTN_OK) return s;
  return from_cuda(e);
}

namespace {

// Output lengths of history compression (host arithmetic, checked): per request, the
// groups of each recency segment, ceil(covered / group).
rec_attn_status compress_layout(int32_t batch, const int64_t* offsets_host, const int64_t* hist_begin_host,
                                const int64_t* hist_len_host, int32_t n_segments, const int64_t* seg_len,
                                const int32_t* seg_group, std::vector<CompressReq>* reqs, int64_t* out_offsets) {
  if (batch < 0 || (batch > 0 && (!offsets_host || !hist_begin_host || !hist_len_host)))
    return REC_ATTN_ERR_INVALID_ARG;
  if (n_segments < 1 || n_segments > kMaxSegments || !seg_len || !seg_group) return REC_ATTN_ERR_INVALID_ARG;
  bool unbounded = false;
  for (int i = 0; i < n_segments; ++i) {
    if (seg_group[i] < 1) return REC_ATTN_ERR_INVALID_ARG;
    if (seg_len[i] < 0) unbounded = true;
  }
  if (batch > 0 && offsets_host[0] != 0) return REC_ATTN_ERR_INVALID_ARG;
  long long out = 0;
  if (out_offsets) out_offsets[0] = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const long long len = offsets_host[b + 1] - offsets_host[b];
    const long long hb = hist_begin_host[b], hl = hist_len_host[b];
    if (len < 0 || hb < 0 || hl < 0 || hb + hl > len) return REC_ATTN_ERR_INVALID_ARG;
    long long covered = 0, groups = 0;
    for (int i = 0; i < n_segments && covered < hl; ++i) {
      const long long room = hl - covered;
      const long long m = (seg_len[i] < 0 || seg_len[i] > room) ? room : seg_len[i];
      groups += (m + seg_group[i] - 1) / seg_group[i];
      covered += m;
    }
    if (covered < hl && !unbounded) return REC_ATTN_ERR_INVALID_ARG;  // the segments must cover the history
    CompressReq r;
    r.in_start = offsets_host[b]; r.len = len; r.hist_begin = hb; r.hist_len = hl;
    r.out_start = out; r.out_len = len - hl + groups;
    out += r.out_len;
    if (reqs) reqs->push_back(r);
    if (out_offsets) out_offsets[b + 1] = out;
  }
  return REC_ATTN_OK;
}

}  // namespace

REC_ATTN_API rec_attn_status rec_attn_compress_lengths(int32_t batch, const int64_t* offsets_host,
                                                       const int64_t* hist_begin_host, const int64_t* hist_len_host,
                                                       int32_t n_segments, const int64_t* seg_len,
                                                       const int32_t* seg_group, int64_t* out_offsets_host) {
  if (!out_offsets_host) return REC_ATTN_ERR_INVALID_ARG;
  return compress_layout(batch, offsets_host, hist_begin_host, hist_len_host, n_segments, seg_len, seg_group,
                         nullptr, out_offsets_host);
}

REC_ATTN_API rec_attn_status rec_attn_compress(int32_t batch, const int64_t* offsets_host,
                                               const int64_t* hist_begin_host, const int64_t* hist_len_host,
                                               int32_t n_segments, const int64_t* seg_len, const int32_t* seg_group,
                                               int32_t dtype, int64_t width, const void* x,
                                               const int64_t* timestamps, const int8_t* types, void* x_out,
                                               int64_t* timestamps_out, int8_t* types_out, void* stream) {
  if (dtype != REC_ATTN_BF16 && dtype != REC_ATTN_FP32) return REC_ATTN_ERR_INVALID_ARG;
  const size_t elem = dtype == REC_ATTN_BF16 ? 2 : 4;
  if (width < 1 || ((size_t)width * elem) % 16 != 0) return REC_ATTN_ERR_INVALID_ARG;
  std::vector<CompressReq> reqs;
  reqs.reserve((size_t)(batch > 0 ? batch : 0));
  rec_attn_status stt = compress_layout(batch, offsets_host, hist_begin_host, hist_len_host, n_segments, seg_len,
                                        seg_group, &reqs, nullptr);
  if (stt != REC_ATTN_OK) return stt;
  const long long rows_out = reqs.empty() ? 0 : reqs.back().out_start + reqs.back().out_len;
  const long long rows_in = batch > 0 ? offsets_host[batch] : 0;
  if (rows_out == 0) return REC_ATTN_OK;
  const void* ptrs[5] = {x, timestamps, types, x_out, timestamps_out};
  for (const void* p : ptrs)
    if (!p) return REC_ATTN_ERR_INVALID_ARG;
  if (!types_out || (reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_out) & 15u) ||
      (reinterpret_cast<uintptr_t>(timestamps) & 7u) || (reinterpret_cast<uintptr_t>(timestamps_out) & 7u))
    return REC_ATTN_ERR_INVALID_ARG;
  if (overlaps(x_out, (size_t)rows_out * width * elem, x, (size_t)rows_in * width * elem))
    return REC_ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  cudaMemPool_t pool;
  if (e == cudaSuccess) e = pool_for(dev, &pool);
  void* dreq = nullptr;
  const size_t req_bytes = sizeof(CompressReq) * reqs.size();
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&dreq, req_bytes, pool, st);
  if (e != cudaSuccess) return from_cuda(e);
  // pageable source: the copy is staged before the call returns, so reqs may go away
  e = cudaMemcpyAsync(dreq, reqs.data(), req_bytes, cudaMemcpyHostToDevice, st);
  CompressArgs a;
  a.req = static_cast<const CompressReq*>(dreq);
  a.batch = batch; a.n_seg = n_segments; a.rows_out = rows_out;
  for (int i = 0; i < kMaxSegments; ++i) {
    a.seg_len[i] = i < n_segments ? seg_len[i] : 0;
    a.seg_group[i] = i < n_segments ? seg_group[i] : 1;
  }
  a.width = width; a.x = x; a.t = reinterpret_cast<const long long*>(timestamps); a.ty = types;
  a.x_out = x_out; a.t_out = reinterpret_cast<long long*>(timestamps_out); a.ty_out = types_out;
  if (e == cudaSuccess) e = launch_compress(a, dtype, st);
  cudaError_t e2 = cudaFreeAsync(dreq, st);
  return from_cuda(e != cudaSuccess ? e : e2);
}

REC_ATTN_API rec_attn_status rec_attn_fwd_compress(rec_attn_plan_t* plan, const void* q, const void* k,
                                                   const void* v, const int64_t* hist_begin_host,
                                                   const int64_t* hist_len_host, int32_t n_segments,
                                                   const int64_t* seg_len, const int32_t* seg_group, void* x_out,
                                                   int64_t* timestamps_out, int8_t* types_out, void* stream) {
  if (!plan) return REC_ATTN_ERR_INVALID_ARG;
  const rec_attn_params& p = plan->p;
  if (p.dtype != REC_ATTN_BF16 || plan->mask.keep_user >= 0) return REC_ATTN_ERR_UNSUPPORTED;
  const int32_t B = plan->batch;
  std::vector<CompressReq> reqs;
  reqs.reserve((size_t)B);
  rec_attn_status s = compress_layout(B, plan->offsets_host.data(), hist_begin_host, hist_len_host, n_segments,
                                      seg_len, seg_group, &reqs, nullptr);
  if (s != REC_ATTN_OK) return s;
  for (int i = 0; i < n_segments; ++i)
    if (seg_group[i] > 32) return REC_ATTN_ERR_UNSUPPORTED;  // a group spans at most two 32-row blocks
  const long long T = plan->T;
  const long long rows_out = reqs.empty() ? 0 : reqs.back().out_start + reqs.back().out_len;
  if (rows_out == 0) return REC_ATTN_OK;
  if (!x_out || !timestamps_out || !types_out || (reinterpret_cast<uintptr_t>(x_out) & 15u) ||
      (reinterpret_cast<uintptr_t>(timestamps_out) & 7u))
    return REC_ATTN_ERR_INVALID_ARG;
  const size_t row_bytes = (size_t)p.num_heads * p.head_dim * 2;
  if (overlaps(x_out, rows_out * row_bytes, q, T * row_bytes) || overlaps(x_out, rows_out * row_bytes, k, T * row_bytes) ||
      overlaps(x_out, rows_out * row_bytes, v, T * row_bytes))
    return REC_ATTN_ERR_INVALID_ARG;
  // per request: where its rows go and its first 32-row block boundary in the fix-up buffer
  std::vector<CmpReq> creq((size_t)B);
  std::vector<int> lens((size_t)B);
  long long n_fix = 0;
  for (int32_t b = 0; b < B; ++b) {
    const CompressReq& r = reqs[b];
    CmpReq& c = creq[b];
    c.out_start = r.out_start;
    c.fix_start = n_fix;
    c.hist_begin = (int)r.hist_begin;
    c.hist_len = (int)r.hist_len;
    c.n_groups = (int)(r.out_len - (r.len - r.hist_len));
    c.pad = 0;
    lens[b] = (int)r.len;
    n_fix += (r.len + 31) / 32;
  }
  const size_t off_len = ws_up(sizeof(CmpReq) * (size_t)B);
  const size_t off_creq = off_len + ws_up(4 * (size_t)B);
  const size_t off_fix = off_creq + ws_up(sizeof(CompressReq) * (size_t)B);
  const size_t fix_bytes = (size_t)n_fix * 2 * p.num_heads * p.head_dim * sizeof(float);
  std::vector<char> up(off_fix, 0);
  std::memcpy(up.data(), creq.data(), sizeof(CmpReq) * (size_t)B);
  std::memcpy(up.data() + off_len, lens.data(), 4 * (size_t)B);
  std::memcpy(up.data() + off_creq, reqs.data(), sizeof(CompressReq) * (size_t)B);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (dev != plan->device) return REC_ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaMemPool_t pool;
  char* buf = nullptr;
  e = pool_for(plan->device, &pool);
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), off_fix + fix_bytes, pool, st);
  if (e != cudaSuccess) return from_cuda(e);
  e = cudaMemcpyAsync(buf, up.data(), up.size(), cudaMemcpyHostToDevice, st);  // staged before the call returns
  CmpArgs c{};
  c.req = reinterpret_cast<const CmpReq*>(buf);
  c.x_out = x_out;
  c.fix = reinterpret_cast<float*>(buf + off_fix);
  c.n_seg = n_segments;
  c.span = 1;
  for (int i = 0; i < kMaxSegments; ++i) {
    c.seg_len[i] = i < n_segments ? seg_len[i] : 0;
    c.seg_group[i] = i < n_segments ? seg_group[i] : 1;
    if (i < n_segments) c.span = std::max(c.span, (int)seg_group[i]);
  }
  if (e == cudaSuccess) s = fwd_impl(plan, q, k, v, nullptr, x_out, nullptr, stream, &c);
  if (e == cudaSuccess && s == REC_ATTN_OK)
    e = launch_cmp_fixup(c, B, reinterpret_cast<const int*>(buf + off_len), n_fix, p.num_heads, p.head_dim, st);
  if (e == cudaSuccess && s == REC_ATTN_OK) {
    // times and types of the output rows (the latest member time, type HIST for merged rows)
    CompressArgs ca;
    ca.req = reinterpret_cast<const CompressReq*>(buf + off_creq);
    ca.batch = B; ca.n_seg = n_segments; ca.rows_out = rows_out;
    for (int i = 0; i < kMaxSegments; ++i) { ca.seg_len[i] = c.seg_len[i]; ca.seg_group[i] = c.seg_group[i]; }
    ca.width = 0; ca.x = nullptr; ca.t = plan->t; ca.ty = plan->ty;
    ca.x_out = nullptr; ca.t_out = reinterpret_cast<long long*>(timestamps_out); ca.ty_out = types_out;
    e = launch_compress(ca, p.dtype, st);
  }
  const cudaError_t ef = cudaFreeAsync(buf, st);
  if (s != REC_ATTN_OK) return s;
  return from_cuda(e != cudaSuccess ? e : ef);
}

REC_ATTN_API rec_attn_status rec_attn_check_wait_timeout(uint32_t limit_ms, int32_t* status_out, void* stream) {
  if (!status_out || limit_ms < 1 || limit_ms > 10000) return REC_ATTN_ERR_INVALID_ARG;
  *status_out = REC_ATTN_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  cudaMemPool_t pool;
  if (e == cudaSuccess) e = pool_for(dev, &pool);
  void* d = nullptr;
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&d, sizeof(int), pool, st);
  if (e != cudaSuccess) return from_cuda(e);
  int h = 0;
  e = cudaMemsetAsync(d, 0, sizeof(int), st);
  if (e == cudaSuccess) e = launch_wait_timeout(static_cast<int*>(d), (unsigned long long)limit_ms * 1000000ull, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, d, sizeof(int), cudaMemcpyDeviceToHost, st);
  cudaError_t e2 = cudaFreeAsync(d, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = e2;
  if (e != cudaSuccess) return from_cuda(e);
  *status_out = h;
  return REC_ATTN_OK;
}

REC_ATTN_API void rec_attn_free(rec_attn_plan_t* plan) {
  if (!plan) return;
  if (plan->ws) {
    cudaStreamWaitEvent(plan->stream, plan->ev_plan, 0);  // planning may still run on the side stream
    cudaFreeAsync(plan->ws, plan->stream);
  }
  if (plan->qk_extra) cudaFreeAsync(plan->qk_extra, plan->stream);
  if (plan->bwd_ws) cudaFreeAsync(plan->bwd_ws, plan->stream);
  for (cudaEvent_t ev : plan->ev)
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : {plan->ev_in, plan->ev_meta, plan->ev_plan})
    if (ev) cudaEventDestroy(ev);
  delete plan;
}

REC_ATTN_API rec_attn_status rec_attn_enable_timing(rec_attn_plan_t* plan) {
  if (!plan) return REC_ATTN_ERR_INVALID_ARG;
  if (plan->timing) return REC_ATTN_OK;
  for (cudaEvent_t& ev : plan->ev) {
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) return from_cuda(e);
  }
  plan->timing = true;
  return REC_ATTN_OK;
}

REC_ATTN_API rec_attn_status rec_attn_read_timings(rec_attn_plan_t* plan, rec_attn_timings* out) {
  if (!plan || !out || !plan->timing || !plan->timed) return REC_ATTN_ERR_INVALID_ARG;
  cudaError_t e = cudaEventSynchronize(plan->ev[3]);
  float a = 0.f, b = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&a, plan->ev[0], plan->ev[1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&b, plan->ev[2], plan->ev[3]);
  if (e != cudaSuccess) return from_cuda(e);
  out->rope_ms = a;
  out->attn_ms = b;
  return REC_ATTN_OK;
}

REC_ATTN_API rec_attn_status rec_attn_tile_classes(rec_attn_plan_t* plan, uint8_t* host_out, size_t capacity,
                                                   size_t* n_needed) {
  if (!plan || !n_needed) return REC_ATTN_ERR_INVALID_ARG;
  *n_needed = (size_t)plan->NC;
  if (!host_out) return REC_ATTN_OK;
  if (capacity < (size_t)plan->NC) return REC_ATTN_ERR_INVALID_ARG;
  if (plan->NC == 0) return REC_ATTN_OK;
  cudaError_t e = cudaStreamWaitEvent(plan->stream, plan->ev_plan, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(host_out, plan->pd.cls, (size_t)plan->NC, cudaMemcpyDeviceToHost, plan->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(plan->stream);
  return from_cuda(e);
}

REC_ATTN_API rec_attn_status rec_attn_visible_pairs(rec_attn_plan_t* plan, uint64_t* host_out) {
  if (!plan || !host_out) return REC_ATTN_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamWaitEvent(plan->stream, plan->ev_plan, 0);
  if (e == cudaSuccess) e = cudaMemsetAsync(plan->pd.pairs, 0, sizeof(unsigned long long), plan->stream);
  if (e == cudaSuccess) e = launch_count_pairs(plan->mask, plan->pd, plan->t, plan->ty, plan->NT, plan->stream);
  unsigned long long n = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&n, plan->pd.pairs, sizeof n, cudaMemcpyDeviceToHost, plan->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(plan->stream);
  if (e == cudaSuccess) *host_out = n;
  return from_cuda(e);
}

REC_ATTN_API rec_attn_status rec_attn_applied_masks(rec_attn_plan_t* plan, int32_t n_pairs, const int32_t* pairs_host,
                                                    int32_t mode, uint32_t* bits_host, uint8_t* list_class_host,
                                                    int32_t* slot_host) {
  if (!plan || n_pairs < 0 || (n_pairs > 0 && (!pairs_host || !bits_host))) return REC_ATTN_ERR_INVALID_ARG;
  if (mode < 0 || mode > 2) return REC_ATTN_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_pairs; ++i) {
    const int32_t b = pairs_host[3 * i], qt = pairs_host[3 * i + 1], kt = pairs_host[3 * i + 2];
    if (b < 0 || b >= plan->batch) return REC_ATTN_ERR_INVALID_ARG;
    const int nt = plan->req_tiles[b];
    if (qt < 0 || qt >= nt || kt < 0 || kt >= nt) return REC_ATTN_ERR_INVALID_ARG;
  }
  if (n_pairs == 0) return REC_ATTN_OK;
  const size_t bits_bytes = (size_t)n_pairs * kTile * 16;
  const size_t pairs_bytes = ((size_t)n_pairs * 12 + 255) & ~(size_t)255;
  const size_t cls_bytes = ((size_t)n_pairs + 255) & ~(size_t)255;
  cudaStream_t st = plan->stream;
  cudaMemPool_t pool;
  char* buf = nullptr;
  cudaError_t e = pool_for(plan->device, &pool);
  if (e == cudaSuccess)
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), bits_bytes + pairs_bytes + cls_bytes +
                                (size_t)n_pairs * 4, pool, st);
  if (e != cudaSuccess) return from_cuda(e);
  int* d_pairs = reinterpret_cast<int*>(buf + bits_bytes);
  uint8_t* d_cls = reinterpret_cast<uint8_t*>(buf + bits_bytes + pairs_bytes);
  int* d_slot = reinterpret_cast<int*>(buf + bits_bytes + pairs_bytes + cls_bytes);
  e = cudaStreamWaitEvent(st, plan->ev_plan, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_pairs, pairs_host, (size_t)n_pairs * 12, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = launch_export_masks(plan->mask, plan->pd, plan->t, plan->ty, d_pairs, n_pairs, mode,
                            reinterpret_cast<uint32_t*>(buf), d_cls, d_slot, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(bits_host, buf, bits_bytes, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && list_class_host)
    e = cudaMemcpyAsync(list_class_host, d_cls, (size_t)n_pairs, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && slot_host)
    e = cudaMemcpyAsync(slot_host, d_slot, (size_t)n_pairs * 4, cudaMemcpyDeviceToHost, st);
  const cudaError_t ef = cudaFreeAsync(buf, st);
  if (e == cudaSuccess) e = ef;
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return from_cuda(e);
}

REC_ATTN_API rec_attn_status rec_attn_device_status(rec_attn_plan_t* plan, int32_t* status_out) {
  if (!plan || !status_out) return REC_ATTN_ERR_INVALID_ARG;
  int s = 0;
  cudaError_t e = cudaStreamWaitEvent(plan->stream, plan->ev_plan, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&s, plan->pd.status, sizeof s, cudaMemcpyDeviceToHost, plan->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(plan->stream);
  if (e == cudaSuccess) *status_out = s;
  return from_cuda(e);
}

// ---------------------------------------------------------------------------------
// Serving with a cached history (M-FALCON, HSTU notes on the blog index page: the
// user's history keys and values are computed once and every candidate micro-batch
// reads them; CADET's serving section scores hundreds of candidates per request).
//
// The cache keeps every request's rows in a combined layout: the history rows, then
// max_cands candidate slots.  Creation rotates the history keys once (K'), copies the
// values, times and types.  A scoring call writes its candidates into the slots
// (rotated Q' and K' against the same per-request reference time, V, time, type
// CAND; unused slots are zero padding that no real token sees), plans a layer in
// which only non-user tokens query (target attention over [history, slots]), runs
// the attention kernel on the cached, already rotated rows, and gathers the
// candidates' outputs back to the caller's packed layout.

struct rec_attn_kv_cache_s {
  rec_attn_params p{};   // the caller's parameters
  rec_attn_params pp{};  // those of the per-call plans: the rows are already rotated
  int device = 0;
  int32_t batch = 0;
  int32_t max_cands = 0;
  long long Tc = 0;                 // rows of the combined layout
  std::vector<int64_t> comb_off;    // [B+1] host: request b owns rows comb_off[b] ..
  std::vector<long long> hist_len;  // [B]
  void* buf = nullptr;              // combined Q', K', V, O, lse, t, types, offsets
  void *q, *k, *v, *o;
  float* lse = nullptr;
  long long* t = nullptr;
  int8_t* ty = nullptr;
  int64_t* off_dev = nullptr;
  float omega[kMaxPairs] = {};
};

namespace {

// Region table of k_rope_slots / k_slots_gather: SlotReq per request, then the
// request and first row of every 128-row chunk; staged through one pool buffer.
struct SlotTable {
  std::vector<char> host;
  size_t off_chunk_req = 0, off_chunk_row0 = 0;
  long long n_chunks = 0;
};

SlotTable slot_table(const std::vector<SlotReq>& reqs) {
  SlotTable st;
  std::vector<int> creq, crow;
  for (size_t b = 0; b < reqs.size(); ++b)
    for (int r0 = 0; r0 < reqs[b].cap; r0 += kTile) {
      creq.push_back((int)b);
      crow.push_back(r0);
    }
  st.n_chunks = (long long)creq.size();
  st.off_chunk_req = ((reqs.size() * sizeof(SlotReq)) + 15) & ~(size_t)15;
  st.off_chunk_row0 = st.off_chunk_req + ((creq.size() * 4 + 15) & ~(size_t)15);
  st.host.assign(st.off_chunk_row0 + crow.size() * 4 + 16, 0);
  std::memcpy(st.host.data(), reqs.data(), reqs.size() * sizeof(SlotReq));
  std::memcpy(st.host.data() + st.off_chunk_req, creq.data(), creq.size() * 4);
  std::memcpy(st.host.data() + st.off_chunk_row0, crow.data(), crow.size() * 4);
  return st;
}

// Upload a region table into pool memory on `st` (freed in stream order by the caller).
cudaError_t upload_table(const SlotTable& tab, int device, cudaStream_t st, void** dev) {
  cudaMemPool_t pool;
  cudaError_t e = pool_for(device, &pool);
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(dev, tab.host.size(), pool, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(*dev, tab.host.data(), tab.host.size(), cudaMemcpyHostToDevice, st);
  return e;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

REC_ATTN_API rec_attn_status rec_attn_cache_create(const rec_attn_params* params, int32_t batch,
                                                   const int64_t* hist_offsets_host, const int64_t* hist_t_dev,
                                                   const int8_t* hist_types_dev, const void* k_hist,
                                                   const void* v_hist, int32_t max_cands, void* stream,
                                                   rec_attn_kv_cache_t** cache_out) {
  if (!cache_out) return REC_ATTN_ERR_INVALID_ARG;
  *cache_out = nullptr;
  rec_attn_status s = check_params(params);
  if (s != REC_ATTN_OK) return s;
  if (batch < 1 || !hist_offsets_host || max_cands < 1) return REC_ATTN_ERR_INVALID_ARG;
  if (hist_offsets_host[0] != 0) return REC_ATTN_ERR_INVALID_ARG;
  long long Th = 0, Tc = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const long long len = hist_offsets_host[b + 1] - hist_offsets_host[b];
    if (len < 0) return REC_ATTN_ERR_INVALID_ARG;
    if (len + max_cands > REC_ATTN_MAX_REQUEST_LEN) return REC_ATTN_ERR_UNSUPPORTED;
    Tc += len + max_cands;
  }
  Th = hist_offsets_host[batch];
  if (Tc >= (1LL << 31)) return REC_ATTN_ERR_UNSUPPORTED;
  if (Th > 0 && (!hist_t_dev || !hist_types_dev || !k_hist || !v_hist || !aligned16(k_hist) || !aligned16(v_hist)))
    return REC_ATTN_ERR_INVALID_ARG;

  rec_attn_kv_cache_s* c = new (std::nothrow) rec_attn_kv_cache_s();
  if (!c) return REC_ATTN_ERR_OOM;
  try {
    c->comb_off.resize((size_t)batch + 1);
    c->hist_len.resize((size_t)batch);
  } catch (...) {
    delete c;
    return REC_ATTN_ERR_OOM;
  }
  c->p = *params;
  if (c->p.softmax_scale == 0.f) c->p.softmax_scale = 1.f / std::sqrt((float)params->head_dim);
  c->pp = c->p;
  c->pp.use_rope = 0;
  c->batch = batch;
  c->max_cands = max_cands;
  c->Tc = Tc;
  c->comb_off[0] = 0;
  for (int32_t b = 0; b < batch; ++b) {
    c->hist_len[b] = hist_offsets_host[b + 1] - hist_offsets_host[b];
    c->comb_off[b + 1] = c->comb_off[b] + c->hist_len[b] + max_cands;
  }
  if (params->use_rope)
    for (int i = 0; i < params->head_dim / 2 && i < kMaxPairs; ++i)
      c->omega[i] = (float)(params->phi_min / params->dt_max_s *
                            std::pow(params->rope_base, 2.0 * i / (double)params->head_dim));
  const size_t elem = params->dtype == REC_ATTN_BF16 ? 2 : 4;
  const size_t rows_bytes = ws_up((size_t)Tc * params->num_heads * params->head_dim * elem);
  const size_t lse_bytes = ws_up((size_t)Tc * params->num_heads * 4);
  const size_t t_bytes = ws_up((size_t)Tc * 8), ty_bytes = ws_up((size_t)Tc), off_bytes = ws_up(8 * ((size_t)batch + 1));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaGetDevice(&c->device);
  cudaMemPool_t pool;
  if (e == cudaSuccess) e = pool_for(c->device, &pool);
  if (e == cudaSuccess)
    e = cudaMallocFromPoolAsync(&c->buf, 4 * rows_bytes + lse_bytes + t_bytes + ty_bytes + off_bytes, pool, st);
  if (e != cudaSuccess) { delete c; return from_cuda(e); }
  char* w = static_cast<char*>(c->buf);
  c->q = w; c->k = w + rows_bytes; c->v = w + 2 * rows_bytes; c->o = w + 3 * rows_bytes;
  c->lse = reinterpret_cast<float*>(w + 4 * rows_bytes);
  c->t = reinterpret_cast<long long*>(w + 4 * rows_bytes + lse_bytes);
  c->ty = reinterpret_cast<int8_t*>(w + 4 * rows_bytes + lse_bytes + t_bytes);
  c->off_dev = reinterpret_cast<int64_t*>(w + 4 * rows_bytes + lse_bytes + t_bytes + ty_bytes);
  // history rows: rotated keys, values, times and types (queries stay zero: no user
  // token queries in a scoring call); the candidate slots are written by each call
  std::vector<SlotReq> reqs((size_t)batch);
  for (int32_t b = 0; b < batch; ++b) {
    SlotReq& r = reqs[b];
    r.src_start = hist_offsets_host[b];
    r.dst_start = c->comb_off[b];
    r.ref_row = hist_offsets_host[b];
    r.ref_dst = 0;
    r.len = r.cap = (int)c->hist_len[b];
    r.pad = 0;
  }
  const SlotTable tab = slot_table(reqs);
  void* dtab = nullptr;
  e = cudaMemsetAsync(c->q, 0, rows_bytes, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->off_dev, c->comb_off.data(), 8 * ((size_t)batch + 1),
                                            cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && tab.n_chunks > 0) {
    e = upload_table(tab, c->device, st, &dtab);
    if (e == cudaSuccess) {
      SlotArgs a{};
      a.req = static_cast<const SlotReq*>(dtab);
      a.chunk_req = reinterpret_cast<const int*>(static_cast<char*>(dtab) + tab.off_chunk_req);
      a.chunk_row0 = reinterpret_cast<const int*>(static_cast<char*>(dtab) + tab.off_chunk_row0);
      a.t_src = reinterpret_cast<const long long*>(hist_t_dev);
      a.ty_src = hist_types_dev;
      a.q_src = nullptr; a.k_src = k_hist; a.v_src = v_hist;
      a.q_dst = nullptr; a.k_dst = c->k; a.v_dst = c->v; a.t_dst = c->t; a.ty_dst = c->ty;
      a.heads = params->num_heads; a.head_dim = params->head_dim;
      std::memcpy(a.omega, c->omega, sizeof a.omega);
      e = launch_rope_slots(a, params->dtype, tab.n_chunks, st);
    }
    if (dtab) {
      const cudaError_t ef = cudaFreeAsync(dtab, st);
      if (e == cudaSuccess) e = ef;
    }
  }
  if (e != cudaSuccess) {
    cudaFreeAsync(c->buf, st);
    delete c;
    return from_cuda(e);
  }
  *cache_out = c;
  return REC_ATTN_OK;
}

REC_ATTN_API rec_attn_status rec_attn_cache_score(rec_attn_kv_cache_t* c, const int64_t* cand_offsets_host,
                                                  const int64_t* cand_t_dev, const void* q_cand, const void* k_cand,
                                                  const void* v_cand, void* out, float* lse, void* stream) {
  if (!c || !cand_offsets_host || cand_offsets_host[0] != 0) return REC_ATTN_ERR_INVALID_ARG;
  for (int32_t b = 0; b < c->batch; ++b) {
    const long long n = cand_offsets_host[b + 1] - cand_offsets_host[b];
    if (n < 0 || n > c->max_cands) return REC_ATTN_ERR_INVALID_ARG;
  }
  const long long Nc = cand_offsets_host[c->batch];
  const rec_attn_params& p = c->p;
  const size_t elem = p.dtype == REC_ATTN_BF16 ? 2 : 4;
  if (Nc > 0) {
    if (!cand_t_dev || !q_cand || !k_cand || !v_cand || !out) return REC_ATTN_ERR_INVALID_ARG;
    const void* ptrs[4] = {q_cand, k_cand, v_cand, out};
    for (const void* x : ptrs)
      if (!aligned16(x)) return REC_ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return REC_ATTN_ERR_INVALID_ARG;
    const size_t bytes = (size_t)Nc * p.num_heads * p.head_dim * elem;
    if (overlaps(out, bytes, q_cand, bytes) || overlaps(out, bytes, k_cand, bytes) ||
        overlaps(out, bytes, v_cand, bytes) || (lse && overlaps(lse, (size_t)Nc * p.num_heads * 4, out, bytes)))
      return REC_ATTN_ERR_INVALID_ARG;
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  if (dev != c->device) return REC_ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the candidate slots: rotated Q' and K' against the request's reference time (its
  // first history row, else its first candidate), V, time and type CAND; padding after
  std::vector<SlotReq> reqs((size_t)c->batch);
  for (int32_t b = 0; b < c->batch; ++b) {
    SlotReq& r = reqs[b];
    r.src_start = cand_offsets_host[b];
    r.dst_start = c->comb_off[b] + c->hist_len[b];
    r.ref_dst = c->hist_len[b] > 0 ? 1 : 0;
    r.ref_row = c->hist_len[b] > 0 ? c->comb_off[b] : cand_offsets_host[b];
    r.len = (int)(cand_offsets_host[b + 1] - cand_offsets_host[b]);
    r.cap = c->max_cands;
    r.pad = 0;
  }
  const SlotTable tab = slot_table(reqs);
  void* dtab = nullptr;
  e = upload_table(tab, c->device, st, &dtab);
  SlotArgs a{};
  if (e == cudaSuccess) {
    a.req = static_cast<const SlotReq*>(dtab);
    a.chunk_req = reinterpret_cast<const int*>(static_cast<char*>(dtab) + tab.off_chunk_req);
    a.chunk_row0 = reinterpret_cast<const int*>(static_cast<char*>(dtab) + tab.off_chunk_row0);
    a.t_src = reinterpret_cast<const long long*>(cand_t_dev);
    a.ty_src = nullptr;
    a.ty_const = REC_ATTN_CAND;
    a.q_src = q_cand; a.k_src = k_cand; a.v_src = v_cand;
    a.q_dst = c->q; a.k_dst = c->k; a.v_dst = c->v; a.t_dst = c->t; a.ty_dst = c->ty;
    a.o_comb = c->o; a.lse_comb = c->lse; a.o_out = out; a.lse_out = lse;
    a.heads = p.num_heads; a.head_dim = p.head_dim;
    std::memcpy(a.omega, c->omega, sizeof a.omega);
    e = launch_rope_slots(a, p.dtype, tab.n_chunks, st);
  }
  // target attention over [history, slots] on the cached rows (no rotation in the plan)
  rec_attn_plan_t* plan = nullptr;
  rec_attn_status s = REC_ATTN_OK;
  if (e == cudaSuccess) {
    s = plan_impl(&c->pp, 0, c->batch, c->comb_off.data(), c->off_dev, reinterpret_cast<const int64_t*>(c->t), c->ty,
                  st, &plan);
    if (s == REC_ATTN_OK) s = fwd_impl(plan, c->q, c->k, c->v, nullptr, c->o, lse ? c->lse : nullptr, st);
    if (s == REC_ATTN_OK) e = launch_slots_gather(a, p.dtype, tab.n_chunks, st);
    if (plan) rec_attn_free(plan);
  }
  if (dtab) {
    const cudaError_t ef = cudaFreeAsync(dtab, st);
    if (e == cudaSuccess) e = ef;
  }
  if (s != REC_ATTN_OK) return s;
  return from_cuda(e);
}

REC_ATTN_API void rec_attn_cache_free(rec_attn_kv_cache_t* c) {
  if (!c) return;
  if (c->buf) cudaFree(c->buf);  // synchronizes: the cache's rows may still be read
  delete c;
}
