// noalloc.cu -- rec_attn_fwd_noalloc: plan, time-RoPE and attention in one call that
// allocates no device memory.
//
// Some callers cannot allocate device memory: a process whose inference runtime has
// reserved the GPU's memory for its own allocator and forbids other cudaMalloc
// calls, or a latency-critical serving loop that must not pay cudaMalloc's latency
// and implicit synchronisation per request.  For them this entry point keeps the
// whole per-call workspace (request table, tile statistics and classes, key-tile
// lists, schedule, rotated Q/K) in one file-scope device array of kScratchBytes,
// which every GPU that loads the library holds until the process exits.  The
// caller still provides inputs and outputs.  The kernels are the same ones
// rec_attn_plan / rec_attn_fwd launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "launchers.cuh"
#include "rec_attn.h"
#include "workspace.cuh"

#define REC_ATTN_API extern "C" __attribute__((visibility("default")))

using namespace recattn;

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB, REC_ATTN_NOALLOC_SCRATCH_BYTES
constexpr int kMaxDevices = 64;
static_assert(kScratchBytes == REC_ATTN_NOALLOC_SCRATCH_BYTES, "header and library disagree");

// The shared workspace.  In host code `g_scratch` names a host-side stand-in, not a
// device address; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

rec_attn_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return REC_ATTN_OK;
  if (e == cudaErrorMemoryAllocation) return REC_ATTN_ERR_OOM;
  return REC_ATTN_ERR_CUDA;
}

// Device address of g_scratch on the current device, looked up once per device.
rec_attn_status scratch_address(int* device, void** out) {
  cudaError_t e = cudaGetDevice(device);
  if (e != cudaSuccess) return status_of(e);
  if (*device < 0 || *device >= kMaxDevices) return REC_ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_dev[*device]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) return e != cudaSuccess ? status_of(e) : REC_ATTN_ERR_CUDA;
    g_scratch_dev[*device] = p;
  }
  *out = g_scratch_dev[*device];
  return REC_ATTN_OK;
}

}  // namespace

REC_ATTN_API rec_attn_status rec_attn_fwd_noalloc(const rec_attn_params* params, int32_t batch,
                                                  const int64_t* offsets_host, const int64_t* offsets_dev,
                                                  const int64_t* timestamps_dev, const int8_t* types_dev,
                                                  const void* q, const void* k, const void* v, void* out,
                                                  float* lse, void* stream) {
  rec_attn_status st = check_params(params);
  if (st != REC_ATTN_OK) return st;
  if (batch < 0 || (batch > 0 && !offsets_host)) return REC_ATTN_ERR_INVALID_ARG;
  // sizes of the workspace pieces (host-only pass over the offsets)
  long long NT = 0, NC = 0, T = 0;
  if (batch > 0) {
    if (offsets_host[0] != 0) return REC_ATTN_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b) {
      const long long len = offsets_host[b + 1] - offsets_host[b];
      if (len < 0) return REC_ATTN_ERR_INVALID_ARG;
      if (len > REC_ATTN_MAX_REQUEST_LEN) return REC_ATTN_ERR_UNSUPPORTED;
      const long long nt = (len + kTile - 1) / kTile;
      NT += nt;
      NC += nt * nt;
    }
    T = offsets_host[batch];
    if (T >= (1LL << 31) || NT * params->num_heads >= (1LL << 31)) return REC_ATTN_ERR_UNSUPPORTED;
  }
  const size_t elem = params->dtype == REC_ATTN_BF16 ? 2 : 4;
  const size_t tensor_bytes = (size_t)T * params->num_heads * params->head_dim * elem;
  // workspace layout inside the static array
  // no mask table here: the kernels build every PARTIAL tile's bits themselves
  const WsLayout lay = ws_layout(batch, NT, NC, params->num_heads, params->use_rope ? tensor_bytes : 0, 0);
  if (lay.total > kScratchBytes) return REC_ATTN_ERR_UNSUPPORTED;  // batch too large for the static workspace
  if (T > 0) {
    if (!offsets_dev || !timestamps_dev || !types_dev || !q || !k || !v || !out) return REC_ATTN_ERR_INVALID_ARG;
    const void* ptrs[4] = {q, k, v, out};
    for (const void* x : ptrs)
      if (reinterpret_cast<uintptr_t>(x) & 15u) return REC_ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return REC_ATTN_ERR_INVALID_ARG;
    const char* o = static_cast<const char*>(out);
    const void* ins[3] = {q, k, v};
    for (const void* x : ins) {
      const char* y = static_cast<const char*>(x);
      if (o < y + tensor_bytes && y < o + tensor_bytes) return REC_ATTN_ERR_INVALID_ARG;
    }
  }
  if (batch == 0 || T == 0) return REC_ATTN_OK;

  int device = 0;
  void* base = nullptr;
  st = scratch_address(&device, &base);
  if (st != REC_ATTN_OK) return st;
  int num_sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return status_of(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(base);
  const PlanDev pd = ws_bind(w, lay);

  // the previous call's counters and status stay in the array: clear them
  e = cudaMemsetAsync(w + lay.hdr, 0, 256, s);
  // request table, uploaded from a stack buffer in chunks (pageable copies are staged
  // before cudaMemcpyAsync returns, so the buffer can be refilled at once)
  ReqMeta chunk[128];
  long long tile = 0, cls = 0;
  for (int32_t b0 = 0; b0 < batch && e == cudaSuccess; b0 += 128) {
    const int n = batch - b0 < 128 ? batch - b0 : 128;
    for (int i = 0; i < n; ++i) {
      const int32_t b = b0 + i;
      ReqMeta& m = chunk[i];
      m.tok_start = offsets_host[b];
      m.len = (int)(offsets_host[b + 1] - offsets_host[b]);
      m.ntiles = (m.len + kTile - 1) / kTile;
      m.tile_start = tile;
      m.cls_start = cls;
      tile += m.ntiles;
      cls += (long long)m.ntiles * m.ntiles;
    }
    e = cudaMemcpyAsync(pd.meta + b0, chunk, sizeof(ReqMeta) * n, cudaMemcpyHostToDevice, s);
  }
  // the request of every tile, uploaded the same way
  {
    int tchunk[2048];
    int nfill = 0;
    long long tdone = 0;
    for (int32_t b = 0; b < batch && e == cudaSuccess; ++b) {
      const long long nt = (offsets_host[b + 1] - offsets_host[b] + kTile - 1) / kTile;
      for (long long i = 0; i < nt && e == cudaSuccess; ++i) {
        tchunk[nfill++] = b;
        if (nfill == 2048) {
          e = cudaMemcpyAsync(pd.treq + tdone, tchunk, sizeof(int) * nfill, cudaMemcpyHostToDevice, s);
          tdone += nfill;
          nfill = 0;
        }
      }
    }
    if (e == cudaSuccess && nfill > 0)
      e = cudaMemcpyAsync(pd.treq + tdone, tchunk, sizeof(int) * nfill, cudaMemcpyHostToDevice, s);
  }
  MaskP mask{};
  mask.use_delay = params->use_delay;
  mask.delay = params->use_delay ? params->delay_s : 0;
  mask.window = params->window;
  mask.bidir = params->hist_bidirectional;
  mask.keep_user = -1;  // every query
  const long long* t = reinterpret_cast<const long long*>(timestamps_dev);
  if (e == cudaSuccess)
    e = launch_plan(mask, params->num_heads, pd, reinterpret_cast<const long long*>(offsets_dev), t, types_dev, batch, NT, nullptr, s);
  if (e != cudaSuccess) return status_of(e);

  const void* qs = q;
  const void* ks = k;
  if (params->use_rope) {
    RopeArgs ra;
    ra.meta = pd.meta; ra.tile_req = pd.treq; ra.batch = batch; ra.t = t;
    ra.ty = types_dev; ra.skip_user_q = 0;
    ra.q = q; ra.k = k; ra.qr = w + lay.rq; ra.kr = w + lay.rk;
    ra.heads = params->num_heads; ra.head_dim = params->head_dim;
    for (int i = 0; i < kMaxPairs; ++i)
      ra.omega[i] = i < params->head_dim / 2
                        ? (float)(params->phi_min / params->dt_max_s *
                                  std::pow(params->rope_base, 2.0 * i / (double)params->head_dim))
                        : 0.f;
    e = launch_rope(ra, params->dtype, NT, s);
    if (e != cudaSuccess) return status_of(e);
    qs = w + lay.rq;
    ks = w + lay.rk;
  }
  AttnArgs a{};
  a.meta = pd.meta; a.qreq = pd.qreq; a.kcount = pd.kcount; a.klist = pd.klist; a.items = pd.items;
  a.counters = pd.counters; a.krec = pd.krec; a.qkeep = pd.qkeep;
  a.kslot = pd.kslot; a.mtab = pd.mtab;
  a.t = t; a.ty = types_dev; a.q = qs; a.k = ks; a.v = v; a.out = out; a.lse = lse; a.status = pd.status;
  a.out_gate = nullptr;
  a.n_items = NT * params->num_heads; a.heads = params->num_heads;
  a.scale = params->softmax_scale > 0.f ? params->softmax_scale : 1.f / std::sqrt((float)params->head_dim);
  a.mask = mask;
  a.long_items = long_items(*params, batch, NT);
  if (params->dtype == REC_ATTN_FP32) return status_of(launch_attn_simt(a, params->head_dim, s));
  CUtensorMap maps[3];
  const long long cols = (long long)params->num_heads * params->head_dim;
  if (!encode_map(&maps[0], qs, T, cols) || !encode_map(&maps[1], ks, T, cols) ||
      !encode_map(&maps[2], v, T, cols))
    return REC_ATTN_ERR_CUDA;
  const int grid = (int)(a.n_items < num_sms ? a.n_items : num_sms);
  return status_of(launch_attn_tc(a, maps[0], maps[1], maps[2], params->head_dim, grid, s));
}
