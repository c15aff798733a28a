// launchers.cuh -- host entry points of the kernels (internal to the library).
#pragma once

#include <cuda.h>

#include "attn_common.cuh"

namespace recattn {

// prologue_ok (may be null) is recorded on st once the RoPE prologue, on another stream,
// may start: before the planner when it is one kernel, after its first kernel when a
// long request's tiles are split over several blocks (so the second kernel's blocks,
// launched first, are not queued behind the prologue's).
cudaError_t launch_plan(const MaskP& mp, int heads, const PlanDev& pd, const long long* offsets_dev,
                        const long long* t, const int8_t* ty, int batch, long long n_tiles,
                        cudaEvent_t prologue_ok, cudaStream_t st);
cudaError_t launch_build_masks(const MaskP& mp, const PlanDev& pd, int num_sms, cudaStream_t st);
cudaError_t launch_count_pairs(const MaskP& mp, const PlanDev& pd, const long long* t,
                               const int8_t* ty, long long n_tiles, cudaStream_t st);
// pairs: device int[n_pairs][3] (request, query tile, key tile), validated by the caller;
// bits: [n_pairs][128][4]; lcls: the pair's class in its query tile's list (0xff: not
// listed, never loaded); lslot: its mask-table slot (-1: none).
cudaError_t launch_export_masks(const MaskP& mp, const PlanDev& pd, const long long* t, const int8_t* ty,
                                const int* pairs, int n_pairs, int mode, uint32_t* bits, uint8_t* lcls, int* lslot,
                                cudaStream_t st);
cudaError_t launch_rope(const RopeArgs& a, int dtype, long long n_tiles, cudaStream_t st);
cudaError_t launch_rope_fused(const RopeArgs& a, const FusedArgs& f, int dtype, long long n_tiles,
                              cudaStream_t st);
// Serving with a cached history: regions of rows into / out of the combined layout
// (n_chunks 128-row chunks listed in a.chunk_req / a.chunk_row0).
cudaError_t launch_rope_slots(const SlotArgs& a, int dtype, long long n_chunks, cudaStream_t st);
cudaError_t launch_slots_gather(const SlotArgs& a, int dtype, long long n_chunks, cudaStream_t st);
cudaError_t launch_attn_simt(const AttnArgs& a, int head_dim, cudaStream_t st);
cudaError_t launch_bwd_delta(const BwdArgs& a, int dtype, int head_dim, cudaStream_t st);
cudaError_t launch_attn_bwd_simt(const BwdArgs& a, int head_dim, long long n_tiles, cudaStream_t st);
cudaError_t launch_bwd_schedule(const BwdSchedArgs& s, int num_sms, cudaStream_t st);
cudaError_t launch_attn_bwd_tc(const BwdArgs& a, const CUtensorMap (&maps)[4], int head_dim, int num_sms,
                               cudaStream_t st);
cudaError_t launch_compress(const CompressArgs& a, int dtype, cudaStream_t st);
cudaError_t launch_bwd_gate(const GateArgs& a, int dtype, cudaStream_t st);
cudaError_t launch_bwd_norm_gate(const NormGateArgs& a, int dtype, cudaStream_t st);
// n_fix 32-row block boundaries (per request ceil(len / 32), from CmpReq::fix_start);
// req_len: device int [B] request lengths.
cudaError_t launch_cmp_fixup(const CmpArgs& c, int batch, const int* req_len, long long n_fix, int heads,
                             int head_dim, cudaStream_t st);
cudaError_t launch_wait_timeout(int* status, unsigned long long limit_ns, cudaStream_t st);
cudaError_t launch_attn_tc(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k,
                           const CUtensorMap& v, int head_dim, int grid, cudaStream_t st);

// Host helpers shared by the entry points (api.cu): the parameter checks of
// rec_attn_params, and a 2-D TMA map over a [T][cols] bf16 tensor (box 64 columns x
// 128 rows, 128-byte swizzle).
rec_attn_status check_params(const rec_attn_params* p);
bool encode_map(CUtensorMap* m, const void* base, long long T, long long cols);
// 1 when the plan's items run over many key tiles (AttnArgs::long_items).
int long_items(const rec_attn_params& p, int batch, long long n_tiles);

}  // namespace recattn
