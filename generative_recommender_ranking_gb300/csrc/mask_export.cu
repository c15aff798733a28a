// mask_export.cu -- copies out the visibility bits the attention kernels apply to named
// (query tile, key tile) pairs, so they can be compared bit for bit with the mask
// predicate (CADET delay rule, SORT U2U/C2U/C2C and local attention, LazFormer
// Eq. 19-21, MTGR hybrid mask).  Each mode walks the same data the kernels walk: the
// query tile's key-tile list (a pair that is not in it is never loaded), its class,
// its mask-table slot, the tiles' planner records, and the same row builder.
#include <climits>

#include "launchers.cuh"
#include "row_mask.cuh"

namespace recattn {

namespace {

// One block per requested pair, one thread per query row of the tile.
__global__ void __launch_bounds__(kTile) k_export_masks(MaskP mp, PlanDev pd, const long long* t, const int8_t* ty,
                                                        const int* pairs, int mode, uint4* bits, uint8_t* lcls,
                                                        int* lslot) {
  const int p = blockIdx.x, r = threadIdx.x;
  const int b = pairs[3 * p], qt = pairs[3 * p + 1], kt = pairs[3 * p + 2];
  const ReqMeta m = pd.meta[b];
  const long long g = m.tile_start + qt;
  // the pair as the kernels see it: an entry of the query tile's list, or nothing
  const int n = pd.kcount[g];
  const uint32_t* list = pd.klist + m.cls_start + (long long)qt * m.ntiles;
  int j = -1;
  for (int e = 0; e < n; ++e)
    if ((int)(list[e] & 0xffffffu) == kt) { j = e; break; }
  const int cl = j < 0 ? -1 : (int)(list[j] >> 24);
  const int slot = j < 0 ? -1 : pd.kslot[m.cls_start + (long long)qt * m.ntiles + j];
  if (r == 0) {
    lcls[p] = (uint8_t)(j < 0 ? 0xff : cl);
    lslot[p] = slot;
  }
  uint32_t vm[4] = {0u, 0u, 0u, 0u};
  const int pi = qt * kTile + r;
  const bool row_ok = pi < m.len;
  if (cl == REC_ATTN_TILE_FULL) {
    vm[0] = vm[1] = vm[2] = vm[3] = ~0u;  // no mask: every key of the (complete) tile
  } else if (cl >= 0 && mode == 2) {
    // the CUDA-core path: the predicate per pair on the tokens' own times and types
    long long ti = 0;
    int tyi = -1;
    if (row_ok) { ti = t[m.tok_start + pi]; tyi = ty[m.tok_start + pi]; }
    bool thr_ok; long long thr;
    delay_bound(ti, mp.delay, thr_ok, thr);
    if (row_ok)
      for (int c = 0; c < kTile; ++c) {
        const int pj = kt * kTile + c;
        const bool ok = pj < m.len;
        const long long tj = ok ? t[m.tok_start + pj] : 0;
        const int tyj = ok ? (int)ty[m.tok_start + pj] : -1;
        if (vis_pred(mp, pi, ti, tyi, thr_ok, thr, pj, tj, tyj)) vm[c >> 5] |= 1u << (c & 31);
      }
  } else if (cl >= 0) {
    if (mode == 0 && slot >= 0) {
      const uint4 w = reinterpret_cast<const uint4*>(pd.mtab)[(long long)slot * kTile + r];
      vm[0] = w.x; vm[1] = w.y; vm[2] = w.z; vm[3] = w.w;
    } else {
      // the row's time and type from the query tile's record, as the softmax reads them
      const KeyTileRec* qr = pd.krec + g;
      const long long ti = qr->t[r];
      int tyi = -1;
#pragma unroll
      for (int c = 0; c < kTypes; ++c)
        if ((qr->typebits[c][r >> 5] >> (r & 31)) & 1u) tyi = c;
      RowMask rm;
      row_mask_setup(mp, row_ok, pi, ti, tyi, rm);
      build_mask(rm, pd.krec + m.tile_start + kt, kt * kTile, vm);
    }
  }
  bits[(long long)p * kTile + r] = make_uint4(vm[0], vm[1], vm[2], vm[3]);
}

}  // namespace

cudaError_t launch_export_masks(const MaskP& mp, const PlanDev& pd, const long long* t, const int8_t* ty,
                                const int* pairs, int n_pairs, int mode, uint32_t* bits, uint8_t* lcls, int* lslot,
                                cudaStream_t st) {
  if (n_pairs <= 0) return cudaSuccess;
  k_export_masks<<<n_pairs, kTile, 0, st>>>(mp, pd, t, ty, pairs, mode, reinterpret_cast<uint4*>(bits), lcls, lslot);
  return cudaGetLastError();
}

}  // namespace recattn
