// workspace.cuh -- layout of a plan's device workspace (shared by the plan-based
// entry points and the no-allocation entry point).
#pragma once

#include <cstddef>

#include "rec_attn_internal.cuh"

namespace recattn {

struct WsLayout {
  size_t hdr, meta, box, rec, cls, kl, kc, qc, qr, it, rc, ro, rf, qk, tr, ks, ps, mi, mt, rq, rk, total;
  int mcap;
};

// Slots of the mask table: enough for a few PARTIAL tile pairs per tile (causal and
// windowed masks have one to five), never more than there are pairs.
inline int mask_capacity(long long NT, long long NC) {
  const long long c = 8 * NT + 1024;
  return (int)(c < NC ? c : NC);
}

inline size_t ws_up(size_t x) { return (x + 255) & ~size_t(255); }

// rot_bytes: bytes of one rotated [T][H][d] copy (0 when the RoPE is off); mcap: slots
// of the mask table (0: none).
inline WsLayout ws_layout(long long batch, long long NT, long long NC, long long heads, size_t rot_bytes,
                          int mcap) {
  WsLayout L;
  L.mcap = mcap;
  size_t off = 0;
  L.hdr = off; off = ws_up(off + 256);
  L.meta = off; off = ws_up(off + sizeof(ReqMeta) * (size_t)batch);
  L.tr = off; off = ws_up(off + 4 * (size_t)NT);  // right after the table: both go up in one copy
  L.box = off; off = ws_up(off + sizeof(TileBox) * kTypes * (size_t)NT);
  L.rec = off; off = ws_up(off + sizeof(KeyTileRec) * (size_t)NT);
  L.cls = off; off = ws_up(off + (size_t)NC);
  L.kl = off; off = ws_up(off + 4 * (size_t)NC);
  L.kc = off; off = ws_up(off + 4 * (size_t)NT);
  L.qc = off; off = ws_up(off + 4 * (size_t)NT);
  L.qr = off; off = ws_up(off + 4 * (size_t)NT);
  L.it = off; off = ws_up(off + 4 * (size_t)NT * (size_t)heads);
  L.rc = off; off = ws_up(off + 4 * (size_t)batch);
  L.ro = off; off = ws_up(off + 4 * (size_t)batch);
  L.rf = off; off = ws_up(off + 4 * ((size_t)batch + 1));
  L.qk = off; off = ws_up(off + 4 * (size_t)batch);
  L.ks = off; off = ws_up(off + 4 * (size_t)NC);
  L.ps = off; off = ws_up(off + 4 * (size_t)NC);
  L.mi = off; off = ws_up(off + 8 * (size_t)mcap);
  L.mt = off; off = ws_up(off + 16 * (size_t)kTile * (size_t)mcap);
  L.rq = off; off = ws_up(off + rot_bytes);
  L.rk = off; off = ws_up(off + rot_bytes);
  L.total = off;
  return L;
}

inline PlanDev ws_bind(char* w, const WsLayout& L) {
  PlanDev pd{};
  pd.counters = reinterpret_cast<int*>(w + L.hdr);
  pd.status = pd.counters + 8;
  pd.pairs = reinterpret_cast<unsigned long long*>(w + L.hdr + 64);
  pd.meta = reinterpret_cast<ReqMeta*>(w + L.meta);
  pd.boxes = reinterpret_cast<TileBox*>(w + L.box);
  pd.krec = reinterpret_cast<KeyTileRec*>(w + L.rec);
  pd.cls = reinterpret_cast<uint8_t*>(w + L.cls);
  pd.klist = reinterpret_cast<uint32_t*>(w + L.kl);
  pd.kcount = reinterpret_cast<int*>(w + L.kc);
  pd.qcost = reinterpret_cast<int*>(w + L.qc);
  pd.qreq = reinterpret_cast<int*>(w + L.qr);
  pd.items = reinterpret_cast<int*>(w + L.it);
  pd.rcost = reinterpret_cast<int*>(w + L.rc);
  pd.rorder = reinterpret_cast<int*>(w + L.ro);
  pd.roff = reinterpret_cast<int*>(w + L.rf);
  pd.qkeep = reinterpret_cast<int*>(w + L.qk);
  pd.treq = reinterpret_cast<int*>(w + L.tr);
  pd.kslot = reinterpret_cast<int*>(w + L.ks);
  pd.pslot = reinterpret_cast<int*>(w + L.ps);
  pd.minfo = reinterpret_cast<int2*>(w + L.mi);
  pd.mtab = reinterpret_cast<uint32_t*>(w + L.mt);
  pd.mcap = L.mcap;
  return pd;
}

}  // namespace recattn
