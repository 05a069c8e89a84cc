// Attention weights, memory-saving variant of "Moebius: Serving
// Mixture-of-Expert Models with Seamless Runtime Parallelism Switch" (paper
// review), §3.1: only the active layout is kept.  EP (DP attention): every
// rank holds the full Wqkv ([Hq query heads][Hkv key heads][Hkv value heads],
// each head Dh rows of H) and Wo [H][Hq*Dh].  TP: rank q holds its query
// heads [q*Hq/P, (q+1)*Hq/P), its KV heads (K then V; replicated over rank
// groups when Hkv < P), and the Wo columns of its query heads.
//
// EP->TP keeps each rank's own shard of its own full copy (no data crosses
// ranks).  TP->EP is the all-gather: every shard element is read once and
// stored into all P full copies (key/value heads from their lowest replica).
// N+1 slots per layer as for the expert weights; layers ascending (EP->TP) or
// descending (TP->EP), one launch per layer, chained (griddep_wait).
#include "umm_internal.cuh"

namespace uk {

struct AParams {
  uint8_t* base;
  uint64_t region_stride, ep_slot, tp_slot;   // slot offsets inside a region
  uint64_t wo_off;                            // Wo offset inside a slot (both views)
  uint64_t head_bytes;                        // Dh * H * 2
  uint64_t full_row_bytes, shard_row_bytes;   // Wo rows: Hq*Dh*2, hq*Dh*2
  uint32_t P, Hq, Hkv, hq, h_tp;
  uint32_t qkv_vec, vr;                       // shard Wqkv vectors, all shard vectors (per rank)
  uint32_t tiles_total;
  FastDiv headv, rowv, tiles_per_rank;
  Span span;                                  // the P regions
};

// the full-layout head held at local head slot b of TP rank q (-1: a key or
// value head that a lower rank also holds, when gathering)
__device__ __forceinline__ int full_head(const AParams& p, uint32_t q, uint32_t b, bool lowest_only) {
  if (b < p.hq) return (int)(q * p.hq + b);
  const uint32_t kvb = b - p.hq, which = kvb / p.h_tp, kv = kvb - which * p.h_tp;
  uint32_t h;
  if (p.Hkv >= p.P) {
    h = q * p.h_tp + kv;
  } else {
    h = q * p.Hkv / p.P;
    if (lowest_only && (h * p.P + p.Hkv - 1) / p.Hkv != q) return -1;   // not the first rank of its group
  }
  return (int)(p.Hq + which * p.Hkv + h);
}

template <int VB, int U, int T>
__global__ void __launch_bounds__(T) attn_kernel(const AParams p, int ep2tp) {
  using V = typename VecT<VB>::T;
  griddep_launch_dependents();
  for (uint32_t tile = blockIdx.x; tile < p.tiles_total; tile += gridDim.x) {
    uint32_t q, lt;
    p.tiles_per_rank.divmod(tile, q, lt);
    uint8_t* const shard = p.base + (uint64_t)q * p.region_stride + p.tp_slot;
    V val[U];
    uint64_t full_off[U];      // offset inside a full (EP) slot
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t v = lt * (uint32_t)(T * U) + threadIdx.x + (uint32_t)(u * T);
      ok[u] = v < p.vr;
      uint64_t shard_off = 0;
      if (ok[u]) {
        if (v < p.qkv_vec) {
          uint32_t b, iv;
          p.headv.divmod(v, b, iv);
          const int hh = full_head(p, q, b, !ep2tp);
          ok[u] = hh >= 0;
          shard_off = (uint64_t)b * p.head_bytes + (uint64_t)iv * VB;
          full_off[u] = (uint64_t)hh * p.head_bytes + (uint64_t)iv * VB;
        } else {
          uint32_t row, cv;
          p.rowv.divmod(v - p.qkv_vec, row, cv);
          shard_off = p.wo_off + (uint64_t)row * p.shard_row_bytes + (uint64_t)cv * VB;
          full_off[u] = p.wo_off + (uint64_t)row * p.full_row_bytes + (uint64_t)q * p.shard_row_bytes +
                        (uint64_t)cv * VB;
        }
      }
      if (ok[u]) {
        const uint8_t* src = ep2tp ? p.base + (uint64_t)q * p.region_stride + p.ep_slot + full_off[u]
                                   : shard + shard_off;
        ok[u] = access_ok<VB>(p.span, src);
        if (ok[u]) val[u] = ld_vec(reinterpret_cast<const V*>(src));
        if (ep2tp) full_off[u] = shard_off;   // from here on: where to store
      }
    }
    griddep_wait();
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!ok[u]) continue;
      if (ep2tp) {
        if (access_ok<VB>(p.span, shard + full_off[u])) st_vec(reinterpret_cast<V*>(shard + full_off[u]), val[u]);
      } else {
        for (uint32_t r = 0; r < p.P; ++r) {
          uint8_t* const dst = p.base + (uint64_t)r * p.region_stride + p.ep_slot + full_off[u];
          if (access_ok<VB>(p.span, dst)) st_vec(reinterpret_cast<V*>(dst), val[u]);
        }
      }
    }
  }
  griddep_wait();
}

cudaError_t launch_attn(const Geo& g, int ep2tp, int layer, cudaStream_t s, bool chained) {
  constexpr int T = 256, U = 4;   // 16 KiB tiles with 16-byte vectors
  const uint64_t Dh = (uint64_t)g.D, H = (uint64_t)g.H;
  const uint32_t hq = (uint32_t)(g.Hq / g.P), h_tp = (uint32_t)g.h_tp;
  const uint64_t head_bytes = Dh * H * 2, shard_row = (uint64_t)hq * Dh * 2;
  int VB = 2;
  for (int cand : {32, 16, 8, 4}) {
    if (head_bytes % cand == 0 && shard_row % cand == 0) {
      VB = cand;
      break;
    }
  }
  AParams p;
  p.base = g.base;
  p.region_stride = g.region_stride;
  p.ep_slot = g.attnslots_off + (uint64_t)(layer + 1) * g.attnslot_stride;
  p.tp_slot = g.attnslots_off + (uint64_t)layer * g.attnslot_stride;
  p.wo_off = g.attn_wo_off;
  p.head_bytes = head_bytes;
  p.full_row_bytes = (uint64_t)g.Hq * Dh * 2;
  p.shard_row_bytes = shard_row;
  p.P = (uint32_t)g.P;
  p.Hq = (uint32_t)g.Hq;
  p.Hkv = (uint32_t)g.Hkv;
  p.hq = hq;
  p.h_tp = h_tp;
  p.qkv_vec = (uint32_t)((uint64_t)(hq + 2 * h_tp) * head_bytes / VB);
  p.vr = p.qkv_vec + (uint32_t)(H * shard_row / VB);
  const uint32_t tile = (uint32_t)(T * (VB == 32 ? U / 2 : U));
  const uint32_t tpr = (p.vr + tile - 1) / tile;
  p.tiles_total = tpr * p.P;
  p.headv = FastDiv((uint32_t)(head_bytes / VB));
  p.rowv = FastDiv((uint32_t)(shard_row / VB));
  p.tiles_per_rank = FastDiv(tpr);
  p.span = g.regions();
  if (p.tiles_total == 0) return cudaSuccess;
  const unsigned grid = p.tiles_total;
  switch (VB) {
    case 32: return launch_chain(attn_kernel<32, U / 2, T>, grid, T, s, chained, p, ep2tp);
    case 16: return launch_chain(attn_kernel<16, U, T>, grid, T, s, chained, p, ep2tp);
    case 8: return launch_chain(attn_kernel<8, U, T>, grid, T, s, chained, p, ep2tp);
    case 4: return launch_chain(attn_kernel<4, U, T>, grid, T, s, chained, p, ep2tp);
    default: return launch_chain(attn_kernel<2, U, T>, grid, T, s, chained, p, ep2tp);
  }
}

}  // namespace uk
