// Expert-weight reshard EP <-> TP, one layer per launch.
//
// "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
// Switch" (paper review): §3.1 (layouts and the permute -> exchange -> scatter
// pipeline), §4.2 Fig. 7 (N+1 slots, in-place layer order), §4.3 Table 1 and
// Fig. 8a (fused direct transfer: one read + one write per element, no staging).
//
// On one GPU the P ranks are P regions of one buffer, so the three stages
// collapse into a single pass: every thread reads 16-byte vectors of the EP
// view and writes them straight to their TP place (EP->TP) or the other way
// round (TP->EP).  Work is walked in EP order, where both W13 and W2 of a
// region are contiguous: the EP side is streamed linearly, the TP side is P
// sequential streams (W13: whole rows of H elements; W2: runs of I/P
// elements), so every DRAM sector moved is fully used.
#include "umm_internal.cuh"

namespace uk {

// TP-side addressing.  The fused path writes (reads) the TP slot of region q
// itself: tp_base = buffer, q_stride = region stride, r_stride = 0,
// expert offset r*El.  The staged path packs into per-peer blocks instead:
// tp_base = staging, block (r, q) at (r*P + q)*block bytes, experts from 0.
struct WParams {
  uint8_t* base;
  uint64_t region_stride, w13_off, w2_off;
  uint64_t ep_slot_off;               // EP slot offset inside a region
  uint8_t* tp_base;
  uint64_t tp_q_stride, tp_r_stride, tp_w13_off, tp_w2_off;
  uint32_t tp_eoff_per_r;             // El (fused) or 0 (staged)
  uint64_t w13_row_bytes;             // H * 2
  uint64_t w2_tp_row_bytes;           // Ip * 2
  uint32_t El, Ip, H;
  uint32_t v13, vr;                   // W13 vectors per region, W13+W2 vectors per region
  uint32_t tiles_total;
  FastDiv hv, two_i, i_d, ip_d, two_ip, iv, ipv, tiles_per_region;
  int split;
  Span ep_span, tp_span;              // where EP-side and TP-side addresses must lie
};

template <int VB, int U, int T>
__global__ void __launch_bounds__(T) weights_kernel(const WParams p, int ep2tp) {
  using V = typename VecT<VB>::T;
  griddep_launch_dependents();
  for (uint32_t tile = blockIdx.x; tile < p.tiles_total; tile += gridDim.x) {
    uint32_t r, lt;
    p.tiles_per_region.divmod(tile, r, lt);
    uint8_t* const region_r = p.base + (uint64_t)r * p.region_stride;
    const uint32_t v0 = lt * (uint32_t)(T * U) + threadIdx.x;

    V val[U];
    uint8_t* tp_addr[U];
    uint8_t* ep_addr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t v = v0 + (uint32_t)(u * T);
      ep_addr[u] = nullptr;
      if (v < p.vr) {
        ep_addr[u] = region_r + p.ep_slot_off +
                     (v < p.v13 ? p.w13_off + (uint64_t)v * VB : p.w2_off + (uint64_t)(v - p.v13) * VB);
      }
    }
    // The TP address of each vector.  EP W13 row (e_l, j) of region r holds
    // expert e = r*El + e_l; with j = g*I + i (g: gate/up), it is TP rank
    // i / Ip's row g*Ip + i % Ip (split 0) or rank j / 2Ip's row j % 2Ip
    // (split 1).  EP W2 row (e_l, h), column i belongs to TP rank i / Ip,
    // row r*El*H + e_l*H + h, column i % Ip.
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t v = v0 + (uint32_t)(u * T);
      tp_addr[u] = nullptr;
      if (v >= p.vr) continue;
      if (v < p.v13) {
        uint32_t row_all, hv, el, j, q, trow;
        p.hv.divmod(v, row_all, hv);
        p.two_i.divmod(row_all, el, j);
        if (p.split == 0) {
          uint32_t g, i, ii;
          p.i_d.divmod(j, g, i);
          p.ip_d.divmod(i, q, ii);
          trow = g * p.Ip + ii;
        } else {
          p.two_ip.divmod(j, q, trow);
        }
        const uint64_t e = (uint64_t)r * p.tp_eoff_per_r + el;
        tp_addr[u] = p.tp_base + (uint64_t)q * p.tp_q_stride + (uint64_t)r * p.tp_r_stride + p.tp_w13_off +
                     (e * 2 * p.Ip + trow) * p.w13_row_bytes + (uint64_t)hv * VB;
      } else {
        uint32_t row_all, iv, q, cc;
        p.iv.divmod(v - p.v13, row_all, iv);
        p.ipv.divmod(iv, q, cc);
        const uint64_t trow = (uint64_t)r * p.tp_eoff_per_r * p.H + row_all;
        tp_addr[u] = p.tp_base + (uint64_t)q * p.tp_q_stride + (uint64_t)r * p.tp_r_stride + p.tp_w2_off +
                     trow * p.w2_tp_row_bytes + (uint64_t)cc * VB;
      }
    }
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      ok[u] = ep_addr[u] && access_ok<VB>(p.ep_span, ep_addr[u]) && access_ok<VB>(p.tp_span, tp_addr[u]);
    if (ep2tp) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) val[u] = ld_vec(reinterpret_cast<const V*>(ep_addr[u]));
      griddep_wait();
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) st_vec(reinterpret_cast<V*>(tp_addr[u]), val[u]);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) val[u] = ld_vec(reinterpret_cast<const V*>(tp_addr[u]));
      griddep_wait();
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) st_vec(reinterpret_cast<V*>(ep_addr[u]), val[u]);
    }
  }
  griddep_wait();
}

namespace {
constexpr int kT = 256;
constexpr int kU = 4;

// One CTA per 16 KiB tile (grid = all tiles of the layer) rather than a
// persistent grid: the block scheduler refills each SM slot the moment a tile
// is done, keeping more loads in flight (measured on GB300, E=128, H=2048,
// I=768: 6.35 TB/s persistent with 8 vectors per thread -> 6.95 TB/s).
template <int VB>
cudaError_t run(const WParams& p, int ep2tp, cudaStream_t s, bool chained) {
  if (p.tiles_total == 0) return cudaSuccess;
  return launch_chain(weights_kernel<VB, kU, kT>, p.tiles_total, kT, s, chained, p, ep2tp);
}
}  // namespace

namespace {

// 16-byte vectors at most: 32-byte ones measured ~1% slower here on GB300
// (E=128, H=2048, I=768: 0.343 -> 0.347 ms per layer; H=4096, I=1536:
// 1.347 -> 1.360 ms), while they pay off in the KV and attention copies.
int vec_bytes(uint32_t H, uint32_t Ip) {
  if (H % 8 == 0 && Ip % 8 == 0) return 16;
  if (H % 4 == 0 && Ip % 4 == 0) return 8;
  if (H % 2 == 0 && Ip % 2 == 0) return 4;
  return 2;
}

// Parameters of one layer's permute: EP slot `layer`+1 <-> the TP side.
WParams layer_params(const Geo& g, int layer, int VB) {
  const uint32_t El = (uint32_t)(g.E / g.P), Ip = (uint32_t)(g.I / g.P), H = (uint32_t)g.H;
  const uint32_t I = (uint32_t)g.I;
  const uint32_t per = (uint32_t)VB / 2;  // elements per vector
  WParams p;
  p.base = g.base;
  p.region_stride = g.region_stride;
  p.w13_off = g.w13_off;
  p.w2_off = g.w2_off;
  p.ep_slot_off = (uint64_t)(layer + 1) * g.wslot_stride;
  p.tp_base = g.base;
  p.tp_q_stride = g.region_stride;
  p.tp_r_stride = 0;
  p.tp_w13_off = (uint64_t)layer * g.wslot_stride + g.w13_off;
  p.tp_w2_off = (uint64_t)layer * g.wslot_stride + g.w2_off;
  p.tp_eoff_per_r = El;
  p.w13_row_bytes = (uint64_t)H * 2;
  p.w2_tp_row_bytes = (uint64_t)Ip * 2;
  p.El = El;
  p.Ip = Ip;
  p.H = H;
  p.v13 = (uint32_t)((uint64_t)El * 2 * I * H / per);
  p.vr = p.v13 + (uint32_t)((uint64_t)El * H * I / per);
  const uint32_t tile = (uint32_t)(kT * kU);
  const uint32_t tpr = (p.vr + tile - 1) / tile;
  p.tiles_total = tpr * (uint32_t)g.P;
  p.hv = FastDiv(H / per);
  p.two_i = FastDiv(2 * I);
  p.i_d = FastDiv(I);
  p.ip_d = FastDiv(Ip);
  p.two_ip = FastDiv(2 * Ip);
  p.iv = FastDiv(I / per);
  p.ipv = FastDiv(Ip / per);
  p.tiles_per_region = FastDiv(tpr);
  p.split = g.w13_split;
  p.ep_span = g.regions();
  p.tp_span = g.regions();
  return p;
}

cudaError_t run_any(const WParams& p, int VB, int ep2tp, cudaStream_t s, bool chained) {
  switch (VB) {
    case 16: return run<16>(p, ep2tp, s, chained);
    case 8: return run<8>(p, ep2tp, s, chained);
    case 4: return run<4>(p, ep2tp, s, chained);
    default: return run<2>(p, ep2tp, s, chained);
  }
}

// Exchange stage of the staged path: block (r, q) of the staging buffer
// holds, in TP layout, the W13 rows then the W2 rows that EP rank r's experts
// contribute to TP rank q.  They are contiguous in TP rank q's slot too (its
// experts r*El .. r*El+El-1), so the exchange is 2*P*P contiguous copies.
struct XParams {
  uint8_t* base;
  const uint8_t* stage;
  uint64_t region_stride, tp_w13_off, tp_w2_off;
  uint64_t seg13, seg2, block;        // bytes: W13 part, W2 part, whole block
  uint32_t P, tiles13, tiles2;        // 16 KiB tiles per part
  uint32_t tiles_total;
  FastDiv tiles_pair;                 // tiles13 + tiles2
  FastDiv pd;                         // P
  Span stage_span, region_span;
};

template <int VB, int U, int T>
__global__ void __launch_bounds__(T) exchange_kernel(const XParams p, int to_tp) {
  using V = typename VecT<VB>::T;
  for (uint32_t tile = blockIdx.x; tile < p.tiles_total; tile += gridDim.x) {
    uint32_t pair, lt, r, q;
    p.tiles_pair.divmod(tile, pair, lt);
    p.pd.divmod(pair, r, q);
    const bool w13 = lt < p.tiles13;
    const uint64_t seg = w13 ? p.seg13 : p.seg2;
    const uint64_t off0 = (uint64_t)(w13 ? lt : lt - p.tiles13) * (uint64_t)(T * U * VB);
    const uint8_t* st = p.stage + (uint64_t)pair * p.block + (w13 ? 0 : p.seg13);
    uint8_t* tp = p.base + (uint64_t)q * p.region_stride +
                  (w13 ? p.tp_w13_off + (uint64_t)r * p.seg13 : p.tp_w2_off + (uint64_t)r * p.seg2);
    V val[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t o = off0 + (uint64_t)(u * T + threadIdx.x) * VB;
      ok[u] = o < seg && access_ok<VB>(p.stage_span, st + o) && access_ok<VB>(p.region_span, tp + o);
      if (ok[u]) val[u] = ld_vec(reinterpret_cast<const V*>((to_tp ? st : tp) + o));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t o = off0 + (uint64_t)(u * T + threadIdx.x) * VB;
      if (ok[u]) st_vec(reinterpret_cast<V*>(const_cast<uint8_t*>(to_tp ? tp : st) + o), val[u]);
    }
  }
}

cudaError_t run_exchange(const Geo& g, int layer, int VB, const uint8_t* stage, int to_tp, cudaStream_t s) {
  const uint64_t El = (uint64_t)(g.E / g.P), Ip = (uint64_t)(g.I / g.P), H = (uint64_t)g.H;
  XParams x;
  x.base = g.base;
  x.stage = stage;
  x.region_stride = g.region_stride;
  x.tp_w13_off = (uint64_t)layer * g.wslot_stride + g.w13_off;
  x.tp_w2_off = (uint64_t)layer * g.wslot_stride + g.w2_off;
  x.seg13 = El * 2 * Ip * H * 2;
  x.seg2 = El * H * Ip * 2;
  x.block = x.seg13 + x.seg2;
  x.P = (uint32_t)g.P;
  const uint64_t tb = (uint64_t)kT * kU * VB;
  x.tiles13 = (uint32_t)((x.seg13 + tb - 1) / tb);
  x.tiles2 = (uint32_t)((x.seg2 + tb - 1) / tb);
  x.tiles_total = (x.tiles13 + x.tiles2) * x.P * x.P;
  x.tiles_pair = FastDiv(x.tiles13 + x.tiles2);
  x.pd = FastDiv(x.P);
  x.stage_span = Span{stage, stage + weights_stage_bytes(g), g.flags};
  x.region_span = g.regions();
  if (x.tiles_total == 0) return cudaSuccess;
  switch (VB) {
    case 16: exchange_kernel<16, kU, kT><<<x.tiles_total, kT, 0, s>>>(x, to_tp); break;
    case 8: exchange_kernel<8, kU, kT><<<x.tiles_total, kT, 0, s>>>(x, to_tp); break;
    case 4: exchange_kernel<4, kU, kT><<<x.tiles_total, kT, 0, s>>>(x, to_tp); break;
    default: exchange_kernel<2, kU, kT><<<x.tiles_total, kT, 0, s>>>(x, to_tp); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_weights(const Geo& g, int ep2tp, int layer, cudaStream_t s, bool chained) {
  const int VB = vec_bytes((uint32_t)g.H, (uint32_t)(g.I / g.P));
  return run_any(layer_params(g, layer, VB), VB, ep2tp, s, chained);
}

uint64_t weights_stage_bytes(const Geo& g) {
  const uint64_t El = (uint64_t)(g.E / g.P), Ip = (uint64_t)(g.I / g.P), H = (uint64_t)g.H;
  return (uint64_t)g.P * (uint64_t)g.P * (El * 2 * Ip * H * 2 + El * H * Ip * 2);
}

cudaError_t launch_weights_staged(const Geo& g, int ep2tp, int layer, uint8_t* stage, cudaStream_t s,
                                  int* launches) {
  const int VB = vec_bytes((uint32_t)g.H, (uint32_t)(g.I / g.P));
  WParams p = layer_params(g, layer, VB);
  const uint64_t El = (uint64_t)(g.E / g.P), Ip = (uint64_t)(g.I / g.P), H = (uint64_t)g.H;
  const uint64_t block = El * 2 * Ip * H * 2 + El * H * Ip * 2;
  p.tp_base = stage;
  p.tp_q_stride = block;
  p.tp_r_stride = (uint64_t)g.P * block;
  p.tp_w13_off = 0;
  p.tp_w2_off = El * 2 * Ip * H * 2;
  p.tp_eoff_per_r = 0;
  p.tp_span = Span{stage, stage + weights_stage_bytes(g), g.flags};
  cudaError_t e;
  if (ep2tp) {   // permute into per-peer blocks, then exchange into the TP slots
    if ((e = run_any(p, VB, 1, s, false)) != cudaSuccess) return e;
    e = run_exchange(g, layer, VB, stage, 1, s);
  } else {       // exchange out of the TP slots, then permute into whole experts
    if ((e = run_exchange(g, layer, VB, stage, 0, s)) != cudaSuccess) return e;
    e = run_any(p, VB, 0, s, false);
  }
  *launches = 2;
  return e;
}

}  // namespace uk
