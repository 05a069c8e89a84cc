// Staged (collective-style) KV reshard, kept for comparison with the fused
// copies in umm_kv.cu.  "Moebius: Serving Mixture-of-Expert Models with
// Seamless Runtime Parallelism Switch" (paper review), §3.2 (the collective
// pipeline: gather scattered slots into per-peer contiguous blocks, one
// exchange, scatter into the target pages) and §4.3, Table 1 (it touches HBM
// more than once per element; the fused kernels do not).
#include "umm_scan.cuh"

namespace uk {

// ------------------------------------------------------------------ staged (collective-style) path
//
// For comparison with the fused copies (§4.3, Table 1: the collective path
// gathers scattered slots into per-peer contiguous blocks, exchanges them
// once, then scatters into the target pages).  One layer is moved one EP rank
// at a time (EP->TP: the source rank; TP->EP: the destination rank), through
// a caller-owned staging buffer holding a send and a receive area:
//   EP->TP  send[c][q][t][h_tp][D]  = rows of rank o's tokens for TP rank q
//   TP->EP  send[c][g][t][h_tp][D]  = rows of head group g (read from its
//                                     lowest replica) for rank o's tokens
// t runs over rank o's live tokens in descriptor order (tokoff + row).

// Per-request token offsets inside their owning rank, in (rank, request)
// order, and each rank's first descriptor, descriptor count and token count.
__global__ void __launch_bounds__(kScanThreads)
kv_stage_prep(Geo g, Ws w, int32_t R, const int32_t* __restrict__ lens, const int32_t* __restrict__ owner,
              int64_t* __restrict__ order_tok, int64_t* __restrict__ rank_info, unsigned int call) {
  DevStatus* st = status_of(g, w);
  if (read_flags(st)) return;
  __shared__ long long carry_t[kMaxGroups];
  __shared__ long long carry_d[kMaxGroups];
  __shared__ long long warp_tot[32 * kMaxGroups];
  const int tid = threadIdx.x, P = g.P;
  if (tid < kMaxGroups) {
    carry_t[tid] = 0;
    carry_d[tid] = 0;
  }
  __syncthreads();
  const int32_t* order_req = reinterpret_cast<const int32_t*>(g.base + w.req_inv);
  for (int base = 0; base < R; base += blockDim.x) {
    const int j = base + tid;
    long long len = 0, np = 0;
    int grp = 0;
    if (j < R) {
      const int k = order_req[j];
      len = lens[k];
      np = pages_of(len, g.ps);
      grp = owner[k];
    }
    const long long tok = group_exclusive_scan(len, grp, P, carry_t, warp_tot);
    group_exclusive_scan(np, grp, P, carry_d, warp_tot);
    if (j < R) order_tok[j] = tok;
  }
  if (tid == 0) {
    long long first = 0;
    int over = 0;
    for (int r = 0; r < P; ++r) {
      rank_info[3 * r + 0] = first;        // first descriptor of rank r
      rank_info[3 * r + 1] = carry_d[r];   // its descriptors
      rank_info[3 * r + 2] = carry_t[r];   // its live tokens
      first += carry_d[r];
      // the staging areas are sized for one rank's full EP pool
      if (carry_t[r] > g.pages_ep * (long long)g.ps) over = 1;
    }
    if (over) raise_flag(st, UMM_FLAG_CAPACITY, call);
  }
}

struct SParams {
  uint8_t* base;
  uint8_t* send;
  uint8_t* recv;
  const umm_kv_desc* desc;
  const DevStatus* st;
  const int32_t* order_req;
  const int64_t* order_start;
  const int64_t* order_tok;
  const int64_t* rank_info;
  int32_t R, rank;
  uint64_t region_stride, kv_v_off, ep_slot, tp_slot, ep_row, tp_row, head_bytes;
  uint32_t ps, Hkv, P, h_tp, rep, groups;   // groups = Hkv / h_tp head groups
  Span regions, staging;                    // the P regions; the caller's staging buffer
};

// token offset of descriptor di inside its rank's stream
__device__ __forceinline__ long long stage_tokoff(const SParams& p, long long di, const umm_kv_desc& d) {
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.order_start[mid] <= di) lo = mid;
    else hi = mid - 1;
  }
  return p.order_tok[lo] + (long long)d.page * p.ps;
}

// stage 1, gather: live rows of rank p.rank's pages -> send.  EP->TP reads the
// EP pages and writes each head once per replica; TP->EP reads each head
// group from its lowest replica's TP page.
template <int VB>
__global__ void __launch_bounds__(256) kv_stage_gather(const SParams p, int dir) {
  using V = typename VecT<VB>::T;
  if (read_flags(p.st)) return;
  const long long first = p.rank_info[3 * p.rank], cnt = p.rank_info[3 * p.rank + 1];
  const long long T = p.rank_info[3 * p.rank + 2];
  const uint32_t rowv = (uint32_t)(p.tp_row / VB);              // vectors per TP row
  for (long long i = blockIdx.x; i < cnt; i += gridDim.x) {
    const long long di = first + i;
    const umm_kv_desc d = p.desc[di];
    const long long t0 = stage_tokoff(p, di, d);
    const uint32_t per_slot = (uint32_t)d.ntok * rowv;           // vectors of one (c, q or g) block
    const uint32_t nslots = 2u * (dir == 0 ? p.P : p.groups);
    for (uint32_t v = threadIdx.x; v < nslots * per_slot; v += blockDim.x) {
      const uint32_t slot = v / per_slot, rv = v - slot * per_slot;
      const uint32_t c = slot / (nslots / 2), qg = slot - c * (nslots / 2);
      const uint32_t tok = rv / rowv, cv = rv - tok * rowv;
      const uint8_t* src;
      if (dir == 0) {   // EP page of rank o; TP rank qg's heads
        const uint32_t h = p.Hkv < p.P ? qg / p.rep : qg * p.h_tp;
        src = p.base + (uint64_t)p.rank * p.region_stride + p.ep_slot + c * p.kv_v_off +
              ((uint64_t)d.src_page * p.ps + tok) * p.ep_row + (uint64_t)h * p.head_bytes + (uint64_t)cv * VB;
      } else {          // TP page of head group qg's lowest replica
        const uint32_t q = p.Hkv < p.P ? qg * p.rep : qg;
        src = p.base + (uint64_t)q * p.region_stride + p.tp_slot + c * p.kv_v_off +
              ((uint64_t)d.src_page * p.ps + tok) * p.tp_row + (uint64_t)cv * VB;
      }
      uint8_t* const dst = p.send + (((uint64_t)slot * T + t0 + tok) * p.tp_row) + (uint64_t)cv * VB;
      if (access_ok<VB>(p.regions, src) && access_ok<VB>(p.staging, dst))
        st_vec(reinterpret_cast<V*>(dst), ld_vec(reinterpret_cast<const V*>(src)));
    }
  }
}

// stage 2, exchange: send -> recv (one contiguous copy of every block).
template <int VB>
__global__ void __launch_bounds__(256) kv_stage_exchange(const SParams p, int dir) {
  using V = typename VecT<VB>::T;
  if (read_flags(p.st)) return;
  const long long T = p.rank_info[3 * p.rank + 2];
  const uint64_t n = 2ull * (dir == 0 ? p.P : p.groups) * (uint64_t)T * p.tp_row / VB;
  for (uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += (uint64_t)gridDim.x * blockDim.x)
    if (access_ok<VB>(p.staging, reinterpret_cast<V*>(p.send) + v) &&
        access_ok<VB>(p.staging, reinterpret_cast<V*>(p.recv) + v))
      st_vec(reinterpret_cast<V*>(p.recv) + v, ld_vec(reinterpret_cast<const V*>(p.send) + v));
}

// stage 3, scatter: recv -> target pages (EP->TP: every TP rank's page;
// TP->EP: the owner's EP page, head group qg at heads qg*h_tp..).
template <int VB>
__global__ void __launch_bounds__(256) kv_stage_scatter(const SParams p, int dir) {
  using V = typename VecT<VB>::T;
  if (read_flags(p.st)) return;
  const long long first = p.rank_info[3 * p.rank], cnt = p.rank_info[3 * p.rank + 1];
  const long long T = p.rank_info[3 * p.rank + 2];
  const uint32_t rowv = (uint32_t)(p.tp_row / VB);
  for (long long i = blockIdx.x; i < cnt; i += gridDim.x) {
    const long long di = first + i;
    const umm_kv_desc d = p.desc[di];
    const long long t0 = stage_tokoff(p, di, d);
    const uint32_t per_slot = (uint32_t)d.ntok * rowv;
    const uint32_t nslots = 2u * (dir == 0 ? p.P : p.groups);
    for (uint32_t v = threadIdx.x; v < nslots * per_slot; v += blockDim.x) {
      const uint32_t slot = v / per_slot, rv = v - slot * per_slot;
      const uint32_t c = slot / (nslots / 2), qg = slot - c * (nslots / 2);
      const uint32_t tok = rv / rowv, cv = rv - tok * rowv;
      const V* src = reinterpret_cast<const V*>(p.recv + (((uint64_t)slot * T + t0 + tok) * p.tp_row) +
                                                (uint64_t)cv * VB);
      uint8_t* dst;
      if (dir == 0)
        dst = p.base + (uint64_t)qg * p.region_stride + p.tp_slot + c * p.kv_v_off +
              ((uint64_t)d.dst_page * p.ps + tok) * p.tp_row + (uint64_t)cv * VB;
      else
        dst = p.base + (uint64_t)p.rank * p.region_stride + p.ep_slot + c * p.kv_v_off +
              ((uint64_t)d.dst_page * p.ps + tok) * p.ep_row + (uint64_t)qg * p.h_tp * p.head_bytes +
              (uint64_t)cv * VB;
      if (access_ok<VB>(p.staging, src) && access_ok<VB>(p.regions, dst))
        st_vec(reinterpret_cast<V*>(dst), ld_vec(src));
    }
  }
}

uint64_t kv_stage_bytes(const Geo& g) {
  // send + receive areas for one rank: its tokens (at most pages_ep * ps)
  // times max(P, Hkv) head rows, K and V
  const uint64_t heads = (uint64_t)(g.Hkv > g.P ? g.Hkv : g.P);
  const uint64_t one = 2ull * (uint64_t)g.pages_ep * g.ps * heads * g.D * 2;
  return 2 * ((one + 255) / 256 * 256);
}

cudaError_t launch_kv_staged(const Geo& g, const Ws& w, int dir, int32_t R, const int32_t* lens,
                             const int32_t* owner, uint8_t* stage, int64_t* order_tok, int64_t* rank_info,
                             unsigned int call, cudaStream_t s, int sms, int* launches) {
  *launches = 0;
  if (R == 0) return cudaSuccess;
  kv_stage_prep<<<1, kScanThreads, 0, s>>>(g, w, R, lens, owner, order_tok, rank_info, call);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches += 1;
  int VB = 2;
  if (g.D % 8 == 0) VB = 16;
  else if (g.D % 4 == 0) VB = 8;
  else if (g.D % 2 == 0) VB = 4;
  SParams p;
  p.base = g.base;
  const uint64_t half = kv_stage_bytes(g) / 2;
  p.send = stage;
  p.recv = stage + half;
  p.regions = g.regions();
  p.staging = Span{stage, stage + 2 * half, g.flags};
  p.desc = reinterpret_cast<const umm_kv_desc*>(g.base + w.desc);
  p.st = reinterpret_cast<const DevStatus*>(g.base + w.status);
  p.order_req = reinterpret_cast<const int32_t*>(g.base + w.req_inv);
  p.order_start = reinterpret_cast<const int64_t*>(g.base + w.req_off);
  p.order_tok = order_tok;
  p.rank_info = rank_info;
  p.R = R;
  p.region_stride = g.region_stride;
  p.kv_v_off = g.kv_v_off;
  p.ep_row = (uint64_t)g.Hkv * g.D * 2;
  p.tp_row = (uint64_t)g.h_tp * g.D * 2;
  p.head_bytes = (uint64_t)g.D * 2;
  p.ps = (uint32_t)g.ps;
  p.Hkv = (uint32_t)g.Hkv;
  p.P = (uint32_t)g.P;
  p.h_tp = (uint32_t)g.h_tp;
  p.rep = g.Hkv < g.P ? (uint32_t)(g.P / g.Hkv) : 1u;
  p.groups = (uint32_t)(g.Hkv / g.h_tp);
  const unsigned grid = (unsigned)sms * 16;
  const int N = g.N;
  for (int t = 0; t < N; ++t) {
    const int layer = dir == 0 ? t : N - 1 - t;
    p.ep_slot = g.kvslots_off + (uint64_t)(layer + 1) * g.kvslot_stride;
    p.tp_slot = g.kvslots_off + (uint64_t)layer * g.kvslot_stride;
    for (int r = 0; r < g.P; ++r) {
      p.rank = r;
      switch (VB) {
#define STAGES(VB_)                                              \
  kv_stage_gather<VB_><<<grid, 256, 0, s>>>(p, dir);             \
  kv_stage_exchange<VB_><<<grid, 256, 0, s>>>(p, dir);           \
  kv_stage_scatter<VB_><<<grid, 256, 0, s>>>(p, dir);            \
  break;
        case 16: STAGES(16)
        case 8: STAGES(8)
        case 4: STAGES(4)
        default: STAGES(2)
#undef STAGES
      }
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      *launches += 3;
    }
  }
  return cudaSuccess;
}

}  // namespace uk
