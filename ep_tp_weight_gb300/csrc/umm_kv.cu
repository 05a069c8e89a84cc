// Paged KV-cache redistribution EP <-> TP.
//
// "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
// Switch" (paper review): §3.2 and Fig. 5 (EP keeps all heads of its requests,
// TP a head shard of every request, heads replicated over rank groups when
// there are fewer KV heads than ranks; the page table drives an index vector
// that gathers scattered token slots per destination and scatters them into
// the target pages), §4.3 Table 1 and Fig. 8b (page-indexed work descriptors
// built from the live request metadata; one read and one direct write).
//
// One switch = one descriptor pass (kv_prep_scan: validation, capacity,
// offsets; kv_prep_emit: one descriptor per live (request, page), page-id
// checks with warp ballots and destination bitmaps, and an index of the
// descriptors by TP page) + one gather/scatter launch per layer (kv_copy_*:
// one CTA per TP page, or per descriptor when the pool is sparsely used).
// Nothing is written to the cache unless the descriptor pass raised no flag.
#include <algorithm>

#include "umm_scan.cuh"

namespace uk {

// ------------------------------------------------------------------ descriptor pass

__global__ void __launch_bounds__(kScanThreads)
kv_prep_scan(Geo g, Ws w, int dir, int32_t R, int32_t maxp, const int32_t* __restrict__ lens,
             const int32_t* __restrict__ owner, unsigned int call) {
  DevStatus* st = status_of(g, w);
  if (read_flags(st)) return;
  __shared__ long long carry[kMaxGroups];    // running page offset per region
  __shared__ long long carry_n[kMaxGroups];  // running request count per region
  __shared__ long long warp_tot[32 * kMaxGroups];
  __shared__ unsigned long long region_pages[kMaxGroups];
  __shared__ unsigned int region_reqs[kMaxGroups];
  __shared__ unsigned long long tokens;
  __shared__ int bad, capfail;
  const int tid = threadIdx.x, P = g.P;
  if (tid < kMaxGroups) {
    region_pages[tid] = 0;
    region_reqs[tid] = 0;
  }
  if (tid == 0) { tokens = 0; bad = 0; capfail = 0; }
  __syncthreads();
  const long long max_len = (long long)maxp * g.ps;
  unsigned long long my_tokens = 0;
  for (int k = tid; k < R; k += blockDim.x) {
    const int len = lens[k], o = owner[k];
    if (len < 0 || (long long)len > max_len || o < 0 || o >= P) {
      bad = 1;
      continue;
    }
    atomicAdd(&region_pages[o], (unsigned long long)((len + g.ps - 1) / g.ps));
    atomicAdd(&region_reqs[o], 1u);
    my_tokens += (unsigned long long)len;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) my_tokens += __shfl_xor_sync(0xffffffffu, my_tokens, d);
  if ((tid & 31) == 0) atomicAdd(&tokens, my_tokens);
  __syncthreads();
  if (bad) {
    if (tid == 0) raise_flag(st, UMM_FLAG_BAD_REQUEST, call);
    return;
  }
  if (tid == 0) {
    unsigned long long total = 0, nreq = 0;
    int fail = 0;
    for (int r = 0; r < P; ++r) {
      carry[r] = (long long)total;  // descriptors of region r start here
      carry_n[r] = (long long)nreq; // and its requests in the (region, request) order
      total += region_pages[r];
      nreq += region_reqs[r];
      if (dir == 1 && (long long)region_pages[r] > g.pages_ep) fail = 1;
    }
    if (dir == 0 && (long long)total > g.pages_tp) fail = 1;
    if ((long long)total > w.desc_cap) fail = 1;
    if (fail) {
      raise_flag(st, UMM_FLAG_CAPACITY, call);
      capfail = 1;
    } else {
      st->ndesc = total;
      st->tokens = tokens;
    }
  }
  __syncthreads();
  if (capfail) return;
  // requests in (owning region, request) order, with their first descriptor:
  // order_req[j] = request, order_start[j] = offset (non-decreasing in j)
  int64_t* order_start = reinterpret_cast<int64_t*>(g.base + w.req_off);
  int32_t* order_req = reinterpret_cast<int32_t*>(g.base + w.req_inv);
  for (int base = 0; base < R; base += blockDim.x) {
    const int k = base + tid;
    long long np = 0;
    int grp = 0;
    if (k < R) {
      np = (lens[k] + g.ps - 1) / g.ps;
      grp = owner[k];
    }
    const long long start = group_exclusive_scan(np, grp, P, carry, warp_tot);
    const long long j = group_exclusive_scan(k < R ? 1 : 0, grp, P, carry_n, warp_tot);
    if (k < R) {
      order_start[j] = start;
      order_req[j] = k;
    }
  }
  // clear the destination-page bitmap (and, for TP->EP, the TP source one)
  const long long bits = dir == 0 ? g.pages_tp : (long long)P * g.pages_ep;
  const long long words = (bits + 31) / 32;
  uint32_t* bm = reinterpret_cast<uint32_t*>(g.base + w.bitmap);
  for (long long i = tid; i < words; i += blockDim.x) bm[i] = 0u;
  if (dir == 1) {
    uint32_t* tb = reinterpret_cast<uint32_t*>(g.base + w.tp_bitmap);
    for (long long i = tid; i < (g.pages_tp + 31) / 32; i += blockDim.x) tb[i] = 0u;
  }
}

// One thread per descriptor: a binary search over the request order finds
// the request whose run holds descriptor d (requests without pages share the
// next request's start, so the last start <= d is the right one).
__global__ void __launch_bounds__(256)
kv_prep_emit(Geo g, Ws w, int dir, int32_t R, int32_t maxp, const int32_t* __restrict__ lens,
             const int32_t* __restrict__ owner, const int32_t* __restrict__ ep_pt,
             const int32_t* __restrict__ tp_pt, unsigned int call, int use_sched) {
  DevStatus* st = status_of(g, w);
  if (read_flags(st)) return;
  const long long nd = (long long)st->ndesc;
  const int lane = threadIdx.x & 31;
  const int64_t* order_start = reinterpret_cast<const int64_t*>(g.base + w.req_off);
  const int32_t* order_req = reinterpret_cast<const int32_t*>(g.base + w.req_inv);
  umm_kv_desc* desc = reinterpret_cast<umm_kv_desc*>(g.base + w.desc);
  uint32_t* bm = reinterpret_cast<uint32_t*>(g.base + w.bitmap);
  uint32_t* tb = reinterpret_cast<uint32_t*>(g.base + w.tp_bitmap);
  unsigned long long* sched = reinterpret_cast<unsigned long long*>(g.base + w.sched);
  unsigned int oob_any = 0, dup_any = 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // every lane runs the same number of iterations (the ballots need them all)
  for (long long base = (long long)blockIdx.x * blockDim.x; base < nd; base += stride) {
    const long long di = base + threadIdx.x;
    bool oob = false, dup = false;
    if (di < nd) {
      int lo = 0, hi = R - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (order_start[mid] <= di) lo = mid;
        else hi = mid - 1;
      }
      const int k = order_req[lo];
      const int p = (int)(di - order_start[lo]);
      const int len = lens[k], o = owner[k];
      const int ep = ep_pt[(int64_t)k * maxp + p], tp = tp_pt[(int64_t)k * maxp + p];
      oob = ep < 0 || ep >= g.pages_ep || tp < 0 || tp >= g.pages_tp;
      if (!oob) {
        const long long bit = dir == 0 ? (long long)tp : (long long)o * g.pages_ep + ep;
        const uint32_t m = 1u << (bit & 31);
        dup = (atomicOr(&bm[bit >> 5], m) & m) != 0;
        if (dir == 1) {   // each TP page belongs to one request
          const uint32_t mt = 1u << (tp & 31);
          dup |= (atomicOr(&tb[tp >> 5], mt) & mt) != 0;
        }
        if (use_sched) sched[tp] = ((unsigned long long)call << 32) | (unsigned long long)di;
      }
      umm_kv_desc d;
      d.req = k;
      d.page = p;
      d.src_region = dir == 0 ? o : -1;
      d.dst_region = dir == 0 ? -1 : o;
      d.src_page = dir == 0 ? ep : tp;
      d.dst_page = dir == 0 ? tp : ep;
      d.ntok = min(g.ps, len - p * g.ps);
      d.reserved = 0;
      desc[di] = d;
    }
    oob_any |= __ballot_sync(0xffffffffu, oob);
    dup_any |= __ballot_sync(0xffffffffu, dup);
  }
  if (lane == 0) {
    if (__popc(oob_any)) raise_flag(st, UMM_FLAG_PAGE_OOB, call);
    if (__popc(dup_any)) raise_flag(st, UMM_FLAG_DUP_PAGE, call);
  }
}

cudaError_t launch_kv_prep(const Geo& g, const Ws& w, int dir, int32_t R, int32_t maxp,
                           const int32_t* lens, const int32_t* owner, const int32_t* ep_pt,
                           const int32_t* tp_pt, unsigned int call, int use_sched, cudaStream_t s, int sms) {
  kv_prep_scan<<<1, kScanThreads, 0, s>>>(g, w, dir, R, maxp, lens, owner, call);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (R == 0) return cudaSuccess;
  // enough threads for every live page (at most min(capacity, R * maxp))
  const long long most = std::min<long long>(w.desc_cap, (long long)R * maxp);
  long long blocks = (most + 255) / 256;
  if (blocks > (long long)sms * 32) blocks = (long long)sms * 32;
  if (blocks < 1) blocks = 1;
  kv_prep_emit<<<(unsigned)blocks, 256, 0, s>>>(g, w, dir, R, maxp, lens, owner, ep_pt, tp_pt, call, use_sched);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ gather / scatter

struct KVParams {
  uint8_t* base;
  const umm_kv_desc* desc;
  const DevStatus* st;
  const unsigned long long* sched;   // TP page -> (call << 32 | descriptor), or null
  unsigned int call;
  uint64_t region_stride, kv_v_off;
  uint64_t ep_slot, tp_slot;   // absolute offsets of the slot inside a region
  uint64_t ep_row, tp_row;     // bytes per token row: Hkv*D*2, h_tp*D*2
  uint64_t head_bytes;         // D*2
  uint32_t ps, Hkv, P, h_tp, rep;   // rep = ranks per head when Hkv < P (else 1)
  uint32_t half_vec;           // vectors in one half (K or V) of an EP page
  long long pages_tp;
  FastDiv half, tok, dv;       // divisors: half_vec, Hkv*Dv, Dv
};

// The descriptor a CTA works on for grid position di: in TP-page order
// through the schedule (false for pages this call does not use), or straight
// from the descriptor list.
__device__ __forceinline__ bool fetch_desc(const KVParams& p, unsigned long long di, umm_kv_desc& d) {
  if (p.sched) {
    const unsigned long long e = p.sched[di];
    const unsigned long long idx = e & 0xffffffffull;
    if ((unsigned int)(e >> 32) != p.call || idx >= p.st->ndesc) return false;
    d = p.desc[idx];
    return true;
  }
  d = p.desc[di];
  return true;
}

// EP -> TP: each source vector of an EP page is loaded once and stored to
// every TP rank holding its head (rank h*rep + j, local head 0, when Hkv < P;
// rank h / h_tp, local head h % h_tp, when Hkv >= P).
template <int VB, int U, int T>
__global__ void __launch_bounds__(T) kv_copy_ep2tp(const KVParams p) {
  using V = typename VecT<VB>::T;
  if (read_flags(p.st)) return;
  const unsigned long long nd = p.sched ? (unsigned long long)p.pages_tp : p.st->ndesc;
  const uint32_t nvec = 2 * p.half_vec;
  for (unsigned long long di = blockIdx.x; di < nd; di += gridDim.x) {
    umm_kv_desc d;
    if (!fetch_desc(p, di, d)) continue;
    uint8_t* const src_region = p.base + (uint64_t)d.src_region * p.region_stride + p.ep_slot;
    const uint64_t src_page = (uint64_t)d.src_page * p.ps * p.ep_row;
    const uint64_t dst_page = (uint64_t)d.dst_page * p.ps * p.tp_row;
    for (uint32_t vb = 0; vb < nvec; vb += T * U) {
      V val[U];
      uint32_t tok[U], h[U], dvv[U], c[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t v = vb + threadIdx.x + u * T;
        uint32_t rem, rem2;
        p.half.divmod(v, c[u], rem);
        p.tok.divmod(rem, tok[u], rem2);
        p.dv.divmod(rem2, h[u], dvv[u]);
        if (v < nvec && tok[u] < (uint32_t)d.ntok)
          val[u] = __ldcs(reinterpret_cast<const V*>(src_region + c[u] * p.kv_v_off + src_page +
                                                      (uint64_t)rem * VB));
        else
          tok[u] = 0xffffffffu;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (tok[u] == 0xffffffffu) continue;
        const uint64_t row_off = dst_page + (uint64_t)tok[u] * p.tp_row + (uint64_t)dvv[u] * VB +
                                 c[u] * p.kv_v_off + p.tp_slot;
        if (p.Hkv < p.P) {
          for (uint32_t j = 0; j < p.rep; ++j) {
            const uint32_t q = h[u] * p.rep + j;
            __stcs(reinterpret_cast<V*>(p.base + (uint64_t)q * p.region_stride + row_off), val[u]);
          }
        } else {
          const uint32_t q = h[u] / p.h_tp, hl = h[u] - q * p.h_tp;
          __stcs(reinterpret_cast<V*>(p.base + (uint64_t)q * p.region_stride + row_off +
                                      (uint64_t)hl * p.head_bytes),
                 val[u]);
        }
      }
    }
  }
}

// TP -> EP: each vector of the destination EP page is read from the lowest TP
// rank holding its head.
template <int VB, int U, int T>
__global__ void __launch_bounds__(T) kv_copy_tp2ep(const KVParams p) {
  using V = typename VecT<VB>::T;
  if (read_flags(p.st)) return;
  const unsigned long long nd = p.sched ? (unsigned long long)p.pages_tp : p.st->ndesc;
  const uint32_t nvec = 2 * p.half_vec;
  for (unsigned long long di = blockIdx.x; di < nd; di += gridDim.x) {
    umm_kv_desc d;
    if (!fetch_desc(p, di, d)) continue;
    uint8_t* const dst_region = p.base + (uint64_t)d.dst_region * p.region_stride + p.ep_slot;
    const uint64_t dst_page = (uint64_t)d.dst_page * p.ps * p.ep_row;
    const uint64_t src_page = (uint64_t)d.src_page * p.ps * p.tp_row;
    for (uint32_t vb = 0; vb < nvec; vb += T * U) {
      V val[U];
      uint32_t rem_[U], c[U];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t v = vb + threadIdx.x + u * T;
        uint32_t rem, rem2, tok, h, dvv;
        p.half.divmod(v, c[u], rem);
        p.tok.divmod(rem, tok, rem2);
        p.dv.divmod(rem2, h, dvv);
        rem_[u] = rem;
        ok[u] = v < nvec && tok < (uint32_t)d.ntok;
        if (ok[u]) {
          uint32_t q, hl;
          if (p.Hkv < p.P) {
            q = h * p.rep;
            hl = 0;
          } else {
            q = h / p.h_tp;
            hl = h - q * p.h_tp;
          }
          val[u] = __ldcs(reinterpret_cast<const V*>(
              p.base + (uint64_t)q * p.region_stride + p.tp_slot + c[u] * p.kv_v_off + src_page +
              (uint64_t)tok * p.tp_row + (uint64_t)hl * p.head_bytes + (uint64_t)dvv * VB));
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u])
          __stcs(reinterpret_cast<V*>(dst_region + c[u] * p.kv_v_off + dst_page + (uint64_t)rem_[u] * VB),
                 val[u]);
    }
  }
}

namespace {
// EP->TP: 128 threads x 8 vectors (half a 32 KiB K+V page per round);
// TP->EP: 256 x 4.  Both picked by measurement on GB300 (within ~1% of the
// neighbouring shapes; 16-vector-per-thread or persistent shapes were slower).
constexpr int kT_ep2tp = 128, kU_ep2tp = 8;
constexpr int kT_tp2ep = 256, kU_tp2ep = 4;

// One CTA per descriptor (grid >= live pages): the block scheduler hands a
// finished CTA's slot to the next page at once, which keeps more loads in
// flight per SM than a persistent grid striding over the descriptors
// (measured on GB300: ~6.72 vs ~6.13 TB/s EP->TP at the full-switch size).
// The kernels still stride by gridDim.x, so any grid size is correct.
template <int VB>
cudaError_t run_copy(const KVParams& p, int dir, int64_t max_desc, cudaStream_t s) {
  if (max_desc <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)(max_desc < 0x7fffffffll ? max_desc : 0x7fffffffll);
  if (dir == 0) kv_copy_ep2tp<VB, kU_ep2tp, kT_ep2tp><<<grid, kT_ep2tp, 0, s>>>(p);
  else kv_copy_tp2ep<VB, kU_tp2ep, kT_tp2ep><<<grid, kT_tp2ep, 0, s>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_kv_copy(const Geo& g, const Ws& w, int dir, int layer, int64_t max_desc, int use_sched,
                           unsigned int call, cudaStream_t s) {
  int VB = 2;
  if (g.D % 8 == 0) VB = 16;
  else if (g.D % 4 == 0) VB = 8;
  else if (g.D % 2 == 0) VB = 4;
  const uint32_t per = (uint32_t)VB / 2;
  const uint32_t Dv = (uint32_t)g.D / per;
  KVParams p;
  p.base = g.base;
  p.desc = reinterpret_cast<const umm_kv_desc*>(g.base + w.desc);
  p.st = reinterpret_cast<const DevStatus*>(g.base + w.status);
  p.sched = use_sched ? reinterpret_cast<const unsigned long long*>(g.base + w.sched) : nullptr;
  p.call = call;
  p.pages_tp = g.pages_tp;
  if (use_sched) max_desc = g.pages_tp;   // one CTA per TP page
  p.region_stride = g.region_stride;
  p.kv_v_off = g.kv_v_off;
  p.ep_slot = g.kvslots_off + (uint64_t)(layer + 1) * g.kvslot_stride;
  p.tp_slot = g.kvslots_off + (uint64_t)layer * g.kvslot_stride;
  p.ep_row = (uint64_t)g.Hkv * g.D * 2;
  p.tp_row = (uint64_t)g.h_tp * g.D * 2;
  p.head_bytes = (uint64_t)g.D * 2;
  p.ps = (uint32_t)g.ps;
  p.Hkv = (uint32_t)g.Hkv;
  p.P = (uint32_t)g.P;
  p.h_tp = (uint32_t)g.h_tp;
  p.rep = g.Hkv < g.P ? (uint32_t)(g.P / g.Hkv) : 1u;
  p.half_vec = (uint32_t)g.ps * (uint32_t)g.Hkv * Dv;
  p.half = FastDiv(p.half_vec);
  p.tok = FastDiv((uint32_t)g.Hkv * Dv);
  p.dv = FastDiv(Dv);
  switch (VB) {
    case 16: return run_copy<16>(p, dir, max_desc, s);
    case 8: return run_copy<8>(p, dir, max_desc, s);
    case 4: return run_copy<4>(p, dir, max_desc, s);
    default: return run_copy<2>(p, dir, max_desc, s);
  }
}

}  // namespace uk
