// Paged KV-cache redistribution EP <-> TP: the descriptor pass.
//
// "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
// Switch" (paper review): §3.2 (the page table drives an index vector that
// gathers scattered token slots per destination), §4.3 and Fig. 8b (page-
// indexed work descriptors built from the live request metadata).
//
// One pass per switch, before any copy: kv_prep_scan (validation, capacity,
// per-region offsets) and kv_prep_emit (one descriptor per live (request,
// page), page-id checks with warp ballots and destination bitmaps, and an
// index of the descriptors by TP page).  Any failed check raises a status flag
// and the copies of the switch then write nothing.
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
  // pages and requests per region: the lanes of a __match_any_sync set (same
  // region) sum their pages with two 16-bit-half reductions (exact: 32 lanes
  // x 2^16 < 2^32) and the set's lowest lane adds them with one shared atomic
  const int lane = tid & 31;
  for (int base = 0; base < R; base += blockDim.x) {
    const int k = base + tid;
    int len = 0, o = -1;
    if (k < R) {
      len = lens[k];
      o = owner[k];
    }
    const bool valid = k < R && len >= 0 && (long long)len <= max_len && o >= 0 && o < P;
    if (k < R && !valid) bad = 1;
    const unsigned int np = valid ? (unsigned int)pages_of(len, g.ps) : 0u;
    const unsigned int same = __match_any_sync(0xffffffffu, valid ? o : -1);
    const unsigned int lo = __reduce_add_sync(same, np & 0xffffu);
    const unsigned int hi = __reduce_add_sync(same, np >> 16);
    if (valid) {
      if (lane == __ffs(same) - 1) {
        atomicAdd(&region_pages[o], ((unsigned long long)hi << 16) + lo);
        atomicAdd(&region_reqs[o], (unsigned int)__popc(same));
      }
      my_tokens += (unsigned long long)len;
    }
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
      np = pages_of(lens[k], g.ps);
      grp = owner[k];
    }
    const long long start = group_exclusive_scan(np, grp, P, carry, warp_tot);
    const long long j = group_exclusive_count(k < R, grp, P, carry_n, warp_tot);
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

}  // namespace uk
