// Request metadata of a switch: the EP->TP global list order, the TP->EP
// greedy placement, and destination page hand-out.
//
// "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
// Switch" (paper review), §3.2: on EP->TP a metadata all-gather gives every
// rank the same ordered in-flight list; on TP->EP the list is sorted by
// sequence length (longest first) and each request goes to the least-loaded
// rank -- deterministic, so every rank computes the same partition without
// communicating.  Requests then move to "reassigned target pages".
//
// These kernels are tiny next to the data movement; each runs as one CTA
// (plus a wide fill for page tables), built on grouped block scans and counts.
#include <algorithm>
#include <atomic>
#include <climits>

#include "umm_place.cuh"

namespace uk {

constexpr int kMaxDevices = 64;

// ------------------------------------------------------------------ list order (EP -> TP)

__global__ void __launch_bounds__(kScanThreads)
order_kernel(Geo g, Ws w, int32_t R, const int32_t* __restrict__ owner, int32_t* __restrict__ tp_pos,
             unsigned int call) {
  DevStatus* st = status_of(g, w);
  if (read_flags(st)) return;
  __shared__ long long carry[kMaxGroups];
  __shared__ long long warp_tot[32 * kMaxGroups];
  __shared__ unsigned long long cnt[kMaxGroups];
  __shared__ int bad;
  const int tid = threadIdx.x, P = g.P;
  if (tid < kMaxGroups) cnt[tid] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  // requests per rank: one shared atomic per rank and warp (the lanes of a
  // __match_any_sync set add their count through the set's lowest lane)
  const int lane = tid & 31;
  for (int base = 0; base < R; base += blockDim.x) {
    const int k = base + tid;
    const int o = k < R ? owner[k] : -1;
    const bool valid = o >= 0 && o < P;
    if (k < R && !valid) bad = 1;
    const unsigned int same = __match_any_sync(0xffffffffu, valid ? o : -1);
    if (valid && lane == __ffs(same) - 1) atomicAdd(&cnt[o], (unsigned long long)__popc(same));
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) raise_flag(st, UMM_FLAG_BAD_REQUEST, call);
    return;
  }
  if (tid == 0) {
    long long run = 0;
    for (int r = 0; r < P; ++r) {
      carry[r] = run;     // rank r's requests follow those of ranks < r
      run += (long long)cnt[r];
    }
  }
  __syncthreads();
  for (int base = 0; base < R; base += blockDim.x) {
    const int k = base + tid;
    const long long pre = group_exclusive_count(k < R, k < R ? owner[k] : 0, P, carry, warp_tot);
    if (k < R) tp_pos[k] = (int32_t)pre;
  }
}

cudaError_t launch_order(const Geo& g, const Ws& w, int32_t R, const int32_t* owner, int32_t* tp_pos,
                         unsigned int call, cudaStream_t s) {
  order_kernel<<<1, kScanThreads, 0, s>>>(g, w, R, owner, tp_pos, call);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(kScanThreads)
place_kernel(Geo g, Ws w, int32_t R, const int32_t* __restrict__ lens, const int32_t* __restrict__ list_pos,
             int32_t* __restrict__ owner, int32_t* __restrict__ local_pos, int keys_in_smem,
             unsigned int call) {
  DevStatus* st = status_of(g, w);
  if (read_flags(st)) return;
  extern __shared__ unsigned long long smem_keys[];
  unsigned long long* keys =
      keys_in_smem ? smem_keys : reinterpret_cast<unsigned long long*>(g.base + w.keys);
  if (!place_block(g.P, R, lens, list_pos, owner, local_pos, reinterpret_cast<int32_t*>(g.base + w.req_inv),
                   g.base + w.choice, keys) &&
      threadIdx.x == 0)
    raise_flag(st, UMM_FLAG_BAD_REQUEST, call);
}

cudaError_t launch_place(const Geo& g, const Ws& w, int32_t R, const int32_t* lens, const int32_t* list_pos,
                         int32_t* owner, int32_t* local_pos, unsigned int call, cudaStream_t s) {
  // keys in shared memory for up to 16 x 1024 requests
  const size_t need = (size_t)sort_span(R) * sizeof(unsigned long long);
  const int in_smem = need <= 128 * 1024;
  const size_t dyn = in_smem ? need : 0;
  // the shared-memory limit is a per-device function attribute: set it once
  // per device.  Handles on one device may be driven from different host
  // threads; setting the same value twice is harmless, so an atomic flag
  // per device is enough
  static std::atomic<bool> attr_set[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  place_kernel<<<1, kScanThreads, dyn, s>>>(g, w, R, lens, list_pos, owner, local_pos, in_smem, call);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ page hand-out

__global__ void __launch_bounds__(kScanThreads)
assign_scan(Geo g, Ws w, int32_t npools, int32_t R, int32_t maxp, const int32_t* __restrict__ lens,
            const int32_t* __restrict__ pool, const int32_t* __restrict__ key, int64_t free_count,
            unsigned int call) {
  DevStatus* st = status_of(g, w);
  if (read_flags(st)) return;
  __shared__ long long carry[kMaxGroups];
  __shared__ long long warp_tot[32 * kMaxGroups];
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  if (tid < kMaxGroups) carry[tid] = 0;
  __syncthreads();
  const long long max_len = (long long)maxp * g.ps;
  for (int k = tid; k < R; k += blockDim.x) {
    const int len = lens[k];
    const int pl = pool ? pool[k] : 0;
    if (len < 0 || (long long)len > max_len || pl < 0 || pl >= npools) bad = 1;
  }
  __syncthreads();
  int32_t* inv = reinterpret_cast<int32_t*>(g.base + w.req_inv);
  bool ok = bad == 0;
  if (ok && key) ok = build_inverse(key, R, inv, &bad);
  if (!ok) {
    if (tid == 0) raise_flag(st, UMM_FLAG_BAD_REQUEST, call);
    return;
  }
  int64_t* start = reinterpret_cast<int64_t*>(g.base + w.req_off);
  for (int base = 0; base < R; base += blockDim.x) {
    const int pos = base + tid;
    int k = 0, grp = 0;
    long long np = 0;
    if (pos < R) {
      k = key ? inv[pos] : pos;
      grp = pool ? pool[k] : 0;
      np = pages_of(lens[k], g.ps);
    }
    const long long pre = group_exclusive_scan(np, grp, npools, carry, warp_tot);
    if (pos < R) start[k] = pre;
  }
  if (tid < npools && carry[tid] > free_count) raise_flag(st, UMM_FLAG_CAPACITY, call);
}

__global__ void __launch_bounds__(256)
assign_emit(Geo g, Ws w, int32_t R, int32_t maxp, const int32_t* __restrict__ lens,
            const int32_t* __restrict__ pool, const int32_t* __restrict__ free_pages, int64_t free_stride,
            int32_t* __restrict__ pt) {
  const DevStatus* st = status_of(g, w);
  if (read_flags(st)) return;
  const int lane = threadIdx.x & 31;
  const int warps_total = (gridDim.x * blockDim.x) >> 5;
  const int64_t* start = reinterpret_cast<const int64_t*>(g.base + w.req_off);
  for (int k = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; k < R; k += warps_total) {
    const int np = pages_of(lens[k], g.ps);
    const int64_t src = (pool ? (int64_t)pool[k] : 0) * free_stride + start[k];
    int32_t* row = pt + (int64_t)k * maxp;
    for (int p = lane; p < maxp; p += 32) row[p] = p < np ? free_pages[src + p] : -1;
  }
}

cudaError_t launch_assign(const Geo& g, const Ws& w, int32_t npools, int32_t R, const int32_t* lens,
                          const int32_t* pool, const int32_t* key, const int32_t* free_pages,
                          int64_t free_stride, int64_t free_count, int32_t* pt, int32_t maxp,
                          unsigned int call, cudaStream_t s, int sms) {
  assign_scan<<<1, kScanThreads, 0, s>>>(g, w, npools, R, maxp, lens, pool, key, free_count, call);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || R == 0) return e;
  // one warp per request, at most 8 CTAs per SM (64-bit: R * 32 reaches 2^31
  // at the largest request count)
  const long long blocks = std::min<long long>(((long long)R * 32 + 255) / 256, (long long)sms * 8);
  assign_emit<<<(unsigned)blocks, 256, 0, s>>>(g, w, R, maxp, lens, pool, free_pages, free_stride, pt);
  return cudaGetLastError();
}

}  // namespace uk
