// TP->EP request placement for callers that cannot allocate device memory.
//
// place_requests_tp2ep() keeps its scratch (the list-position -> request map)
// in the workspace of a unified buffer, which somebody had to cudaMalloc.  A
// request scheduler that only holds metadata (say, a process that is handed
// device pointers by the serving engine, or code that runs while a CUDA graph
// is being built or while an allocator must not be entered) has no such
// buffer and may not call cudaMalloc itself.  This variant computes the same
// result with its scratch in a fixed array of this library's own device
// memory, reserved when the library is loaded.
//
// Limits and caveats:
//  - at most kNoAllocMaxRequests (16,384) requests and P <= 64 ranks; larger
//    calls are refused with UMM_ERR_CAPACITY / UMM_ERR_INVALID_ARG before
//    anything is enqueued;
//  - the scratch array (64 KiB) exists once per GPU that loads the library,
//    for the life of the process, and every call on that GPU shares it: two
//    calls whose kernels overlap on the GPU (different streams without an
//    ordering between them) race and may produce wrong results;
//  - the first call on a device looks up the array's device address and
//    raises the kernel's shared-memory limit (no allocation); make that first
//    call before capturing a stream into a CUDA graph.
#include <climits>
#include <mutex>

#include "umm_scan.cuh"

namespace {

constexpr int kNoAllocMaxRequests = 16384;
constexpr int kMaxDevices = 64;

// list position -> request index, one entry per request.  It holds no state
// between calls: every entry a call reads is written by that call first.
static __device__ __align__(256) int32_t g_place_scratch[kNoAllocMaxRequests];

std::mutex g_setup_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Greedy list scheduling with the loads held in registers (PB >= P).
template <int PB>
__device__ void greedy_lpt(const unsigned long long* keys, int32_t R, int P, const int32_t* inv,
                           int32_t* owner) {
  long long load[PB];
#pragma unroll
  for (int q = 0; q < PB; ++q) load[q] = q < P ? 0 : LLONG_MAX;
  for (int i = 0; i < R; ++i) {
    const unsigned long long key = keys[i];
    const int pos = (int)(key & 0xffffffffu);
    const long long len = 0x7fffffffll - (long long)(key >> 32);
    int best = 0;
    long long bl = load[0];
#pragma unroll
    for (int q = 1; q < PB; ++q)
      if (load[q] < bl) { bl = load[q]; best = q; }
#pragma unroll
    for (int q = 0; q < PB; ++q)
      if (q == best) load[q] += len;
    owner[inv ? inv[pos] : pos] = best;
  }
}

__global__ void __launch_bounds__(uk::kScanThreads)
place_noalloc_kernel(int P, int32_t R, const int32_t* __restrict__ lens, const int32_t* __restrict__ list_pos,
                     int32_t* __restrict__ owner, int32_t* __restrict__ local_pos, int32_t* inv,
                     int32_t* status) {
  extern __shared__ unsigned long long keys[];
  __shared__ long long carry[uk::kMaxGroups];
  __shared__ long long warp_tot[32 * uk::kMaxGroups];
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  if (tid < uk::kMaxGroups) carry[tid] = 0;
  __syncthreads();
  for (int k = tid; k < R; k += blockDim.x)
    if (lens[k] < 0) bad = 1;
  __syncthreads();
  if (!bad && list_pos) {
    for (int k = tid; k < R; k += blockDim.x) {
      const int pos = list_pos[k];
      if (pos < 0 || pos >= R) bad = 1;
      else inv[pos] = k;
    }
    __syncthreads();
    if (!bad)
      for (int k = tid; k < R; k += blockDim.x)
        if (inv[list_pos[k]] != k) bad = 1;   // a repeated position
    __syncthreads();
  }
  if (bad) {
    if (tid == 0 && status) *status = UMM_ERR_BAD_REQUEST;
    return;
  }
  int n2 = 1;
  while (n2 < R) n2 <<= 1;
  for (int i = tid; i < n2; i += blockDim.x) {
    unsigned long long kk = ~0ull;
    if (i < R) {
      const unsigned long long pos = list_pos ? (unsigned long long)list_pos[i] : (unsigned long long)i;
      kk = ((unsigned long long)(0x7fffffffll - lens[i]) << 32) | pos;   // length desc, position asc
    }
    keys[i] = kk;
  }
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n2; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const unsigned long long a = keys[i], b = keys[j];
          if ((a > b) == up) { keys[i] = b; keys[j] = a; }
        }
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    const int32_t* iv = list_pos ? inv : nullptr;
    if (P <= 8) greedy_lpt<8>(keys, R, P, iv, owner);
    else if (P <= 16) greedy_lpt<16>(keys, R, P, iv, owner);
    else if (P <= 32) greedy_lpt<32>(keys, R, P, iv, owner);
    else greedy_lpt<64>(keys, R, P, iv, owner);
  }
  __syncthreads();
  for (int base = 0; base < R; base += blockDim.x) {
    const int pos = base + tid;
    int k = 0, grp = 0;
    if (pos < R) {
      k = list_pos ? inv[pos] : pos;
      grp = owner[k];
    }
    const long long pre = uk::group_exclusive_scan(pos < R ? 1 : 0, grp, P, carry, warp_tot);
    if (pos < R) local_pos[k] = (int32_t)pre;
  }
  if (tid == 0 && status) *status = UMM_OK;
}

// Once per device, with that device current: the device address of the
// scratch array, and the kernel's dynamic shared-memory limit.
int setup_device(int32_t** scratch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UMM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_place_scratch) != cudaSuccess || !p) return UMM_ERR_CUDA;
    if (cudaFuncSetAttribute(place_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kNoAllocMaxRequests * (int)sizeof(unsigned long long)) != cudaSuccess)
      return UMM_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *scratch = g_scratch_ptr[dev];
  return UMM_OK;
}

}  // namespace

extern "C" int place_requests_tp2ep_noalloc(int32_t P, int32_t R, const int32_t* d_seq_lens,
                                            const int32_t* d_list_pos, int32_t* d_owner, int32_t* d_local_pos,
                                            int32_t* d_status, void* stream) {
  if (P < 1 || P > uk::kMaxGroups || R < 0) return UMM_ERR_INVALID_ARG;
  if (R > kNoAllocMaxRequests) return UMM_ERR_CAPACITY;
  if (R > 0 && (!d_seq_lens || !d_owner || !d_local_pos)) return UMM_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  const int rc = setup_device(&scratch);
  if (rc != UMM_OK) return rc;
  if (R == 0) return UMM_OK;
  int n2 = 1;
  while (n2 < R) n2 <<= 1;
  place_noalloc_kernel<<<1, uk::kScanThreads, (size_t)n2 * sizeof(unsigned long long),
                         reinterpret_cast<cudaStream_t>(stream)>>>(P, R, d_seq_lens, d_list_pos, d_owner,
                                                                   d_local_pos, scratch, d_status);
  return cudaGetLastError() == cudaSuccess ? UMM_OK : UMM_ERR_CUDA;
}
