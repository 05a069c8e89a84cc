// TP->EP request placement for callers that cannot allocate device memory.
//
// place_requests_tp2ep() keeps its scratch (the list-position -> request map)
// in the workspace of a unified buffer, which somebody had to cudaMalloc.  A
// request scheduler that only holds metadata (say, a process that is handed
// device pointers by the serving engine, or code that runs while a CUDA graph
// is being built or while an allocator must not be entered) has no such
// buffer and may not call cudaMalloc itself.  This variant computes the same
// result with its scratch in two fixed arrays of this library's own device
// memory (statically sized `__device__` arrays, 80 KiB together).
//
// Limits and caveats:
//  - at most kNoAllocMaxRequests (16,384) requests and P <= 64 ranks; larger
//    calls are refused with UMM_ERR_CAPACITY / UMM_ERR_INVALID_ARG before
//    anything is enqueued;
//  - the scratch arrays exist once per GPU that uses this entry point, for
//    the life of the process, and every call on that GPU shares them: two
//    calls whose kernels overlap on the GPU (different streams without an
//    ordering between them) race and may produce wrong results;
//  - the first call on a device (R == 0 included) does the set-up: it looks
//    up the arrays' device addresses and raises the kernel's shared-memory
//    limit.  With CUDA's lazy module loading (the default), that is when the
//    driver loads this file's device code and arrays onto the device, which
//    may take device memory; make that first call at start-up, before any
//    stream capture.  Later calls take no device memory.
#include <mutex>

#include "umm_place.cuh"

namespace {

constexpr int kNoAllocMaxRequests = 16384;
constexpr int kMaxDevices = 64;

// list position -> request index, and the rank per sorted position, one
// entry per request.  They hold no state between calls: every entry a call
// reads is written by that call first.
static __device__ __align__(256) int32_t g_place_scratch[kNoAllocMaxRequests];
static __device__ __align__(256) uint8_t g_place_choice[kNoAllocMaxRequests + 4];

std::mutex g_setup_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};
uint8_t* g_choice_ptr[kMaxDevices] = {};

// The placement of place_requests_tp2ep (same code, same results) with the
// scratch above and the sort keys in shared memory.
__global__ void __launch_bounds__(uk::kScanThreads)
place_noalloc_kernel(int P, int32_t R, const int32_t* __restrict__ lens, const int32_t* __restrict__ list_pos,
                     int32_t* __restrict__ owner, int32_t* __restrict__ local_pos, int32_t* inv, uint8_t* choice,
                     int32_t* status) {
  extern __shared__ unsigned long long keys[];
  const bool ok = uk::place_block(P, R, lens, list_pos, owner, local_pos, inv, choice, keys);
  if (threadIdx.x == 0 && status) *status = ok ? UMM_OK : UMM_ERR_BAD_REQUEST;
}

// Once per device, with that device current: the device addresses of the
// scratch arrays, and the kernel's dynamic shared-memory limit.
int setup_device(int32_t** scratch, uint8_t** choice) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return UMM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    void* c = nullptr;
    if (cudaGetSymbolAddress(&p, g_place_scratch) != cudaSuccess || !p) return UMM_ERR_CUDA;
    if (cudaGetSymbolAddress(&c, g_place_choice) != cudaSuccess || !c) return UMM_ERR_CUDA;
    if (cudaFuncSetAttribute(place_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kNoAllocMaxRequests * (int)sizeof(unsigned long long)) != cudaSuccess)
      return UMM_ERR_CUDA;
    g_choice_ptr[dev] = static_cast<uint8_t*>(c);
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *scratch = g_scratch_ptr[dev];
  *choice = g_choice_ptr[dev];
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
  uint8_t* choice = nullptr;
  const int rc = setup_device(&scratch, &choice);
  if (rc != UMM_OK) return rc;
  if (R == 0) return UMM_OK;
  place_noalloc_kernel<<<1, uk::kScanThreads, (size_t)uk::sort_span(R) * sizeof(unsigned long long),
                         reinterpret_cast<cudaStream_t>(stream)>>>(P, R, d_seq_lens, d_list_pos, d_owner,
                                                                   d_local_pos, scratch, choice, d_status);
  return cudaGetLastError() == cudaSuccess ? UMM_OK : UMM_ERR_CUDA;
}
