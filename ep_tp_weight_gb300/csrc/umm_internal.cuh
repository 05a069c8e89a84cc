// Internal declarations shared by the libumm translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "umm.h"

namespace uk {

constexpr int kMaxGroups = 64;     // bound on P and on page-pool counts
constexpr int kScanThreads = 1024; // threads of the single-CTA metadata kernels

// Division by a runtime constant 1 <= d < 2^31 for numerators n < 2^31, by
// multiply-high (round-up method, Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994).  With
// s = ceil(log2 d) >= 1 and m = ceil(2^(31+s) / d) (< 2^32):
//   n*m / 2^(31+s) = n/d + eps, 0 <= eps < n / 2^(31+s) < 2^-s <= 1/d,
// which never carries the fraction of n/d past an integer, so
//   floor(n/d) = umulhi(n, m) >> (s-1).   d == 1 is passed through.
struct FastDiv {
  uint32_t d, m, sh;
  FastDiv() = default;
  __host__ explicit FastDiv(uint32_t div) : d(div), m(0), sh(0) {
    if (div <= 1) return;
    uint32_t s = 0;
    while ((1ull << s) < div) ++s;
    m = (uint32_t)(((1ull << (31 + s)) + div - 1) / div);
    sh = s - 1;
  }
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    return d <= 1 ? n : (__umulhi(n, m) >> sh);
#else
    return d <= 1 ? n : (uint32_t)(((uint64_t)n * m) >> 32) >> sh;
#endif
  }
  __host__ __device__ __forceinline__ void divmod(uint32_t n, uint32_t& q, uint32_t& r) const {
    q = div(n);
    r = n - q * d;
  }
};

// Vector type moved per access (VB bytes); data is never interpreted.
template <int VB> struct VecT;
template <> struct VecT<16> { using T = uint4; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<4> { using T = uint32_t; };
template <> struct VecT<2> { using T = unsigned short; };

// 32-byte vectors: 256-bit global loads and stores (sm_100 and later).
struct alignas(32) u256 {
  uint32_t w[8];
};
template <> struct VecT<32> { using T = u256; };

// Vector loads and stores with the default cache policy.  The streaming
// (evict-first, .cs) hints were measured on GB300 against it: the same for the
// KV and attention copies, while the weights copy inside the full-switch
// buffer ran 0.350 ms per layer with them and 0.342 ms without (plain loads
// with streaming stores: 0.361 ms).
template <typename V>
__device__ __forceinline__ V ld_vec(const V* p) {
  return *p;
}
template <>
__device__ __forceinline__ u256 ld_vec<u256>(const u256* p) {
  u256 v;
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                 "=r"(v.w[6]), "=r"(v.w[7])
               : "l"(p));
  return v;
}
template <typename V>
__device__ __forceinline__ void st_vec(V* p, const V& v) {
  *p = v;
}
template <>
__device__ __forceinline__ void st_vec<u256>(u256* p, const u256& v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :
               : "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]),
                 "r"(v.w[6]), "r"(v.w[7])
               : "memory");
}

// Programmatic dependent launch (griddepcontrol, sm_90 and later).  The layer
// copies of one reshard call run as a chain: layer k+1 is launched with
// programmatic stream serialization, so its CTAs may start while layer k's
// last wave drains.  Layer k+1 only reads a slot that no launch of the chain
// writes (ascending: EP slot k+2; descending: TP slot k-1), so it loads before
// waiting; it writes the slot layer k reads, so every store comes after
// griddep_wait(), which returns once the previous grid has completed and its
// memory is visible (at once when the launch carried no such attribute).
// Every CTA passes griddep_wait() before it exits, so a chained grid never
// completes ahead of its predecessor.  A hardware dependency, not a spin.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches kern<<<grid, block, 0, s>>>(args...), as a programmatic dependent
// of the previous launch on s when `chained`.
template <typename... KArgs, typename... Args>
cudaError_t launch_chain(void (*kern)(KArgs...), unsigned grid, unsigned block, cudaStream_t s, bool chained,
                         Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = chained ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Device view of the workspace status block.
struct DevStatus {
  unsigned int flags;
  unsigned int fail_call;
  unsigned long long ndesc;
  unsigned long long tokens;
  unsigned long long reserved[5];
};
static_assert(sizeof(DevStatus) == sizeof(umm_status_block), "status block layout");

__device__ __forceinline__ void raise_flag(DevStatus* st, unsigned int flag, unsigned int call) {
  atomicOr(&st->flags, flag);
  atomicCAS(&st->fail_call, 0u, call);
}

// Pages of a request of `len` tokens (len >= 0), without int32 overflow for
// lengths near 2^31.
__device__ __forceinline__ int pages_of(int32_t len, int32_t ps) {
  return (int)(((long long)len + ps - 1) / ps);
}

// The buffer a kernel's vector accesses must lie in.  In the checked build
// (UMM_CHECKED) every access is tested against it and against the vector's
// alignment; a failing access is skipped and raises UMM_FLAG_ACCESS.  In the
// normal build the test compiles away.
struct Span {
  const uint8_t* lo;
  const uint8_t* hi;
  unsigned int* flags;
};

template <int VB>
__device__ __forceinline__ bool access_ok(const Span& s, const void* a) {
#ifdef UMM_CHECKED
  const uint8_t* b = static_cast<const uint8_t*>(a);
  if (b < s.lo || b + VB > s.hi || (reinterpret_cast<uintptr_t>(b) & (uintptr_t)(VB - 1))) {
    atomicOr(s.flags, UMM_FLAG_ACCESS);
    return false;
  }
#else
  (void)s;
  (void)a;
#endif
  return true;
}

// The same test for an n-byte bulk (TMA) copy starting at a (16-byte aligned).
__device__ __forceinline__ bool range_ok(const Span& s, const void* a, uint64_t n) {
#ifdef UMM_CHECKED
  const uint8_t* b = static_cast<const uint8_t*>(a);
  if (b < s.lo || b + n > s.hi || (reinterpret_cast<uintptr_t>(b) & 15u) || (n & 15u)) {
    atomicOr(s.flags, UMM_FLAG_ACCESS);
    return false;
  }
#else
  (void)s;
  (void)a;
  (void)n;
#endif
  return true;
}

// Everything a kernel needs to address the unified buffer.
struct Geo {
  uint8_t* base;
  uint64_t region_stride, wslot_stride, w13_off, w2_off;
  uint64_t kvslot_stride, kv_v_off, kvslots_off;
  int32_t P, E, H, I, N, Hkv, D, ps, w13_split, Hq;
  int64_t pages_ep, pages_tp, h_tp;
  uint64_t attnslot_stride, attn_wo_off, attnslots_off;
  unsigned int* flags;     // the workspace status block's flags word

  // the P regions: every fused copy stays inside them
  __host__ __device__ Span regions() const {
    return Span{base, base + (uint64_t)P * region_stride, flags};
  }
};

// Workspace carve-up (byte offsets from the buffer base).
struct Ws {
  uint64_t status;     // DevStatus
  uint64_t desc;       // umm_kv_desc[desc_cap]
  int64_t desc_cap;
  uint64_t req_off;    // int64[max_requests]   per-request start offsets
  uint64_t req_inv;    // int32[max_requests]   list position -> request
  uint64_t keys;       // uint64[keys_cap]      sort keys (placement)
  int64_t keys_cap;    // power of two >= max_requests
  uint64_t choice;     // uint8[max_requests]   placement: rank per sorted position
  uint64_t bitmap;     // uint32[bitmap_words]  destination-page use bits
  int64_t bitmap_words;
  uint64_t tp_bitmap;  // uint32[(pages_tp+31)/32] TP source pages read by TP->EP
  uint64_t sched;      // uint64[pages_tp]      TP page -> (call << 32 | descriptor)
  uint64_t order_tok;  // int64[max_requests]   staged path: token offsets in rank order
  uint64_t rank_info;  // int64[3 * kMaxGroups] staged path: per-rank descriptor/token counts
  int32_t max_requests;
};

// ---- launchers (enqueue only; all arguments already validated) ----
// chained: launch as a programmatic dependent of the previous layer's copy
// (griddep_wait above); false for the first layer of a call.
cudaError_t launch_attn(const Geo& g, int ep2tp, int layer, cudaStream_t s, bool chained);
cudaError_t launch_weights(const Geo& g, int ep2tp, int layer, cudaStream_t s, bool chained);
// The staged comparison path (permute + exchange through `stage`).
uint64_t weights_stage_bytes(const Geo& g);
cudaError_t launch_weights_staged(const Geo& g, int ep2tp, int layer, uint8_t* stage, cudaStream_t s,
                                  int* launches);

// use_sched: also index the descriptors by TP page (see launch_kv_copy).
cudaError_t launch_kv_prep(const Geo& g, const Ws& w, int dir, int32_t R, int32_t maxp,
                           const int32_t* lens, const int32_t* owner, const int32_t* ep_pt,
                           const int32_t* tp_pt, unsigned int call, int use_sched, cudaStream_t s, int sms);
// max_desc: an upper bound on the descriptors of the call.  With use_sched
// the grid walks the TP page pool (descriptors in TP-page order, empty pages
// exit at once); otherwise it walks the descriptor list.  stall_polls (checked
// build, tests only): the TMA copy's extra wait that runs out (0 = off).
cudaError_t launch_kv_copy(const Geo& g, const Ws& w, int dir, int layer, int64_t max_desc, int use_sched,
                           unsigned int call, cudaStream_t s, bool chained, bool allow_tma = true,
                           uint32_t stall_polls = 0);
// Host-side choices of launch_kv_copy: whether KV EP->TP can run through the
// TMA copy, and the vector width (bytes) of the LSU copies.
bool ep2tp_tma_shape(const Geo& g);
int kv_vector_bytes(const Geo& g);

// The staged comparison path for the KV cache (gather -> exchange -> scatter
// per rank through `stage`; the descriptor pass must have run first).
uint64_t kv_stage_bytes(const Geo& g);
cudaError_t launch_kv_staged(const Geo& g, const Ws& w, int dir, int32_t R, const int32_t* lens,
                             const int32_t* owner, uint8_t* stage, int64_t* order_tok, int64_t* rank_info,
                             unsigned int call, cudaStream_t s, int sms, int* launches);

cudaError_t launch_order(const Geo& g, const Ws& w, int32_t R, const int32_t* owner, int32_t* tp_pos,
                         unsigned int call, cudaStream_t s);
cudaError_t launch_place(const Geo& g, const Ws& w, int32_t R, const int32_t* lens,
                         const int32_t* list_pos, int32_t* owner, int32_t* local_pos,
                         unsigned int call, cudaStream_t s);
cudaError_t launch_assign(const Geo& g, const Ws& w, int32_t npools, int32_t R, const int32_t* lens,
                          const int32_t* pool, const int32_t* key, const int32_t* free_pages,
                          int64_t free_stride, int64_t free_count, int32_t* pt, int32_t maxp,
                          unsigned int call, cudaStream_t s, int sms);

}  // namespace uk
