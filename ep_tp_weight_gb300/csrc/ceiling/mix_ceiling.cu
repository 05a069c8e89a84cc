// Ceilings of HBM read:write mixes on one GPU: what a plain streaming copy
// reaches for the access pattern of each reshard kernel, so that a kernel's
// rate can be read against the mix it must move rather than against a 1:1
// copy.  A standalone program (not part of libumm), built and run by
// `python bench.py --ceilings`; one JSON line per case on stdout.
//
// Every case moves 16 KiB per CTA (256 threads x 2 x 32-byte vectors), one
// CTA per chunk, over buffers of 8 GiB each by default (64x the L2), with the
// default cache policy:
//   read sequential / shuffled: CTA b reads source chunk b, or chunk perm[b]
//   (a fixed random permutation of the chunks: scattered 16 KiB pages);
//   write sequential / shuffled: likewise for the destination chunk;
//   nd destinations: the chunk is stored to nd buffers (replicas).
// Mapping to the reshard kernels: weights and attention EP->TP = 1 read,
// 1 write, sequential; KV EP->TP = shuffled reads, 2 writes (two replicas of
// each head); KV TP->EP = sequential reads, shuffled writes; attention
// TP->EP = 1 read, 8 writes (all-gather into every rank's full copy).
// Cases 7-9 are the other orders KV EP->TP could walk its pages in: each
// 16 KiB read split into 4 KiB pieces written to shuffled places (the same
// place in both destinations, as a head's two replicas share a TP page id).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>

namespace {

struct alignas(32) u256 {
  uint32_t w[8];
};

__device__ __forceinline__ u256 ld32(const u256* p) {
  u256 v;
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                 "=r"(v.w[6]), "=r"(v.w[7])
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st32(u256* p, const u256& v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :
               : "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]),
                 "r"(v.w[6]), "r"(v.w[7])
               : "memory");
}

constexpr int kT = 256, kU = 2, kMaxDst = 8;
constexpr size_t kChunkVec = (size_t)kT * kU;   // 32-byte vectors per chunk
constexpr size_t kChunk = kChunkVec * 32;       // 16 KiB

struct Dsts {
  u256* d[kMaxDst];
};

// wpiece: vectors per shuffled write piece (kChunkVec: whole 16 KiB chunks;
// kChunkVec / 4: 4 KiB pieces, wperm then permutes pieces, not chunks)
__global__ void __launch_bounds__(kT) mix_copy(const u256* src, Dsts dst, int nd, const uint32_t* rperm,
                                               const uint32_t* wperm, uint32_t wpiece, uint32_t nchunks) {
  const uint32_t b = blockIdx.x;
  if (b >= nchunks) return;
  const uint32_t rc = rperm ? rperm[b] : b;
  const u256* s = src + (size_t)rc * kChunkVec;
  u256 v[kU];
  size_t at[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const uint32_t i = threadIdx.x + u * kT;   // vector in the chunk
    v[u] = ld32(s + i);
    const size_t piece = (size_t)b * (kChunkVec / wpiece) + i / wpiece;
    at[u] = (wperm ? (size_t)wperm[piece] : piece) * wpiece + i % wpiece;
  }
#pragma unroll
  for (int k = 0; k < kMaxDst; ++k) {
    if (k < nd) {
#pragma unroll
      for (int u = 0; u < kU; ++u) st32(dst.d[k] + at[u], v[u]);
    }
  }
}

// The 1R1W sequential case through TMA: one thread per CTA bulk-loads its
// 16 KiB chunk into shared memory (mbarrier, bounded wait) and bulk-stores it.
__global__ void __launch_bounds__(32) bulk_copy(const u256* src, u256* dst, uint32_t nchunks) {
  extern __shared__ __align__(128) uint8_t buf[];
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x != 0 || blockIdx.x >= nchunks) return;
  const uint32_t s0 = ((uint32_t)__cvta_generic_to_shared(buf) + 127u) & ~127u;
  const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
  const u256* from = src + (size_t)blockIdx.x * kChunkVec;
  u256* to = dst + (size_t)blockIdx.x * kChunkVec;
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"((uint32_t)kChunk) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(s0), "l"(from), "r"((uint32_t)kChunk), "r"(b)
               : "memory");
  for (uint32_t i = 0; i < (1u << 22); ++i) {   // bounded wait for the load
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
                 "selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done)
                 : "r"(b)
                 : "memory");
    if (done) {
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(to), "r"(s0),
                   "r"((uint32_t)kChunk)
                   : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      return;
    }
  }
  for (uint32_t i = 0; i < (1u << 22); ++i) {   // never expected: wait as long again for the load, then leave
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
                 "selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done)
                 : "r"(b)
                 : "memory");
    if (done) return;
  }
}

struct Case {
  const char* name;
  const char* kernels;   // reshard kernels with this pattern
  int nd;
  bool shuffled_reads, shuffled_writes;
  bool tma = false;      // bulk_copy instead of mix_copy (1R1W sequential only)
  bool pieces4k = false; // shuffled writes in 4 KiB pieces instead of 16 KiB chunks
};

}  // namespace

#define CK(x)                                                                        \
  do {                                                                               \
    cudaError_t e_ = (x);                                                            \
    if (e_ != cudaSuccess) {                                                         \
      std::fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                                      \
    }                                                                                \
  } while (0)

int main(int argc, char** argv) {
  // argv[1]: GiB per buffer (1..16, default 8); argv[2] (optional): run only
  // case k of the list below (0..9), allocating only the buffers it uses
  const int gib = argc > 1 ? std::max(1, std::min(16, std::atoi(argv[1]))) : 8;
  const int only = argc > 2 ? std::atoi(argv[2]) : -1;
  const size_t S = (size_t)gib << 30;
  const uint32_t n = (uint32_t)(S / kChunk);
  u256* src = nullptr;
  Dsts dst{};
  uint32_t *rperm = nullptr, *wperm = nullptr;
  CK(cudaMalloc(&src, S));
  CK(cudaMemset(src, 0x5a, S));
  const int ndst = only == 0 || only == 1 || only == 2 || only == 6 ? 1
                   : only == 3 || only == 4 || only >= 7   ? 2
                                                          : kMaxDst;
  for (int k = 0; k < ndst; ++k) {
    CK(cudaMalloc(&dst.d[k], S));
    CK(cudaMemset(dst.d[k], 0, S));
  }
  std::vector<uint32_t> p1(n), p2(n), p3((size_t)n * 4);
  for (uint32_t i = 0; i < n; ++i) p1[i] = p2[i] = i;
  for (uint32_t i = 0; i < 4 * n; ++i) p3[i] = i;
  std::mt19937_64 rng(20251);
  std::shuffle(p1.begin(), p1.end(), rng);
  std::shuffle(p2.begin(), p2.end(), rng);
  std::shuffle(p3.begin(), p3.end(), rng);
  uint32_t* wperm4 = nullptr;
  CK(cudaMalloc(&rperm, (size_t)n * 4));
  CK(cudaMalloc(&wperm, (size_t)n * 4));
  CK(cudaMalloc(&wperm4, (size_t)n * 16));
  CK(cudaMemcpy(rperm, p1.data(), (size_t)n * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(wperm, p2.data(), (size_t)n * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(wperm4, p3.data(), (size_t)n * 16, cudaMemcpyHostToDevice));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  const Case cases[] = {
      {"1R1W sequential", "weights_kernel, attn_kernel EP->TP", 1, false, false},
      {"1R1W shuffled reads", "", 1, true, false},
      {"1R1W shuffled writes", "kv_copy_tp2ep", 1, false, true},
      {"1R2W sequential", "", 2, false, false},
      {"1R2W shuffled reads", "kv_copy_ep2tp", 2, true, false},
      {"1R8W sequential", "attn_kernel TP->EP", 8, false, false},
      {"1R1W sequential, TMA bulk copies", "", 1, false, false, true},
      {"1R2W shuffled writes", "", 2, false, true},
      {"1R2W shuffled 4 KiB writes", "", 2, false, true, false, true},
      {"1R2W shuffled reads, shuffled 4 KiB writes", "", 2, true, true, false, true},
  };
  const int reps = 10;
  for (int ci = 0; ci < (int)(sizeof(cases) / sizeof(cases[0])); ++ci) {
    if (only >= 0 && ci != only) continue;
    const Case& c = cases[ci];
    const uint32_t* rp = c.shuffled_reads ? rperm : nullptr;
    const uint32_t* wp = c.shuffled_writes ? (c.pieces4k ? wperm4 : wperm) : nullptr;
    const uint32_t wpiece = c.pieces4k ? (uint32_t)(kChunkVec / 4) : (uint32_t)kChunkVec;
    auto launch = [&]() {
      if (c.tma) bulk_copy<<<n, 32, kChunk + 128>>>(src, dst.d[0], n);
      else mix_copy<<<n, kT>>>(src, dst, c.nd, rp, wp, wpiece, n);
    };
    for (int w = 0; w < 3; ++w) launch();
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(e0));
    for (int r = 0; r < reps; ++r) launch();
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double per = ms / reps, bytes = (double)S * (1 + c.nd);
    std::printf("{\"ceiling\": \"%s\", \"kernels\": \"%s\", \"read_bytes\": %zu, \"write_bytes\": %zu, "
                "\"ms_per_launch\": %.4f, \"GB_s\": %.1f}\n",
                c.name, c.kernels, S, S * (size_t)c.nd, per, bytes / (per * 1e-3) / 1e9);
  }
  for (int k = 0; k < ndst; ++k) CK(cudaFree(dst.d[k]));
  CK(cudaFree(src));
  CK(cudaFree(rperm));
  CK(cudaFree(wperm));
  CK(cudaFree(wperm4));
  return 0;
}
