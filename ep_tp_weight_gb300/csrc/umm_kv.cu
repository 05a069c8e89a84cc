// Paged KV-cache redistribution EP <-> TP: the gather/scatter copies.
//
// "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
// Switch" (paper review): §3.2 and Fig. 5 (EP keeps all heads of its requests,
// TP a head shard of every request, heads replicated over rank groups when
// there are fewer KV heads than ranks; the page table drives an index vector
// that gathers scattered token slots per destination and scatters them into
// the target pages), §4.3 Table 1 and Fig. 8b (one read and one direct write
// per element).
//
// One launch per layer (kv_copy_*: one CTA per TP page, or per descriptor when
// the pool is sparsely used; layers after the first chained, griddep_wait;
// EP -> TP through TMA when every TP rank holds one head, kv_copy_ep2tp_tma),
// driven by the descriptors of the descriptor pass
// (umm_kv_prep.cu).  Nothing is written to the cache unless that pass raised
// no flag.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "umm_scan.cuh"

namespace uk {

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
  Span span;                   // the P regions
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
  griddep_launch_dependents();
  if (read_flags(p.st)) {
    griddep_wait();
    return;
  }
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
        if (v < nvec && tok[u] < (uint32_t)d.ntok) {
          const uint8_t* const src = src_region + c[u] * p.kv_v_off + src_page + (uint64_t)rem * VB;
          if (access_ok<VB>(p.span, src)) val[u] = ld_vec(reinterpret_cast<const V*>(src));
          else tok[u] = 0xffffffffu;
        } else {
          tok[u] = 0xffffffffu;
        }
      }
      griddep_wait();
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (tok[u] == 0xffffffffu) continue;
        const uint64_t row_off = dst_page + (uint64_t)tok[u] * p.tp_row + (uint64_t)dvv[u] * VB +
                                 c[u] * p.kv_v_off + p.tp_slot;
        if (p.Hkv < p.P) {
          for (uint32_t j = 0; j < p.rep; ++j) {
            const uint32_t q = h[u] * p.rep + j;
            uint8_t* const dst = p.base + (uint64_t)q * p.region_stride + row_off;
            if (access_ok<VB>(p.span, dst)) st_vec(reinterpret_cast<V*>(dst), val[u]);
          }
        } else {
          const uint32_t q = h[u] / p.h_tp, hl = h[u] - q * p.h_tp;
          uint8_t* const dst = p.base + (uint64_t)q * p.region_stride + row_off + (uint64_t)hl * p.head_bytes;
          if (access_ok<VB>(p.span, dst)) st_vec(reinterpret_cast<V*>(dst), val[u]);
        }
      }
    }
  }
  griddep_wait();
}

// TP -> EP: each vector of the destination EP page is read from the lowest TP
// rank holding its head.
template <int VB, int U, int T>
__global__ void __launch_bounds__(T) kv_copy_tp2ep(const KVParams p) {
  using V = typename VecT<VB>::T;
  griddep_launch_dependents();
  if (read_flags(p.st)) {
    griddep_wait();
    return;
  }
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
          const uint8_t* const src = p.base + (uint64_t)q * p.region_stride + p.tp_slot + c[u] * p.kv_v_off +
                                     src_page + (uint64_t)tok * p.tp_row + (uint64_t)hl * p.head_bytes +
                                     (uint64_t)dvv * VB;
          ok[u] = access_ok<VB>(p.span, src) &&
                  access_ok<VB>(p.span, dst_region + c[u] * p.kv_v_off + dst_page + (uint64_t)rem * VB);
          if (ok[u]) val[u] = ld_vec(reinterpret_cast<const V*>(src));
        }
      }
      griddep_wait();
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u])
          st_vec(reinterpret_cast<V*>(dst_region + c[u] * p.kv_v_off + dst_page + (uint64_t)rem_[u] * VB),
                 val[u]);
    }
  }
  griddep_wait();
}

// ------------------------------------------------------------------ EP -> TP through TMA

// When every TP rank holds one head (Hkv <= P), a TP page of one head is
// [ps rows][D] contiguous, while the same head is a strided column of the EP
// page [ps][Hkv][D].  The TMA engine de-interleaves it: one tensor-map load
// per (half, head) brings the head's ps rows of the EP page into a dense
// shared-memory tile, and one bulk store per replica writes the tile's live
// rows to the TP page.  One CTA (one thread issuing) per TP page and half
// (K or V); with Hkv = 4, ps = 16, D = 128 a CTA holds 16 KiB of tiles.
// Measured on GB300 against kv_copy_ep2tp with 32-byte vectors: 6.145 vs
// 6.164 ms per layer (full-switch workload), 3.971 vs 3.989 ms (256 requests
// of 1k-32k tokens), with one CTA per page; one per page and half then
// measured 6.141 vs 6.147 ms and 3.968 vs 3.972 ms.
//
// Tensor coordinates are signed 32-bit.  Each half (K, V) has its own map
// whose dimensions are {element, head, row in page, page, region}, so a load
// is addressed by the page id itself, never by page * page_size: every
// coordinate stays below 2^31 for every pool size the handle accepts
// (kv_pages_tp < 2^31, and pages_ep <= pages_tp).
struct TmaKVParams {
  uint8_t* base;
  const umm_kv_desc* desc;
  const DevStatus* st;
  unsigned int* flags;
  const unsigned long long* sched;
  unsigned int call;
  uint64_t region_stride, kv_v_off, tp_slot;
  uint32_t ps, Hkv, rep, tile_bytes, row_bytes;
  uint32_t tile_stride;   // tile_bytes rounded up to 128 (TMA destination alignment)
  uint32_t stall_polls;   // checked build, tests only: see kv_copy_ep2tp_tma (0 = off)
  long long pages_tp;
  Span span;
};

constexpr uint32_t kTmaWaitTries = 1u << 22;   // bound of each mbarrier wait

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Waits, at most `tries` polls, for the phase `parity` of the mbarrier at
// `bar` to complete; false if it did not.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t tries) {
  for (uint32_t i = 0; i < tries; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__global__ void __launch_bounds__(32) kv_copy_ep2tp_tma(const __grid_constant__ CUtensorMap map_k,
                                                        const __grid_constant__ CUtensorMap map_v,
                                                        const TmaKVParams p) {
  extern __shared__ __align__(1024) uint8_t tiles[];   // [Hkv heads][tile_stride] of half c
  __shared__ __align__(8) unsigned long long bar;
  griddep_launch_dependents();
  if (threadIdx.x != 0) return;
  if (read_flags(p.st)) {
    griddep_wait();
    return;
  }
  const unsigned long long nd = p.sched ? (unsigned long long)p.pages_tp : p.st->ndesc;
  const uint32_t b = smem_addr(&bar);
  const uint32_t t0 = (smem_addr(tiles) + 127u) & ~127u;   // TMA destinations: 128-byte aligned
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  uint32_t parity = 0;
  const uint32_t c = blockIdx.x & 1u;
  const CUtensorMap* const map = c ? &map_v : &map_k;
  for (unsigned long long di = blockIdx.x >> 1; di < nd; di += gridDim.x >> 1) {
    umm_kv_desc d;
    if (p.sched) {
      const unsigned long long e = p.sched[di];
      const unsigned long long idx = e & 0xffffffffull;
      if ((unsigned int)(e >> 32) != p.call || idx >= p.st->ndesc) continue;
      d = p.desc[idx];
    } else {
      d = p.desc[di];
    }
    // loads: tensor coordinates (dim 0 first) {element, head, row in page, page, region}
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(p.Hkv * p.tile_bytes)
                 : "memory");
    for (uint32_t h = 0; h < p.Hkv; ++h)
        asm volatile(
            "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(t0 + h * p.tile_stride),
            "l"(map), "r"(0), "r"((int)h), "r"(0), "r"(d.src_page), "r"(d.src_region), "r"(b)
            : "memory");
    bool landed = mbar_wait(b, parity, kTmaWaitTries);
#ifdef UMM_CHECKED
    // test hook (checked build only): after the loads above have landed, one
    // more wait, on a barrier that expects two arrivals and gets one, which
    // therefore runs out after p.stall_polls polls and takes the timeout exit
    // below with no copy in flight
    if (landed && p.stall_polls) {
      __shared__ __align__(8) unsigned long long never;
      const uint32_t nb = smem_addr(&never);
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;" ::"r"(nb) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(nb) : "memory");
      landed = mbar_wait(nb, 0, p.stall_polls);
    }
#endif
    if (!landed) {
      // Never expected.  Flag it; wait, again at most kTmaWaitTries polls,
      // for this CTA's loads; store nothing and leave.  Later kernels of the
      // call see the flag and do nothing.  Should that wait run out as well,
      // a load may still be writing this CTA's shared memory after it exits:
      // the status (UMM_ERR_TIMEOUT) then tells the caller that this call's
      // KV contents are undefined.
      atomicOr(p.flags, UMM_FLAG_TIMEOUT);
      mbar_wait(b, parity, kTmaWaitTries);
      griddep_wait();
      return;
    }
    parity ^= 1u;
    griddep_wait();
    // stores: the live rows of each head's tile to every TP rank holding it
    const uint32_t nbytes = (uint32_t)d.ntok * p.row_bytes;
    for (uint32_t h = 0; h < p.Hkv; ++h)
        for (uint32_t j = 0; j < p.rep; ++j) {
          uint8_t* const g = p.base + (uint64_t)(h * p.rep + j) * p.region_stride + p.tp_slot + c * p.kv_v_off +
                             (uint64_t)d.dst_page * p.tile_bytes;
          if (range_ok(p.span, g, nbytes))
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(g),
                         "r"(t0 + h * p.tile_stride), "r"(nbytes)
                         : "memory");
        }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // tiles free for the next page
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  griddep_wait();
}

// cuTensorMapEncodeTiled, from the driver through the runtime (no link to
// libcuda); null if the driver does not offer it.  Looked up once per
// process; the static's initialisation is thread-safe, so handles used from
// different host threads may call this at the same time.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return nullptr;
  }();
  return fn;
}

// Shared memory a block gets without an opt-in, static and dynamic together.
constexpr uint64_t kDefaultSmemPerBlock = 48 * 1024;
// The TMA copy's static shared memory: its mbarriers, rounded up to the
// 1024-byte alignment of the tile array that follows (ptxas reports 1024
// bytes).  The launcher checks the kernel's real figure before each launch.
constexpr uint64_t kTmaStaticSmem = 1024;

// Whether the shape lets KV EP->TP run through kv_copy_ep2tp_tma: one head
// per TP rank (Hkv <= P), a head row a multiple of 16 bytes (bulk-copy
// sizes), boxes of at most 256 per dimension, the tiles (plus 128 bytes to
// align them, plus the static part) within the 48 KiB a block gets without
// an opt-in, and every tensor coordinate below 2^31.
bool ep2tp_tma_shape(const Geo& g) {
  const uint64_t tile = (uint64_t)g.ps * (uint64_t)g.D * 2;
  const uint64_t stride = (tile + 127) / 128 * 128;
  const uint64_t smem = (uint64_t)g.Hkv * stride;
  return g.Hkv >= 1 && g.Hkv <= g.P && g.D <= 256 && g.ps <= 256 && (g.D * 2) % 16 == 0 &&
         smem + 128 + kTmaStaticSmem <= kDefaultSmemPerBlock && g.pages_ep >= 1 && g.pages_ep <= 0x7fffffffll &&
         g.P <= 0x7fffffff;
}

// The TMA copy's static shared memory as the runtime reports it (looked up
// once; the initialisation of the static is thread-safe), or ~0 if the
// lookup fails, which sends every shape to the LSU copy.
uint64_t tma_static_smem() {
  static const uint64_t bytes = []() -> uint64_t {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kv_copy_ep2tp_tma) != cudaSuccess) {
      cudaGetLastError();
      return ~0ull;
    }
    return (uint64_t)fa.sharedSizeBytes;
  }();
  return bytes;
}

// Launches the TMA copy for one layer when the shape allows it; *done = false
// (nothing enqueued) otherwise, and the caller uses kv_copy_ep2tp.
cudaError_t launch_ep2tp_tma(const Geo& g, const KVParams& p, int layer, int64_t max_desc, cudaStream_t s,
                             bool chained, uint32_t stall_polls, bool* done) {
  *done = false;
  if (!ep2tp_tma_shape(g) || max_desc <= 0) return cudaSuccess;
  const uint64_t tile = (uint64_t)g.ps * (uint64_t)g.D * 2;
  const uint64_t stride = (tile + 127) / 128 * 128;
  const uint64_t smem = (uint64_t)g.Hkv * stride;
  const uint64_t stat = tma_static_smem();
  if (stat > kDefaultSmemPerBlock || smem + 128 + stat > kDefaultSmemPerBlock) return cudaSuccess;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaSuccess;
  // the EP view of layer `layer` in every region, one map per half (K, V):
  // [region][page][row in page][head][element]
  CUtensorMap map[2];
  const cuuint64_t dims[5] = {(cuuint64_t)g.D, (cuuint64_t)g.Hkv, (cuuint64_t)g.ps, (cuuint64_t)g.pages_ep,
                              (cuuint64_t)g.P};
  const cuuint64_t row = (cuuint64_t)g.Hkv * g.D * 2;
  const cuuint64_t strides[4] = {(cuuint64_t)g.D * 2, row, row * (cuuint64_t)g.ps, (cuuint64_t)g.region_stride};
  const cuuint32_t box[5] = {(cuuint32_t)g.D, 1, (cuuint32_t)g.ps, 1, 1};
  const cuuint32_t unit[5] = {1, 1, 1, 1, 1};
  uint8_t* const ep_slot = g.base + g.kvslots_off + (uint64_t)(layer + 1) * g.kvslot_stride;
  for (int c = 0; c < 2; ++c)
    if (encode(&map[c], CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, ep_slot + (uint64_t)c * g.kv_v_off, dims, strides, box,
               unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaSuccess;
  TmaKVParams t;
  t.base = g.base;
  t.desc = p.desc;
  t.st = p.st;
  t.flags = g.flags;
  t.sched = p.sched;
  t.call = p.call;
  t.region_stride = g.region_stride;
  t.kv_v_off = g.kv_v_off;
  t.tp_slot = p.tp_slot;
  t.ps = (uint32_t)g.ps;
  t.Hkv = (uint32_t)g.Hkv;
  t.rep = p.rep;
  t.tile_bytes = (uint32_t)tile;
  t.tile_stride = (uint32_t)stride;
  t.row_bytes = (uint32_t)g.D * 2;
  t.stall_polls = stall_polls;
  t.pages_tp = g.pages_tp;
  t.span = g.regions();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * max_desc < 0x7fffffffll ? 2 * max_desc : 0x7ffffffell));
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = (size_t)smem + 128;   // room to align the tiles
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = chained ? 1 : 0;
  *done = true;
  return cudaLaunchKernelEx(&cfg, kv_copy_ep2tp_tma, map[0], map[1], t);
}

namespace {
// Threads and vectors per thread of the copies; one round of a CTA loads
// 16 KiB in every shape below.  Picked by
// measurement on GB300, full-switch workload, ms per layer EP->TP / TP->EP:
//   16-byte vectors, 128 x 8 / 256 x 4 (the best 16-byte shapes): 6.211 / 4.131
//   32-byte vectors: EP->TP 64 x 8: 6.170, 32 x 8: 6.190, 64 x 4: 6.189,
//   128 x 4: 6.195, 256 x 2: 6.196, 96 x 8: 6.211, 128 x 8: 6.211;
//   TP->EP 256 x 2: 4.015, 128 x 4: 4.027, 256 x 4: 4.053, 512 x 1: 4.226.
// 32-byte vectors are used whenever the head size allows them.
template <int VB>
struct Shape {
  static constexpr int T_ep2tp = VB == 32 ? 64 : 128, U_ep2tp = 8;
  static constexpr int T_tp2ep = 256, U_tp2ep = VB == 32 ? 2 : 4;
};

// One CTA per descriptor (grid >= live pages): the block scheduler hands a
// finished CTA's slot to the next page at once, which keeps more loads in
// flight per SM than a persistent grid striding over the descriptors
// (measured on GB300: ~6.72 vs ~6.13 TB/s EP->TP at the full-switch size).
// The kernels still stride by gridDim.x, so any grid size is correct.
template <int VB>
cudaError_t run_copy(const KVParams& p, int dir, int64_t max_desc, cudaStream_t s, bool chained) {
  if (max_desc <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)(max_desc < 0x7fffffffll ? max_desc : 0x7fffffffll);
  using S = Shape<VB>;
  if (dir == 0) return launch_chain(kv_copy_ep2tp<VB, S::U_ep2tp, S::T_ep2tp>, grid, S::T_ep2tp, s, chained, p);
  return launch_chain(kv_copy_tp2ep<VB, S::U_tp2ep, S::T_tp2ep>, grid, S::T_tp2ep, s, chained, p);
}
}  // namespace

int kv_vector_bytes(const Geo& g) {
  if (g.D % 16 == 0) return 32;
  if (g.D % 8 == 0) return 16;
  if (g.D % 4 == 0) return 8;
  if (g.D % 2 == 0) return 4;
  return 2;
}

cudaError_t launch_kv_copy(const Geo& g, const Ws& w, int dir, int layer, int64_t max_desc, int use_sched,
                           unsigned int call, cudaStream_t s, bool chained, bool allow_tma, uint32_t stall_polls) {
  const int VB = kv_vector_bytes(g);
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
  p.span = g.regions();
  if (dir == 0 && allow_tma) {
    bool done = false;
    const cudaError_t e = launch_ep2tp_tma(g, p, layer, max_desc, s, chained, stall_polls, &done);
    if (done || e != cudaSuccess) return e;
  }
  switch (VB) {
    case 32: return run_copy<32>(p, dir, max_desc, s, chained);
    case 16: return run_copy<16>(p, dir, max_desc, s, chained);
    case 8: return run_copy<8>(p, dir, max_desc, s, chained);
    case 4: return run_copy<4>(p, dir, max_desc, s, chained);
    default: return run_copy<2>(p, dir, max_desc, s, chained);
  }
}

}  // namespace uk
