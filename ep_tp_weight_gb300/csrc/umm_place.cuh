// TP->EP request placement, shared by place_requests_tp2ep (scratch in a
// unified buffer's workspace) and place_requests_tp2ep_noalloc (scratch in
// the library's own device memory).
//
// "Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
// Switch" (paper review), §3.2: the request list is sorted by sequence length,
// longest first, and each request goes to the least-loaded rank; the rule is
// deterministic, so every rank computes the same partition without
// communicating.  Ties: equal lengths keep list order, equal loads go to the
// lowest rank; a rank's requests keep list order (local positions).
#pragma once

#include "umm_scan.cuh"

namespace uk {

// ------------------------------------------------------------------ shared checks

// inv[pos] = k for the list positions pos = key[k]; returns false unless the
// keys are a permutation of 0..R-1.  Block-wide; all threads return the same.
static __device__ bool build_inverse(const int32_t* __restrict__ key, int32_t R, int32_t* inv, int* bad_flag) {
  for (int k = threadIdx.x; k < R; k += blockDim.x) {
    const int pos = key[k];
    if (pos < 0 || pos >= R) *bad_flag = 1;
    else inv[pos] = k;
  }
  __syncthreads();
  if (!*bad_flag)
    for (int k = threadIdx.x; k < R; k += blockDim.x)
      if (inv[key[k]] != k) *bad_flag = 1;   // a repeated position left another k there
  __syncthreads();
  return *bad_flag == 0;
}

// ------------------------------------------------------------------ placement (TP -> EP)

// Greedy list scheduling over the sorted keys, one thread.  Each rank's load
// is packed with its index, (load << S) | q, so keys are unique and the
// smallest key is the least-loaded rank with ties towards the lowest rank.
// The P keys are kept sorted in registers: the head a[0] is the rank chosen
// for the next request; its key grows by the request's length and is merged
// back into a[1..] by one min/max per position, b[i] = max(a[i],
// min(a[i+1], x)).  The loop-carried chain is one add and one min, and the
// other positions update in parallel.  Requests go in batches of four: the
// next batch's keys are loaded while this one runs, and the four choices
// (choice[i] = rank of sorted position i) are stored as one word.  Past the
// last request the increment is 0, which leaves the sorted keys as they are.
template <typename Word, int PB, int S>
__device__ void greedy_sorted(const unsigned long long* __restrict__ keys, int32_t R, int P,
                              uint32_t* __restrict__ choice4) {
  Word a[PB];
#pragma unroll
  for (int q = 0; q < PB; ++q) a[q] = q < P ? (Word)q : (Word)~(Word)0;
  unsigned long long nk[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) nk[u] = u < R ? keys[u] : 0ull;
  for (int i0 = 0; i0 < R; i0 += 4) {
    unsigned long long kk[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      kk[u] = nk[u];
      nk[u] = i0 + 4 + u < R ? keys[i0 + 4 + u] : 0ull;
    }
    uint32_t pack = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const Word inc = i0 + u < R ? (Word)(0x7fffffffull - (kk[u] >> 32)) << S : (Word)0;
      pack |= (uint32_t)(a[0] & (Word)((1u << S) - 1u)) << (8 * u);
      const Word x = a[0] + inc;
      a[0] = a[1] < x ? a[1] : x;
#pragma unroll
      for (int q = 1; q < PB - 1; ++q) {
        const Word lo = a[q + 1] < x ? a[q + 1] : x;
        a[q] = a[q] > lo ? a[q] : lo;
      }
      a[PB - 1] = a[PB - 1] > x ? a[PB - 1] : x;
    }
    choice4[i0 >> 2] = pack;
  }
}

// The variants out of line, so that each gets the kernel's whole register
// budget and none weighs on the others.
static __device__ __noinline__ void greedy_sorted8(const unsigned long long* __restrict__ keys, int32_t R, int P,
                                            uint32_t* __restrict__ choice4) {
  greedy_sorted<uint32_t, 8, 3>(keys, R, P, choice4);
}

static __device__ __noinline__ void greedy_sorted16(const unsigned long long* __restrict__ keys, int32_t R, int P,
                                             uint32_t* __restrict__ choice4) {
  greedy_sorted<uint32_t, 16, 4>(keys, R, P, choice4);
}

static __device__ __noinline__ void greedy_sorted_wide16(const unsigned long long* __restrict__ keys, int32_t R, int P,
                                                  uint32_t* __restrict__ choice4) {
  greedy_sorted<unsigned long long, 16, 6>(keys, R, P, choice4);
}

// The same rule with one rank per lane of a warp (P <= 32, 32-bit packed
// loads): the least-loaded rank of each step is one warp reduce-min.
template <int S>
__device__ void greedy_warp(const unsigned long long* __restrict__ keys, int32_t R, int P,
                            uint32_t* __restrict__ choice4) {
  const int lane = threadIdx.x & 31;
  uint32_t k = lane < P ? (uint32_t)lane : 0xffffffffu;
  uint32_t pack = 0;
  unsigned long long next = R > 0 ? keys[0] : 0ull;
  for (int i = 0; i < R; ++i) {
    const unsigned long long key = next;
    if (i + 1 < R) next = keys[i + 1];
    const uint32_t len = (uint32_t)(0x7fffffffull - (key >> 32));
    const uint32_t m = __reduce_min_sync(0xffffffffu, k);
    const int best = (int)(m & ((1u << S) - 1u));
    if (lane == best) k += len << S;
    pack |= (uint32_t)best << (8 * (i & 3));
    if ((i & 3) == 3 || i + 1 == R) {
      if (lane == 0) choice4[i >> 2] = pack;
      pack = 0;
    }
  }
}

// The same rule for P > 16, with the loads in local memory.
static __device__ __noinline__ void greedy_wide(const unsigned long long* __restrict__ keys, int32_t R, int P,
                                         uint32_t* __restrict__ choice4) {
  unsigned long long k[kMaxGroups];
  for (int q = 0; q < P; ++q) k[q] = (unsigned long long)q;
  uint32_t pack = 0;
  for (int i = 0; i < R; ++i) {
    const unsigned long long len = 0x7fffffffull - (keys[i] >> 32);
    unsigned long long m = k[0];
    for (int q = 1; q < P; ++q) m = k[q] < m ? k[q] : m;
    const int best = (int)(m & 63u);
    k[best] += len << 6;
    pack |= (uint32_t)best << (8 * (i & 3));
    if ((i & 3) == 3 || i + 1 == R) {
      choice4[i >> 2] = pack;
      pack = 0;
    }
  }
}

// Compare-exchange of two register-held keys that are `S` apart inside a
// thread (elements e and e + S): ascending when `up`.
template <int E, int S>
__device__ __forceinline__ void cx_local(unsigned long long (&x)[E], int t, int size) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (e & S) continue;
    const bool up = (((t * E + e) & size) == 0);
    const unsigned long long lo = x[e] < x[e + S] ? x[e] : x[e + S];
    const unsigned long long hi = x[e] < x[e + S] ? x[e + S] : x[e];
    x[e] = up ? lo : hi;
    x[e + S] = up ? hi : lo;
  }
}

// Bitonic sort, ascending, of the E * blockDim.x keys in keys[] (thread t
// holds elements t*E .. t*E+E-1 in registers).  Exchanges between elements
// of one thread stay in registers, between threads of one warp go through
// shuffles, and only the wider ones through shared memory.  Every thread
// runs the same sequence of stages, so every shuffle and barrier is reached
// by the whole block.
template <int E>
static __device__ __noinline__ void sort_keys_regs(unsigned long long* keys) {
  const int t = threadIdx.x;
  const int n = E * (int)blockDim.x;
  unsigned long long x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = keys[t * E + e];
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * E) {
        __syncthreads();                       // earlier readers of keys[] are done
#pragma unroll
        for (int e = 0; e < E; ++e) keys[t * E + e] = x[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int gi = t * E + e;
          const unsigned long long v = keys[gi ^ stride];
          const bool keep_min = ((gi & stride) == 0) == ((gi & size) == 0);
          x[e] = keep_min ? (v < x[e] ? v : x[e]) : (v < x[e] ? x[e] : v);
        }
      } else if (stride >= E) {
        const int lanes = stride / E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int gi = t * E + e;
          const unsigned long long v = __shfl_xor_sync(0xffffffffu, x[e], lanes);
          const bool keep_min = ((gi & stride) == 0) == ((gi & size) == 0);
          x[e] = keep_min ? (v < x[e] ? v : x[e]) : (v < x[e] ? x[e] : v);
        }
      } else {
        if constexpr (E > 2) if (stride == 2) cx_local<E, (E > 2 ? 2 : 1)>(x, t, size);
        if constexpr (E > 1) if (stride == 1) cx_local<E, 1>(x, t, size);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e) keys[t * E + e] = x[e];
  __syncthreads();
}

// Elements per thread of the register sort for R keys; 0 selects the
// bitonic network in memory, which measured faster from 8 elements per thread
// on (GB300: 8192 keys 192k vs 231k cycles, 16384 keys 411k vs 748k, the
// register version spilling), while the register sort wins below (2048
// keys: 33k vs 45k cycles).
__host__ __device__ __forceinline__ int sort_elems(int32_t R) {
  return R <= 1024 ? 1 : R <= 2048 ? 2 : R <= 4096 ? 4 : 0;
}

// Keys the sort covers: E * 1024 for the register sort, else the next power
// of two; they sit in shared memory up to 16 x 1024 keys.
__host__ __device__ __forceinline__ int sort_span(int32_t R) {
  int n2 = 1;
  while (n2 < R) n2 <<= 1;
  const int E = sort_elems(R);
  return E ? E * kScanThreads : n2;
}

// ------------------------------------------------------------------ the whole placement, one CTA

// One CTA of kScanThreads threads places R requests on P ranks: owner[k] and
// local_pos[k] for request k (lens[k] tokens; list position list_pos[k], or
// k when list_pos is null).  Scratch: inv (R entries, list position ->
// request), choice (R + 4 bytes, rank per sorted position), keys (sort_span(R)
// entries, shared memory when they fit, else global).  Returns false, the
// same in every thread and before anything is written, when a length is
// negative or the list positions are not a permutation of 0..R-1.
__device__ __forceinline__ bool place_block(int P, int32_t R, const int32_t* __restrict__ lens,
                                            const int32_t* __restrict__ list_pos, int32_t* __restrict__ owner,
                                            int32_t* __restrict__ local_pos, int32_t* inv, uint8_t* choice,
                                            unsigned long long* keys) {
  __shared__ long long carry[kMaxGroups];
  __shared__ long long warp_tot[32 * kMaxGroups];
  __shared__ int bad;
  __shared__ unsigned long long total_len_s;
  const int tid = threadIdx.x;
  if (tid == 0) {
    bad = 0;
    total_len_s = 0;
  }
  if (tid < kMaxGroups) carry[tid] = 0;
  __syncthreads();
  unsigned long long my_len = 0;
  for (int k = tid; k < R; k += blockDim.x) {
    if (lens[k] < 0) bad = 1;
    else my_len += (unsigned long long)lens[k];
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) my_len += __shfl_xor_sync(0xffffffffu, my_len, d);
  if ((tid & 31) == 0) atomicAdd(&total_len_s, my_len);
  __syncthreads();
  const unsigned long long total_len = total_len_s;
  bool ok = bad == 0;
  if (ok && list_pos) ok = build_inverse(list_pos, R, inv, &bad);
  if (!ok) return false;
  // keys: (length descending, list position ascending), unique; sorted in
  // registers for up to 4 x 1024 keys, else by a bitonic network
  const int E = sort_elems(R);
  const int nk = sort_span(R);
  for (int i = tid; i < nk; i += blockDim.x) {
    unsigned long long kk = ~0ull;
    if (i < R) {
      const unsigned long long pos = list_pos ? (unsigned long long)list_pos[i] : (unsigned long long)i;
      kk = ((unsigned long long)(0x7fffffffll - lens[i]) << 32) | pos;
    }
    keys[i] = kk;
  }
  __syncthreads();
  if (E == 1) sort_keys_regs<1>(keys);
  else if (E == 2) sort_keys_regs<2>(keys);
  else if (E == 4) sort_keys_regs<4>(keys);
  else {
    for (int size = 2; size <= nk; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < nk; i += blockDim.x) {
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
  }
  // the rank chosen for sorted position i, then scattered to request order;
  // 32-bit packed loads when the total of all lengths, shifted, fits.  The
  // variant depends on P and the total only, so it is the same for every
  // thread; warp 0 runs the warp variant whole, thread 0 the others.
  uint32_t* c4 = reinterpret_cast<uint32_t*>(choice);
  const int variant = P <= 8 && total_len < (1ull << 29)    ? 0
                      : P <= 16 && total_len < (1ull << 28) ? 1
                      : P <= 16                             ? 2
                      : P <= 32 && total_len < (1ull << 27) ? 3
                                                            : 4;
  if (variant == 3) {
    if (tid < 32) greedy_warp<5>(keys, R, P, c4);
  } else if (tid == 0) {
    if (variant == 0) greedy_sorted8(keys, R, P, c4);
    else if (variant == 1) greedy_sorted16(keys, R, P, c4);
    else if (variant == 2) greedy_sorted_wide16(keys, R, P, c4);
    else greedy_wide(keys, R, P, c4);
  }
  __syncthreads();
  for (int i = tid; i < R; i += blockDim.x) {
    const int pos = (int)(keys[i] & 0xffffffffu);
    owner[list_pos ? inv[pos] : pos] = choice[i];
  }
  __syncthreads();
  // local position = rank among the owner's requests in list order
  for (int base = 0; base < R; base += blockDim.x) {
    const int pos = base + tid;
    int k = 0, grp = 0;
    if (pos < R) {
      k = list_pos ? inv[pos] : pos;
      grp = owner[k];
    }
    const long long pre = group_exclusive_count(pos < R, grp, P, carry, warp_tot);
    if (pos < R) local_pos[k] = (int32_t)pre;
  }
  return true;
}

}  // namespace uk
