// Block-wide building blocks for the single-CTA metadata kernels.
#pragma once

#include "umm_internal.cuh"

namespace uk {


__device__ __forceinline__ long long warp_incl_scan(long long x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  return x;
}

// Grouped exclusive prefix sum over one chunk of blockDim.x items (item i is
// thread i).  For every item, returns carry[grp] + the sum of `val` over the
// earlier items of this chunk in the same group, then advances carry[] by the
// chunk's group totals.  All threads of the block must call it; `warp_tot`
// holds 32 * ngroups entries of shared memory.  Items that do not exist pass
// val = 0.
__device__ __forceinline__ long long group_exclusive_scan(long long val, int grp, int ngroups, long long* carry,
                                          long long* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  long long mine = 0;
  for (int g = 0; g < ngroups; ++g) {
    long long x = warp_incl_scan(grp == g ? val : 0);
    if (grp == g) mine = x - val;
    if (lane == 31) warp_tot[warp * ngroups + g] = x;
  }
  __syncthreads();
  if (threadIdx.x < ngroups) {
    const int g = threadIdx.x;
    long long run = carry[g];
    for (int w = 0; w < nwarps; ++w) {
      long long t = warp_tot[w * ngroups + g];
      warp_tot[w * ngroups + g] = run;
      run += t;
    }
    carry[g] = run;
  }
  __syncthreads();
  long long out = warp_tot[warp * ngroups + grp] + mine;
  __syncthreads();
  return out;
}

// The same for val = 1 on the items that exist (a grouped count): an item's
// rank among the earlier items of its group in this warp is the number of
// lower lanes in its __match_any_sync set, and the warp's count per group is
// one ballot per group.  Items that do not exist pass present = false.
__device__ __forceinline__ long long group_exclusive_count(bool present, int grp, int ngroups, long long* carry,
                                                           long long* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const unsigned int same = __match_any_sync(0xffffffffu, present ? grp : -1);
  const long long mine = __popc(same & ((1u << lane) - 1u));
  for (int g = 0; g < ngroups; ++g) {
    const unsigned int b = __ballot_sync(0xffffffffu, present && grp == g);
    if (lane == 0) warp_tot[warp * ngroups + g] = __popc(b);
  }
  __syncthreads();
  if (threadIdx.x < ngroups) {
    const int g = threadIdx.x;
    long long run = carry[g];
    for (int w = 0; w < nwarps; ++w) {
      long long t = warp_tot[w * ngroups + g];
      warp_tot[w * ngroups + g] = run;
      run += t;
    }
    carry[g] = run;
  }
  __syncthreads();
  long long out = present ? warp_tot[warp * ngroups + grp] + mine : 0;
  __syncthreads();
  return out;
}

__device__ __forceinline__ DevStatus* status_of(const Geo& g, const Ws& w) {
  return reinterpret_cast<DevStatus*>(g.base + w.status);
}

__device__ __forceinline__ unsigned int read_flags(const DevStatus* st) {
  return *reinterpret_cast<const volatile unsigned int*>(&st->flags);
}

}  // namespace uk
