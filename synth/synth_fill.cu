// Device twin of synth.fill_host: counter-form SplitMix64 over 16-bit element
// indices (Steele, Lea, Flood, OOPSLA 2014).  Test/benchmark input generator;
// holds none of the reshard method's arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

__device__ __forceinline__ uint64_t sm64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Each thread writes 8 consecutive elements (one 16-byte store when aligned).
__global__ void synth_fill_kernel(uint16_t* __restrict__ p, uint64_t n, uint64_t base,
                                  uint64_t seed, int mode, const uint16_t* __restrict__ table) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x * 8ull;
  for (uint64_t s = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8ull; s < n; s += stride) {
    uint16_t v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint64_t z = sm64(seed, base + s + k);
      v[k] = mode == 0 ? (uint16_t)(z & 0xFFFFu) : table[z >> 48];
    }
    if (s + 8 <= n && ((reinterpret_cast<uintptr_t>(p + s) & 15u) == 0)) {
      uint4 w;
      w.x = v[0] | ((uint32_t)v[1] << 16);
      w.y = v[2] | ((uint32_t)v[3] << 16);
      w.z = v[4] | ((uint32_t)v[5] << 16);
      w.w = v[6] | ((uint32_t)v[7] << 16);
      *reinterpret_cast<uint4*>(p + s) = w;
    } else {
      for (int k = 0; k < 8 && s + k < n; ++k) p[s + k] = v[k];
    }
  }
}

extern "C" int synth_fill_u16(void* p, uint64_t n, uint64_t base, uint64_t seed, int mode,
                              const void* table, void* stream) {
  if (n == 0) return 0;
  if (mode != 0 && table == nullptr) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t want = (n + 8 * 256 - 1) / (8 * 256);
  uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 8;
  unsigned grid = (unsigned)(want < cap ? want : cap);
  synth_fill_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>((uint16_t*)p, n, base, seed, mode,
                                                            (const uint16_t*)table);
  return (int)cudaGetLastError();
}
