// GPU version of the seeded value generator of the `workloads` module (the
// numpy version in __init__.py is the definition; both produce the same
// bits).  Input generation only: fills a device buffer with elements
// [e0, e0 + n) of one value stream, value = table[mix64(key + (e+1)*GAMMA) >> 48],
// where mix64 is the SplitMix64 output function.  Used to populate
// multi-gigabyte synthetic caches quickly; the oracle regenerates the same
// elements on the host with numpy.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

template <typename T>
__global__ void fill_kernel(uint64_t key, int64_t e0, int64_t n, const T* __restrict__ table,
                            T* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t e = (uint64_t)(e0 + i) + 1ull;
    out[i] = table[mix64(key + e * 0x9E3779B97F4A7C15ull) >> 48];
  }
}

}  // namespace

extern "C" int synth_fill(uint64_t key, int64_t e0, int64_t n, const void* table, int elem_bytes,
                          void* out, cudaStream_t stream) {
  if (n <= 0) return 0;
  if (!table || !out || (elem_bytes != 2 && elem_bytes != 4)) return -1;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  if (elem_bytes == 2)
    fill_kernel<uint16_t><<<(int)blocks, 256, 0, stream>>>(key, e0, n, (const uint16_t*)table,
                                                           (uint16_t*)out);
  else
    fill_kernel<uint32_t><<<(int)blocks, 256, 0, stream>>>(key, e0, n, (const uint32_t*)table,
                                                           (uint32_t*)out);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
