// Test program: the kernels' bounded mbarrier wait (dcp::mbar_wait) on a
// phase that nothing completes gives up after its iteration limit and
// reports it, the kernel returns, and the context stays usable: a second
// launch whose barrier does complete runs normally.  No fault, trap or
// unbounded loop is involved; every access is to the kernel's own shared
// barrier and a 2-int status buffer.
#include <chrono>
#include <cstdio>

#include <cuda_runtime.h>

#include "dcp_ptx.cuh"

// status[0] = 1 if the wait saw the phase complete, 2 if it gave up
__global__ void wait_on_nothing(int* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = dcp::smem_u32(&bar);
  if (threadIdx.x == 0) {
    dcp::mbar_init(b, 1);
    dcp::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) status[0] = dcp::mbar_wait(b, 0) ? 1 : 2;   // nothing arrives
}

// status[1] = 1 if the wait saw the phase complete (it does: one arrival)
__global__ void wait_on_arrival(int* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = dcp::smem_u32(&bar);
  if (threadIdx.x == 0) {
    dcp::mbar_init(b, 1);
    dcp::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    dcp::mbar_arrive(b);
    status[1] = dcp::mbar_wait(b, 0) ? 1 : 2;
  }
}

int main() {
  int* d = nullptr;
  if (cudaMalloc(&d, 2 * sizeof(int)) != cudaSuccess) return 3;
  cudaMemset(d, 0, 2 * sizeof(int));
  const auto t0 = std::chrono::steady_clock::now();
  wait_on_nothing<<<1, 32>>>(d);
  const cudaError_t e0 = cudaDeviceSynchronize();
  const double s = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  wait_on_arrival<<<1, 32>>>(d);
  const cudaError_t e1 = cudaDeviceSynchronize();
  int h[2] = {0, 0};
  const cudaError_t e2 = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  printf("errors %d %d %d status %d %d seconds %.3f\n", (int)e0, (int)e1, (int)e2, h[0], h[1], s);
  cudaFree(d);
  return 0;
}
