// Allocation-free variant of the fused GQA decode step.
//
// Some callers cannot allocate device memory at the point where they decode:
// code running inside a CUDA-graph replay or a custom allocator's critical
// section, runtimes that hand the library a fixed memory budget, or C
// callers without a device allocator at all.  For them this file offers
// dcp_decode_gqa_noalloc: the same computation as dcp_decode_gqa, with the
// split-KV workspace taken from a fixed array in the library's own device
// memory instead of a caller buffer.
//
// The array is a file-scope __device__ object of kNoallocScratchBytes; every
// GPU that loads the library holds it until the process exits.  Host code
// may not use its name as a device address, so its address is looked up with
// cudaGetSymbolAddress once per device (on the first call made on that
// device, with that device current) and passed to the kernels like any
// workspace.  No call here allocates memory.
#include <mutex>

#include "dcp_common.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DCP_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DCP_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DCP_OK;
}

}  // namespace

extern "C" int dcp_decode_gqa_noalloc(dcp_layout_t layout, const void* q, int32_t num_reqs,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, float scale, dcp_dtype_t dtype,
                                      dcp_paged_kv_t kv, const int32_t* local_lens,
                                      const float* sink, void* out, dcp_dtype_t out_dtype,
                                      float* out_lse, int32_t* err_count, dcp_stream_t stream) {
  size_t need = 0;
  const int rc = dcp_decode_workspace_size(layout, DCP_KIND_GQA, num_reqs, num_q_heads,
                                           num_kv_heads, head_dim, &need);
  if (rc != DCP_OK) return rc;
  if (need > kNoallocScratchBytes) return DCP_EWORKSPACE;  // batch too large for the fixed array
  void* scratch = nullptr;
  const int src = scratch_for_current_device(&scratch);
  if (src != DCP_OK) return src;
  return dcp_decode_gqa(layout, q, num_reqs, num_q_heads, num_kv_heads, head_dim, scale, dtype,
                        kv, local_lens, sink, out, out_dtype, out_lse, scratch,
                        kNoallocScratchBytes, err_count, stream);
}
