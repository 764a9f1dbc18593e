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
// The array is a file-scope __device__ object of kNoallocScratchBytes.  The
// library's device code is loaded lazily, so the array is reserved on a
// device by the first call made there (the cudaGetSymbolAddress below loads
// this file's module); from then on the device holds it until the process
// exits.  That first call returns DCP_ECUDA when the 16 MiB cannot be
// reserved, and it should come before any stream capture, as a warm-up.
// Host code may not use the array's name as a device address, so the address
// is looked up with cudaGetSymbolAddress, with the device current, and passed
// to the kernels like any workspace.  It is cached per device together with
// the unique id of the CUDA context it was looked up in; a call made in
// another context (after cudaDeviceReset, or under a context the caller
// created) looks it up again.  No call here allocates memory.
#include <cudaTypedefs.h>

#include <mutex>

#include "dcp_common.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;
  bool keyed = false;  // ctx_id is valid
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// cuCtxGetId through the runtime's driver entry point (no -lcuda needed).
PFN_cuCtxGetId_v12000 ctx_id_getter() {
  static PFN_cuCtxGetId_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuCtxGetId_v12000)p;
    cudaGetLastError();
  }
  return fn;
}

bool current_ctx_id(unsigned long long* id) {
  PFN_cuCtxGetId_v12000 fn = ctx_id_getter();
  return fn != nullptr && fn(nullptr, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's current context.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DCP_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot& slot = g_scratch[dev];
  unsigned long long id = 0;
  const bool have_id = current_ctx_id(&id);
  if (!(have_id && slot.keyed && slot.ptr != nullptr && slot.ctx_id == id)) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // not sticky: leave no error for the next call to misread
      return DCP_ECUDA;
    }
    // the lookup may have initialised the device's context: key on it now
    slot.ptr = p;
    slot.keyed = current_ctx_id(&slot.ctx_id);
  }
  *out = slot.ptr;
  return DCP_OK;
}

}  // namespace

extern "C" int dcp_decode_gqa_noalloc(dcp_layout_t layout, const void* q, int32_t num_reqs,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, float scale, dcp_dtype_t dtype,
                                      dcp_paged_kv_t kv, const int32_t* local_lens,
                                      const float* sink, void* out, dcp_dtype_t out_dtype,
                                      float* out_lse, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_decode_gqa_noalloc");
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
