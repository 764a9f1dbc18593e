// Shared device/host helpers of libdcp (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dcp.h"

#ifndef DCP_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace dcp {

// ---------------------------------------------------------------------------
// host-side argument checks
// ---------------------------------------------------------------------------

inline bool layout_ok(const dcp_layout_t& L) {
  return L.dcp_size >= 1 && L.dcp_size <= DCP_MAX_RANKS && L.block_size >= 1 &&
         L.interleave >= 1 && L.block_size % L.interleave == 0;
}

inline bool ranks_ok(const dcp_rank_ptrs_t& p, int dcp) {
  for (int r = 0; r < dcp; ++r)
    if (p.ptr[r] == nullptr) return false;
  return true;
}

// DCP_OK, or DCP_ECUDA if the last runtime call or launch failed (the error
// text goes to stderr when the environment sets DCP_VERBOSE).
int launch_status_report(cudaError_t e);
inline int launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DCP_OK : launch_status_report(e);
}

int num_sms();  // SM count of the current device (cached per device)

// Host-side NVTX range around one public call: with a profiler attached the
// call's kernels are grouped under its name; without one a push or pop costs
// a check of a function pointer.  -DDCP_NO_NVTX compiles the ranges out.
struct NvtxRange {
#ifndef DCP_NO_NVTX
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
#else
  explicit NvtxRange(const char*) {}
#endif
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// layout ("Decode Context Parallel (DCP)", section "KV-cache layout")
// ---------------------------------------------------------------------------

struct Layout {
  int dcp, bs, I;
};

// Owner rank, virtual block and in-block local offset of global token x.
__device__ __forceinline__ void place_token(int64_t x, const Layout& L, int& rank, int64_t& vb,
                                            int& loc) {
  const int64_t vbs = (int64_t)L.bs * L.dcp;
  vb = x / vbs;
  const int off = (int)(x - vb * vbs);    // offset_in_virtual_block
  const int lbi = off / L.I;              // local_block_index
  rank = lbi % L.dcp;                     // target_rank
  loc = (lbi / L.dcp) * L.I + off % L.I;  // offset inside the rank's block
}

__device__ __forceinline__ void count_error(int32_t* err) {
  if (err) atomicAdd(err, 1);
}

// ---------------------------------------------------------------------------
// numerics
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// split-KV plan shared by the decode kernels
// ---------------------------------------------------------------------------
//
// A work item is a run of local positions [p0, p1) of request b on rank r
// for head group g.  Items are ordered by (b, g, r, chunk) so that the items
// of one (b, g) -- over all ranks -- and of one (b, g, r) are contiguous.
// Workspace layout (each part 256-byte aligned):
//   int32 hdr[4]         n_items, chunk_tokens, item counter, stuck counter
//   int32 off[B*G*dcp+1] first item of (b, g, r)
//   int4  item[max_items] {b, g << 8 | r, p0, p1}
//   int32 ipart[max_items]   run of each item (balanced-parts plans only)
//   int32 pfirst[kMaxParts+1] first item of each run (balanced-parts plans only)
//   float lse[max_items * heads_per_item]
//   float o[max_items * heads_per_item * dv]

constexpr int kMaxParts = 1024;

struct Plan {
  int32_t* hdr;
  int32_t* off;
  int4* item;
  int32_t* ipart;
  int32_t* pfirst;
  float* lse;
  float* o;
  int max_items;
};

inline size_t plan_bytes(int entries, int max_items, int heads_per_item, int dv) {
  size_t b = 256;
  b += align_up(sizeof(int32_t) * (size_t)(entries + 1), 256);
  b += align_up(sizeof(int4) * (size_t)max_items, 256);
  b += align_up(sizeof(int32_t) * (size_t)max_items, 256);
  b += align_up(sizeof(int32_t) * (size_t)(kMaxParts + 1), 256);
  b += align_up(sizeof(float) * (size_t)max_items * heads_per_item, 256);
  b += align_up(sizeof(float) * (size_t)max_items * heads_per_item * dv, 256);
  return b;
}

inline Plan plan_carve(void* ws, int entries, int max_items, int heads_per_item) {
  Plan p;
  char* c = (char*)ws;
  p.hdr = (int32_t*)c;
  c += 256;
  p.off = (int32_t*)c;
  c += align_up(sizeof(int32_t) * (size_t)(entries + 1), 256);
  p.item = (int4*)c;
  c += align_up(sizeof(int4) * (size_t)max_items, 256);
  p.ipart = (int32_t*)c;
  c += align_up(sizeof(int32_t) * (size_t)max_items, 256);
  p.pfirst = (int32_t*)c;
  c += align_up(sizeof(int32_t) * (size_t)(kMaxParts + 1), 256);
  p.lse = (float*)c;
  c += align_up(sizeof(float) * (size_t)max_items * heads_per_item, 256);
  p.o = (float*)c;
  p.max_items = max_items;
  return p;
}

// Launch the plan kernel: chunk = max(min_chunk, ceil(sum_tokens*G/target)),
// rounded up to `tile`; items never cross a rank.
int launch_plan(const int32_t* local_lens, int B, int dcp, int G, int tile, int min_chunk,
                int target_items, const Plan& plan, cudaStream_t s);

// Balanced-parts plan (G = 1): the local ranges of all (b, r), concatenated in
// (b, r) order, are cut into `parts` runs of about equal cost, where a
// non-empty range costs its tokens plus `overhead` (the fixed cost of an item,
// in tokens); a cut inside a range falls on a multiple of `tile` positions.
// Items are the pieces between cuts, in (b, r) order; run k owns items
// [pfirst[k], pfirst[k+1]).  At most B*dcp + parts - 1 items; 1 <= parts <= kMaxParts.
int launch_plan_parts(const int32_t* local_lens, int B, int dcp, int tile, int parts,
                      int overhead, const Plan& plan, cudaStream_t s);

// Largest item count the MLA plan can produce (sizes its workspace).
int mla_max_items(int B, int dcp);

// Merge item partials: mode 0 -> one output per (b, h) over all ranks (with
// sink), mode 1 -> one output per (r, b, h) (no sink).
// dcp_lse_merge for callers inside the library: with pdl, the launch is a
// programmatic dependent of the previous kernel in the stream (the merge
// waits for it before reading the partials).
int launch_dense_merge(int num_parts, const float* part_o, const float* part_lse, int B, int H,
                       int dv, const float* sink, void* out, int out_dtype, float* out_lse,
                       cudaStream_t s, bool pdl);
int launch_item_merge(const Plan& plan, int mode, int B, int dcp, int Hq, int G_per_item,
                      int groups, int dv, const float* sink, void* out, int out_dtype,
                      float* out_lse, cudaStream_t s);

}  // namespace dcp
