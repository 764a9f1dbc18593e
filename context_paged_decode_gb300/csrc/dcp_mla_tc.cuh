// tcgen05 (5th-generation tensor core) MLA decode kernel: interface.
#pragma once

#include "dcp_common.cuh"

namespace dcp {

constexpr int kMlaTcTile = 64;  // run boundaries of the balanced-parts plan fall on this

// True when the tensor-core kernel handles this call (bf16, 128 heads,
// 576/512 latent, block_size a multiple of the tile, driver TMA available).
bool mla_tc_supported(const dcp_layout_t& layout, int B, int Hq, int dk, int dv, dcp_dtype_t dtype,
                      const dcp_paged_kv_t& kv);

// Clusters the kernel runs on this device (one run of the balanced-parts
// plan each); -1 if the kernel cannot be configured.
int mla_tc_clusters();

// Launch on a plan made by launch_plan_parts with parts == clusters.
int launch_mla_tc(const dcp_layout_t& layout, const void* q, int B, int Hq, float scale,
                  const dcp_paged_kv_t& kv, const Plan& plan, int clusters, int32_t* err,
                  cudaStream_t s);

}  // namespace dcp
