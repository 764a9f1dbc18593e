// tcgen05 SFA decode kernel: interface.
#pragma once

#include "dcp_common.cuh"
#include "dcp_ptx.cuh"

namespace dcp {

constexpr int kSfaTcMaxSel = 2048;     // selected tokens per request on this path

struct SfaTcArgs {
  CUtensorMap qmap;                     // q [B*Hq rows][576] bf16, box 64 x 64, 128 B swizzle
  const uint8_t* pool[DCP_MAX_RANKS];   // per-rank latent pools [num_blocks*bs rows][576] bf16
  int B, Hq, hblocks, bs, K;
  int dcp, rpc;                         // ranks; ranks per CTA (set by launch_sfa_tc)
  float sl2;                            // softmax scale * log2(e)
  int64_t num_blocks;
  const int32_t* sel_rank;               // [B][K] remapped owner rank (-1: not selected)
  const int32_t* sel_slot;               // [B][K] slot on that rank
  float* part_o;                        // [dcp][B][Hq][512]
  float* part_lse;                      // [dcp][B][Hq]
  int32_t* err;
  // merge inside the kernel (set by launch_sfa_tc): the ngroups CTAs of a
  // (request, head block) form a cluster, and after every one has written
  // its ranks' partials each merges its share of the rows into out / out_lse
  int fuse, ngroups;
  const float* sink;                    // [Hq] or null
  void* out;                            // [B][Hq][512] of out_dtype
  int out_dtype;
  float* out_lse;                       // [B][Hq] or null
};

// bf16, 576-wide latent rows with a 512-wide value, Hq a multiple of 64,
// at most 2048 selected tokens per request, 16-byte aligned q and pools.
bool sfa_tc_supported(int Hq, int dk, int dv, dcp_dtype_t dtype, int K, int64_t pool_rows,
                      const void* q, const dcp_rank_ptrs_t& pool, int dcp);
// pdl: launched as a programmatic dependent of the previous kernel in the
// stream, which must be the dcp_sfa_remap that produced sel_rank / sel_slot
// (the kernel reads q and sets up before waiting for it).
int launch_sfa_tc(const SfaTcArgs& A, const void* q, int dcp, cudaStream_t s, bool pdl = false);
// The same, merging the partials inside the kernel into out / out_lse with the
// sink applied once when the shape allows (a cluster of the CTAs of a request:
// at most 8 of them); *merged tells whether it did (otherwise the caller
// merges the partials).
int launch_sfa_tc_merged(const SfaTcArgs& A, const void* q, int dcp, cudaStream_t s, bool pdl,
                         const float* sink, void* out, int out_dtype, float* out_lse, bool* merged);
// Ranks one CTA of the kernel covers for this shape (host side).
int sfa_tc_ranks_per_cta(int dcp, int B, int hblocks);

}  // namespace dcp
