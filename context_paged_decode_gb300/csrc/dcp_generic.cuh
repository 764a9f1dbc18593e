// Arguments of the CUDA-core decode kernels (any shape, f32 or bf16).
#pragma once

#include "dcp_common.cuh"

namespace dcp {

struct GenericArgs {
  const void* q;  // [B][Hq][dk]
  int B, Hq, G, groups, dcp, bs;
  int dk, dv;
  int64_t k_stride, v_stride;  // elements between consecutive cache rows
  float sl2;                   // softmax scale * log2(e)
  dcp_rank_ptrs_t k, v;        // per-rank pools (v == k for latent caches)
  const int32_t* bt;
  int max_vb;
  int64_t bt_rank_stride;
  int64_t num_blocks;
  int32_t* err;
};

// Row of (physical block, head group g, in-block offset) in a pool is
// (phys*groups + g)*bs + off: HND for GQA, [block][bs][row] for latent caches.
int launch_split_generic(const GenericArgs& A, const Plan& plan, bool bf16, cudaStream_t s);

// Selected tokens of SFA: either remapped pairs (sel_rank/sel_slot) or, when
// topk != nullptr, global top-k indices remapped inside the kernel.
struct SfaSel {
  const int32_t* sel_rank;
  const int32_t* sel_slot;
  const int32_t* topk;
  const int32_t* seq_lens;
  int K;
  Layout L;
};

int launch_sfa_generic(const GenericArgs& A, const SfaSel& S, float* part_o, float* part_lse,
                       bool bf16, cudaStream_t s);

}  // namespace dcp
