// Tensor-core SFA decode kernel: interface.
#pragma once

#include "dcp_common.cuh"

namespace dcp {

struct SfaMmaArgs {
  const __nv_bfloat16* q;  // [B][Hq][576]
  int B, Hq, hblocks, dcp, bs, K;
  float sl2;               // softmax scale * log2(e)
  dcp_rank_ptrs_t pool;    // per-rank latent pools [num_blocks*bs][576]
  int64_t num_blocks;
  // selected tokens: remapped pairs, or global top-k remapped in the kernel
  const int32_t* sel_rank;
  const int32_t* sel_slot;
  const int32_t* topk;
  const int32_t* seq_lens;
  const int32_t* bt;
  int max_vb;
  int64_t bt_rank_stride;
  Layout L;
  float* part_o;           // [dcp][B][Hq][512]
  float* part_lse;         // [dcp][B][Hq]
  int32_t* err;
};

// Does top-k entry k of request b belong to rank r?  Sets its slot (-2 when
// the block-table entry is unusable).
__device__ __forceinline__ bool sfa_select(const SfaMmaArgs& A, int b, int k, int r,
                                           int64_t& slot) {
  if (A.topk == nullptr) {
    if (__ldg(A.sel_rank + (int64_t)b * A.K + k) != r) return false;
    slot = __ldg(A.sel_slot + (int64_t)b * A.K + k);
    return true;
  }
  const int64_t g = __ldg(A.topk + (int64_t)b * A.K + k);
  if (g < 0 || g >= __ldg(A.seq_lens + b)) return false;
  int rk, loc;
  int64_t vb;
  place_token(g, A.L, rk, vb, loc);
  if (rk != r) return false;
  const int64_t phys =
      vb < A.max_vb ? (int64_t)__ldg(A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb + vb)
                    : (int64_t)-1;
  slot = (phys >= 0 && phys < A.num_blocks) ? phys * A.bs + loc : (int64_t)-2;
  return true;
}

bool sfa_mma_supported(int Hq, int dk, int dv, dcp_dtype_t dtype, int K);
int launch_sfa_mma(const SfaMmaArgs& A, cudaStream_t s);

}  // namespace dcp
