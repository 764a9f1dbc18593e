// SFA (sparse flash attention) decode under DCP.
//
// Page "Decode Context Parallel (DCP)", section "GLM-5.2 SFA DCP replicated
// indexer": the indexer sees the full sequence on every rank and picks the
// same global top-k tokens as without DCP; the SFA KV cache stays sharded,
// so the global indices are remapped to local KV indices before SFA runs,
// and decode-only batches keep the Q-gather and result-merge path.  The
// attention sink is applied once, at the merge (page "DeepSeek V4.1 context
// parallelism", section "Decode computation").
#include <string.h>

#include "dcp_generic.cuh"
#include "dcp_sfa_mma.cuh"
#include "dcp_sfa_tc.cuh"

using namespace dcp;

namespace {

bool sfa_args_ok(const dcp_layout_t& layout, const void* q, int B, int Hq, int dk, int dv,
                 dcp_dtype_t dtype, const dcp_paged_kv_t& kv, int K) {
  if (!layout_ok(layout) || B < 0 || Hq < 1 || dk < 32 || dk % 32 || dk > 1024 || dv < 32 ||
      dv % 32 || dv > dk || K < 0 || (dtype != DCP_F32 && dtype != DCP_BF16) ||
      kv.num_blocks < 0)
    return false;
  if (B == 0) return true;
  return q && ranks_ok(kv.k, layout.dcp_size);
}

GenericArgs sfa_generic_args(const dcp_layout_t& layout, const void* q, int B, int Hq, int dk,
                             int dv, float scale, const dcp_paged_kv_t& kv, int32_t* err) {
  GenericArgs A;
  A.q = q;
  A.B = B;
  A.Hq = Hq;
  A.G = Hq;
  A.groups = 1;
  A.dcp = layout.dcp_size;
  A.bs = layout.block_size;
  A.dk = dk;
  A.dv = dv;
  A.k_stride = dk;
  A.v_stride = dk;
  A.sl2 = scale * kLog2e;
  A.k = kv.k;
  A.v = kv.k;
  A.bt = kv.block_table;
  A.max_vb = kv.max_vblocks;
  A.bt_rank_stride = kv.bt_rank_stride;
  A.num_blocks = kv.num_blocks;
  A.err = err;
  return A;
}

bool sfa_fast_ok(const dcp_layout_t& layout, const void* q, int Hq, int dk, int dv,
                 dcp_dtype_t dtype, const dcp_paged_kv_t& kv, int K) {
  if (!sfa_mma_supported(Hq, dk, dv, dtype, K)) return false;
  if ((int64_t)kv.num_blocks * layout.block_size >= (int64_t(1) << 31)) return false;
  if ((uintptr_t)q & 15) return false;
  for (int r = 0; r < layout.dcp_size; ++r)
    if ((uintptr_t)kv.k.ptr[r] & 15) return false;
  return true;
}

SfaMmaArgs sfa_mma_args(const dcp_layout_t& layout, const void* q, int B, int Hq, float scale,
                        const dcp_paged_kv_t& kv, int K, float* part_o, float* part_lse,
                        int32_t* err) {
  SfaMmaArgs A;
  memset(&A, 0, sizeof(A));
  A.q = (const __nv_bfloat16*)q;
  A.B = B;
  A.Hq = Hq;
  A.dcp = layout.dcp_size;
  A.bs = layout.block_size;
  A.K = K;
  A.sl2 = scale * kLog2e;
  A.pool = kv.k;
  A.num_blocks = kv.num_blocks;
  A.bt = kv.block_table;
  A.max_vb = kv.max_vblocks;
  A.bt_rank_stride = kv.bt_rank_stride;
  A.L = Layout{layout.dcp_size, layout.block_size, layout.interleave};
  A.part_o = part_o;
  A.part_lse = part_lse;
  A.err = err;
  return A;
}

bool sfa_tc_ok(const dcp_layout_t& layout, const void* q, int Hq, int dk, int dv,
               dcp_dtype_t dtype, const dcp_paged_kv_t& kv, int K) {
  return sfa_tc_supported(Hq, dk, dv, dtype, K, (int64_t)kv.num_blocks * layout.block_size, q,
                          kv.k, layout.dcp_size);
}

SfaTcArgs sfa_tc_args(const dcp_layout_t& layout, int B, int Hq, float scale,
                      const dcp_paged_kv_t& kv, int K, float* part_o, float* part_lse,
                      int32_t* err) {
  SfaTcArgs A;
  memset(&A, 0, sizeof(A));
  for (int r = 0; r < layout.dcp_size; ++r) A.pool[r] = (const uint8_t*)kv.k.ptr[r];
  A.B = B;
  A.Hq = Hq;
  A.bs = layout.block_size;
  A.K = K;
  A.sl2 = scale * kLog2e;
  A.num_blocks = kv.num_blocks;
  A.part_o = part_o;
  A.part_lse = part_lse;
  A.err = err;
  return A;
}

}  // namespace

extern "C" {

int dcp_sfa_decode_partial(dcp_layout_t layout, const void* q, int32_t num_reqs,
                           int32_t num_q_heads, int32_t kv_dim, int32_t v_dim, float scale,
                           dcp_dtype_t dtype, dcp_paged_kv_t kv, const int32_t* sel_rank,
                           const int32_t* sel_slot, int32_t topk_len, float* part_o,
                           float* part_lse, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_sfa_decode_partial");
  if (!sfa_args_ok(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, dtype, kv, topk_len))
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!part_o || !part_lse || (topk_len > 0 && (!sel_rank || !sel_slot))) return DCP_EINVAL;
  if (sfa_tc_ok(layout, q, num_q_heads, kv_dim, v_dim, dtype, kv, topk_len)) {
    SfaTcArgs T = sfa_tc_args(layout, num_reqs, num_q_heads, scale, kv, topk_len, part_o, part_lse,
                              err_count);
    T.sel_rank = sel_rank;
    T.sel_slot = sel_slot;
    return launch_sfa_tc(T, q, layout.dcp_size, (cudaStream_t)stream);
  }
  if (sfa_fast_ok(layout, q, num_q_heads, kv_dim, v_dim, dtype, kv, topk_len)) {
    SfaMmaArgs M = sfa_mma_args(layout, q, num_reqs, num_q_heads, scale, kv, topk_len, part_o,
                                part_lse, err_count);
    M.sel_rank = sel_rank;
    M.sel_slot = sel_slot;
    return launch_sfa_mma(M, (cudaStream_t)stream);
  }
  const GenericArgs A =
      sfa_generic_args(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, scale, kv, err_count);
  SfaSel S{sel_rank, sel_slot, nullptr, nullptr, topk_len,
           Layout{layout.dcp_size, layout.block_size, layout.interleave}};
  return launch_sfa_generic(A, S, part_o, part_lse, dtype == DCP_BF16, (cudaStream_t)stream);
}

int dcp_sfa_decode(dcp_layout_t layout, const void* q, int32_t num_reqs, int32_t num_q_heads,
                   int32_t kv_dim, int32_t v_dim, float scale, dcp_dtype_t dtype,
                   dcp_paged_kv_t kv, const int32_t* topk, int32_t topk_len,
                   const int32_t* seq_lens, const float* sink, void* out,
                   dcp_dtype_t out_dtype, float* out_lse, void* workspace,
                   size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_sfa_decode");
  if (!sfa_args_ok(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, dtype, kv, topk_len) ||
      (out_dtype != DCP_F32 && out_dtype != DCP_BF16) || kv.max_vblocks < 0 ||
      kv.bt_rank_stride < 0)
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!out || (topk_len > 0 && (!topk || !seq_lens || !kv.block_table))) return DCP_EINVAL;
  size_t need = 0;
  dcp_decode_workspace_size(layout, DCP_KIND_SFA, num_reqs, num_q_heads, 1, v_dim, &need);
  if (!workspace || workspace_bytes < need) return DCP_EWORKSPACE;
  const int dcp = layout.dcp_size;
  float* part_o = (float*)workspace;
  float* part_lse =
      (float*)((char*)workspace +
               align_up(sizeof(float) * (size_t)dcp * num_reqs * num_q_heads * v_dim, 256));
  cudaStream_t s = (cudaStream_t)stream;
  int rc;
  if (sfa_tc_ok(layout, q, num_q_heads, kv_dim, v_dim, dtype, kv, topk_len)) {
    // remap once per selected token, then every CTA of a request reads the pairs
    int32_t* sel_rank =
        (int32_t*)((char*)part_lse +
                   align_up(sizeof(float) * (size_t)dcp * num_reqs * num_q_heads, 256));
    int32_t* sel_slot =
        (int32_t*)((char*)sel_rank + align_up(sizeof(int32_t) * (size_t)num_reqs * kSfaTcMaxSel, 256));
    rc = dcp_sfa_remap(layout, topk, num_reqs, topk_len, seq_lens, kv.block_table, kv.max_vblocks,
                       kv.bt_rank_stride, kv.num_blocks, sel_rank, sel_slot, err_count, stream);
    if (rc) return rc;
    SfaTcArgs T = sfa_tc_args(layout, num_reqs, num_q_heads, scale, kv, topk_len, part_o, part_lse,
                              err_count);
    T.sel_rank = sel_rank;
    T.sel_slot = sel_slot;
    // the remap, the partials and the merge overlap their launch boundaries:
    // each dependent waits for its predecessor before reading its output.
    // With no top-k entries the remap launches nothing, and the partials
    // kernel must not overlap whatever the caller ran last.
    const bool after_remap = (int64_t)num_reqs * topk_len > 0;
    bool merged = false;
    rc = launch_sfa_tc_merged(T, q, layout.dcp_size, s, after_remap, sink, out, (int)out_dtype,
                              out_lse, &merged);
    if (rc || merged) return rc;
    return launch_dense_merge(dcp, part_o, part_lse, num_reqs, num_q_heads, v_dim, sink, out,
                              (int)out_dtype, out_lse, s, true);
  } else if (sfa_fast_ok(layout, q, num_q_heads, kv_dim, v_dim, dtype, kv, topk_len)) {
    SfaMmaArgs M = sfa_mma_args(layout, q, num_reqs, num_q_heads, scale, kv, topk_len, part_o,
                                part_lse, err_count);
    M.topk = topk;
    M.seq_lens = seq_lens;
    rc = launch_sfa_mma(M, s);
  } else {
    const GenericArgs A =
        sfa_generic_args(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, scale, kv, err_count);
    SfaSel S{nullptr, nullptr, topk, seq_lens, topk_len,
             Layout{layout.dcp_size, layout.block_size, layout.interleave}};
    rc = launch_sfa_generic(A, S, part_o, part_lse, dtype == DCP_BF16, s);
  }
  if (rc) return rc;
  return dcp_lse_merge(dcp, part_o, part_lse, num_reqs, num_q_heads, v_dim, sink, out, out_dtype,
                       out_lse, stream);
}

}  // extern "C"
