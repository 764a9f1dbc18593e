// MLA decode under DCP: per-rank split-KV partials and the fused decode step.
//
// vLLM DCP blog post, section 1: MLA keeps one latent KV head shared by all
// query heads, which tensor parallelism replicates in full; DCP instead
// shards it along the sequence.  Page "Decode Context Parallel (DCP)",
// section "Decode": each rank attends its local shard and emits a partial
// output plus LSE; the partials are merged by LSE.
//
// Key = the whole latent row (512 latent + 64 rope), value = its first 512
// entries.  The tensor-core kernel for the 128-head bf16 shape lives in
// dcp_mla_tc.cu; every other shape runs the CUDA-core split kernel.
#include "dcp_generic.cuh"
#include "dcp_mla_tc.cuh"

namespace dcp {

int mla_target_items() { return 4 * num_sms(); }

// What an item costs a cluster beyond its tokens (Q reload, epilogue and
// ring refill), in tokens, for balancing the runs of the tensor-core kernel.
// On GB300 (B=64, 128 heads, bimodal lengths, 3-22 items per run) a step took
// 1.770 ms with runs of equal tokens; 1.707, 1.677, 1.670, 1.677, 1.687 and
// 1.707 ms at 256, 384, 512, 640, 768 and 1024.
constexpr int kMlaItemOverhead = 512;

// The balanced-parts plan makes at most B*dcp + clusters - 1 items and the
// chunked plan at most target + B*dcp; clusters <= SMs/2 < target.
int mla_max_items(int B, int dcp) { return mla_target_items() + B * dcp; }

}  // namespace dcp

using namespace dcp;

namespace {

bool mla_args_ok(const dcp_layout_t& layout, const void* q, int B, int Hq, int dk, int dv,
                 dcp_dtype_t dtype, const dcp_paged_kv_t& kv, const int32_t* local_lens) {
  if (!layout_ok(layout) || B < 0 || Hq < 1 || dk < 32 || dk % 32 || dk > 1024 || dv < 32 ||
      dv % 32 || dv > dk || (dtype != DCP_F32 && dtype != DCP_BF16) || kv.num_blocks < 0 ||
      kv.max_vblocks < 0 || kv.bt_rank_stride < 0)
    return false;
  if (B == 0) return true;
  return q && local_lens && kv.block_table && ranks_ok(kv.k, layout.dcp_size);
}

int mla_split(const dcp_layout_t& layout, const void* q, int B, int Hq, int dk, int dv,
              float scale, dcp_dtype_t dtype, const dcp_paged_kv_t& kv, const int32_t* local_lens,
              const Plan& plan, int32_t* err, cudaStream_t s) {
  if (mla_tc_supported(layout, B, Hq, dk, dv, dtype, kv)) {
    const int clusters = mla_tc_clusters();
    if (clusters < 1) return DCP_ECUDA;
    int rc = launch_plan_parts(local_lens, B, layout.dcp_size, kMlaTcTile, clusters,
                               kMlaItemOverhead, plan, s);
    if (rc) return rc;
    return launch_mla_tc(layout, q, B, Hq, scale, kv, plan, clusters, err, s);
  }
  int rc = launch_plan(local_lens, B, layout.dcp_size, 1, 1, 64, mla_target_items(), plan, s);
  if (rc) return rc;
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
  return launch_split_generic(A, plan, dtype == DCP_BF16, s);
}

}  // namespace

extern "C" {

int dcp_decode_partial_mla(dcp_layout_t layout, const void* q, int32_t num_reqs,
                           int32_t num_q_heads, int32_t kv_dim, int32_t v_dim, float scale,
                           dcp_dtype_t dtype, dcp_paged_kv_t kv, const int32_t* local_lens,
                           float* part_o, float* part_lse, void* workspace,
                           size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_decode_partial_mla");
  if (!mla_args_ok(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, dtype, kv, local_lens))
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!part_o || !part_lse) return DCP_EINVAL;
  size_t need = 0;
  dcp_decode_workspace_size(layout, DCP_KIND_MLA, num_reqs, num_q_heads, 1, v_dim, &need);
  if (!workspace || workspace_bytes < need) return DCP_EWORKSPACE;
  const int dcp = layout.dcp_size;
  const Plan plan =
      plan_carve(workspace, num_reqs * dcp, mla_max_items(num_reqs, dcp), num_q_heads);
  cudaStream_t s = (cudaStream_t)stream;
  int rc = mla_split(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, scale, dtype, kv,
                     local_lens, plan, err_count, s);
  if (rc) return rc;
  return launch_item_merge(plan, 1, num_reqs, dcp, num_q_heads, num_q_heads, 1, v_dim, nullptr,
                           part_o, DCP_F32, part_lse, s);
}

int dcp_decode_mla(dcp_layout_t layout, const void* q, int32_t num_reqs, int32_t num_q_heads,
                   int32_t kv_dim, int32_t v_dim, float scale, dcp_dtype_t dtype,
                   dcp_paged_kv_t kv, const int32_t* local_lens, const float* sink, void* out,
                   dcp_dtype_t out_dtype, float* out_lse, void* workspace,
                   size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_decode_mla");
  if (!mla_args_ok(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, dtype, kv, local_lens) ||
      (out_dtype != DCP_F32 && out_dtype != DCP_BF16))
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!out) return DCP_EINVAL;
  size_t need = 0;
  dcp_decode_workspace_size(layout, DCP_KIND_MLA, num_reqs, num_q_heads, 1, v_dim, &need);
  if (!workspace || workspace_bytes < need) return DCP_EWORKSPACE;
  const int dcp = layout.dcp_size;
  const Plan plan =
      plan_carve(workspace, num_reqs * dcp, mla_max_items(num_reqs, dcp), num_q_heads);
  cudaStream_t s = (cudaStream_t)stream;
  int rc = mla_split(layout, q, num_reqs, num_q_heads, kv_dim, v_dim, scale, dtype, kv,
                     local_lens, plan, err_count, s);
  if (rc) return rc;
  return launch_item_merge(plan, 0, num_reqs, dcp, num_q_heads, num_q_heads, 1, v_dim, sink, out,
                           out_dtype, out_lse, s);
}

}  // extern "C"
