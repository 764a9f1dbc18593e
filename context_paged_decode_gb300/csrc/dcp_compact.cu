// SFA prefill compaction: keep only the KV blocks the selected tokens refer to.
//
// Page "Decode Context Parallel (DCP)", section "GLM-5.2 SFA DCP replicated
// indexer": during prefill or a mixed batch, only the KV blocks referenced
// by the sparse block table are compacted and all-gathered after the layer
// writes its KV cache.  This is the single-GPU part: mark every (rank,
// physical block) a valid selected token refers to, number the marked
// blocks (ranks in order, increasing block id within a rank), copy them
// into one contiguous buffer, and rewrite every selected token as a row of
// that buffer.  Four launches: mark, scan (one CTA), copy, remap.
#include "dcp_common.cuh"

namespace dcp {

struct CompactArgs {
  Layout L;
  const int32_t* topk;
  const int32_t* q_req;
  int Q, K;
  const int32_t* seq_lens;
  int B;
  const int32_t* bt;
  int max_vb;
  int64_t bt_rank_stride;
  int64_t nb;          // physical blocks per rank
  int32_t* mark;       // [dcp][nb]: 1 when referenced, then the compact index or -1
  int32_t* bounds;     // [dcp+1]: first compact index of each rank; bounds[dcp] = total
  int64_t max_blocks;  // capacity of the output buffer
  int32_t* err;
};

// (rank, physical block, in-block offset) of entry i, false when it does not resolve
__device__ __forceinline__ bool compact_entry(const CompactArgs& A, int64_t i, int& r,
                                              int64_t& phys, int& loc, bool& bad) {
  bad = false;
  const int q = (int)(i / A.K);
  const int b = __ldg(A.q_req + q);
  const int64_t g = __ldg(A.topk + i);
  if (b < 0 || b >= A.B || g < 0 || g >= __ldg(A.seq_lens + b)) return false;  // padding
  int64_t vb;
  place_token(g, A.L, r, vb, loc);
  phys = vb < A.max_vb ? (int64_t)__ldg(A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb + vb)
                       : (int64_t)-1;
  if (phys < 0 || phys >= A.nb) {
    bad = true;
    return false;
  }
  return true;
}

__global__ void compact_mark_kernel(CompactArgs A) {
  const int64_t n = (int64_t)A.Q * A.K;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int r, loc;
    int64_t phys;
    bool bad;
    if (compact_entry(A, i, r, phys, loc, bad)) A.mark[r * A.nb + phys] = 1;
  }
}

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) compact_scan_kernel(CompactArgs A, int dcp,
                                                                    int32_t* ids,
                                                                    int32_t* counts) {
  __shared__ int wsum[32];
  const int64_t n = (int64_t)dcp * A.nb;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t per = (n + kScanThreads - 1) / kScanThreads;
  const int64_t e0 = min(n, (int64_t)tid * per), e1 = min(n, e0 + per);
  int mine = 0;
  for (int64_t e = e0; e < e1; ++e) mine += A.mark[e] != 0;
  int x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wsum[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  int base = (w > 0 ? wsum[w - 1] : 0) + x - mine;
  if (A.nb == 0 && tid == 0)
    for (int r = 0; r < dcp; ++r) A.bounds[r] = 0;
  for (int64_t e = e0; e < e1; ++e) {
    if (e % A.nb == 0) A.bounds[e / A.nb] = base;  // first compact index of rank e / nb
    if (A.mark[e] != 0) {
      if (base < A.max_blocks) ids[base] = (int32_t)(e % A.nb);
      A.mark[e] = base++;
    } else {
      A.mark[e] = -1;
    }
  }
  __syncthreads();
  if (tid == 0) {
    A.bounds[dcp] = wsum[31];
    for (int r = 0; r < dcp; ++r) counts[r] = A.bounds[r + 1] - A.bounds[r];
  }
}

// one warp per compact block: bs rows of `row_chunks` 16-byte pieces
__global__ void compact_copy_kernel(CompactArgs A, int dcp, const int32_t* __restrict__ ids,
                                    dcp_rank_ptrs_t pools, int row_chunks, uint4* __restrict__ out) {
  const int total = A.bounds[dcp];
  const int64_t lim = total < A.max_blocks ? total : A.max_blocks;
  const int lane = threadIdx.x & 31;
  const int64_t per_block = (int64_t)A.L.bs * row_chunks;
  for (int64_t c = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); c < lim;
       c += (int64_t)gridDim.x * (blockDim.x >> 5)) {
    int r = 0;
    while (r + 1 < dcp && A.bounds[r + 1] <= c) ++r;
    const uint4* src = reinterpret_cast<const uint4*>(pools.ptr[r]) + (int64_t)ids[c] * per_block;
    uint4* dst = out + c * per_block;
    for (int64_t i = lane; i < per_block; i += 32) dst[i] = __ldg(src + i);
  }
}

__global__ void compact_remap_kernel(CompactArgs A, int64_t* __restrict__ index) {
  const int64_t n = (int64_t)A.Q * A.K;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int r, loc;
    int64_t phys;
    bool bad;
    int64_t out = -1;
    if (compact_entry(A, i, r, phys, loc, bad)) {
      const int64_t c = A.mark[r * A.nb + phys];
      if (c >= 0 && c < A.max_blocks)
        out = c * A.L.bs + loc;
      else
        bad = true;  // beyond the output capacity
    }
    if (bad) count_error(A.err);
    index[i] = out;
  }
}

}  // namespace dcp

using namespace dcp;

extern "C" {

int dcp_sfa_compact_workspace_size(dcp_layout_t layout, int64_t num_blocks, size_t* bytes) {
  if (!bytes || !layout_ok(layout) || num_blocks < 0) return DCP_EINVAL;
  *bytes = 256 + align_up(sizeof(int32_t) * (size_t)layout.dcp_size * (size_t)num_blocks, 256);
  return DCP_OK;
}

int dcp_sfa_compact_blocks(dcp_layout_t layout, const int32_t* topk, const int32_t* q_req,
                           int32_t num_queries, int32_t topk_len, const int32_t* seq_lens,
                           int32_t num_reqs, dcp_paged_kv_t kv, int32_t kv_dim, dcp_dtype_t dtype,
                           int64_t max_blocks, void* out_blocks, int32_t* out_block_ids,
                           int32_t* out_counts, int64_t* out_index, void* workspace,
                           size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_sfa_compact_blocks");
  const int es = dtype == DCP_F32 ? 4 : (dtype == DCP_BF16 ? 2 : 0);
  if (!layout_ok(layout) || es == 0 || num_queries < 0 || topk_len < 0 || num_reqs < 0 ||
      kv_dim < 1 || max_blocks < 0 || kv.num_blocks < 0 || kv.max_vblocks < 0 ||
      kv.bt_rank_stride < 0)
    return DCP_EINVAL;
  if ((kv_dim * es) % 16 != 0) return DCP_EUNSUPPORTED;
  if (!out_counts || !ranks_ok(kv.k, layout.dcp_size)) return DCP_EINVAL;
  size_t need = 0;
  dcp_sfa_compact_workspace_size(layout, kv.num_blocks, &need);
  if (!workspace || workspace_bytes < need) return DCP_EWORKSPACE;
  const int64_t n = (int64_t)num_queries * topk_len;
  if (n > 0 && (!topk || !q_req || !seq_lens || !kv.block_table || !out_index)) return DCP_EINVAL;
  if (max_blocks > 0 && (!out_blocks || !out_block_ids)) return DCP_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  CompactArgs A;
  A.L = Layout{layout.dcp_size, layout.block_size, layout.interleave};
  A.topk = topk;
  A.q_req = q_req;
  A.Q = num_queries;
  A.K = topk_len;
  A.seq_lens = seq_lens;
  A.B = num_reqs;
  A.bt = kv.block_table;
  A.max_vb = kv.max_vblocks;
  A.bt_rank_stride = kv.bt_rank_stride;
  A.nb = kv.num_blocks;
  A.bounds = (int32_t*)workspace;
  A.mark = (int32_t*)((char*)workspace + 256);
  A.max_blocks = max_blocks;
  A.err = err_count;
  const size_t mark_bytes = sizeof(int32_t) * (size_t)layout.dcp_size * (size_t)kv.num_blocks;
  if (cudaMemsetAsync(A.mark, 0, mark_bytes, s) != cudaSuccess) return DCP_ECUDA;
  const int sms = num_sms();
  if (n > 0) {
    const int64_t blocks = (n + 255) / 256;
    compact_mark_kernel<<<(int)(blocks < 8 * sms ? blocks : 8 * sms), 256, 0, s>>>(A);
  }
  compact_scan_kernel<<<1, kScanThreads, 0, s>>>(A, layout.dcp_size, out_block_ids, out_counts);
  if (max_blocks > 0) {
    const int64_t blocks = (max_blocks + 7) / 8;
    compact_copy_kernel<<<(int)(blocks < 8 * sms ? blocks : 8 * sms), 256, 0, s>>>(
        A, layout.dcp_size, out_block_ids, kv.k, kv_dim * es / 16, (uint4*)out_blocks);
  }
  if (n > 0) {
    const int64_t blocks = (n + 255) / 256;
    compact_remap_kernel<<<(int)(blocks < 8 * sms ? blocks : 8 * sms), 256, 0, s>>>(A, out_index);
  }
  return launch_status();
}

}  // extern "C"
