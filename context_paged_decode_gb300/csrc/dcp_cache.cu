// Owner-masked reshape-and-cache into the per-rank paged pools.
//
// Page "DeepSeek V4.1 context parallelism" (TokenSpeed), section "Cache
// ownership": every rank sees the write, writes translate virtual slots to
// local slots, and non-owners are masked.  The slot of each token on each
// rank comes from dcp_slot_mapping (-1 on non-owners).
#include "dcp_common.cuh"

namespace dcp {

// One thread moves one 16-byte chunk of one head row of one token, for every
// rank whose slot is valid.  Pools are [num_blocks][H][bs][row] per rank.
template <int NSRC>
__global__ void cache_write_kernel(const uint4* __restrict__ src0, const uint4* __restrict__ src1,
                                   int64_t T, int H, int chunks_per_row, int bs, int dcp,
                                   const int64_t* __restrict__ slot, int64_t num_slots,
                                   dcp_rank_ptrs_t dst0, dcp_rank_ptrs_t dst1, int32_t* err) {
  const int64_t per_tok = (int64_t)H * chunks_per_row;
  const int64_t n = T * per_tok;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / per_tok;
    const int rem = (int)(i - t * per_tok);
    const int h = rem / chunks_per_row, c = rem % chunks_per_row;
    const uint4 a = __ldg(src0 + i);
    uint4 b = make_uint4(0, 0, 0, 0);
    if (NSRC == 2) b = __ldg(src1 + i);
    for (int r = 0; r < dcp; ++r) {
      const int64_t s = __ldg(slot + (int64_t)r * T + t);
      if (s < 0 || s >= num_slots) {
        if (s != -1 && rem == 0) count_error(err);
        continue;
      }
      const int64_t blk = s / bs, off = s - blk * bs;
      const int64_t e = (((blk * H + h) * bs + off) * chunks_per_row) + c;
      reinterpret_cast<uint4*>(dst0.ptr[r])[e] = a;
      if (NSRC == 2) reinterpret_cast<uint4*>(dst1.ptr[r])[e] = b;
    }
  }
}

static int launch_cache_write(int nsrc, const void* s0, const void* s1, int64_t T, int H,
                              int row_bytes, int bs, int dcp, const int64_t* slot,
                              int64_t num_blocks, const dcp_rank_ptrs_t& d0,
                              const dcp_rank_ptrs_t& d1, int32_t* err, cudaStream_t st) {
  const int cpr = row_bytes / 16;
  const int64_t n = T * H * cpr;
  const int64_t blocks = (n + 255) / 256;
  const int grid = (int)(blocks < 16 * num_sms() ? blocks : 16 * num_sms());
  const int64_t num_slots = num_blocks * bs;
  if (nsrc == 2)
    cache_write_kernel<2><<<grid, 256, 0, st>>>((const uint4*)s0, (const uint4*)s1, T, H, cpr, bs,
                                                dcp, slot, num_slots, d0, d1, err);
  else
    cache_write_kernel<1><<<grid, 256, 0, st>>>((const uint4*)s0, nullptr, T, H, cpr, bs, dcp,
                                                slot, num_slots, d0, d0, err);
  return launch_status();
}

}  // namespace dcp

using namespace dcp;

static inline int elem_bytes(dcp_dtype_t d) { return d == DCP_F32 ? 4 : (d == DCP_BF16 ? 2 : 0); }

extern "C" {

int dcp_cache_write_gqa(dcp_layout_t layout, const void* k, const void* v, int64_t num_tokens,
                        int32_t num_kv_heads, int32_t head_dim, dcp_dtype_t dtype,
                        const int64_t* slot, int64_t num_blocks, dcp_rank_ptrs_t k_cache,
                        dcp_rank_ptrs_t v_cache, int32_t* err_count, dcp_stream_t stream) {
  const int es = elem_bytes(dtype);
  if (!layout_ok(layout) || es == 0 || num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 ||
      num_blocks < 0)
    return DCP_EINVAL;
  if ((head_dim * es) % 16 != 0) return DCP_EUNSUPPORTED;
  if (num_tokens == 0) return DCP_OK;
  if (!k || !v || !slot || !ranks_ok(k_cache, layout.dcp_size) ||
      !ranks_ok(v_cache, layout.dcp_size))
    return DCP_EINVAL;
  return launch_cache_write(2, k, v, num_tokens, num_kv_heads, head_dim * es, layout.block_size,
                            layout.dcp_size, slot, num_blocks, k_cache, v_cache, err_count,
                            (cudaStream_t)stream);
}

int dcp_cache_write_mla(dcp_layout_t layout, const void* kv, int64_t num_tokens, int32_t kv_dim,
                        dcp_dtype_t dtype, const int64_t* slot, int64_t num_blocks,
                        dcp_rank_ptrs_t cache, int32_t* err_count, dcp_stream_t stream) {
  const int es = elem_bytes(dtype);
  if (!layout_ok(layout) || es == 0 || num_tokens < 0 || kv_dim < 1 || num_blocks < 0)
    return DCP_EINVAL;
  if ((kv_dim * es) % 16 != 0) return DCP_EUNSUPPORTED;
  if (num_tokens == 0) return DCP_OK;
  if (!kv || !slot || !ranks_ok(cache, layout.dcp_size)) return DCP_EINVAL;
  return launch_cache_write(1, kv, nullptr, num_tokens, 1, kv_dim * es, layout.block_size,
                            layout.dcp_size, slot, num_blocks, cache, cache, err_count,
                            (cudaStream_t)stream);
}

}  // extern "C"
