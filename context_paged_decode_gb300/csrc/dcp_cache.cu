// Owner-masked reshape-and-cache into the per-rank paged pools.
//
// Page "DeepSeek V4.1 context parallelism" (TokenSpeed), section "Cache
// ownership": every rank sees the write, writes translate virtual slots to
// local slots, and non-owners are masked.  The slot of each token on each
// rank comes from dcp_slot_mapping (-1 on non-owners).
#include "dcp_common.cuh"
#include "dcp_ptx.cuh"

namespace dcp {

// One thread moves one 16-byte chunk of one head row of one token, for every
// rank whose slot is valid.  Pools are [num_blocks][H][bs][row] per rank.
template <int NSRC>
__global__ void cache_write_kernel(const uint4* __restrict__ src0, const uint4* __restrict__ src1,
                                   int64_t T, int H, int chunks_per_row, int bs, int dcp,
                                   const int64_t* __restrict__ slot, int64_t num_slots,
                                   dcp_rank_ptrs_t dst0, dcp_rank_ptrs_t dst1, int32_t* err) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  griddep_wait();                // launched chained: the preceding kernel completed
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
    // every rank's slot is loaded before any store, so the thread waits for
    // memory once rather than once per rank
    int64_t sl[DCP_MAX_RANKS];
#pragma unroll
    for (int r = 0; r < DCP_MAX_RANKS; ++r) sl[r] = r < dcp ? __ldg(slot + (int64_t)r * T + t) : -1;
#pragma unroll
    for (int r = 0; r < DCP_MAX_RANKS; ++r) {
      if (r >= dcp) break;
      const int64_t s = sl[r];
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
  const uint4* u0 = (const uint4*)s0;
  const uint4* u1 = nsrc == 2 ? (const uint4*)s1 : nullptr;
  const cudaError_t e =
      nsrc == 2 ? launch_chained(cache_write_kernel<2>, (unsigned)grid, 256, 0, st, u0, u1, T, H,
                                 cpr, bs, dcp, slot, num_slots, d0, d1, err)
                : launch_chained(cache_write_kernel<1>, (unsigned)grid, 256, 0, st, u0, u1, T, H,
                                 cpr, bs, dcp, slot, num_slots, d0, d0, err);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

// Context gather: one warp per requested token resolves its owner rank and
// slot once, then copies the row in 16-byte pieces.  Unresolvable tokens get
// a zero row and are counted.
__global__ void gather_rows_kernel(Layout L, dcp_rank_ptrs_t pools, int64_t num_blocks,
                                   const int32_t* __restrict__ bt, int B, int max_vb,
                                   int64_t bt_rank_stride, const int32_t* __restrict__ req,
                                   const int64_t* __restrict__ pos, int64_t T, int cpr,
                                   uint4* __restrict__ out, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
       t += nwarps) {
    int owner = -1;
    int64_t slot = -1;
    if (lane == 0) {
      const int b = req[t];
      const int64_t x = pos[t];
      if (b >= 0 && b < B && x >= 0) {
        int r, loc;
        int64_t vb;
        place_token(x, L, r, vb, loc);
        const int64_t phys =
            vb < max_vb ? (int64_t)bt[r * bt_rank_stride + (int64_t)b * max_vb + vb] : -1;
        if (phys >= 0 && phys < num_blocks) {
          owner = r;
          slot = phys * L.bs + loc;
        }
      }
      if (owner < 0) count_error(err);
    }
    owner = __shfl_sync(0xffffffffu, owner, 0);
    slot = __shfl_sync(0xffffffffu, slot, 0);
    uint4* dst = out + t * cpr;
    if (owner < 0) {
      for (int c = lane; c < cpr; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(pools.ptr[owner]) + slot * cpr;
      for (int c = lane; c < cpr; c += 32) dst[c] = __ldg(src + c);
    }
  }
}

}  // namespace dcp

using namespace dcp;

static inline int elem_bytes(dcp_dtype_t d) { return d == DCP_F32 ? 4 : (d == DCP_BF16 ? 2 : 0); }

extern "C" {

int dcp_cache_write_gqa(dcp_layout_t layout, const void* k, const void* v, int64_t num_tokens,
                        int32_t num_kv_heads, int32_t head_dim, dcp_dtype_t dtype,
                        const int64_t* slot, int64_t num_blocks, dcp_rank_ptrs_t k_cache,
                        dcp_rank_ptrs_t v_cache, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_cache_write_gqa");
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
  dcp::NvtxRange nvtx_range("dcp_cache_write_mla");
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

int dcp_gather_context_mla(dcp_layout_t layout, dcp_paged_kv_t kv, int32_t num_reqs,
                           int32_t kv_dim, dcp_dtype_t dtype, const int32_t* req_idx,
                           const int64_t* positions, int64_t num_tokens, void* out,
                           int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_gather_context_mla");
  const int es = elem_bytes(dtype);
  if (!layout_ok(layout) || es == 0 || num_reqs < 0 || num_tokens < 0 || kv_dim < 1 ||
      kv.num_blocks < 0 || kv.max_vblocks < 0 || kv.bt_rank_stride < 0)
    return DCP_EINVAL;
  if ((kv_dim * es) % 16 != 0) return DCP_EUNSUPPORTED;
  if (num_tokens == 0) return DCP_OK;
  if (!req_idx || !positions || !out || !kv.block_table || !ranks_ok(kv.k, layout.dcp_size))
    return DCP_EINVAL;
  const Layout L{layout.dcp_size, layout.block_size, layout.interleave};
  const int64_t blocks = (num_tokens + 7) / 8;
  const int grid = (int)(blocks < 16 * num_sms() ? blocks : 16 * num_sms());
  gather_rows_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
      L, kv.k, kv.num_blocks, kv.block_table, num_reqs, kv.max_vblocks, kv.bt_rank_stride,
      req_idx, positions, num_tokens, kv_dim * es / 16, (uint4*)out, err_count);
  return launch_status();
}

}  // extern "C"
