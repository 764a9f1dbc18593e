// Exact LSE merge of partial attention results (+ optional sink applied once).
//
// Page "Decode Context Parallel (DCP)", section "Backend structure" (the
// common partial-output/LSE merge) and page "DeepSeek V4.1 context
// parallelism", section "Decode computation" (the sink is applied once when
// the partial outputs are merged by log-sum-exp):
//     lse = ln(sum_i exp(lse_i) + exp(sink)),  o = sum_i exp(lse_i - lse) o_i.
// HBM-bound: one warp per output row (or per 128-value chunk of a row when
// there are at most 16 parts), 16-byte loads of the partials.
#include <utility>

#include "dcp_common.cuh"
#include "dcp_merge.cuh"
#include "dcp_ptx.cuh"

namespace dcp {

struct DensePlusOne {  // n dense parts [n][B][H][dv] and one more part [B][H][dv]
  const float* o;
  const float* lse;
  int64_t stride;  // B*H
  int n;
  const float* xo;
  const float* xlse;
  __device__ __forceinline__ float lse_at(int i, int64_t row) const {
    return i < n ? lse[i * stride + row] : xlse[row];
  }
  __device__ __forceinline__ const float* o_at(int i, int64_t row, int dv) const {
    return i < n ? o + (i * stride + row) * dv : xo + row * dv;
  }
  __device__ __forceinline__ float4 load4(const float4* p) const { return __ldg(p); }
};

struct ItemParts {  // plan items: lse [item][G], o [item][G][dv]
  const float* o;
  const float* lse;
  int first, G, hh;
  __device__ __forceinline__ float lse_at(int i, int64_t) const {
    return lse[(int64_t)(first + i) * G + hh];
  }
  __device__ __forceinline__ const float* o_at(int i, int64_t, int dv) const {
    return o + ((int64_t)(first + i) * G + hh) * dv;
  }
};

// Parts read per round of loads: 16 for rows of up to 128 values (one float4
// per lane and part), fewer for wider rows, so a round holds 16 float4 per lane.
template <int CH>
constexpr int parts_per_round() {
  return CH == 1 ? 16 : (CH == 2 ? 8 : 4);
}

// One warp per output row.  With at most 32 parts, lane i holds part i's
// LSE, so the maximum, the sum and every part's weight come from one round
// of loads and warp shuffles; the partial rows are then read PG parts at a
// time, all loads of a group issued before any is used.  More parts take the
// same steps in blocks of 32.
template <int CH, class Parts>
__device__ __forceinline__ void merge_row(const Parts& P, int n, int64_t row, int dv,
                                          bool has_sink, float sink, void* out, int out_dtype,
                                          int64_t out_row, float* out_lse) {
  constexpr int PG = parts_per_round<CH>();
  const int lane = threadIdx.x & 31;
  const int nv = dv >> 2;
  const float l_mine = lane < n ? P.lse_at(lane, row) : -INFINITY;
  float m = has_sink ? sink : -INFINITY;
  m = fmaxf(m, l_mine);
  for (int i = 32 + lane; i < n; i += 32) m = fmaxf(m, P.lse_at(i, row));
  m = warp_max(m);
  if (m == -INFINITY) {  // nothing attended and no sink
    for (int c = lane; c < nv; c += 32) {
      if (out_dtype == DCP_F32)
        reinterpret_cast<float4*>(out)[out_row * nv + c] = make_float4(0.f, 0.f, 0.f, 0.f);
      else
        reinterpret_cast<uint2*>(out)[out_row * nv + c] = make_uint2(0u, 0u);
    }
    if (out_lse && lane == 0) out_lse[out_row] = -INFINITY;
    return;
  }
  float s = l_mine != -INFINITY ? expf(l_mine - m) : 0.f;
  for (int i = 32 + lane; i < n; i += 32) {
    const float l = P.lse_at(i, row);
    if (l != -INFINITY) s += expf(l - m);
  }
  s = warp_sum(s);  // identical on every lane
  if (has_sink) s += expf(sink - m);
  const float lse = m + logf(s);
  float4 acc[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int blk = 0; blk < n; blk += 32) {
    float wl = 0.f;
    if (blk + lane < n) {
      const float l = blk == 0 ? l_mine : P.lse_at(blk + lane, row);
      wl = l == -INFINITY ? 0.f : expf(l - lse);
    }
    const int cnt = min(32, n - blk);
    for (int i0 = 0; i0 < cnt; i0 += PG) {
      // up to PG parts: every load first, then the weighted sums in part order
      float4 v[PG][CH];
#pragma unroll
      for (int q = 0; q < PG; ++q) {
        const float4* src =
            reinterpret_cast<const float4*>(P.o_at(blk + min(i0 + q, cnt - 1), row, dv));
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int idx = lane + 32 * c;
          v[q][c] = (i0 + q < cnt && idx < nv) ? __ldg(src + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < PG; ++q) {
        const float w = __shfl_sync(0xffffffffu, wl, min(i0 + q, 31));
        if (i0 + q < cnt && w != 0.f) {  // an empty part adds nothing, whatever its o holds
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            acc[c].x = fmaf(w, v[q][c].x, acc[c].x);
            acc[c].y = fmaf(w, v[q][c].y, acc[c].y);
            acc[c].z = fmaf(w, v[q][c].z, acc[c].z);
            acc[c].w = fmaf(w, v[q][c].w, acc[c].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int idx = lane + 32 * c;
    if (idx < nv) {
      if (out_dtype == DCP_F32)
        reinterpret_cast<float4*>(out)[out_row * nv + idx] = acc[c];
      else
        reinterpret_cast<uint2*>(out)[out_row * nv + idx] =
            make_uint2(pack_bf16(acc[c].x, acc[c].y), pack_bf16(acc[c].z, acc[c].w));
    }
  }
  if (out_lse && lane == 0) out_lse[out_row] = lse;
}

// The same merge with one CTA of kWideWarps warps per output row, for calls
// with too few rows to fill the GPU one warp per row (a long request split
// into hundreds of parts).  Warp w takes parts [n w / W, n (w+1) / W); the
// warps' maxima, sums and weighted partial rows are combined in shared
// memory in warp order, so the result does not depend on timing.
constexpr int kWideWarps = 8;

template <int CH, class Parts>
__device__ __forceinline__ void merge_row_wide(const Parts& P, int n, int64_t row, int dv,
                                               bool has_sink, float sink, void* out,
                                               int out_dtype, int64_t out_row, float* out_lse) {
  extern __shared__ float4 wide_acc[];               // [kWideWarps][nv]
  __shared__ float wm[kWideWarps], ws[kWideWarps];
  constexpr int PG = parts_per_round<CH>();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nv = dv >> 2;
  const int p0 = (int)((int64_t)n * w / kWideWarps), p1 = (int)((int64_t)n * (w + 1) / kWideWarps);
  float m = -INFINITY;
  for (int i = p0 + lane; i < p1; i += 32) m = fmaxf(m, P.lse_at(i, row));
  m = warp_max(m);
  if (lane == 0) wm[w] = m;
  __syncthreads();
  m = has_sink ? sink : -INFINITY;
  for (int i = 0; i < kWideWarps; ++i) m = fmaxf(m, wm[i]);
  if (m == -INFINITY) {  // nothing attended and no sink
    for (int c = threadIdx.x; c < nv; c += blockDim.x) {
      if (out_dtype == DCP_F32)
        reinterpret_cast<float4*>(out)[out_row * nv + c] = make_float4(0.f, 0.f, 0.f, 0.f);
      else
        reinterpret_cast<uint2*>(out)[out_row * nv + c] = make_uint2(0u, 0u);
    }
    if (out_lse && threadIdx.x == 0) out_lse[out_row] = -INFINITY;
    return;
  }
  float s = 0.f;
  for (int i = p0 + lane; i < p1; i += 32) {
    const float l = P.lse_at(i, row);
    if (l != -INFINITY) s += expf(l - m);
  }
  s = warp_sum(s);
  if (lane == 0) ws[w] = s;
  __syncthreads();
  s = 0.f;
  for (int i = 0; i < kWideWarps; ++i) s += ws[i];
  if (has_sink) s += expf(sink - m);
  const float lse = m + logf(s);
  float4 acc[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int blk = p0; blk < p1; blk += 32) {
    float wl = 0.f;
    if (blk + lane < p1) {
      const float l = P.lse_at(blk + lane, row);
      wl = l == -INFINITY ? 0.f : expf(l - lse);
    }
    const int cnt = min(32, p1 - blk);
    for (int i0 = 0; i0 < cnt; i0 += PG) {
      float4 v[PG][CH];
#pragma unroll
      for (int q = 0; q < PG; ++q) {
        const float4* src =
            reinterpret_cast<const float4*>(P.o_at(blk + min(i0 + q, cnt - 1), row, dv));
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int idx = lane + 32 * c;
          v[q][c] = (i0 + q < cnt && idx < nv) ? __ldg(src + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < PG; ++q) {
        const float wt = __shfl_sync(0xffffffffu, wl, min(i0 + q, 31));
        if (i0 + q < cnt && wt != 0.f) {
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            acc[c].x = fmaf(wt, v[q][c].x, acc[c].x);
            acc[c].y = fmaf(wt, v[q][c].y, acc[c].y);
            acc[c].z = fmaf(wt, v[q][c].z, acc[c].z);
            acc[c].w = fmaf(wt, v[q][c].w, acc[c].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int idx = lane + 32 * c;
    if (idx < nv) wide_acc[w * nv + idx] = acc[c];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nv; c += blockDim.x) {
    float4 t = wide_acc[c];
    for (int i = 1; i < kWideWarps; ++i) {
      const float4 u = wide_acc[i * nv + c];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    if (out_dtype == DCP_F32)
      reinterpret_cast<float4*>(out)[out_row * nv + c] = t;
    else
      reinterpret_cast<uint2*>(out)[out_row * nv + c] =
          make_uint2(pack_bf16(t.x, t.y), pack_bf16(t.z, t.w));
  }
  if (out_lse && threadIdx.x == 0) out_lse[out_row] = lse;
}

template <int CH>
__global__ void dense_merge_kernel(int n, const float* __restrict__ po,
                                   const float* __restrict__ pl, int B, int H, int dv,
                                   const float* __restrict__ sink, void* out, int out_dtype,
                                   float* out_lse) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  griddep_wait();   // launched as a dependent: the partials are complete past this point
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= (int64_t)B * H) return;
  const int h = (int)(row % H);
  DenseParts P{po, pl, (int64_t)B * H};
  merge_row<CH>(P, n, row, dv, sink != nullptr, sink ? sink[h] : 0.f, out, out_dtype, row,
                out_lse);
}

template <int CH>
__global__ void dense_plus_one_merge_kernel(int n, const float* __restrict__ po,
                                            const float* __restrict__ pl,
                                            const float* __restrict__ xo,
                                            const float* __restrict__ xl, int B, int H, int dv,
                                            const float* __restrict__ sink, void* out,
                                            int out_dtype, float* out_lse) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= (int64_t)B * H) return;
  const int h = (int)(row % H);
  DensePlusOne P{po, pl, (int64_t)B * H, n, xo, xl};
  merge_row<CH>(P, n + 1, row, dv, sink != nullptr, sink ? sink[h] : 0.f, out, out_dtype, row,
                out_lse);
}

template <int NP>
__global__ void dense_merge_chunk_kernel(int n, const float* __restrict__ po,
                                         const float* __restrict__ pl, int B, int H, int dv,
                                         int chunks, const float* __restrict__ sink, void* out,
                                         int out_dtype, float* out_lse) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  griddep_wait();   // launched as a dependent: the partials are complete past this point
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t row = wid / chunks;
  if (row >= (int64_t)B * H) return;
  const int chunk = (int)(wid - row * chunks);
  const int h = (int)(row % H);
  DenseParts P{po, pl, (int64_t)B * H};
  merge_chunk<NP>(P, n, row, dv, chunk, sink != nullptr, sink ? sink[h] : 0.f, out, out_dtype,
                  row, out_lse);
}

template <int NP>
__global__ void dense_plus_one_merge_chunk_kernel(int n, const float* __restrict__ po,
                                                  const float* __restrict__ pl,
                                                  const float* __restrict__ xo,
                                                  const float* __restrict__ xl, int B, int H,
                                                  int dv, int chunks,
                                                  const float* __restrict__ sink, void* out,
                                                  int out_dtype, float* out_lse) {
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t row = wid / chunks;
  if (row >= (int64_t)B * H) return;
  const int chunk = (int)(wid - row * chunks);
  const int h = (int)(row % H);
  DensePlusOne P{po, pl, (int64_t)B * H, n, xo, xl};
  merge_chunk<NP>(P, n + 1, row, dv, chunk, sink != nullptr, sink ? sink[h] : 0.f, out,
                  out_dtype, row, out_lse);
}

// mode 0: row = (b, h), parts = all items of (b, g) over every rank; sink applies.
// mode 1: row = (r, b, h), parts = items of (b, g, r); output is float32 per rank.
template <int CH>
__global__ void item_merge_kernel(Plan plan, int mode, int B, int dcp, int Hq, int G, int groups,
                                  int dv, const float* __restrict__ sink, void* out,
                                  int out_dtype, float* out_lse) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nrows = (int64_t)(mode == 0 ? 1 : dcp) * B * Hq;
  if (row >= nrows) return;
  const int h = (int)(row % Hq);
  const int b = (int)((row / Hq) % B);
  const int r = mode == 0 ? 0 : (int)(row / ((int64_t)B * Hq));
  const int g = h / G, hh = h % G;
  const int e = (b * groups + g) * dcp;
  const int first = plan.off[e + r];
  const int last = plan.off[e + (mode == 0 ? dcp : r + 1)];
  ItemParts P{plan.o, plan.lse, first, G, hh};
  const bool hs = (mode == 0) && sink != nullptr;
  merge_row<CH>(P, last - first, row, dv, hs, hs ? sink[h] : 0.f, out,
            mode == 0 ? out_dtype : (int)DCP_F32, row, out_lse);
}

// item_merge_kernel with one CTA per output row (merge_row_wide).
template <int CH>
__global__ void __launch_bounds__(kWideWarps * 32)
item_merge_wide_kernel(Plan plan, int mode, int B, int dcp, int Hq, int G, int groups, int dv,
                       const float* __restrict__ sink, void* out, int out_dtype, float* out_lse) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  const int64_t row = blockIdx.x;
  const int h = (int)(row % Hq);
  const int b = (int)((row / Hq) % B);
  const int r = mode == 0 ? 0 : (int)(row / ((int64_t)B * Hq));
  const int g = h / G, hh = h % G;
  const int e = (b * groups + g) * dcp;
  const int first = plan.off[e + r];
  const int last = plan.off[e + (mode == 0 ? dcp : r + 1)];
  ItemParts P{plan.o, plan.lse, first, G, hh};
  const bool hs = (mode == 0) && sink != nullptr;
  merge_row_wide<CH>(P, last - first, row, dv, hs, hs ? sink[h] : 0.f, out,
                     mode == 0 ? out_dtype : (int)DCP_F32, row, out_lse);
}

int launch_item_merge(const Plan& plan, int mode, int B, int dcp, int Hq, int G, int groups,
                      int dv, const float* sink, void* out, int out_dtype, float* out_lse,
                      cudaStream_t s) {
  const int64_t rows = (int64_t)(mode == 0 ? 1 : dcp) * B * Hq;
  if (rows == 0) return DCP_OK;
  const int nv = dv / 4;
  if (rows < 4 * (int64_t)num_sms()) {
    // few rows (few, long requests): one CTA of kWideWarps warps per row
    const size_t smem = (size_t)kWideWarps * nv * sizeof(float4);
#define DCP_ITEM_WIDE(CH)                                                                      \
  item_merge_wide_kernel<CH><<<(unsigned)rows, kWideWarps * 32, smem, s>>>(                    \
      plan, mode, B, dcp, Hq, G, groups, dv, sink, out, out_dtype, out_lse)
    if (nv <= 32)
      DCP_ITEM_WIDE(1);
    else if (nv <= 64)
      DCP_ITEM_WIDE(2);
    else if (nv <= 128)
      DCP_ITEM_WIDE(4);
    else
      DCP_ITEM_WIDE(8);
#undef DCP_ITEM_WIDE
    return launch_status();
  }
  const int wpb = 8;
  const unsigned grid = (unsigned)((rows + wpb - 1) / wpb);
  if (nv <= 32)
    item_merge_kernel<1><<<grid, wpb * 32, 0, s>>>(plan, mode, B, dcp, Hq, G, groups, dv, sink,
                                                   out, out_dtype, out_lse);
  else if (nv <= 64)
    item_merge_kernel<2><<<grid, wpb * 32, 0, s>>>(plan, mode, B, dcp, Hq, G, groups, dv, sink,
                                                   out, out_dtype, out_lse);
  else if (nv <= 128)
    item_merge_kernel<4><<<grid, wpb * 32, 0, s>>>(plan, mode, B, dcp, Hq, G, groups, dv, sink,
                                                   out, out_dtype, out_lse);
  else
    item_merge_kernel<8><<<grid, wpb * 32, 0, s>>>(plan, mode, B, dcp, Hq, G, groups, dv, sink,
                                                   out, out_dtype, out_lse);
  return launch_status();
}

}  // namespace dcp

using namespace dcp;

namespace dcp {

namespace {

template <typename... Exp, typename... Act>
cudaError_t launch_maybe_pdl(bool pdl, void (*kernel)(Exp...), unsigned grid, unsigned block,
                             cudaStream_t st, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

}  // namespace

int launch_dense_merge(int num_parts, const float* part_o, const float* part_lse, int B, int H,
                       int dv, const float* sink, void* out, int out_dtype, float* out_lse,
                       cudaStream_t st, bool pdl) {
  const int64_t rows = (int64_t)B * H;
  if (rows == 0) return DCP_OK;
  const int wpb = 8;
  const int nv = dv / 4;
  cudaError_t e;
  if (num_parts <= 16) {
    const int chunks = (nv + 31) / 32;
    const unsigned cgrid = (unsigned)((rows * chunks + wpb - 1) / wpb);
    auto k = num_parts <= 4 ? dense_merge_chunk_kernel<4>
             : num_parts <= 8 ? dense_merge_chunk_kernel<8> : dense_merge_chunk_kernel<16>;
    e = launch_maybe_pdl(pdl, k, cgrid, wpb * 32, st, num_parts, part_o, part_lse, B, H, dv,
                         chunks, sink, out, out_dtype, out_lse);
  } else {
    const unsigned grid = (unsigned)((rows + wpb - 1) / wpb);
    auto k = nv <= 32 ? dense_merge_kernel<1>
             : nv <= 64 ? dense_merge_kernel<2> : nv <= 128 ? dense_merge_kernel<4>
                                                            : dense_merge_kernel<8>;
    e = launch_maybe_pdl(pdl, k, grid, wpb * 32, st, num_parts, part_o, part_lse, B, H, dv, sink,
                         out, out_dtype, out_lse);
  }
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

}  // namespace dcp

extern "C" int dcp_lse_merge(int32_t num_parts, const float* part_o, const float* part_lse,
                             int32_t num_reqs, int32_t num_heads, int32_t head_dim_v,
                             const float* sink, void* out, dcp_dtype_t out_dtype, float* out_lse,
                             dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_lse_merge");
  if (num_parts < 0 || num_reqs < 0 || num_heads < 0 || head_dim_v < 4 || head_dim_v % 4 != 0 ||
      head_dim_v > 1024 || (out_dtype != DCP_F32 && out_dtype != DCP_BF16))
    return DCP_EINVAL;
  const int64_t rows = (int64_t)num_reqs * num_heads;
  if (rows == 0) return DCP_OK;
  if (!out || (num_parts > 0 && (!part_o || !part_lse))) return DCP_EINVAL;
  return launch_dense_merge(num_parts, part_o, part_lse, num_reqs, num_heads, head_dim_v, sink,
                            out, (int)out_dtype, out_lse, (cudaStream_t)stream, false);
}

extern "C" int dcp_lse_merge_swa(int32_t num_parts, const float* part_o, const float* part_lse,
                                 const float* swa_o, const float* swa_lse, int32_t num_reqs,
                                 int32_t num_heads, int32_t head_dim_v, const float* sink,
                                 void* out, dcp_dtype_t out_dtype, float* out_lse,
                                 dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_lse_merge_swa");
  if (num_parts < 0 || num_reqs < 0 || num_heads < 0 || head_dim_v < 4 || head_dim_v % 4 != 0 ||
      head_dim_v > 1024 || (out_dtype != DCP_F32 && out_dtype != DCP_BF16))
    return DCP_EINVAL;
  const int64_t rows = (int64_t)num_reqs * num_heads;
  if (rows == 0) return DCP_OK;
  if (!out || !swa_o || !swa_lse || (num_parts > 0 && (!part_o || !part_lse))) return DCP_EINVAL;
  const int wpb = 8;
  cudaStream_t st = (cudaStream_t)stream;
  const int nv = head_dim_v / 4;
  if (num_parts + 1 <= 16) {
    const int chunks = (nv + 31) / 32;
    const unsigned cgrid = (unsigned)((rows * chunks + wpb - 1) / wpb);
#define DCP_MERGE_SWA_CHUNK(NP)                                                                  \
  dense_plus_one_merge_chunk_kernel<NP><<<cgrid, wpb * 32, 0, st>>>(                             \
      num_parts, part_o, part_lse, swa_o, swa_lse, num_reqs, num_heads, head_dim_v, chunks, sink, \
      out, (int)out_dtype, out_lse)
    if (num_parts + 1 <= 4)
      DCP_MERGE_SWA_CHUNK(4);
    else if (num_parts + 1 <= 8)
      DCP_MERGE_SWA_CHUNK(8);
    else
      DCP_MERGE_SWA_CHUNK(16);
#undef DCP_MERGE_SWA_CHUNK
    return launch_status();
  }
  const unsigned grid = (unsigned)((rows + wpb - 1) / wpb);
#define DCP_MERGE_SWA(CH)                                                                  \
  dense_plus_one_merge_kernel<CH><<<grid, wpb * 32, 0, st>>>(                              \
      num_parts, part_o, part_lse, swa_o, swa_lse, num_reqs, num_heads, head_dim_v, sink, \
      out, (int)out_dtype, out_lse)
  if (nv <= 32)
    DCP_MERGE_SWA(1);
  else if (nv <= 64)
    DCP_MERGE_SWA(2);
  else if (nv <= 128)
    DCP_MERGE_SWA(4);
  else
    DCP_MERGE_SWA(8);
#undef DCP_MERGE_SWA
  return launch_status();
}
