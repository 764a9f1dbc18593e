// Exact LSE merge of partial attention results for one 128-value chunk of
// an output row (shared by the merge kernels and the fused SFA decode).
//
// Page "Decode Context Parallel (DCP)", section "Backend structure" (the
// common partial-output/LSE merge) and page "DeepSeek V4.1 context
// parallelism", section "Decode computation" (the sink is applied once when
// the partial outputs are merged by log-sum-exp):
//     lse = ln(sum_i exp(lse_i) + exp(sink)),  o = sum_i exp(lse_i - lse) o_i.
#pragma once

#include "dcp_common.cuh"

namespace dcp {

struct DenseParts {  // part_o [n][B][H][dv], part_lse [n][B][H]
  const float* o;
  const float* lse;
  int64_t stride;  // B*H
  __device__ __forceinline__ float lse_at(int i, int64_t row) const { return lse[i * stride + row]; }
  __device__ __forceinline__ const float* o_at(int i, int64_t row, int dv) const {
    return o + (i * stride + row) * dv;
  }
  // partials written by an earlier kernel: the read-only path
  __device__ __forceinline__ float4 load4(const float4* p) const { return __ldg(p); }
};

// The same partials written earlier in the same kernel by other CTAs: loads
// that bypass the SM's L1 (read at L2, the point of coherence).
struct DensePartsL2 : DenseParts {
  __device__ __forceinline__ float lse_at(int i, int64_t row) const {
    return __ldcg(lse + i * stride + row);
  }
  __device__ __forceinline__ float4 load4(const float4* p) const { return __ldcg(p); }
};


// The same merge with one warp per (output row, 128-value chunk), for calls
// with at most NP parts: every part's LSE and its 128 values are loaded
// before any is used, so a warp waits for memory once, and there are four
// warps per 512-wide row to hide that wait.  The arithmetic and its order are
// those of merge_row, so the output is bitwise the same.
template <int NP, class Parts>
__device__ __forceinline__ void merge_chunk(const Parts& P, int n, int64_t row, int dv, int chunk,
                                            bool has_sink, float sink, void* out, int out_dtype,
                                            int64_t out_row, float* out_lse) {
  const int lane = threadIdx.x & 31;
  const int nv = dv >> 2;
  const int idx = chunk * 32 + lane;                 // float4 of the row
  const bool act = idx < nv;
  const float l_mine = lane < n ? P.lse_at(lane, row) : -INFINITY;
  float4 v[NP];
#pragma unroll
  for (int i = 0; i < NP; ++i)
    v[i] = (i < n && act) ? P.load4(reinterpret_cast<const float4*>(P.o_at(i, row, dv)) + idx)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
  float m = has_sink ? sink : -INFINITY;
  m = fmaxf(m, l_mine);
  m = warp_max(m);
  if (m == -INFINITY) {  // nothing attended and no sink
    if (act) {
      if (out_dtype == DCP_F32)
        reinterpret_cast<float4*>(out)[out_row * nv + idx] = make_float4(0.f, 0.f, 0.f, 0.f);
      else
        reinterpret_cast<uint2*>(out)[out_row * nv + idx] = make_uint2(0u, 0u);
    }
    if (out_lse && chunk == 0 && lane == 0) out_lse[out_row] = -INFINITY;
    return;
  }
  float s = l_mine != -INFINITY ? expf(l_mine - m) : 0.f;
  s = warp_sum(s);
  if (has_sink) s += expf(sink - m);
  const float lse = m + logf(s);
  const float wl = l_mine == -INFINITY ? 0.f : expf(l_mine - lse);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const float w = __shfl_sync(0xffffffffu, wl, i);
    if (i < n && w != 0.f) {  // an empty part adds nothing, whatever its o holds
      acc.x = fmaf(w, v[i].x, acc.x);
      acc.y = fmaf(w, v[i].y, acc.y);
      acc.z = fmaf(w, v[i].z, acc.z);
      acc.w = fmaf(w, v[i].w, acc.w);
    }
  }
  if (act) {
    if (out_dtype == DCP_F32)
      reinterpret_cast<float4*>(out)[out_row * nv + idx] = acc;
    else
      reinterpret_cast<uint2*>(out)[out_row * nv + idx] =
          make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  }
  if (out_lse && chunk == 0 && lane == 0) out_lse[out_row] = lse;
}

// merge_chunk for every chunk of a row at once (CH chunks of 128 values):
// every part's values of the whole row are loaded before any is used, so a
// warp waits for memory once per row.  The arithmetic and its order are those
// of merge_chunk, chunk by chunk, so the output is bitwise the same.
template <int NP, int CH, class Parts>
__device__ __forceinline__ void merge_row_chunks(const Parts& P, int n, int64_t row, bool has_sink,
                                                 float sink, void* out, int out_dtype,
                                                 int64_t out_row, float* out_lse) {
  constexpr int nv = CH * 32;                        // float4 of the row
  const int lane = threadIdx.x & 31;
  const float l_mine = lane < n ? P.lse_at(lane, row) : -INFINITY;
  float4 v[CH][NP];
#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int i = 0; i < NP; ++i)
      v[c][i] = i < n ? P.load4(reinterpret_cast<const float4*>(P.o_at(i, row, 4 * nv)) + c * 32 +
                                lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  float m = has_sink ? sink : -INFINITY;
  m = fmaxf(m, l_mine);
  m = warp_max(m);
  if (m == -INFINITY) {  // nothing attended and no sink
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (out_dtype == DCP_F32)
        reinterpret_cast<float4*>(out)[out_row * nv + c * 32 + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
      else
        reinterpret_cast<uint2*>(out)[out_row * nv + c * 32 + lane] = make_uint2(0u, 0u);
    }
    if (out_lse && lane == 0) out_lse[out_row] = -INFINITY;
    return;
  }
  float s = l_mine != -INFINITY ? expf(l_mine - m) : 0.f;
  s = warp_sum(s);
  if (has_sink) s += expf(sink - m);
  const float lse = m + logf(s);
  const float wl = l_mine == -INFINITY ? 0.f : expf(l_mine - lse);
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const float w = __shfl_sync(0xffffffffu, wl, i);
      if (i < n && w != 0.f) {  // an empty part adds nothing, whatever its o holds
        acc.x = fmaf(w, v[c][i].x, acc.x);
        acc.y = fmaf(w, v[c][i].y, acc.y);
        acc.z = fmaf(w, v[c][i].z, acc.z);
        acc.w = fmaf(w, v[c][i].w, acc.w);
      }
    }
    if (out_dtype == DCP_F32)
      reinterpret_cast<float4*>(out)[out_row * nv + c * 32 + lane] = acc;
    else
      reinterpret_cast<uint2*>(out)[out_row * nv + c * 32 + lane] =
          make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  }
  if (out_lse && lane == 0) out_lse[out_row] = lse;
}

}  // namespace dcp
