// CUDA-core split-KV decode partials for any supported shape and dtype.
//
// Used for fp32 caches and for shapes the tensor-core kernels do not cover.
// One warp per (work item, query head): lane i holds dims i, i+32, ... of q
// and of the running output; each token costs one warp reduction.  Slow but
// exact in fp32 arithmetic.  Work items come from the split-KV plan (items
// never cross a rank: each shard attends only its local tokens, page "Decode
// Context Parallel (DCP)", section "Decode").
#include "dcp_generic.cuh"

namespace dcp {

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}

constexpr int kGenWarps = 8;
constexpr int kGenMaxPerLane = 32;  // dims up to 1024

template <typename T>
__global__ void __launch_bounds__(kGenWarps * 32)
split_generic_kernel(GenericArgs A, Plan plan) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_items = plan.hdr[0];
  const int kpl = (A.dk + 31) >> 5, vpl = (A.dv + 31) >> 5;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int4 d = plan.item[it];
    const int b = d.x, g = d.y >> 8, r = d.y & 255, p0 = d.z, p1 = d.w;
    const T* kp = (const T*)A.k.ptr[r];
    const T* vp = (const T*)A.v.ptr[r];
    const int32_t* bt = A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb;
    for (int hh = warp; hh < A.G; hh += kGenWarps) {
      const int h = g * A.G + hh;
      const T* qp = (const T*)A.q + ((int64_t)b * A.Hq + h) * A.dk;
      float qv[kGenMaxPerLane], ov[kGenMaxPerLane];
#pragma unroll
      for (int i = 0; i < kGenMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        qv[i] = (i < kpl && c < A.dk) ? ld_elem(qp + c) : 0.f;
        ov[i] = 0.f;
      }
      float m = -INFINITY, l = 0.f;
      for (int p = p0; p < p1; ++p) {
        const int j = p / A.bs, off = p - j * A.bs;
        const int64_t phys = (j < A.max_vb) ? (int64_t)__ldg(bt + j) : -1;
        if (phys < 0 || phys >= A.num_blocks) {
          if (lane == 0 && hh == 0) count_error(A.err);
          continue;
        }
        const int64_t row = (phys * A.groups + g) * A.bs + off;
        const T* kr = kp + row * A.k_stride;
        const T* vr = vp + row * A.v_stride;
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < kGenMaxPerLane; ++i) {
          const int c = lane + 32 * i;
          if (i < kpl && c < A.dk) dot = fmaf(qv[i], ld_elem(kr + c), dot);
        }
        const float s = warp_sum(dot) * A.sl2;
        const float mn = fmaxf(m, s);
        const float alpha = exp2f(m - mn);
        const float pw = exp2f(s - mn);
        l = l * alpha + pw;
        m = mn;
#pragma unroll
        for (int i = 0; i < kGenMaxPerLane; ++i) {
          const int c = lane + 32 * i;
          if (i < vpl && c < A.dv) ov[i] = fmaf(pw, ld_elem(vr + c), ov[i] * alpha);
        }
      }
      float* out = plan.o + ((int64_t)it * A.G + hh) * A.dv;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int i = 0; i < kGenMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        if (i < vpl && c < A.dv) out[c] = ov[i] * inv;
      }
      if (lane == 0) plan.lse[(int64_t)it * A.G + hh] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  }
}

int launch_split_generic(const GenericArgs& A, const Plan& plan, bool bf16, cudaStream_t s) {
  const int grid = num_sms() * 4 < plan.max_items ? num_sms() * 4 : plan.max_items;
  if (grid <= 0) return DCP_OK;
  if (bf16)
    split_generic_kernel<__nv_bfloat16><<<grid, kGenWarps * 32, 0, s>>>(A, plan);
  else
    split_generic_kernel<float><<<grid, kGenWarps * 32, 0, s>>>(A, plan);
  return launch_status();
}

// SFA: one CTA per (rank, request); each warp walks the selected entries of
// its heads and keeps those the rank owns.  Writes the per-rank partial.
__device__ __forceinline__ bool sfa_entry(const GenericArgs& A, const SfaSel& S, int b, int k,
                                          int r, int64_t& slot) {
  if (S.topk == nullptr) {
    if (__ldg(S.sel_rank + (int64_t)b * S.K + k) != r) return false;
    slot = __ldg(S.sel_slot + (int64_t)b * S.K + k);
    return true;
  }
  const int64_t g = __ldg(S.topk + (int64_t)b * S.K + k);
  if (g < 0 || g >= __ldg(S.seq_lens + b)) return false;
  int rk, loc;
  int64_t vb;
  place_token(g, S.L, rk, vb, loc);
  if (rk != r) return false;
  const int64_t phys =
      vb < A.max_vb ? (int64_t)__ldg(A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb + vb)
                    : (int64_t)-1;
  slot = (phys >= 0 && phys < A.num_blocks) ? phys * A.bs + loc : (int64_t)-2;
  return true;
}

template <typename T>
__global__ void __launch_bounds__(kGenWarps * 32)
sfa_generic_kernel(GenericArgs A, SfaSel S, float* __restrict__ part_o,
                   float* __restrict__ part_lse) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x / A.B, b = blockIdx.x % A.B;
  const T* kp = (const T*)A.k.ptr[r];
  const int64_t num_slots = A.num_blocks * A.bs;
  const int kpl = (A.dk + 31) >> 5, vpl = (A.dv + 31) >> 5;
  for (int h = warp; h < A.Hq; h += kGenWarps) {
    const T* qp = (const T*)A.q + ((int64_t)b * A.Hq + h) * A.dk;
    float qv[kGenMaxPerLane], ov[kGenMaxPerLane];
#pragma unroll
    for (int i = 0; i < kGenMaxPerLane; ++i) {
      const int c = lane + 32 * i;
      qv[i] = (i < kpl && c < A.dk) ? ld_elem(qp + c) : 0.f;
      ov[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int k = 0; k < S.K; ++k) {
      int64_t s;
      if (!sfa_entry(A, S, b, k, r, s)) continue;
      if (s < 0 || s >= num_slots) {
        if (lane == 0 && h == 0) count_error(A.err);
        continue;
      }
      const T* kr = kp + s * A.k_stride;
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < kGenMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        if (i < kpl && c < A.dk) dot = fmaf(qv[i], ld_elem(kr + c), dot);
      }
      const float sc = warp_sum(dot) * A.sl2;
      const float mn = fmaxf(m, sc);
      const float alpha = exp2f(m - mn);
      const float pw = exp2f(sc - mn);
      l = l * alpha + pw;
      m = mn;
#pragma unroll
      for (int i = 0; i < kGenMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        if (i < vpl && c < A.dv) ov[i] = fmaf(pw, ld_elem(kr + c), ov[i] * alpha);
      }
    }
    const int64_t row = ((int64_t)r * A.B + b) * A.Hq + h;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < kGenMaxPerLane; ++i) {
      const int c = lane + 32 * i;
      if (i < vpl && c < A.dv) part_o[row * A.dv + c] = ov[i] * inv;
    }
    if (lane == 0) part_lse[row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

int launch_sfa_generic(const GenericArgs& A, const SfaSel& S, float* part_o, float* part_lse,
                       bool bf16, cudaStream_t s) {
  const int grid = A.B * A.dcp;
  if (grid <= 0) return DCP_OK;
  if (bf16)
    sfa_generic_kernel<__nv_bfloat16><<<grid, kGenWarps * 32, 0, s>>>(A, S, part_o, part_lse);
  else
    sfa_generic_kernel<float><<<grid, kGenWarps * 32, 0, s>>>(A, S, part_o, part_lse);
  return launch_status();
}

}  // namespace dcp
