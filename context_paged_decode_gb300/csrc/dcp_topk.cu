// Exact distributed top-k over the DCP ranks.
//
// Page "DeepSeek V4.1 context parallelism", section "Decode computation":
// each rank computes local top-k candidates and the scores and logical ids
// are merged across ranks; this is exact top-k selection under the score /
// tie rule, not a reduced candidate budget (the global top-k is always
// inside the union of the local top-k sets).
//
// Rule: a higher score ranks first; equal scores rank the smaller logical
// (global) token id first; NaN counts as -inf and -0 as +0.  Both are folded into one
// 64-bit key, larger = better:
//     key = (order(score) << 32) | (0xFFFFFFFF - id),
// order() mapping IEEE floats monotonically onto unsigned integers.  Keys
// are distinct, so the k-th largest key is a unique threshold.
//
// One CTA selects the top-k of a key list: an 8-bit MSB-first radix select
// finds the threshold in 8 passes of shared-memory histograms, the keys at
// or above it are collected, and a bitonic sort orders them.  Stage 1 runs
// one CTA per (rank, request) over the rank's local scores (local position
// p of rank r is global token x through the inverse of the layout
// formulas); stage 2 one CTA per request over the dcp x k candidates.
#include "dcp_common.cuh"

namespace dcp {

constexpr int kTopkThreads = 1024;
constexpr int kTopkMax = 4096;  // largest k (shared-memory sort buffer)

__device__ __forceinline__ uint32_t order_f32(float f) {
  uint32_t u = __float_as_uint(f);
  if (f != f) u = 0xFF800000u;  // NaN -> -inf
  if (f == 0.f) u = 0u;         // -0 and +0 are equal scores
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unorder_f32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ uint64_t topk_key(float s, uint32_t id) {
  return ((uint64_t)order_f32(s) << 32) | (uint64_t)(0xFFFFFFFFu - id);
}

// Global token of local position p on rank r (inverse of the layout formulas).
__device__ __forceinline__ int64_t global_of_local(int64_t p, int r, const Layout& L) {
  const int64_t vb = p / L.bs;
  const int loc = (int)(p - vb * L.bs);
  const int lbi = (loc / L.I) * L.dcp + r;
  return vb * L.bs * L.dcp + (int64_t)lbi * L.I + loc % L.I;
}

struct LocalSrc {  // rank r's local scores of request b
  const float* s;
  int64_t n;
  int r;
  Layout L;
  __device__ __forceinline__ uint64_t operator()(int64_t p) const {
    return topk_key(__ldg(s + p), (uint32_t)global_of_local(p, r, L));
  }
};

struct CandSrc {  // dcp candidate lists of request b
  const uint64_t* c;
  int64_t per;       // k
  int64_t rstride;   // B * k
  __device__ __forceinline__ uint64_t operator()(int64_t i) const {
    return __ldg(reinterpret_cast<const unsigned long long*>(c) + (i / per) * rstride + i % per);
  }
};

// Top-k keys of src(0..n-1), sorted descending, into out[0..k) (0 = none).
template <class Src>
__device__ void cta_topk(const Src& src, int64_t n, int k, uint64_t* out) {
  __shared__ uint64_t keys[kTopkMax];
  __shared__ int hist[256];
  __shared__ int sh[4];
  const int tid = threadIdx.x;
  uint64_t thr = 0;  // keys >= thr are taken
  if (n > k) {
    uint64_t prefix = 0, mask = 0;
    int kk = k;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int64_t i = tid; i < n; i += blockDim.x) {
        const uint64_t key = src(i);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int cum = 0;
        for (int d = 255; d >= 0; --d) {
          if (cum + hist[d] >= kk) {
            sh[0] = d;
            sh[1] = kk - cum;
            break;
          }
          cum += hist[d];
        }
      }
      __syncthreads();
      prefix |= (uint64_t)sh[0] << shift;
      mask |= (uint64_t)0xFF << shift;
      kk = sh[1];
      __syncthreads();
    }
    thr = prefix;  // the k-th largest key
  }
  if (tid == 0) sh[2] = 0;
  int npow = 1;
  while (npow < k) npow <<= 1;
  for (int i = tid; i < npow; i += blockDim.x) keys[i] = 0;
  __syncthreads();
  for (int64_t i = tid; i < n; i += blockDim.x) {
    const uint64_t key = src(i);
    if (key >= thr && key != 0) {
      const int pos = atomicAdd(&sh[2], 1);
      if (pos < k) keys[pos] = key;
    }
  }
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= npow; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < npow / 2; t += blockDim.x) {
        const int lo = 2 * stride * (t / stride) + (t % stride), hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = keys[lo], b = keys[hi];
        if ((a < b) == desc) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  for (int i = tid; i < k; i += blockDim.x) out[i] = keys[i];
}

__global__ void __launch_bounds__(kTopkThreads)
topk_local_kernel(Layout L, const float* __restrict__ scores, int B, int max_local,
                  const int32_t* __restrict__ local_lens, int k, uint64_t* __restrict__ cand) {
  const int r = blockIdx.x / B, b = blockIdx.x % B;
  int64_t n = local_lens[b * L.dcp + r];
  if (n < 0) n = 0;
  if (n > max_local) n = max_local;
  LocalSrc src{scores + ((int64_t)r * B + b) * max_local, n, r, L};
  cta_topk(src, n, k, cand + ((int64_t)r * B + b) * k);
}

__global__ void __launch_bounds__(kTopkThreads)
topk_merge_kernel(int dcp, const uint64_t* __restrict__ cand, int B, int k,
                  uint64_t* __restrict__ tmp, int32_t* __restrict__ out_ids,
                  float* __restrict__ out_scores) {
  const int b = blockIdx.x;
  CandSrc src{cand + (int64_t)b * k, k, (int64_t)B * k};
  uint64_t* best = tmp + (int64_t)b * k;
  cta_topk(src, (int64_t)dcp * k, k, best);
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    const uint64_t key = best[i];
    out_ids[(int64_t)b * k + i] = key ? (int32_t)(0xFFFFFFFFu - (uint32_t)key) : -1;
    if (out_scores)
      out_scores[(int64_t)b * k + i] = key ? unorder_f32((uint32_t)(key >> 32)) : -INFINITY;
  }
}

}  // namespace dcp

using namespace dcp;

extern "C" {

int dcp_topk_workspace_size(dcp_layout_t layout, int32_t num_reqs, int32_t k, size_t* bytes) {
  if (!bytes || !layout_ok(layout) || num_reqs < 0 || k < 1 || k > kTopkMax) return DCP_EINVAL;
  *bytes = sizeof(uint64_t) * (size_t)(layout.dcp_size + 1) * num_reqs * k;
  return DCP_OK;
}

int dcp_topk_local(dcp_layout_t layout, const float* local_scores, int32_t num_reqs,
                   int32_t max_local, const int32_t* local_lens, int32_t k, uint64_t* cand_keys,
                   dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_topk_local");
  if (!layout_ok(layout) || num_reqs < 0 || max_local < 0 || k < 1 || k > kTopkMax)
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!local_scores || !local_lens || !cand_keys) return DCP_EINVAL;
  const Layout L{layout.dcp_size, layout.block_size, layout.interleave};
  topk_local_kernel<<<layout.dcp_size * num_reqs, kTopkThreads, 0, (cudaStream_t)stream>>>(
      L, local_scores, num_reqs, max_local, local_lens, k, cand_keys);
  return launch_status();
}

int dcp_topk_merge(int32_t dcp_size, const uint64_t* cand_keys, int32_t num_reqs, int32_t k,
                   void* workspace, size_t workspace_bytes, int32_t* out_ids, float* out_scores,
                   dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_topk_merge");
  if (dcp_size < 1 || dcp_size > DCP_MAX_RANKS || num_reqs < 0 || k < 1 || k > kTopkMax)
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!cand_keys || !out_ids) return DCP_EINVAL;
  if (!workspace || workspace_bytes < sizeof(uint64_t) * (size_t)num_reqs * k)
    return DCP_EWORKSPACE;
  topk_merge_kernel<<<num_reqs, kTopkThreads, 0, (cudaStream_t)stream>>>(
      dcp_size, cand_keys, num_reqs, k, (uint64_t*)workspace, out_ids, out_scores);
  return launch_status();
}

int dcp_topk(dcp_layout_t layout, const float* local_scores, int32_t num_reqs, int32_t max_local,
             const int32_t* local_lens, int32_t k, int32_t* out_ids, float* out_scores,
             void* workspace, size_t workspace_bytes, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_topk");
  size_t need = 0;
  const int rc0 = dcp_topk_workspace_size(layout, num_reqs, k, &need);
  if (rc0) return rc0;
  if (!workspace || workspace_bytes < need) return DCP_EWORKSPACE;
  uint64_t* cand = (uint64_t*)workspace;
  int rc = dcp_topk_local(layout, local_scores, num_reqs, max_local, local_lens, k, cand, stream);
  if (rc) return rc;
  return dcp_topk_merge(layout.dcp_size, cand, num_reqs, k,
                        cand + (size_t)layout.dcp_size * num_reqs * k,
                        sizeof(uint64_t) * (size_t)num_reqs * k, out_ids, out_scores, stream);
}

}  // extern "C"
