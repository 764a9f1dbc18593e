// Integer side of the DCP hot path: per-rank context lengths, slot mapping,
// SFA index remap, and the split-KV work plan.
//
// Layout formulas: page "Decode Context Parallel (DCP)" (vLLM Ascend design
// documents), section "KV-cache layout".  Owner masking: page "DeepSeek V4.1
// context parallelism" (TokenSpeed), section "Cache ownership".  Remap:
// "Decode Context Parallel (DCP)", section "GLM-5.2 SFA DCP replicated
// indexer".
#include <stdio.h>
#include <stdlib.h>

#include "dcp_common.cuh"
#include "dcp_ptx.cuh"

namespace dcp {

int launch_status_report(cudaError_t e) {
  if (getenv("DCP_VERBOSE")) fprintf(stderr, "libdcp: CUDA error %d: %s\n", (int)e, cudaGetErrorString(e));
  return DCP_ECUDA;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// local_lens[b][r]: closed form of the number of tokens x < L with rank(x) == r.
__global__ void local_seq_lens_kernel(Layout L, const int32_t* __restrict__ seq_lens, int B,
                                      int32_t* __restrict__ out, int32_t* err) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  griddep_wait();                // launched chained: the preceding kernel completed
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * L.dcp) return;
  const int b = i / L.dcp, r = i % L.dcp;
  int64_t len = seq_lens[b];
  if (len < 0) {
    if (r == 0) count_error(err);
    len = 0;
  }
  const int64_t vbs = (int64_t)L.bs * L.dcp;
  const int64_t full = len / vbs;
  const int rem = (int)(len % vbs);
  const int c = rem / L.I, p = rem % L.I;  // complete interleave groups, leftover tokens
  int64_t n = full * L.bs + (int64_t)(c / L.dcp) * L.I;
  if (c % L.dcp > r) n += L.I;
  if (c % L.dcp == r) n += p;
  out[i] = (int32_t)n;
}

__global__ void slot_mapping_kernel(Layout L, const int32_t* __restrict__ req,
                                    const int64_t* __restrict__ pos, int64_t T,
                                    const int32_t* __restrict__ bt, int B, int max_vb,
                                    int64_t bt_rank_stride, int64_t num_blocks,
                                    int32_t* __restrict__ out_rank, int64_t* __restrict__ out_slot,
                                    int32_t* err) {
  griddep_launch_dependents();
  griddep_wait();
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < T;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int b = req[t];
    const int64_t x = pos[t];
    int owner = -1;
    int64_t s = -1;
    if (b >= 0 && b < B && x >= 0) {
      int r, loc;
      int64_t vb;
      place_token(x, L, r, vb, loc);
      if (vb < max_vb) {
        const int64_t phys = bt[r * bt_rank_stride + (int64_t)b * max_vb + vb];
        if (phys >= 0 && phys < num_blocks) {
          owner = r;
          s = phys * L.bs + loc;
        }
      }
    }
    if (owner < 0) count_error(err);
    out_rank[t] = owner;
    for (int r = 0; r < L.dcp; ++r) out_slot[(int64_t)r * T + t] = (r == owner) ? s : -1;
  }
}

__global__ void sfa_remap_kernel(Layout L, const int32_t* __restrict__ topk, int B, int K,
                                 const int32_t* __restrict__ seq_lens,
                                 const int32_t* __restrict__ bt, int max_vb,
                                 int64_t bt_rank_stride, int64_t num_blocks,
                                 int32_t* __restrict__ out_rank, int32_t* __restrict__ out_slot,
                                 int32_t* err) {
  griddep_launch_dependents();   // a dependent sparse-attention launch may start its prologue
  griddep_wait();                // launched chained: the preceding kernel completed
  const int64_t n = (int64_t)B * K;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / K);
    const int64_t g = topk[i];
    int owner = -1, s = -1;
    if (g >= 0 && g < seq_lens[b]) {
      int r, loc;
      int64_t vb;
      place_token(g, L, r, vb, loc);
      const int64_t phys =
          vb < max_vb ? bt[r * bt_rank_stride + (int64_t)b * max_vb + vb] : (int64_t)-1;
      if (phys >= 0 && phys < num_blocks) {
        owner = r;
        s = (int)(phys * L.bs + loc);
      } else {
        count_error(err);
      }
    }
    out_rank[i] = owner;
    out_slot[i] = s;
  }
}

// ---------------------------------------------------------------------------
// split-KV plan (one CTA)
// ---------------------------------------------------------------------------

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int64_t block_sum_i64(int64_t v, int64_t* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    v = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh[32] = v;
  }
  __syncthreads();
  const int64_t r = sh[32];
  __syncthreads();
  return r;
}

// Exclusive block scan of one int per thread; returns the prefix, *total the sum.
__device__ __forceinline__ int block_scan_excl(int v, int* sh, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  const int warp_prefix = w > 0 ? sh[w - 1] : 0;
  *total = sh[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ local_lens, int B, int dcp, int G, int tile,
            int min_chunk, int target_items, Plan plan) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int64_t sh64[33];
  __shared__ int sh[32];
  const int n = B * G * dcp;  // entries (b, g, r)
  // total tokens over (b, r), each counted once per head group
  int64_t tot = 0;
  for (int i = threadIdx.x; i < B * dcp; i += blockDim.x) tot += max(local_lens[i], 0);
  tot = block_sum_i64(tot, sh64) * G;
  int64_t chunk = (tot + target_items - 1) / max(target_items, 1);
  if (chunk < min_chunk) chunk = min_chunk;
  chunk = (chunk + tile - 1) / tile * tile;
  if (chunk > (1 << 30)) chunk = 1 << 30;

  // contiguous segment of entries per thread
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int e0 = min(n, (int)threadIdx.x * per), e1 = min(n, e0 + per);
  int mine = 0;
  for (int e = e0; e < e1; ++e) {
    const int r = e % dcp, b = e / (G * dcp);
    const int len = max(local_lens[b * dcp + r], 0);
    mine += (int)((len + chunk - 1) / chunk);
  }
  int total;
  int base = block_scan_excl(mine, sh, &total);
  if (total > plan.max_items) total = plan.max_items;  // cannot happen with the sized bound
  for (int e = e0; e < e1; ++e) {
    const int r = e % dcp, g = (e / dcp) % G, b = e / (G * dcp);
    const int len = max(local_lens[b * dcp + r], 0);
    plan.off[e] = min(base, plan.max_items);
    for (int64_t p0 = 0; p0 < len; p0 += chunk) {
      if (base < plan.max_items)
        plan.item[base] = make_int4(b, (g << 8) | r, (int)p0, (int)((int64_t)len < p0 + chunk ? (int64_t)len : p0 + chunk));
      ++base;
    }
  }
  if (threadIdx.x == 0) {
    plan.off[n] = total;
    plan.hdr[0] = total;
    plan.hdr[1] = (int)chunk;
    plan.hdr[2] = 0;  // dynamic item counter of the split kernels
    plan.hdr[3] = 0;  // stuck-wait counter when the caller passes no err_count
  }
}

int launch_plan(const int32_t* local_lens, int B, int dcp, int G, int tile, int min_chunk,
                int target_items, const Plan& plan, cudaStream_t s) {
  const cudaError_t e = launch_chained(plan_kernel, 1, kPlanThreads, 0, s, local_lens, B, dcp, G,
                                       tile, min_chunk, target_items, plan);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

// Exclusive block scan of one int64 per thread; *total gets the sum.
__device__ __forceinline__ int64_t block_scan_excl_i64(int64_t v, int64_t* sh, int64_t* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int64_t s = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh[lane] = s;
  }
  __syncthreads();
  const int64_t warp_prefix = w > 0 ? sh[w - 1] : 0;
  *total = sh[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

// Balanced-parts plan: entry e = b*dcp + r owns the global token range
// [S_e, S_e + len_e) of the concatenation; tile t of the entry starts at
// S_e + t*tile and belongs to run floor((S_e + t*tile) / per), with per =
// ceil(total / parts) rounded up to the tile (so consecutive tiles differ by
// at most one run and no run boundary splits a tile).
__global__ void __launch_bounds__(kPlanThreads)
plan_parts_kernel(const int32_t* __restrict__ local_lens, int B, int dcp, int tile, int parts,
                  int overhead, Plan plan) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int64_t sh64[33];
  __shared__ int sh[32];
  const int n = B * dcp;
  const int per_thr = (n + blockDim.x - 1) / blockDim.x;
  const int e0 = min(n, (int)threadIdx.x * per_thr), e1 = min(n, e0 + per_thr);
  int64_t mine = 0;
  for (int e = e0; e < e1; ++e) {
    const int64_t len = max(local_lens[e], 0);
    mine += len > 0 ? len + overhead : 0;
  }
  int64_t tot;
  const int64_t start0 = block_scan_excl_i64(mine, sh64, &tot);
  int64_t per = (tot + parts - 1) / parts;
  per = (per + tile - 1) / tile * tile;
  if (per < tile) per = tile;
  // pieces of each entry: runs kf..kl of its first and last tile
  int cnt = 0;
  {
    int64_t S = start0;
    for (int e = e0; e < e1; ++e) {
      const int64_t len = max(local_lens[e], 0);
      if (len > 0) {
        const int64_t S0 = S + overhead;       // position of the entry's first token
        const int64_t last = S0 + (len - 1) / tile * tile;
        cnt += (int)(last / per - S0 / per + 1);
        S += len + overhead;
      }
    }
  }
  int total;
  int base = block_scan_excl(cnt, sh, &total);
  if (total > plan.max_items) total = plan.max_items;  // cannot happen with the sized bound
  {
    int64_t S = start0;
    for (int e = e0; e < e1; ++e) {
      const int64_t len = max(local_lens[e], 0);
      plan.off[e] = min(base, plan.max_items);
      if (len > 0) {
        const int64_t S0 = S + overhead;
        const int64_t ntiles = (len + tile - 1) / tile;
        const int64_t kf = S0 / per, kl = (S0 + (ntiles - 1) * tile) / per;
        for (int64_t k = kf; k <= kl; ++k) {
          const int64_t t0 = k == kf ? 0 : (k * per - S0 + tile - 1) / tile;
          const int64_t t1 = k == kl ? ntiles : ((k + 1) * per - S0 + tile - 1) / tile;
          if (base < plan.max_items) {
            plan.item[base] = make_int4(e / dcp, e % dcp, (int)(t0 * tile),
                                        (int)(t1 * tile < len ? t1 * tile : len));
            plan.ipart[base] = (int)k;
          }
          ++base;
        }
        S += len + overhead;
      }
    }
  }
  __syncthreads();
  // pfirst[k] = first item whose run is >= k
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int k = plan.ipart[i], kp = i > 0 ? plan.ipart[i - 1] : -1;
    for (int q = kp + 1; q <= k && q <= parts; ++q) plan.pfirst[q] = i;
  }
  if (threadIdx.x == 0) {
    const int kl = total > 0 ? plan.ipart[total - 1] : -1;
    for (int q = kl + 1; q <= parts; ++q) plan.pfirst[q] = total;
    plan.off[n] = total;
    plan.hdr[0] = total;
    plan.hdr[1] = (int)(per < (1 << 30) ? per : (1 << 30));
    plan.hdr[2] = 0;
    plan.hdr[3] = 0;
  }
}

int launch_plan_parts(const int32_t* local_lens, int B, int dcp, int tile, int parts,
                      int overhead, const Plan& plan, cudaStream_t s) {
  if (parts < 1 || parts > kMaxParts || tile < 1 || overhead < 0) return DCP_EINVAL;
  const cudaError_t e = launch_chained(plan_parts_kernel, 1, kPlanThreads, 0, s, local_lens, B, dcp,
                                       tile, parts, overhead, plan);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

}  // namespace dcp

using namespace dcp;

extern "C" {

const char* dcp_strerror(int code) {
  switch (code) {
    case DCP_OK: return "ok";
    case DCP_EINVAL: return "invalid argument or layout";
    case DCP_EWORKSPACE: return "workspace missing or too small";
    case DCP_ECUDA: return "CUDA launch or driver call failed";
    case DCP_EUNSUPPORTED: return "shape or dtype not supported by this build";
    default: return "unknown error";
  }
}

int dcp_version(void) { return 100; }

int dcp_local_seq_lens(dcp_layout_t layout, const int32_t* seq_lens, int32_t num_reqs,
                       int32_t* local_lens, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_local_seq_lens");
  if (!layout_ok(layout) || num_reqs < 0) return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!seq_lens || !local_lens) return DCP_EINVAL;
  const Layout L{layout.dcp_size, layout.block_size, layout.interleave};
  const int n = num_reqs * layout.dcp_size;
  const cudaError_t e = launch_chained(local_seq_lens_kernel, (unsigned)((n + 255) / 256), 256, 0,
                                       (cudaStream_t)stream, L, seq_lens, num_reqs, local_lens,
                                       err_count);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

int dcp_slot_mapping(dcp_layout_t layout, const int32_t* req_idx, const int64_t* positions,
                     int64_t num_tokens, const int32_t* block_table, int32_t num_reqs,
                     int32_t max_vblocks, int64_t bt_rank_stride, int64_t num_blocks,
                     int32_t* out_rank, int64_t* out_slot, int32_t* err_count,
                     dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_slot_mapping");
  if (!layout_ok(layout) || num_tokens < 0 || num_reqs < 0 || max_vblocks < 0 ||
      bt_rank_stride < 0 || num_blocks < 0)
    return DCP_EINVAL;
  if (num_tokens == 0) return DCP_OK;
  if (!req_idx || !positions || !out_rank || !out_slot || (!block_table && num_reqs > 0))
    return DCP_EINVAL;
  const Layout L{layout.dcp_size, layout.block_size, layout.interleave};
  const int64_t blocks = (num_tokens + 255) / 256;
  const int grid = (int)(blocks < 8 * num_sms() ? blocks : 8 * num_sms());
  const cudaError_t e = launch_chained(slot_mapping_kernel, (unsigned)grid, 256, 0,
                                       (cudaStream_t)stream, L, req_idx, positions, num_tokens,
                                       block_table, num_reqs, max_vblocks, bt_rank_stride,
                                       num_blocks, out_rank, out_slot, err_count);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

int dcp_sfa_remap(dcp_layout_t layout, const int32_t* topk, int32_t num_reqs, int32_t topk_len,
                  const int32_t* seq_lens, const int32_t* block_table, int32_t max_vblocks,
                  int64_t bt_rank_stride, int64_t num_blocks, int32_t* out_rank,
                  int32_t* out_slot, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_sfa_remap");
  if (!layout_ok(layout) || num_reqs < 0 || topk_len < 0 || max_vblocks < 0 ||
      bt_rank_stride < 0 || num_blocks < 0)
    return DCP_EINVAL;
  if (num_blocks * (int64_t)layout.block_size >= (int64_t(1) << 31)) return DCP_EINVAL;
  const int64_t n = (int64_t)num_reqs * topk_len;
  if (n == 0) return DCP_OK;
  if (!topk || !seq_lens || !block_table || !out_rank || !out_slot) return DCP_EINVAL;
  const Layout L{layout.dcp_size, layout.block_size, layout.interleave};
  const int64_t blocks = (n + 255) / 256;
  const int grid = (int)(blocks < 8 * num_sms() ? blocks : 8 * num_sms());
  const cudaError_t e = launch_chained(sfa_remap_kernel, (unsigned)grid, 256, 0, (cudaStream_t)stream,
                                       L, topk, num_reqs, topk_len, seq_lens, block_table,
                                       max_vblocks, bt_rank_stride, num_blocks, out_rank, out_slot,
                                       err_count);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

}  // extern "C"
