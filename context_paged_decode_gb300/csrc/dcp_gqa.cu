// GQA decode under DCP: per-rank split-KV partials and the fused decode step.
//
// Page "Decode Context Parallel (DCP)", section "Decode": each rank attends
// its local KV shard and produces partial outputs plus LSE values, which are
// then combined; vLLM DCP blog post, section 5.4: the shared KV heads are
// broadcast to their query heads.
//
// Fast path (bf16, head_dim 128, block_size % 16 == 0): each warp streams
// 16-token tiles of one (block, kv head) page through its own ring of shared-
// memory stages, filled by TMA (2-D tensor maps over each rank's HND pool,
// 128-byte swizzle so ldmatrix reads are bank-conflict free).  Scores and
// P.V run on mma.sync (m16n8k16, bf16 in / fp32 accumulate) with the group's
// query heads as the M rows: a CUDA-core version spends ~5 issue slots per
// KV element (convert + 4 FMA per head) plus cross-lane reductions, which is
// more than the issue budget of one 8-KB page at HBM speed; the tensor-core
// form needs ~100 warp instructions per page.  Online softmax in fp32 with
// exp2; P is rounded to bf16 for the P.V product.
#include <mutex>

#include "dcp_generic.cuh"
#include "dcp_ptx.cuh"
#include "dcp_sfa_tc.cuh"

namespace dcp {

// ---------------------------------------------------------------------------
// host: tensor maps
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

bool encode_2d_bf16_sw128(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                          uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  if (((uintptr_t)base & 15) || (row_bytes & 15) || rows == 0 || rows > (1ull << 32)) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// tensor-core split kernel
// ---------------------------------------------------------------------------

struct GqaTmaArgs {
  CUtensorMap kmap[DCP_MAX_RANKS];
  CUtensorMap vmap[DCP_MAX_RANKS];
  const __nv_bfloat16* q;
  int B, Hq, Hkv, G, bs, dcp;
  float sl2;
  const int32_t* bt;
  int max_vb;
  int64_t bt_rank_stride;
  int64_t num_blocks;
  int32_t* err;
};

constexpr int kTile = 16;             // tokens per tile (one MMA k-step of P.V)
constexpr int kStageBytes = 8192;     // K tile 4 KB + V tile 4 KB
constexpr int kGqaWarps = 4;
constexpr int kGqaStages = 3;         // per warp
constexpr int kStuck = 1 << 20;       // err_count increment for a wait that timed out

__host__ __device__ constexpr int gqa_smem_bytes(int nw, int d) {
  return 1024 + nw * d * kStageBytes + nw * d * 8 + nw * 2 * 16 * 4;
}

// Swizzled byte offset of 16-byte chunk c (0..15) of row `row` in a tile
// stored as two 64-column halves of [16 rows][128 B] (TMA SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw_off(int row, int c) {
  return (uint32_t)((c >> 3) * 2048 + row * 128 + (((c & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

template <int NW, int D, bool kUpper>
__global__ void __launch_bounds__(NW * 32)
gqa_tma_kernel(const __grid_constant__ GqaTmaArgs A, Plan plan) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ int s_item;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t stage0 = smem_u32(smem) + warp * D * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * D * kStageBytes);
  float* ml = reinterpret_cast<float*>(bars + NW * D);  // [NW][2][16]
  const uint32_t bar0 = smem_u32(bars + warp * D);
  if (lane == 0) {
    for (int s = 0; s < D; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    for (int r = 0; r < A.dcp; ++r) {
      prefetch_tmap(&A.kmap[r]);
      prefetch_tmap(&A.vmap[r]);
    }
  }
  __syncthreads();
  const uint64_t pol = policy_evict_first();
  const int n_items = plan.hdr[0];
  uint32_t seq = 0;    // tiles this warp has consumed so far
  bool dead = false;   // a wait timed out: stop waiting and issuing
  const int r0 = lane >> 2, cq = 2 * (lane & 3);

  for (;;) {
    if (threadIdx.x == 0) s_item = atomicAdd(&plan.hdr[2], 1);
    __syncthreads();
    const int it = s_item;
    if (it >= n_items) break;
    const int4 d = plan.item[it];
    const int b = d.x, g = d.y >> 8, r = d.y & 255, p0 = d.z, p1 = d.w;
    const int ntiles = (p1 - p0 + kTile - 1) / kTile;
    const int my_n = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
    const void* km = &A.kmap[r];
    const void* vm = &A.vmap[r];
    const int32_t* btr = A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb;

    // row of the k-th tile of this warp in the rank's pool, false if the
    // block-table entry is unusable
    auto tile_row = [&](int k, int& row) -> bool {
      const int p = p0 + (warp + k * NW) * kTile;
      const int j = p / A.bs, off = p - j * A.bs;
      const int64_t phys = j < A.max_vb ? (int64_t)__ldg(btr + j) : -1;
      if (phys < 0 || phys >= A.num_blocks) return false;
      row = (int)((phys * A.Hkv + g) * A.bs + off);
      return true;
    };
    auto issue = [&](int k) {  // lane 0
      const uint32_t st = (seq + k) % D;
      const uint32_t bar = bar0 + 8 * st, dst = stage0 + st * kStageBytes;
      int row;
      if (tile_row(k, row)) {
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d_hint(dst, km, 0, row, bar, pol);
        tma_load_2d_hint(dst + 2048, km, 64, row, bar, pol);
        tma_load_2d_hint(dst + 4096, vm, 0, row, bar, pol);
        tma_load_2d_hint(dst + 6144, vm, 64, row, bar, pol);
      } else {
        count_error(A.err);
        mbar_arrive(bar);
      }
    };
    if (lane == 0 && !dead) {
      fence_proxy_async_smem();  // order the last item's generic smem traffic before TMA
      for (int k = 0; k < D && k < my_n; ++k) issue(k);
    }

    // query heads of this group as the A operand (rows >= G are zero)
    uint32_t qa[8][4];
    {
      const __nv_bfloat16* qb = A.q + ((int64_t)b * A.Hq + (int64_t)g * A.G) * 128;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const bool lo = r0 < A.G, hi = kUpper && (r0 + 8 < A.G);
        qa[ks][0] = lo ? ld_u32(qb + r0 * 128 + ks * 16 + cq) : 0u;
        qa[ks][1] = hi ? ld_u32(qb + (r0 + 8) * 128 + ks * 16 + cq) : 0u;
        qa[ks][2] = lo ? ld_u32(qb + r0 * 128 + ks * 16 + 8 + cq) : 0u;
        qa[ks][3] = hi ? ld_u32(qb + (r0 + 8) * 128 + ks * 16 + 8 + cq) : 0u;
      }
    }
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int k = 0; k < my_n; ++k) {
      const uint32_t st = (seq + k) % D;
      const uint32_t par = ((seq + k) / D) & 1;
      if (!dead && !mbar_wait(bar0 + 8 * st, par)) {
        dead = true;
        if (lane == 0) atomicAdd(A.err ? A.err : plan.hdr + 3, kStuck);
      }
      int row;
      const bool valid = !dead && tile_row(k, row);
      if (valid) {
        const uint32_t kb = stage0 + st * kStageBytes, vb = kb + 4096;
        const int nvalid = min(kTile, p1 - (p0 + (warp + k * NW) * kTile));
        if (nvalid < kTile) {  // zero V rows past the end so 0 * garbage stays 0
          for (int i = lane; i < (kTile - nvalid) * 16; i += 32) {
            const int rr = nvalid + (i >> 4);
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vb + sw_off(rr, i & 15)),
                         "r"(0u)
                         : "memory");
          }
          __syncwarp();
        }
        // S = Q K^T for 16 tokens: 2 n-tiles x 8 k-steps
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int mi = lane >> 3;
        const int krow = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + sw_off(krow, ks * 2 + (mi & 1)), b0, b1, b2, b3);
          mma_bf16_16816(s[0], qa[ks], b0, b1);
          mma_bf16_16816(s[1], qa[ks], b2, b3);
        }
        // online softmax (base 2); rows r0 (c0,c1) and r0+8 (c2,c3)
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = nt * 8 + cq + (e & 1);
            x[nt][e] = col < nvalid ? s[nt][e] * A.sl2 : -INFINITY;
          }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        const float mn0 = fmaxf(m0, mx0);
        const float a0 = exp2f(m0 - mn0);
        float p[2][4];
        p[0][0] = exp2f(x[0][0] - mn0);
        p[0][1] = exp2f(x[0][1] - mn0);
        p[1][0] = exp2f(x[1][0] - mn0);
        p[1][1] = exp2f(x[1][1] - mn0);
        l0 = l0 * a0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        m0 = mn0;
        float a1 = 1.f;
        if (kUpper) {
          float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
          const float mn1 = fmaxf(m1, mx1);
          a1 = exp2f(m1 - mn1);
          p[0][2] = exp2f(x[0][2] - mn1);
          p[0][3] = exp2f(x[0][3] - mn1);
          p[1][2] = exp2f(x[1][2] - mn1);
          p[1][3] = exp2f(x[1][3] - mn1);
          l1 = l1 * a1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
          m1 = mn1;
        } else {
          p[0][2] = p[0][3] = p[1][2] = p[1][3] = 0.f;
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][0] *= a0;
          o[n][1] *= a0;
          if (kUpper) {
            o[n][2] *= a1;
            o[n][3] *= a1;
          }
        }
        uint32_t pa[4];
        pa[0] = pack_bf16(p[0][0], p[0][1]);
        pa[1] = pack_bf16(p[0][2], p[0][3]);
        pa[2] = pack_bf16(p[1][0], p[1][1]);
        pa[3] = pack_bf16(p[1][2], p[1][3]);
        // O += P V: 16 n-tiles of 8 dims, k = the 16 tokens
        const int vrow = (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + sw_off(vrow, 2 * j + (mi >> 1)), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * j], pa, b0, b1);
          mma_bf16_16816(o[2 * j + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0 && !dead && k + D < my_n) {
        fence_proxy_async_smem();
        issue(k + D);
      }
    }
    seq += my_n;

    // this warp's state -> its first stage (all its loads have landed)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    if (kUpper) {
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    float* ost = reinterpret_cast<float*>(smem + warp * D * kStageBytes);
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      *reinterpret_cast<float2*>(ost + r0 * 128 + n * 8 + cq) = make_float2(o[n][0], o[n][1]);
      if (kUpper)
        *reinterpret_cast<float2*>(ost + (r0 + 8) * 128 + n * 8 + cq) =
            make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
      ml[(warp * 2 + 0) * 16 + r0] = m0;
      ml[(warp * 2 + 1) * 16 + r0] = l0;
      if (kUpper) {
        ml[(warp * 2 + 0) * 16 + r0 + 8] = m1;
        ml[(warp * 2 + 1) * 16 + r0 + 8] = l1;
      }
    }
    __syncthreads();
    // combine the warps: exact LSE algebra over disjoint token subsets
    for (int idx = threadIdx.x; idx < A.G * 128; idx += NW * 32) {
      const int row = idx >> 7, col = idx & 127;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, ml[(w * 2) * 16 + row]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = ml[(w * 2) * 16 + row];
        if (mw == -INFINITY) continue;
        const float sc = exp2f(mw - M);
        L = fmaf(ml[(w * 2 + 1) * 16 + row], sc, L);
        O = fmaf(reinterpret_cast<const float*>(smem + w * D * kStageBytes)[row * 128 + col], sc, O);
      }
      const bool any = L > 0.f;
      plan.o[((int64_t)it * A.G + row) * 128 + col] = any ? O / L : 0.f;
      if (col == 0) plan.lse[(int64_t)it * A.G + row] = any ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    __syncthreads();
  }
}

template <int NW, int D, bool U>
static int launch_gqa_tma(const GqaTmaArgs& A, const Plan& plan, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = gqa_smem_bytes(NW, D);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(gqa_tma_kernel<NW, D, U>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return DCP_ECUDA;
    attr_done[dev] = true;
  }
  const int per_sm = (228 * 1024) / (smem + 1024);
  int grid = num_sms() * (per_sm > 0 ? per_sm : 1);
  if (grid > plan.max_items) grid = plan.max_items;
  if (grid <= 0) return DCP_OK;
  gqa_tma_kernel<NW, D, U><<<grid, NW * 32, smem, s>>>(A, plan);
  return launch_status();
}

// ---------------------------------------------------------------------------
// split plan sizing (shared with the MLA path through dcp_common.cuh users)
// ---------------------------------------------------------------------------

static int gqa_target_items() { return 16 * 2 * num_sms(); }

static int gqa_max_items(int B, int Hkv, int dcp) { return gqa_target_items() + B * Hkv * dcp; }

}  // namespace dcp

using namespace dcp;

namespace {

bool gqa_args_ok(const dcp_layout_t& layout, const void* q, int B, int Hq, int Hkv, int d,
                 dcp_dtype_t dtype, const dcp_paged_kv_t& kv, const int32_t* local_lens) {
  if (!layout_ok(layout) || B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > 16 ||
      d < 32 || d % 32 != 0 || d > 256 || (dtype != DCP_F32 && dtype != DCP_BF16) ||
      kv.num_blocks < 0 || kv.max_vblocks < 0 || kv.bt_rank_stride < 0)
    return false;
  if (B == 0) return true;
  return q && local_lens && kv.block_table && ranks_ok(kv.k, layout.dcp_size) &&
         ranks_ok(kv.v, layout.dcp_size);
}

bool gqa_fast_ok(const dcp_layout_t& layout, int Hkv, int d, dcp_dtype_t dtype,
                 const dcp_paged_kv_t& kv) {
  if (dtype != DCP_BF16 || d != 128 || layout.block_size % kTile != 0) return false;
  if ((int64_t)kv.num_blocks * Hkv * layout.block_size >= (int64_t(1) << 31)) return false;
  for (int r = 0; r < layout.dcp_size; ++r)
    if (((uintptr_t)kv.k.ptr[r] & 15) || ((uintptr_t)kv.v.ptr[r] & 15)) return false;
  return tensor_map_encoder() != nullptr;
}

// plan + split kernels; fills plan partials
int gqa_split(const dcp_layout_t& layout, const void* q, int B, int Hq, int Hkv, int d,
              float scale, dcp_dtype_t dtype, const dcp_paged_kv_t& kv, const int32_t* local_lens,
              const Plan& plan, int32_t* err, cudaStream_t s) {
  const int G = Hq / Hkv;
  const bool fast = gqa_fast_ok(layout, Hkv, d, dtype, kv);
  int rc = launch_plan(local_lens, B, layout.dcp_size, Hkv, kTile, fast ? 256 : 64,
                       gqa_target_items(), plan, s);
  if (rc) return rc;
  if (fast) {
    GqaTmaArgs A;
    memset(&A, 0, sizeof(A));
    const uint64_t rows = (uint64_t)kv.num_blocks * Hkv * layout.block_size;
    for (int r = 0; r < layout.dcp_size; ++r) {
      if (!encode_2d_bf16_sw128(&A.kmap[r], kv.k.ptr[r], 128, rows > 0 ? rows : 1, 256, 64, 16) ||
          !encode_2d_bf16_sw128(&A.vmap[r], kv.v.ptr[r], 128, rows > 0 ? rows : 1, 256, 64, 16))
        return DCP_ECUDA;
    }
    A.q = (const __nv_bfloat16*)q;
    A.B = B;
    A.Hq = Hq;
    A.Hkv = Hkv;
    A.G = G;
    A.bs = layout.block_size;
    A.dcp = layout.dcp_size;
    A.sl2 = scale * kLog2e;
    A.bt = kv.block_table;
    A.max_vb = kv.max_vblocks;
    A.bt_rank_stride = kv.bt_rank_stride;
    A.num_blocks = kv.num_blocks;
    A.err = err;
    return G > 8 ? launch_gqa_tma<kGqaWarps, kGqaStages, true>(A, plan, s)
                 : launch_gqa_tma<kGqaWarps, kGqaStages, false>(A, plan, s);
  }
  GenericArgs A;
  A.q = q;
  A.B = B;
  A.Hq = Hq;
  A.G = G;
  A.groups = Hkv;
  A.dcp = layout.dcp_size;
  A.bs = layout.block_size;
  A.dk = d;
  A.dv = d;
  A.k_stride = d;
  A.v_stride = d;
  A.sl2 = scale * kLog2e;
  A.k = kv.k;
  A.v = kv.v;
  A.bt = kv.block_table;
  A.max_vb = kv.max_vblocks;
  A.bt_rank_stride = kv.bt_rank_stride;
  A.num_blocks = kv.num_blocks;
  A.err = err;
  return launch_split_generic(A, plan, dtype == DCP_BF16, s);
}

}  // namespace

extern "C" {

int dcp_decode_workspace_size(dcp_layout_t layout, dcp_kind_t kind, int32_t num_reqs,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim_v,
                              size_t* bytes) {
  if (!bytes || !layout_ok(layout) || num_reqs < 0 || num_q_heads < 1 || head_dim_v < 1)
    return DCP_EINVAL;
  const int dcp = layout.dcp_size;
  if (kind == DCP_KIND_GQA) {
    if (num_kv_heads < 1 || num_q_heads % num_kv_heads) return DCP_EINVAL;
    const int entries = num_reqs * num_kv_heads * dcp;
    *bytes = plan_bytes(entries, gqa_max_items(num_reqs, num_kv_heads, dcp),
                        num_q_heads / num_kv_heads, head_dim_v);
    return DCP_OK;
  }
  if (kind == DCP_KIND_MLA) {
    const int entries = num_reqs * dcp;
    *bytes = plan_bytes(entries, mla_max_items(num_reqs, dcp), num_q_heads, head_dim_v);
    return DCP_OK;
  }
  if (kind == DCP_KIND_SFA) {
    // per-rank partials (o and lse) plus the remapped (rank, slot) pairs of
    // the tensor-core path (at most 2048 selected tokens per request)
    *bytes = align_up(sizeof(float) * (size_t)dcp * num_reqs * num_q_heads * head_dim_v, 256) +
             align_up(sizeof(float) * (size_t)dcp * num_reqs * num_q_heads, 256) +
             2 * align_up(sizeof(int32_t) * (size_t)num_reqs * kSfaTcMaxSel, 256);
    return DCP_OK;
  }
  return DCP_EINVAL;
}

int dcp_decode_partial_gqa(dcp_layout_t layout, const void* q, int32_t num_reqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           float scale, dcp_dtype_t dtype, dcp_paged_kv_t kv,
                           const int32_t* local_lens, float* part_o, float* part_lse,
                           void* workspace, size_t workspace_bytes, int32_t* err_count,
                           dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_decode_partial_gqa");
  if (!gqa_args_ok(layout, q, num_reqs, num_q_heads, num_kv_heads, head_dim, dtype, kv,
                   local_lens))
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!part_o || !part_lse) return DCP_EINVAL;
  size_t need = 0;
  dcp_decode_workspace_size(layout, DCP_KIND_GQA, num_reqs, num_q_heads, num_kv_heads, head_dim,
                            &need);
  if (!workspace || workspace_bytes < need) return DCP_EWORKSPACE;
  const int dcp = layout.dcp_size;
  const Plan plan = plan_carve(workspace, num_reqs * num_kv_heads * dcp,
                               gqa_max_items(num_reqs, num_kv_heads, dcp),
                               num_q_heads / num_kv_heads);
  cudaStream_t s = (cudaStream_t)stream;
  int rc = gqa_split(layout, q, num_reqs, num_q_heads, num_kv_heads, head_dim, scale, dtype, kv,
                     local_lens, plan, err_count, s);
  if (rc) return rc;
  // per-rank output: part_o is [dcp][B][Hq][d] = rows (r, b, h) in mode 1
  return launch_item_merge(plan, 1, num_reqs, dcp, num_q_heads, num_q_heads / num_kv_heads,
                           num_kv_heads, head_dim, nullptr, part_o, DCP_F32, part_lse, s);
}

int dcp_decode_gqa(dcp_layout_t layout, const void* q, int32_t num_reqs, int32_t num_q_heads,
                   int32_t num_kv_heads, int32_t head_dim, float scale, dcp_dtype_t dtype,
                   dcp_paged_kv_t kv, const int32_t* local_lens, const float* sink, void* out,
                   dcp_dtype_t out_dtype, float* out_lse, void* workspace,
                   size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream) {
  dcp::NvtxRange nvtx_range("dcp_decode_gqa");
  if (!gqa_args_ok(layout, q, num_reqs, num_q_heads, num_kv_heads, head_dim, dtype, kv,
                   local_lens) ||
      (out_dtype != DCP_F32 && out_dtype != DCP_BF16))
    return DCP_EINVAL;
  if (num_reqs == 0) return DCP_OK;
  if (!out) return DCP_EINVAL;
  size_t need = 0;
  dcp_decode_workspace_size(layout, DCP_KIND_GQA, num_reqs, num_q_heads, num_kv_heads, head_dim,
                            &need);
  if (!workspace || workspace_bytes < need) return DCP_EWORKSPACE;
  const int dcp = layout.dcp_size;
  const Plan plan = plan_carve(workspace, num_reqs * num_kv_heads * dcp,
                               gqa_max_items(num_reqs, num_kv_heads, dcp),
                               num_q_heads / num_kv_heads);
  cudaStream_t s = (cudaStream_t)stream;
  int rc = gqa_split(layout, q, num_reqs, num_q_heads, num_kv_heads, head_dim, scale, dtype, kv,
                     local_lens, plan, err_count, s);
  if (rc) return rc;
  return launch_item_merge(plan, 0, num_reqs, dcp, num_q_heads, num_q_heads / num_kv_heads,
                           num_kv_heads, head_dim, sink, out, out_dtype, out_lse, s);
}

}  // extern "C"
