// tcgen05 MLA decode kernel: per-rank split-KV partials for 128 query heads
// sharing one 576-wide latent KV head (512 latent + 64 rope; value = the
// first 512 entries), bf16 in, fp32 accumulate.
//
// Why tensor cores here: all 128 heads of a request read the same latent
// rows, so S = Q K^T (M=128 heads, K=576) and O = P V (N=512) are dense
// contractions with ~242 flop per KV byte, near the bf16 ridge point
// (vLLM DCP blog post, section 1: one latent KV head for all query heads).
//
// Shape of the kernel:
//  * one work item = a run of local positions of one request on one rank
//    (the split-KV plan); items never cross a rank (each shard attends only
//    its local KV, page "Decode Context Parallel (DCP)", section "Decode");
//  * two CTAs per item, one per half of the 512 value columns: the fp32
//    output tile 128 x 512 would fill all of tensor memory, so each CTA
//    keeps 128 x 256 of it (256 columns) next to two 32-column score
//    buffers and two 16-column bf16 P buffers.  Both CTAs compute the same
//    scores, so their softmax decisions agree bit for bit;
//  * warp 0 issues TMA (Q once per request, then 32-token KV stages through a
//    double buffer), warp 1 issues tcgen05.mma (QK^T of stage j+1 overlaps
//    the softmax of stage j), warps 2-5 run the online softmax (one head row
//    per thread, scores read from tensor memory, P written back to tensor
//    memory as the A operand of P.V) and the epilogue;
//  * the output is rescaled only when the running maximum grows by more
//    than 8 (log2 units), so P stays <= 256 and the rare rescale waits for
//    the in-flight P.V.
// Every mbarrier wait is bounded; a timed-out wait adds 1<<20 to the error
// counter and that role stops waiting, so the kernel always terminates.
#include <stdlib.h>
#include <string.h>

#include "dcp_mla_tc.cuh"
#include "dcp_ptx.cuh"

namespace dcp {

struct MlaTcArgs {
  CUtensorMap qmap;                  // [B*128 rows][576] bf16, box 64 x 128
  CUtensorMap kvmap[DCP_MAX_RANKS];  // [num_blocks*bs rows][576] bf16, box 64 x 32
  int B, bs, dcp;
  float sl2;
  const int32_t* bt;
  int max_vb;
  int64_t bt_rank_stride;
  int64_t num_blocks;
  int32_t* err;
};

constexpr int kHeads = 128;
constexpr int kDk = 576;
constexpr int kDvHalf = 256;
constexpr int kChunks = kDk / 64;                   // 9 column chunks of 64 (128 B)
constexpr int kSt = 32;                             // tokens per KV stage
constexpr int kQChunkBytes = kHeads * 128;          // 16 KB
constexpr int kQBytes = kChunks * kQChunkBytes;     // 147456
constexpr int kKvChunkBytes = kSt * 128;            // 4 KB
constexpr int kKvStageBytes = kChunks * kKvChunkBytes;  // 36864
constexpr int kKvOff = kQBytes;
constexpr int kBarOff = kKvOff + 2 * kKvStageBytes;  // 221184
constexpr int kNumBars = 16;
constexpr int kMlaSmem = 1024 + kBarOff + kNumBars * 8 + 16;
constexpr int kMlaThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320;
constexpr float kRescaleThreshold = 8.f;
constexpr int kStuckMla = 1 << 20;

// barrier slots
enum : int {
  B_KV_FULL = 0,   // +stage
  B_KV_EMPTY = 2,  // +stage
  B_Q_FULL = 4,
  B_Q_EMPTY = 5,
  B_S_FULL = 6,    // +buffer
  B_S_FREE = 8,    // +buffer
  B_P_FULL = 10,   // +buffer
  B_PV_DONE = 12,  // +buffer
  B_O_FULL = 14,
  B_O_FREE = 15
};

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kSt, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kDvHalf, false, true);

__global__ void __launch_bounds__(kMlaThreads, 1)
mla_tc_kernel(const __grid_constant__ MlaTcArgs A, Plan plan) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int n_items = plan.hdr[0];
  int32_t* errp = A.err ? A.err : plan.hdr + 3;

  if (threadIdx.x == 0) {
    const uint32_t counts[kNumBars] = {1, 1, 1, 1, 1, 1, 1, 1, 128, 128, 128, 128, 1, 1, 1, 128};
    for (int i = 0; i < kNumBars; ++i) mbar_init(bars + 8 * i, counts[i]);
    fence_mbar_init();
    prefetch_tmap(&A.qmap);
    for (int r = 0; r < A.dcp; ++r) prefetch_tmap(&A.kvmap[r]);
  }
  if (warp == 1) {
    tc_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // physical row of stage j of an item, false if the block-table entry is unusable
  auto stage_row = [&](int b, int r, int p0, int j, int& row) -> bool {
    const int p = p0 + j * kSt;
    const int vb = p / A.bs, off = p - vb * A.bs;
    const int64_t phys =
        vb < A.max_vb ? (int64_t)__ldg(A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb + vb)
                      : (int64_t)-1;
    if (phys < 0 || phys >= A.num_blocks) return false;
    row = (int)(phys * A.bs + off);
    return true;
  };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    uint32_t g = 0, k = 0;
    int prev_b = -1;
    bool dead = false;
    for (int it = pair; it < n_items && !dead; it += npairs, ++k) {
      const int4 d = plan.item[it];
      const int b = d.x, r = d.y & 255, p0 = d.z, p1 = d.w;
      const int nst = (p1 - p0 + kSt - 1) / kSt;
      if (!mbar_wait(bars + 8 * B_Q_EMPTY, (k & 1) ^ 1)) {
        dead = true;
        break;
      }
      if (b != prev_b) {
        mbar_arrive_expect_tx(bars + 8 * B_Q_FULL, kQBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_2d(sbase + c * kQChunkBytes, &A.qmap, 64 * c, b * kHeads, bars + 8 * B_Q_FULL);
        prev_b = b;
      } else {
        mbar_arrive(bars + 8 * B_Q_FULL);
      }
      for (int j = 0; j < nst; ++j, ++g) {
        const uint32_t st = g & 1, u = g >> 1;
        if (!mbar_wait(bars + 8 * (B_KV_EMPTY + st), (u & 1) ^ 1)) {
          dead = true;
          break;
        }
        const uint32_t full = bars + 8 * (B_KV_FULL + st);
        int row;
        if (stage_row(b, r, p0, j, row)) {
          mbar_arrive_expect_tx(full, kKvStageBytes);
          const uint32_t dst = sbase + kKvOff + st * kKvStageBytes;
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(dst + c * kKvChunkBytes, &A.kvmap[r], 64 * c, row, full);
        } else {
          if (half == 0) count_error(A.err);
          mbar_arrive(full);
        }
      }
    }
    if (dead) atomicAdd(errp, kStuckMla);
  } else if (warp == 1 && lane == 0) {
    // ---------------- tcgen05.mma issuer ----------------
    uint32_t g = 0, k = 0;
    bool dead = false;
    const uint32_t d_o = tmem + kColO;
    auto qk = [&](uint32_t gs) -> bool {
      const uint32_t st = gs & 1, u = gs >> 1;
      if (!mbar_wait(bars + 8 * (B_KV_FULL + st), u & 1)) return false;
      if (!mbar_wait(bars + 8 * (B_S_FREE + st), (u & 1) ^ 1)) return false;
      tc_fence_after();
      const uint32_t d_s = tmem + kColS + st * kSt;
      const uint32_t kv = sbase + kKvOff + st * kKvStageBytes;
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t a = sdesc_sw128(sbase + c * kQChunkBytes + kk * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(kv + c * kKvChunkBytes + kk * 32, 0, 1024);
          tc_mma_ss(d_s, a, bd, kIdescQK, (c | kk) != 0);
        }
      }
      tc_commit(bars + 8 * (B_S_FULL + st));
      return true;
    };
    auto pv = [&](uint32_t gs, bool first) -> bool {
      const uint32_t st = gs & 1, u = gs >> 1;
      if (!mbar_wait(bars + 8 * (B_P_FULL + st), u & 1)) return false;
      if (first && !mbar_wait(bars + 8 * B_O_FREE, (k & 1) ^ 1)) return false;
      tc_fence_after();
      const uint32_t v = sbase + kKvOff + st * kKvStageBytes + (4 * half) * kKvChunkBytes;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        // V as the MN-major B operand: 64-column atoms kKvChunkBytes apart,
        // 8-token groups 1024 B apart; the second k-step starts 16 tokens in.
        const uint64_t bd = sdesc_sw128(v + kk * 16 * 128, kKvChunkBytes, 1024);
        tc_mma_ts(d_o, tmem + kColP + st * 16 + kk * 8, bd, kIdescPV, (!first || kk) ? 1u : 0u);
      }
      tc_commit(bars + 8 * (B_KV_EMPTY + st));
      tc_commit(bars + 8 * (B_PV_DONE + st));
      return true;
    };
    for (int it = pair; it < n_items && !dead; it += npairs, ++k) {
      const int4 d = plan.item[it];
      const int nst = (d.w - d.z + kSt - 1) / kSt;
      if (!mbar_wait(bars + 8 * B_Q_FULL, k & 1)) {
        dead = true;
        break;
      }
      tc_fence_after();
      if (!qk(g)) {
        dead = true;
        break;
      }
      for (int j = 0; j < nst; ++j) {
        if (j + 1 < nst && !qk(g + j + 1)) {
          dead = true;
          break;
        }
        if (!pv(g + j, j == 0)) {
          dead = true;
          break;
        }
      }
      if (dead) break;
      g += nst;
      tc_commit(bars + 8 * B_O_FULL);
      tc_commit(bars + 8 * B_Q_EMPTY);
    }
    if (dead) atomicAdd(errp, kStuckMla);
  } else if (warp >= 2) {
    // ---------------- softmax + epilogue (one head row per thread) ----------------
    const int q4 = warp & 3;                 // tensor-memory lane quarter of this warp
    const int head = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int tid = threadIdx.x - 64;        // 0..127
    uint32_t g = 0, k = 0;
    bool dead = false;
    // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform
    auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par));
    };
    for (int it = pair; it < n_items && !dead; it += npairs, ++k) {
      const int4 d = plan.item[it];
      const int b = d.x, r = d.y & 255, p0 = d.z, p1 = d.w;
      const int nst = (p1 - p0 + kSt - 1) / kSt;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nst; ++j, ++g) {
        const uint32_t st = g & 1, u = g >> 1;
        if (!wwait(bars + 8 * (B_S_FULL + st), u & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        uint32_t s[32];
        tc_ld32(tmem + lane_off + kColS + st * kSt, s);
        tc_wait_ld(s);
        tc_fence_before();
        mbar_arrive(bars + 8 * (B_S_FREE + st));
        int row;
        const int nvalid = stage_row(b, r, p0, j, row) ? min(kSt, p1 - (p0 + j * kSt)) : 0;
        float x[32];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = i < nvalid ? __uint_as_float(s[i]) * A.sl2 : -INFINITY;
          mx = fmaxf(mx, x[i]);
        }
        const bool grow = mx > m + kRescaleThreshold;
        const bool need = grow && j > 0 && l > 0.f;  // O already holds this row's sums
        if (__any_sync(0xffffffffu, need)) {
          // wait for the in-flight P.V, then rescale the rows that need it
          const uint32_t gp = g - 1;
          if (!wwait(bars + 8 * (B_PV_DONE + (gp & 1)), (gp >> 1) & 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
          const float sc = need ? exp2f(m - mx) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < kDvHalf / 32; ++cc) {
            uint32_t o[32];
            tc_ld32(tmem + lane_off + kColO + cc * 32, o);
            tc_wait_ld(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * sc);
            tc_st32(tmem + lane_off + kColO + cc * 32, o);
          }
          tc_wait_st();
          l *= sc;
        }
        if (grow) m = mx;
        const float mb = (m == -INFINITY) ? 0.f : m;
        uint32_t pk[16];
        float ls = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float pa = exp2f(x[2 * i] - mb), pb = exp2f(x[2 * i + 1] - mb);
          ls += pa + pb;
          pk[i] = pack_bf16(pa, pb);
        }
        l += ls;
        // P buffer st is free once the P.V of two stages ago completed
        if (!wwait(bars + 8 * (B_PV_DONE + st), (u & 1) ^ 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        tc_st16(tmem + lane_off + kColP + st * 16, pk);
        tc_wait_st();
        if (nvalid < kSt) {
          // rows past the end may hold anything: zero this CTA's V columns so 0 * x stays 0
          const uint32_t v = sbase + kKvOff + st * kKvStageBytes + (4 * half) * kKvChunkBytes;
          const int total = (kSt - nvalid) * 4 * 8;
          for (int i = tid; i < total; i += 128) {
            const int rr = nvalid + (i >> 5), ch = (i >> 3) & 3, part = i & 7;
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                             v + ch * kKvChunkBytes + rr * 128 + part * 16),
                         "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(bars + 8 * (B_P_FULL + st));
      }
      if (dead) break;
      // epilogue: O / l -> item partial, LSE in natural log
      if (!wwait(bars + 8 * B_O_FULL, k & 1)) {
        dead = true;
        break;
      }
      tc_fence_after();
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      float* dst = plan.o + ((int64_t)it * kHeads + head) * (2 * kDvHalf) + half * kDvHalf;
#pragma unroll 1
      for (int cc = 0; cc < kDvHalf / 32; ++cc) {
        uint32_t o[32];
        tc_ld32(tmem + lane_off + kColO + cc * 32, o);
        tc_wait_ld(o);
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + cc * 32 + i) =
              make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                          __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
      }
      if (half == 0) plan.lse[(int64_t)it * kHeads + head] = any ? (m + log2f(l)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(bars + 8 * B_O_FREE);
    }
    if (dead && lane == 0) atomicAdd(errp, kStuckMla);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kTmemCols);
  }
}

bool mla_tc_supported(const dcp_layout_t& layout, int B, int Hq, int dk, int dv,
                      dcp_dtype_t dtype, const dcp_paged_kv_t& kv) {
  if (dtype != DCP_BF16 || Hq != kHeads || dk != kDk || dv != 2 * kDvHalf) return false;
  if (layout.block_size % kSt != 0 || B < 1) return false;
  if ((int64_t)kv.num_blocks * layout.block_size >= (int64_t(1) << 31)) return false;
  if ((int64_t)B * kHeads >= (int64_t(1) << 31)) return false;
  for (int r = 0; r < layout.dcp_size; ++r)
    if ((uintptr_t)kv.k.ptr[r] & 15) return false;
  if (getenv("DCP_DISABLE_TCGEN05")) return false;
  return tensor_map_encoder() != nullptr;
}

int launch_mla_tc(const dcp_layout_t& layout, const void* q, int B, int Hq, float scale,
                  const dcp_paged_kv_t& kv, const Plan& plan, int32_t* err, cudaStream_t s) {
  (void)Hq;
  if ((uintptr_t)q & 15) return DCP_EUNSUPPORTED;
  MlaTcArgs A;
  memset(&A, 0, sizeof(A));
  if (!encode_2d_bf16_sw128(&A.qmap, q, kDk, (uint64_t)B * kHeads, kDk * 2, 64, kHeads))
    return DCP_ECUDA;
  const uint64_t rows = (uint64_t)kv.num_blocks * layout.block_size;
  for (int r = 0; r < layout.dcp_size; ++r)
    if (!encode_2d_bf16_sw128(&A.kvmap[r], kv.k.ptr[r], kDk, rows > 0 ? rows : 1, kDk * 2, 64,
                              kSt))
      return DCP_ECUDA;
  A.B = B;
  A.bs = layout.block_size;
  A.dcp = layout.dcp_size;
  A.sl2 = scale * kLog2e;
  A.bt = kv.block_table;
  A.max_vb = kv.max_vblocks;
  A.bt_rank_stride = kv.bt_rank_stride;
  A.num_blocks = kv.num_blocks;
  A.err = err;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMlaSmem) != cudaSuccess)
      return DCP_ECUDA;
    attr_done[dev] = true;
  }
  const int pairs = num_sms() / 2;
  mla_tc_kernel<<<2 * (pairs > 0 ? pairs : 1), kMlaThreads, kMlaSmem, s>>>(A, plan);
  return launch_status();
}

}  // namespace dcp
