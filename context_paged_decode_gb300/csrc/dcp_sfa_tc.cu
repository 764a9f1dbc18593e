// tcgen05 SFA decode partials: per (rank, request, 64 query heads), sparse
// attention over the selected tokens that rank owns, MLA-shaped latent rows
// (576 bf16: key = whole row, value = first 512 entries), bf16 in, fp32
// accumulate.
//
// Page "Decode Context Parallel (DCP)", section "GLM-5.2 SFA DCP replicated
// indexer": the global top-k indices are remapped to local KV indices
// before SFA runs; each rank attends only the selected tokens it stores and
// the per-rank results are merged by LSE (the sink is applied once, at the
// merge: page "DeepSeek V4.1 context parallelism", section "Decode
// computation").
//
// The contraction runs transposed so that the gathered tokens are the M
// dimension of the tensor core:
//   S^T [tokens x 64 heads]          = K_stage . Q^T      (9 chunks x 4 MMAs)
//   O^T [512 value rows x 64 heads] += V_stage^T . P^T    (4 row blocks x 4 MMAs)
// Shape of the kernel:
//  * one CTA per (rank, request, 64 heads).  The CTA first lists its selected
//    slots in top-k order (from the remapped (rank, slot) pairs), then walks
//    them in 64-token stages through a two-slot ring;
//  * shared memory: Q (64 heads x 576 as nine 8 KB chunks, 128-byte swizzle,
//    one TMA box each), two 72 KB stage slots (nine 8 KB chunks of 64 token
//    rows x 64 columns in the same layout) and the selection list.  The
//    ninth (rope) chunk of a slot is dead once that stage's S^T is complete,
//    and P^T (64 tokens x 64 heads, bf16) takes its place;
//  * Q.K^T runs at M=128 although a stage has 64 tokens: rows 64-127 of the
//    A operand are whatever follows the chunk in shared memory, and the
//    matching rows of S^T (tensor-memory lanes 64-127) are never read;
//  * seven warps gather with 16-byte cp.async (whole 1152-byte rows;
//    unselected, unusable and tail rows are zero-filled): four fill slot 0
//    and three slot 1, so two stages are in flight and a stage's barrier
//    never waits for the other slot.  Each gather thread waits for its own
//    copies and fences them for the tensor core before its warp arrives;
//  * tensor memory: two S^T buffers (64 columns each), O^T (4 x 64 columns);
//  * warps 0-1: softmax, one token (tensor-memory lane) per thread; the
//    per-head stage maximum is a warp max (redux.sync) combined over the two
//    warps in shared memory.  Warp 2 issues P V, warp 4 issues Q.K^T;
//    warps 0-3 each own one lane quarter of O^T for the rescale and the
//    epilogue.  O^T columns (heads) are rescaled only when a head's running
//    maximum grows by more than 8 (log2 units), which keeps P <= 256.
// Every mbarrier wait is bounded; a timed-out wait adds 1<<20 to the error
// counter and that role stops waiting, so the kernel always terminates.
#include <stdlib.h>
#include <string.h>

#include "dcp_sfa_tc.cuh"

namespace dcp {

namespace {

constexpr int kHB = 64;                                // heads per CTA (N)
constexpr int kRowE = 576;
constexpr int kRowB = kRowE * 2;                       // 1152 bytes per latent row
constexpr int kChunks = 9;                             // 64-column chunks of a row
constexpr int kSt = 64;                                // tokens per stage
constexpr int kChunkB = kSt * 128;                     // 8 KB
constexpr int kStageB = kChunks * kChunkB;             // 72 KB
constexpr int kPieces = kSt * kRowB / 16;              // 16-byte pieces per stage
constexpr int kQOff = 0;
constexpr int kSlotOff = kChunks * kHB * 128;          // 72 KB
constexpr int kSelOff = kSlotOff + 2 * kStageB;        // 216 KB
constexpr int kMaxSelTc = kSfaTcMaxSel;
constexpr int kWMaxOff = kSelOff + kMaxSelTc * 4;      // [parity][warp][head] floats
constexpr int kFacOff = kWMaxOff + 2 * 2 * kHB * 4;    // [parity][head] rescale factors
constexpr int kMiscOff = kFacOff + 2 * kHB * 4;        // count, flags[2], rescale stage
constexpr int kBarOff = kMiscOff + 32;
constexpr int kNumBars = 17;
constexpr int kSfaTcSmem = 1024 + kBarOff + kNumBars * 8 + 16;
constexpr int kFirstGather = 5;
constexpr int kGatherWarps = 7;
constexpr int kGather0 = 4;                            // gather warps of slot 0 (the rest: slot 1)
constexpr int kSfaTcThreads = 32 * (kFirstGather + kGatherWarps);   // 384
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 2 * kSt;
constexpr float kRescaleThreshold = 8.f;
constexpr int kStuck = 1 << 20;

static_assert(kSfaTcSmem + 64 <= 227 * 1024, "shared memory overflow");
static_assert(kSlotOff % 1024 == 0 && kStageB % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kColO + 4 * kHB <= kTmemCols, "tensor memory overflow");

// barrier slots
enum : int {
  B_Q_FULL = 0,
  B_FULL = 1,        // +slot: the stage in the slot landed (gather warps)
  B_SLOT_FREE = 3,   // +slot: the P V that read the slot completed
  B_S_FULL = 5,      // +buffer: S^T of the stage is complete
  B_S_FREE = 7,      // +buffer: both softmax warps read it
  B_P_FULL = 9,      // +stage parity: P^T, the factors and the rescale flag are stored
  B_PVD = 11,        // one phase per P V completed
  B_MX = 12,         // the two softmax warps published their stage maxima (per stage)
  B_RS_GO = 13,      // the P V warp: rescale now (rescale stages), or O^T is complete (last)
  B_RS_DONE = 14,    // warps 0, 1 and 3 rescaled their quarters
  B_LX = 15,         // the softmax warps published their row sums
  B_IX = 16          // softmax warp 0 published 1 / l per head
};

__device__ __forceinline__ int arrivals(int i) {
  if (i == B_FULL) return kGather0;
  if (i == B_FULL + 1) return kGatherWarps - kGather0;
  if (i == B_S_FREE || i == B_S_FREE + 1 || i == B_P_FULL || i == B_P_FULL + 1 || i == B_MX ||
      i == B_LX)
    return 2;
  if (i == B_RS_DONE) return 3;
  return 1;
}

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kHB, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kHB, true, true);

__device__ __forceinline__ float warp_max_f32(float v) {
  float m;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}

// 16 bytes global -> shared; bytes == 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16_fill(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace

// Twelve warps put three on every SM sub-partition (16K registers each), so a
// thread may hold up to 168 registers.
__global__ void __launch_bounds__(kSfaTcThreads, 1) sfa_tc_kernel(const __grid_constant__ SfaTcArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  int32_t* sel = reinterpret_cast<int32_t*>(smem + kSelOff);
  volatile int32_t* misc = reinterpret_cast<volatile int32_t*>(smem + kMiscOff);
  float* wmax = reinterpret_cast<float*>(smem + kWMaxOff);
  const float* fac = reinterpret_cast<const float*>(smem + kFacOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = blockIdx.x / (A.B * A.hblocks);
  const int rem = blockIdx.x % (A.B * A.hblocks);
  const int b = rem / A.hblocks, h0 = (rem % A.hblocks) * kHB;
  const int64_t num_slots = A.num_blocks * A.bs;
  int32_t* errp = A.err;

  griddep_launch_dependents();   // a dependent merge launch may start waiting
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bars + 8 * i, arrivals(i));
    fence_mbar_init();
    prefetch_tmap(&A.qmap);
    misc[0] = 0;
    // Q of heads h0 .. h0+63: nine 64 x 64 boxes (awaited by the Q.K^T issuer,
    // or at the end when the rank selected no token)
    mbar_arrive_expect_tx(bars + 8 * B_Q_FULL, kChunks * kHB * 128);
    for (int c = 0; c < kChunks; ++c)
      tma_load_2d(sbase + kQOff + c * kHB * 128, &A.qmap, 64 * c, b * A.Hq + h0,
                  bars + 8 * B_Q_FULL);
  }
  if (warp == 4) {
    tc_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as a dependent of the remap: its pairs are complete past this
  // point (Q, a caller input, was ready before the remap started)
  griddep_wait();

  // ---- this rank's selected slots, in top-k order (-1: unusable, attended as masked) ----
  {
    constexpr int kPer = 6;
    static_assert(kPer * kSfaTcThreads >= kMaxSelTc, "selection runs must cover kMaxSelTc");
    const int per = (A.K + kSfaTcThreads - 1) / kSfaTcThreads;
    const int k0 = min(A.K, tid * per), k1 = min(A.K, k0 + per);
    int64_t slot[kPer];
    uint32_t own = 0;
    {
      int rk[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int k = k0 + i;
        rk[i] = k < k1 ? __ldg(A.sel_rank + (int64_t)b * A.K + k) : -1;
        slot[i] = k < k1 ? (int64_t)__ldg(A.sel_slot + (int64_t)b * A.K + k) : -1;
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (rk[i] == r) own |= 1u << i;
    }
    const int mine = __popc(own);
    __shared__ int wsum[kSfaTcThreads / 32];
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += wsum[w];
    base += x - mine;
    if (tid == kSfaTcThreads - 1) misc[0] = base + mine;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (own >> i & 1) {
        int64_t sl = slot[i];
        if (sl < 0 || sl >= num_slots) {
          if (h0 == 0) count_error(errp);
          sl = -1;
        }
        if (base < kMaxSelTc) sel[base] = (int32_t)sl;
        ++base;
      }
    }
  }
  __syncthreads();
  const int n_sel = min((int)misc[0], kMaxSelTc);
  const int nst = (n_sel + kSt - 1) / kSt;

  // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform
  auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, par));
  };
  auto warp_arrive = [&](uint32_t bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };
  // multiply the O^T columns of lane quarter q by the per-head factors f[64]
  auto rescale = [&](int q, const float* f) {
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o[32];
        const uint32_t ta = tmem + lane_off + kColO + 64 * blk + 32 * hh;
        tc_ld32(ta, o);
        tc_wait_ld(o);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[i] = __float_as_uint(__uint_as_float(o[i]) * f[32 * hh + i]);
        tc_st32(ta, o);
      }
    }
    tc_wait_st();
  };
  // o = O^T / l per head for the value rows of lane quarter q, with 1 / l
  // per head from the factor slots (unused when the rank has no token)
  auto epilogue = [&](int q, bool have) {
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int64_t orow = ((int64_t)r * A.B + b) * A.Hq + h0;   // row of head h0
    float inv[64];
#pragma unroll
    for (int h = 0; h < 64; ++h) inv[h] = have ? fac[h] : 0.f;
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
      const int d = 128 * mb + 32 * q + lane;                  // value column
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o[32];
        if (have) {
          tc_ld32(tmem + lane_off + kColO + 64 * mb + 32 * hh, o);
          tc_wait_ld(o);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          A.part_o[(orow + 32 * hh + i) * 512 + d] =
              have ? __uint_as_float(o[i]) * inv[32 * hh + i] : 0.f;
      }
    }
  };

  if (warp >= kFirstGather) {
    // ---------------- gather: warp group `slot` fills slot n & 1 ----------------
    // Two groups, one per slot, each with one stage in flight: a stage's
    // barrier then never waits for the other slot to drain.
    const int slot = warp - kFirstGather < kGather0 ? 0 : 1;
    const int gthreads = 32 * (slot == 0 ? kGather0 : kGatherWarps - kGather0);
    const int gt = tid - 32 * (kFirstGather + (slot == 0 ? 0 : kGather0));
    const uint8_t* pool = A.pool[r];
    bool dead = false;
    for (int n = slot; n < nst; n += 2) {
      // the slot is free once the P V of stage n - 2 completed
      if (!wwait(bars + 8 * (B_SLOT_FREE + slot), ((n >> 1) & 1) ^ 1)) {
        dead = true;
        break;
      }
      const uint32_t dst0 = sbase + kSlotOff + slot * kStageB;
      // a warp takes groups of 4 token rows (one slot-list read per lane and
      // group); each copy instruction moves chunk c of the 4 rows: lane l
      // copies 16-byte unit l % 8 of row 4 g + l / 8, swizzled by the row & 7.
      // All 32 lanes copy in every instruction: the load pipe's cost is per
      // instruction, whatever its active lanes.
      const int gw_in = gt >> 5, gwarps = gthreads >> 5;
      const int rsub = lane >> 3, un = lane & 7;
#pragma unroll 1
      for (int rg = gw_in; rg < kSt / 4; rg += gwarps) {
        const int rr = rg * 4 + rsub;
        const int t = n * kSt + rr;
        const int row = t < n_sel ? sel[t] : -1;
        const uint8_t* rsrc = row >= 0 ? pool + (int64_t)row * kRowB + un * 16 : pool;
        const uint32_t bytes = row >= 0 ? 16u : 0u;
        const uint32_t rdst = dst0 + rr * 128 + ((uint32_t)(un ^ (rr & 7)) << 4);
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          cp_async16_fill(rdst + c * kChunkB, row >= 0 ? rsrc + c * 128 : pool, bytes);
      }
      cp_async_commit();
      // the stage landed: make it visible to the tensor core
      cp_async_wait<0>();
      fence_proxy_async_smem();
      warp_arrive(bars + 8 * (B_FULL + slot));
    }
    if (dead && lane == 0) atomicAdd(errp, kStuck);
  } else if (warp == 4) {
    // ---------------- Q.K^T issuer ----------------
    if (lane == 0) {
      bool dead = nst > 0 && !mbar_wait(bars + 8 * B_Q_FULL, 0);
      for (int n = 0; n < nst && !dead; ++n) {
        const int sb = n & 1;                                  // slot and S^T buffer
        const uint32_t u = (uint32_t)(n >> 1) & 1u;
        if (!mbar_wait2_cluster(bars + 8 * (B_FULL + sb), u, bars + 8 * (B_S_FREE + sb), u ^ 1u)) {
          dead = true;
          break;
        }
        tc_fence_after();
        const uint32_t st = sbase + kSlotOff + sb * kStageB;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          const uint64_t ad = sdesc_sw128(st + c * kChunkB, 0, 1024);
          const uint64_t bd = sdesc_sw128(sbase + kQOff + c * kHB * 128, 0, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_ss(tmem + kColS + sb * kSt, ad + (uint64_t)((kk * 32) >> 4),
                      bd + (uint64_t)((kk * 32) >> 4), kIdescQK, (c | kk) != 0);
        }
        tc_commit(bars + 8 * (B_S_FULL + sb));
      }
      if (dead) atomicAdd(errp, kStuck);
    }
  } else if (warp == 2) {
    // ---------------- P V issuer (lane 0), rescale and epilogue of quarter 2 ----------------
    uint32_t pvd_seen = 0, rsc = 0;
    bool dead = false;
    // Observe every phase of B_PVD in order, up to the P V of stage k.  A
    // parity wait is unambiguous only while the barrier is at most one phase
    // past the last one observed, so the P V of stage n is issued only after
    // that of stage n - 1 was seen to complete.
    auto pvd_upto = [&](int k) -> bool {
      while ((int)pvd_seen <= k) {
        if (!wwait(bars + 8 * B_PVD, pvd_seen & 1)) return false;
        ++pvd_seen;
      }
      return true;
    };
    for (int n = 0; n < nst; ++n) {
      const int sb = n & 1;
      if (!wwait(bars + 8 * (B_P_FULL + sb), (n >> 1) & 1) || !pvd_upto(n - 1)) {
        dead = true;
        break;
      }
      if (misc[1 + sb] != 0) {
        // rescale stage: all four quarters multiply their O^T columns by the
        // stage's factors (the P V of stage n - 1 completed)
        if (lane == 0) misc[3] = n;
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * B_RS_GO);
        tc_fence_after();
        rescale(2, fac + sb * kHB);
        tc_fence_before();
        if (!wwait(bars + 8 * B_RS_DONE, rsc & 1)) {
          dead = true;
          break;
        }
        ++rsc;
      }
      tc_fence_after();
      if (lane == 0) {
        // O^T[mb] += V^T . P^T: V^T is MN-major (value columns contiguous, the
        // two 64-column chunks of row block mb one chunk apart); P^T is
        // MN-major (heads contiguous); k-step kk = tokens 16kk .. 16kk+15
        const uint32_t st = sbase + kSlotOff + sb * kStageB;
#pragma unroll
        for (int kk = 0; kk < kSt / 16; ++kk) {
          const uint64_t pd = sdesc_sw128(st + 8 * kChunkB + kk * 2048, kChunkB, 1024);
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
            const uint64_t vd = sdesc_sw128(st + 2 * mb * kChunkB + kk * 2048, kChunkB, 1024);
            tc_mma_ss(tmem + kColO + 64 * mb, vd, pd, kIdescPV, (n > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc_commit(bars + 8 * (B_SLOT_FREE + sb));
        tc_commit(bars + 8 * B_PVD);
      }
      __syncwarp();
    }
    // O^T is complete once the last P V completed: release the other row warps
    if (!dead && nst > 0 && !pvd_upto(nst - 1)) dead = true;
    if (lane == 0) misc[3] = -1;
    __syncwarp();
    if (lane == 0 && nst > 0) mbar_arrive(bars + 8 * B_RS_GO);
    if (!dead && nst > 0 && !wwait(bars + 8 * B_IX, 0)) dead = true;
    tc_fence_after();
    epilogue(2, !dead && nst > 0);
    if (dead && lane == 0) atomicAdd(errp, kStuck);
  } else if (warp == 3) {
    // ---------------- rescale and epilogue of quarter 3 ----------------
    uint32_t rsc = 0;
    bool dead = false;
    while (nst > 0) {
      if (!wwait(bars + 8 * B_RS_GO, rsc & 1)) {
        dead = true;
        break;
      }
      ++rsc;
      const int n = misc[3];
      if (n < 0) break;
      tc_fence_after();
      rescale(3, fac + (n & 1) * kHB);
      tc_fence_before();
      warp_arrive(bars + 8 * B_RS_DONE);
    }
    if (!dead && nst > 0 && !wwait(bars + 8 * B_IX, 0)) dead = true;
    tc_fence_after();
    epilogue(3, !dead && nst > 0);
    if (dead && lane == 0) atomicAdd(errp, kStuck);
  } else {
    // ---------------- softmax (warps 0-1): one token (lane) per thread ----------------
    float* facw = reinterpret_cast<float*>(smem + kFacOff);
    const int tok = 32 * warp + lane;                          // row of S^T / P^T
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // per-head state of heads 2*lane and 2*lane + 1: the running maximum
    // (the same in both warps) and this warp's share of the sum
    float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};
    uint32_t mxc = 0, rsc = 0;
    bool dead = false;
    for (int n = 0; n < nst; ++n) {
      const int sb = n & 1;
      if (!wwait(bars + 8 * (B_S_FULL + sb), (n >> 1) & 1)) {
        dead = true;
        break;
      }
      tc_fence_after();
      float s[64];
      {
        uint32_t u0[32], u1[32];
        tc_ld32(tmem + lane_off + kColS + sb * kSt, u0);
        tc_ld32(tmem + lane_off + kColS + sb * kSt + 32, u1);
        tc_wait_ld(u0);
        tc_wait_ld(u1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(u0[i]);
          s[32 + i] = __uint_as_float(u1[i]);
        }
      }
      tc_fence_before();
      warp_arrive(bars + 8 * (B_S_FREE + sb));
      const int t = n * kSt + tok;
      const bool valid = t < n_sel && sel[t] >= 0;
      // per-head maximum over this warp's 32 tokens (raw scores; the scale is positive)
      float mine[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        const float wm = warp_max_f32(valid ? s[h] : -INFINITY);
        if (lane == (h >> 1)) mine[h & 1] = wm;
      }
      float* wm_st = wmax + sb * 2 * kHB;
      wm_st[warp * kHB + 2 * lane] = mine[0];
      wm_st[warp * kHB + 2 * lane + 1] = mine[1];
      warp_arrive(bars + 8 * B_MX);
      if (!wwait(bars + 8 * B_MX, mxc & 1)) {
        dead = true;
        break;
      }
      ++mxc;
      float f2[2], mb2[2];
      bool need_any = false;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * lane + e;
        const float tm = fmaxf(wm_st[h], wm_st[kHB + h]) * A.sl2;
        const bool grow = tm > m2[e] + kRescaleThreshold;
        const bool need = grow && m2[e] > -INFINITY;         // O^T already holds this head's sums
        f2[e] = need ? exp2f(m2[e] - tm) : 1.f;
        if (grow) m2[e] = tm;
        l2[e] *= f2[e];
        need_any |= need;
        mb2[e] = m2[e] == -INFINITY ? 0.f : m2[e];
      }
      const bool rs = __any_sync(0xffffffffu, need_any);      // the same in both warps
      if (warp == 0) {
        facw[sb * kHB + 2 * lane] = f2[0];
        facw[sb * kHB + 2 * lane + 1] = f2[1];
        if (lane == 0) misc[1 + sb] = rs ? 1 : 0;
      }
      // P (fp32, kept in s) and P^T row `tok` in the slot's rope chunk: 64
      // heads (bf16), 16-byte units swizzled by tok & 7
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        const float mh = __shfl_sync(0xffffffffu, mb2[h & 1], h >> 1);
        s[h] = valid ? ex2_ftz(fmaf(s[h], A.sl2, -mh)) : 0.f;
      }
      const uint32_t prow = sbase + kSlotOff + sb * kStageB + 8 * kChunkB + tok * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(prow + ((u ^ (tok & 7)) << 4)),
                     "r"(pack_bf16(s[8 * u], s[8 * u + 1])),
                     "r"(pack_bf16(s[8 * u + 2], s[8 * u + 3])),
                     "r"(pack_bf16(s[8 * u + 4], s[8 * u + 5])),
                     "r"(pack_bf16(s[8 * u + 6], s[8 * u + 7]))
                     : "memory");
      fence_proxy_async_smem();
      warp_arrive(bars + 8 * (B_P_FULL + sb));
      // this warp's per-head sums of P over its 32 tokens: recursive halving
      // leaves heads 2*lane and 2*lane + 1 in this lane
#pragma unroll
      for (int w = 32, o = 16; o > 0; w >>= 1, o >>= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
          const float send = hi ? s[i] : s[w + i];
          const float keep = hi ? s[w + i] : s[i];
          s[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      l2[0] += s[0];
      l2[1] += s[1];
      if (rs) {
        if (!wwait(bars + 8 * B_RS_GO, rsc & 1)) {
          dead = true;
          break;
        }
        ++rsc;
        tc_fence_after();
        rescale(warp, fac + sb * kHB);
        tc_fence_before();
        warp_arrive(bars + 8 * B_RS_DONE);
      }
    }
    // O^T is complete (the P V warp's last phase of B_RS_GO); publish the sums
    // then warp 0 adds the two warps' sums, publishes 1 / l per head for the
    // four epilogue warps and writes the LSE
    float lt[2] = {0.f, 0.f};
    if (!dead && nst > 0) {
      if (!wwait(bars + 8 * B_RS_GO, rsc & 1)) {
        dead = true;
      } else {
        wmax[warp * kHB + 2 * lane] = l2[0];
        wmax[warp * kHB + 2 * lane + 1] = l2[1];
        warp_arrive(bars + 8 * B_LX);
        if (warp == 0) {
          if (!wwait(bars + 8 * B_LX, 0)) {
            dead = true;
          } else {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int h = 2 * lane + e;
              lt[e] = wmax[h] + wmax[kHB + h];
              facw[h] = lt[e] > 0.f ? 1.f / lt[e] : 0.f;
            }
            warp_arrive(bars + 8 * B_IX);
          }
        } else if (!wwait(bars + 8 * B_IX, 0)) {
          dead = true;
        }
      }
    }
    tc_fence_after();
    epilogue(warp, !dead && nst > 0);
    if (warp == 0) {
      const int64_t orow = ((int64_t)r * A.B + b) * A.Hq + h0;
#pragma unroll
      for (int e = 0; e < 2; ++e)
        A.part_lse[orow + 2 * lane + e] =
            lt[e] > 0.f ? (m2[e] + log2f(lt[e])) * kLn2 : -INFINITY;
    }
    if (dead && lane == 0) atomicAdd(errp, kStuck);
  }
  if (tid == 0 && nst == 0 && !mbar_wait(bars + 8 * B_Q_FULL, 0)) atomicAdd(errp, kStuck);
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kTmemCols);
  }
}

namespace {

bool encode_q(CUtensorMap* map, const void* base, uint64_t rows) {
  auto enc = tensor_map_encoder();
  if (!enc || ((uintptr_t)base & 15) || rows == 0 || rows > (1ull << 31)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kRowE, rows};
  cuuint64_t strides[1] = {(cuuint64_t)kRowB};
  cuuint32_t box[2] = {64, (cuuint32_t)kHB};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool sfa_tc_supported(int Hq, int dk, int dv, dcp_dtype_t dtype, int K, int64_t pool_rows,
                      const void* q, const dcp_rank_ptrs_t& pool, int dcp) {
  if (dtype != DCP_BF16 || dk != kRowE || dv != 512 || Hq % kHB != 0 || K > kMaxSelTc) return false;
  if (pool_rows <= 0 || pool_rows >= (int64_t(1) << 31)) return false;
  if ((uintptr_t)q & 15) return false;
  for (int r = 0; r < dcp; ++r)
    if (!pool.ptr[r] || ((uintptr_t)pool.ptr[r] & 15)) return false;
  if (getenv("DCP_DISABLE_TCGEN05")) return false;
  return tensor_map_encoder() != nullptr;
}

int launch_sfa_tc(const SfaTcArgs& A0, const void* q, int dcp, cudaStream_t s, bool pdl) {
  SfaTcArgs A = A0;
  A.hblocks = A.Hq / kHB;
  if (!encode_q(&A.qmap, q, (uint64_t)A.B * A.Hq)) return DCP_ECUDA;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(sfa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSfaTcSmem);
    if (e != cudaSuccess) {
      launch_status_report(e);
      return DCP_ECUDA;
    }
    attr_done[dev] = true;
  }
  const int grid = dcp * A.B * A.hblocks;
  if (grid <= 0) return DCP_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kSfaTcThreads);
  cfg.dynamicSmemBytes = kSfaTcSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sfa_tc_kernel, A);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

}  // namespace dcp
