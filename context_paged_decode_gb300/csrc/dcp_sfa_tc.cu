// tcgen05 SFA decode partials: per (group of ranks, request, 64 query heads),
// sparse attention over the selected tokens each rank owns, MLA-shaped
// latent rows (576 bf16: key = whole row, value = first 512 entries), bf16
// in, fp32 accumulate.
//
// Page "Decode Context Parallel (DCP)", section "GLM-5.2 SFA DCP replicated
// indexer": the global top-k indices are remapped to local KV indices
// before SFA runs; each rank attends only the selected tokens it stores and
// the per-rank results are merged by LSE (the sink is applied once, at the
// merge: page "DeepSeek V4.1 context parallelism", section "Decode
// computation").
//
// The two products per 64-token stage:
//   S   [64 heads x 64 tokens]       = Q . K_stage^T    (M=64: 9 chunks x 4 MMAs)
//   O^T [512 value rows x 64 heads] += V_stage^T . P^T  (4 row blocks x 4 MMAs)
// Shape of the kernel:
//  * one CTA per (group of ranks, request, 64 query heads).  The host picks
//    the fewest ranks per group for which the grid fits in one wave of one
//    CTA per SM (two ranks for 32 requests of 64 heads on 8 ranks: 128
//    CTAs on 152 SMs), so no CTA waits for a second wave and the ranks of a
//    group share one load of Q and one pass over the request's pairs.  The
//    CTA lists each rank's selected slots in top-k order, one segment per
//    rank, and walks the segments' 64-token stages through a two-slot ring
//    without draining it between ranks.  A segment's output is written as
//    that rank's partial when its last P V completed; the next segment's
//    first P V waits for those tensor-memory reads;
//  * shared memory: Q (64 heads x 576 as nine 8 KB chunks, 128-byte swizzle,
//    one TMA box each), two 72 KB stage slots (nine 8 KB chunks of 64 token
//    rows x 64 columns in the same layout) and the selection list.  The
//    ninth (rope) chunk of a slot is dead once that stage's S is complete,
//    and P^T takes its place: 64 head rows of 64 tokens (bf16), K-major;
//  * S runs at M=64 with the heads as rows, so that a stage's scores of one
//    head sit in one thread: tensor-memory lanes 0-15 of each lane quarter
//    hold heads 16q .. 16q+15 (the M=64 accumulator layout), and the
//    softmax's maximum and sum need no exchange between threads;
//  * four warps gather with 16-byte cp.async (whole 1152-byte rows;
//    unselected, unusable and tail rows are zero-filled).  Each walks every
//    stage, taking a quarter of its rows, and never waits for its copies:
//    cp.async.mbarrier.arrive.noinc arrives on the slot's barrier once the
//    thread's copies have landed, so all four warps start on a slot the
//    moment it is free.  The threads that wait on that barrier fence the
//    data for the tensor core.  The rows carry an L2 evict-first hint and
//    the partials an evict-last hint, so the merge finds the partials in L2;
//  * one thread issues a tcgen05.mma only every ~55-100 cycles, so Q.K^T is
//    split between two issuing warps (latent chunks 0-4 and 5-8) into two
//    partial accumulators that the softmax adds, in a fixed order, and P V
//    between two more (O^T value rows 0-255 and 256-511);
//  * tensor memory: two pairs of partial S buffers (64 columns each), O^T
//    (4 x 64 columns);
//  * in the fused decode the CTAs of a (request, head block) form a cluster:
//    once each has written its ranks' partials (and a cluster barrier made
//    them visible), each merges its share of the request's head rows by LSE
//    from L2 (one warp per row, every part loaded before any is used), with
//    the sink applied once, so no separate merge launch waits for the whole
//    grid;
//  * warps 0-3: softmax of their lane quarter's 16 heads (threads l and
//    l + 16 take tokens 0-31 and 32-63 of head 16 q + l), rescale and
//    epilogue of their quarter of O^T (value rows).  Warps 4 and 6 issue
//    Q.K^T, warps 5 and 7 P V.  O^T columns (heads) are rescaled
//    only when a head's running maximum grows by more than 8 (log2 units),
//    which keeps P <= 256; the leading P V warp orders that rescale between
//    two P Vs.
// Every mbarrier wait is bounded; a timed-out wait adds 1<<20 to the error
// counter and that role stops waiting, so the kernel always terminates.
#include <stdlib.h>
#include <string.h>

#include "dcp_merge.cuh"
#include "dcp_sfa_tc.cuh"

namespace dcp {

namespace {

constexpr int kHB = 64;                                // heads per CTA
constexpr int kRowE = 576;
constexpr int kRowB = kRowE * 2;                       // 1152 bytes per latent row
constexpr int kChunks = 9;                             // 64-column chunks of a row
constexpr int kSt = 64;                                // tokens per stage
constexpr int kChunkB = kSt * 128;                     // 8 KB
constexpr int kStageB = kChunks * kChunkB;             // 72 KB
constexpr int kQOff = 0;
constexpr int kSlotOff = kChunks * kHB * 128;          // 72 KB
constexpr int kSelOff = kSlotOff + 2 * kStageB;        // 216 KB
constexpr int kMaxSelTc = kSfaTcMaxSel;
// stages of one CTA: every selected entry belongs to one rank, and each rank
// adds at most one partly filled stage
constexpr int kMaxStages = kMaxSelTc / kSt + DCP_MAX_RANKS;
constexpr int kTabOff = kSelOff + kMaxSelTc * 4;       // stage table, one word per stage
constexpr int kFacOff = kTabOff + kMaxStages * 4;      // [parity][head] rescale factors
constexpr int kFlagOff = kFacOff + 2 * kHB * 4;        // [parity][softmax warp] rescale flags
constexpr int kInvOff = kFlagOff + 2 * 4 * 4;          // 1 / l per head of the segment
// misc words: 4 the stage count; 8 .. 8 + DCP_MAX_RANKS - 1 the selected
// entries of each rank of the group
constexpr int kMiscWords = 8 + DCP_MAX_RANKS;
constexpr int kMiscOff = kInvOff + kHB * 4;
constexpr int kBarOff = kMiscOff + kMiscWords * 4;
constexpr int kNumBars = 16;
constexpr int kSfaTcSmem = 1024 + kBarOff + kNumBars * 8 + 16;
constexpr int kSoftmaxWarps = 4;
constexpr int kQkWarpA = 4, kPvWarp = 5, kQkWarpB = 6, kPvWarpB = 7;
constexpr int kQkSplit = 5;                            // chunks [0, 5) -> S_a, [5, 9) -> S_b
constexpr int kFirstGather = 8;
constexpr int kGatherWarps = 4;
constexpr bool kL2Hints = true;   // gathered rows evict first; partials (read by the merge) last
constexpr int kSfaTcThreads = 32 * (kFirstGather + kGatherWarps);   // 384
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColSa = 0, kColSb = 2 * kSt, kColO = 4 * kSt;
constexpr float kRescaleThreshold = 8.f;
constexpr int kStuck = 1 << 20;

static_assert(kSfaTcSmem <= 227 * 1024, "shared memory overflow");
static_assert(kSlotOff % 1024 == 0 && kStageB % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kColO + 4 * kHB <= kTmemCols, "tensor memory overflow");
static_assert(kSfaTcThreads <= 384, "three warps per sub-partition keep 168 registers a thread");
static_assert(kMaxSelTc <= 4096 && kSt < 128 && DCP_MAX_RANKS <= 32, "stage-table fields");

// barrier slots
enum : int {
  B_Q_FULL = 0,
  B_FULL = 1,        // +slot: the stage in the slot landed (every gather thread's copies)
  B_SLOT_FREE = 3,   // +slot: both halves of the P V that read the slot completed
  B_S_FULL = 5,      // +buffer: both partial S of the stage are complete
  B_S_FREE = 7,      // +buffer: the softmax warps read it
  B_P_FULL = 9,      // +stage parity: P^T, the factors and the rescale flags are stored
  B_PVD = 11,        // one phase per P V completed (both halves)
  B_RS_GO = 12,      // the P V warp: rescale now (rescale stages), or O^T is complete
  B_RS_DONE = 13,    // the softmax warps rescaled their quarters
  B_IX = 14,         // the softmax warps published 1 / l of their heads (per segment)
  B_DRAIN = 15       // the softmax warps read the segment's O^T (its epilogue is done)
};

__device__ __forceinline__ int arrivals(int i) {
  if (i == B_FULL || i == B_FULL + 1) return 32 * kGatherWarps;
  if (i == B_S_FULL || i == B_S_FULL + 1 || i == B_SLOT_FREE || i == B_SLOT_FREE + 1 ||
      i == B_PVD)
    return 2;
  if (i == B_S_FREE || i == B_S_FREE + 1 || i == B_P_FULL || i == B_P_FULL + 1 ||
      i == B_RS_DONE || i == B_IX || i == B_DRAIN)
    return kSoftmaxWarps;
  return 1;
}

// S = Q . K^T: A = Q (64 head rows, K-major), B = K (64 token rows, K-major)
constexpr uint32_t kIdescQK = idesc_bf16_f32(64, kSt, false, false);
// O^T += V^T . P^T: A = V^T (MN-major), B = P^T (64 head rows of tokens, K-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kHB, true, false);

// 16 bytes global -> shared; bytes == 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16_fill(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
// The same with an L2 eviction policy.
__device__ __forceinline__ void cp_async16_fill_hint(uint32_t dst, const void* src, uint32_t bytes,
                                                     uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
               "l"(src), "r"(bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_f32_hint(float* dst, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst), "f"(v), "l"(policy)
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// One word per stage: first entry of the stage in the selection list (12
// bits), entries in the stage (7), segment (5), first / last stage of its
// segment (1 + 1).
__device__ __forceinline__ int st_pack(int start, int n, int seg, bool first, bool last) {
  return start | (n << 12) | (seg << 19) | ((first ? 1 : 0) << 24) | ((last ? 1 : 0) << 25);
}
__device__ __forceinline__ int st_start(int e) { return e & 0xFFF; }
__device__ __forceinline__ int st_count(int e) { return (e >> 12) & 0x7F; }
__device__ __forceinline__ int st_seg(int e) { return (e >> 19) & 0x1F; }
__device__ __forceinline__ bool st_first(int e) { return (e >> 24) & 1; }
__device__ __forceinline__ bool st_last(int e) { return (e >> 25) & 1; }

}  // namespace

// Twelve warps put three on every SM sub-partition (16K registers each), so
// a thread may hold up to 168 registers.
__global__ void __launch_bounds__(kSfaTcThreads, 1) sfa_tc_kernel(const __grid_constant__ SfaTcArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  int32_t* sel = reinterpret_cast<int32_t*>(smem + kSelOff);
  int32_t* tab = reinterpret_cast<int32_t*>(smem + kTabOff);
  volatile int32_t* misc = reinterpret_cast<volatile int32_t*>(smem + kMiscOff);
  float* fac = reinterpret_cast<float*>(smem + kFacOff);
  volatile int32_t* flags = reinterpret_cast<volatile int32_t*>(smem + kFlagOff);
  float* invl = reinterpret_cast<float*>(smem + kInvOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // block -> (group of ranks, request, head block); in a fused launch the
  // groups of one (request, head block) are consecutive blocks (one cluster)
  const int per_group = A.B * A.hblocks;
  const int grp = A.fuse ? (int)(blockIdx.x % A.ngroups) : (int)(blockIdx.x / per_group);
  const int rem = A.fuse ? (int)(blockIdx.x / A.ngroups) : (int)(blockIdx.x % per_group);
  const int r0 = grp * A.rpc;                                 // first rank of the group
  const int nr = min(A.rpc, A.dcp - r0);                      // ranks in the group
  const int b = rem / A.hblocks, h0 = (rem % A.hblocks) * kHB;
  const int64_t num_slots = A.num_blocks * A.bs;
  int32_t* errp = A.err;

  griddep_launch_dependents();   // a dependent merge launch may start waiting
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bars + 8 * i, arrivals(i));
    fence_mbar_init();
    prefetch_tmap(&A.qmap);
    // Q of heads h0 .. h0+63: nine 64 x 64 boxes (awaited by the Q.K^T issuer,
    // or at the end when the group selected no token)
    mbar_arrive_expect_tx(bars + 8 * B_Q_FULL, kChunks * kHB * 128);
    for (int c = 0; c < kChunks; ++c)
      tma_load_2d(sbase + kQOff + c * kHB * 128, &A.qmap, 64 * c, b * A.Hq + h0,
                  bars + 8 * B_Q_FULL);
  }
  if (warp == kQkWarpA) {
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

  // ---- the group's selected slots: one segment per rank, each in top-k order
  // (-1: unusable, attended as masked), then one table word per stage ----
  {
    constexpr int kPer = 6;
    static_assert(kPer * kSfaTcThreads >= kMaxSelTc, "selection runs must cover kMaxSelTc");
    const int per = (A.K + kSfaTcThreads - 1) / kSfaTcThreads;
    const int k0 = min(A.K, tid * per), k1 = min(A.K, k0 + per);
    int64_t slot[kPer];
    int rel[kPer];                                            // rank - r0, or -1
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int k = k0 + i;
      const int rk = k < k1 ? __ldg(A.sel_rank + (int64_t)b * A.K + k) : -1;
      slot[i] = k < k1 ? (int64_t)__ldg(A.sel_slot + (int64_t)b * A.K + k) : -1;
      rel[i] = (rk >= r0 && rk < r0 + nr) ? rk - r0 : -1;
    }
    int* wsum = reinterpret_cast<int*>(fac);                  // free until the first stage
    int off = 0;
    for (int j = 0; j < nr; ++j) {
      int mine = 0;
#pragma unroll
      for (int i = 0; i < kPer; ++i) mine += rel[i] == j ? 1 : 0;
      int x = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wsum[warp] = x;
      __syncthreads();
      int base = 0, total = 0;
      for (int w = 0; w < kSfaTcThreads / 32; ++w) {
        const int c = wsum[w];
        if (w < warp) base += c;
        total += c;
      }
      base += off + x - mine;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        if (rel[i] == j) {
          int64_t sl = slot[i];
          if (sl < 0 || sl >= num_slots) {
            if (h0 == 0) count_error(errp);
            sl = -1;
          }
          if (base < kMaxSelTc) sel[base] = (int32_t)sl;
          ++base;
        }
      }
      if (tid == 0) misc[8 + j] = total;
      off += total;
      __syncthreads();                                        // wsum is rewritten next
    }
    if (tid == 0) {
      int n = 0, start = 0;
      for (int j = 0; j < nr; ++j) {
        const int c = min((int)misc[8 + j], kMaxSelTc - start);
        const int ns = (c + kSt - 1) / kSt;
        for (int t = 0; t < ns && n < kMaxStages; ++t)
          tab[n++] = st_pack(start + t * kSt, min(kSt, c - t * kSt), j, t == 0, t == ns - 1);
        start += c;
      }
      misc[4] = n;
    }
    __syncthreads();
  }
  const int nst = misc[4];

  // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform
  auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, par));
  };
  auto warp_arrive = [&](uint32_t bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };

  if (warp >= kFirstGather) {
    // ---------------- gather: every warp takes part in every stage ----------------
    const int gw = warp - kFirstGather;
    bool dead = false;
    for (int n = 0; n < nst; ++n) {
      const int slot = n & 1;
      // the slot is free once the P V of stage n - 2 completed
      if (!wwait(bars + 8 * (B_SLOT_FREE + slot), ((n >> 1) & 1) ^ 1)) {
        dead = true;
        break;
      }
      const int e = tab[n];
      const int s0 = st_start(e), cnt = st_count(e);
      const uint8_t* pool = A.pool[r0 + st_seg(e)];
      const uint32_t dst0 = sbase + kSlotOff + slot * kStageB;
      // a warp takes groups of 4 token rows (one slot-list read per lane and
      // group); each copy instruction moves chunk c of the 4 rows: lane l
      // copies 16-byte unit l % 8 of row 4 g + l / 8, swizzled by the row & 7.
      // All 32 lanes copy in every instruction: the load pipe's cost is per
      // instruction, whatever its active lanes.  16 groups over four warps,
      // four each, which groups rotating from stage to stage.
      const int rsub = lane >> 3, un = lane & 7;
#pragma unroll 1
      for (int rg = (gw + n) % kGatherWarps; rg < kSt / 4; rg += kGatherWarps) {
        const int rr = rg * 4 + rsub;
        const int row = rr < cnt ? sel[s0 + rr] : -1;
        const uint8_t* rsrc = row >= 0 ? pool + (int64_t)row * kRowB + un * 16 : pool;
        const uint32_t bytes = row >= 0 ? 16u : 0u;
        const uint32_t rdst = dst0 + rr * 128 + ((uint32_t)(un ^ (rr & 7)) << 4);
        if (kL2Hints) {
          const uint64_t pol = policy_evict_first();
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
            cp_async16_fill_hint(rdst + c * kChunkB, row >= 0 ? rsrc + c * 128 : pool, bytes, pol);
        } else {
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
            cp_async16_fill(rdst + c * kChunkB, row >= 0 ? rsrc + c * 128 : pool, bytes);
        }
      }
      cp_async_arrive_noinc(bars + 8 * (B_FULL + slot));
    }
    cp_async_wait<0>();
    if (dead && lane == 0) atomicAdd(errp, kStuck);
    // ranks of the group with no selected token: o = 0, lse = -inf
    const int zt = tid - 32 * kFirstGather, zn = 32 * kGatherWarps;
    for (int j = 0; j < nr; ++j) {
      if (misc[8 + j] != 0) continue;
      const int64_t orow = ((int64_t)(r0 + j) * A.B + b) * A.Hq + h0;
      float4* dst = reinterpret_cast<float4*>(A.part_o + orow * 512);
      for (int i = zt; i < kHB * 512 / 4; i += zn) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = zt; i < kHB; i += zn) A.part_lse[orow + i] = -INFINITY;
    }
  } else if (warp == kQkWarpA || warp == kQkWarpB) {
    // ---------------- Q.K^T issuers: chunks [c0, c1) into partial S ----------------
    if (lane == 0) {
      const int c0 = warp == kQkWarpA ? 0 : kQkSplit, c1 = warp == kQkWarpA ? kQkSplit : kChunks;
      const uint32_t col = warp == kQkWarpA ? kColSa : kColSb;
      bool dead = nst > 0 && !mbar_wait(bars + 8 * B_Q_FULL, 0);
      for (int n = 0; n < nst && !dead; ++n) {
        const int sb = n & 1;                                  // slot and S buffer
        const uint32_t u = (uint32_t)(n >> 1) & 1u;
        if (!mbar_wait2_cluster(bars + 8 * (B_FULL + sb), u, bars + 8 * (B_S_FREE + sb), u ^ 1u)) {
          dead = true;
          break;
        }
        // the gathered rows were written by cp.async (generic proxy): make
        // them visible to the tensor core's reads
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t st = sbase + kSlotOff + sb * kStageB;
#pragma unroll 1
        for (int c = c0; c < c1; ++c) {
          const uint64_t ad = sdesc_sw128(sbase + kQOff + c * kHB * 128, 0, 1024);
          const uint64_t bd = sdesc_sw128(st + c * kChunkB, 0, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_ss(tmem + col + sb * kSt, ad + (uint64_t)((kk * 32) >> 4),
                      bd + (uint64_t)((kk * 32) >> 4), kIdescQK, (c > c0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bars + 8 * (B_S_FULL + sb));
      }
      if (dead) atomicAdd(errp, kStuck);
    }
  } else if (warp == kPvWarp || warp == kPvWarpB) {
    // ---------------- P V issuers: O^T row blocks [2 half, 2 half + 2) ----------------
    // The first (the leader) orders the rescales and announces the end of a
    // segment; both wait for the rescale they need before their P V.
    if (lane == 0) {
      const bool leader = warp == kPvWarp;
      const int mb0 = leader ? 0 : 2;
      uint32_t pvd_seen = 0, rsc = 0, drc = 0;
      bool dead = false;
      // Observe every phase of B_PVD in order, up to the P V of stage k (the
      // leader only).  A parity wait is unambiguous only while the barrier is
      // at most one phase past the last one observed, so the leader issues
      // the P V of stage n only after that of stage n - 1 was seen to complete.
      auto pvd_upto = [&](int k) -> bool {
        while ((int)pvd_seen <= k) {
          if (!mbar_wait(bars + 8 * B_PVD, pvd_seen & 1)) return false;
          ++pvd_seen;
        }
        return true;
      };
      for (int n = 0; n < nst && !dead; ++n) {
        const int sb = n & 1;
        const int e = tab[n];
        // a segment's first P V overwrites O^T: the previous segment's
        // epilogue must have read it
        if (st_first(e) && n > 0) {
          if (!mbar_wait(bars + 8 * B_DRAIN, drc & 1)) {
            dead = true;
            break;
          }
          ++drc;
        }
        if (!mbar_wait(bars + 8 * (B_P_FULL + sb), (n >> 1) & 1) || (leader && !pvd_upto(n - 1))) {
          dead = true;
          break;
        }
        if ((flags[sb * 4 + 0] | flags[sb * 4 + 1] | flags[sb * 4 + 2] | flags[sb * 4 + 3]) != 0) {
          // rescale stage: the softmax warps multiply their O^T quarters by
          // the stage's factors once both halves of P V n - 1 completed
          if (leader) mbar_arrive(bars + 8 * B_RS_GO);
          if (!mbar_wait(bars + 8 * B_RS_DONE, rsc & 1)) {
            dead = true;
            break;
          }
          ++rsc;
        }
        fence_proxy_async_smem();
        tc_fence_after();
        // O^T[mb] += V^T . P^T: V^T is MN-major (value columns contiguous, the
        // two 64-column chunks of row block mb one chunk apart); P^T is
        // K-major (each head's 64 tokens contiguous); k-step kk = tokens
        // 16kk .. 16kk+15
        const uint32_t st = sbase + kSlotOff + sb * kStageB;
        const uint64_t pd0 = sdesc_sw128(st + 8 * kChunkB, 0, 1024);
        const bool first = st_first(e);
#pragma unroll
        for (int kk = 0; kk < kSt / 16; ++kk) {
#pragma unroll
          for (int mb = mb0; mb < mb0 + 2; ++mb) {
            const uint64_t vd = sdesc_sw128(st + 2 * mb * kChunkB + kk * 2048, kChunkB, 1024);
            tc_mma_ss(tmem + kColO + 64 * mb, vd, pd0 + (uint64_t)((kk * 32) >> 4), kIdescPV,
                      (first && kk == 0) ? 0u : 1u);
          }
        }
        tc_commit(bars + 8 * (B_SLOT_FREE + sb));
        tc_commit(bars + 8 * B_PVD);
        if (leader && st_last(e)) {
          // the segment's O^T is complete once both halves of this P V
          // completed: release the softmax warps for the epilogue
          if (!pvd_upto(n)) {
            dead = true;
            break;
          }
          mbar_arrive(bars + 8 * B_RS_GO);
        }
      }
      if (dead) atomicAdd(errp, kStuck);
    }
  } else {
    // ---------------- softmax, rescale, epilogue (warps 0-3, lane quarter = warp) --------
    // Threads l and l + 16 of warp w own head hl = 16 w + l: tokens 0-31 and
    // 32-63 of every stage, the running maximum m (log2 units, the same in
    // both) and a share of the sum l.  Every lane takes part in the rescale
    // and the epilogue of the quarter's value rows.
    const int hl = 16 * warp + (lane & 15);
    const bool hi = lane >= 16;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m2 = -INFINITY, l2 = 0.f;
    uint32_t rsc = 0, ixc = 0;
    bool dead = false;
    // multiply this quarter's O^T columns by the per-head factors f[64]
    auto rescale = [&](const float* f) {
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
    for (int n = 0; n < nst; ++n) {
      const int sb = n & 1;
      const int e = tab[n];
      if (st_first(e)) {
        m2 = -INFINITY;
        l2 = 0.f;
      }
      if (!wwait(bars + 8 * (B_S_FULL + sb), (n >> 1) & 1)) {
        dead = true;
        break;
      }
      tc_fence_after();
      // S = S_a + S_b: head hl's row sits in tensor-memory lane hl % 16 of
      // the quarter (M=64 layout); the 16x32bx2 load gives thread l its
      // tokens 0-31 and thread l + 16 its tokens 32-63
      float s[32];
      {
        uint32_t a[32], c[32];
        tc_ld16x2_32<32>(tmem + lane_off + kColSa + sb * kSt, a);
        tc_ld16x2_32<32>(tmem + lane_off + kColSb + sb * kSt, c);
        tc_wait_ld(a);
        tc_wait_ld(c);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(a[i]) + __uint_as_float(c[i]);
      }
      tc_fence_before();
      // tokens of the stage that are attended: lane t checks tokens t, t + 32
      const int cnt = st_count(e), s0 = st_start(e);
      const uint32_t v_lo =
          __ballot_sync(0xffffffffu, lane < cnt && sel[s0 + lane] >= 0);
      const uint32_t v_hi =
          __ballot_sync(0xffffffffu, lane + 32 < cnt && sel[s0 + lane + 32] >= 0);
      const uint32_t vm = hi ? v_hi : v_lo;
      // this head's stage maximum (raw scores; the scale is positive), in
      // four independent chains
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int t = 0; t < 32; ++t) mq[t & 3] = fmaxf(mq[t & 3], ((vm >> t) & 1u) ? s[t] : -INFINITY);
      float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float tm = mx * A.sl2;
      const bool grow = tm > m2 + kRescaleThreshold;
      const bool need = grow && m2 > -INFINITY;                 // O^T already holds its sums
      const float f = need ? exp2f(m2 - tm) : 1.f;
      if (grow) m2 = tm;
      l2 *= f;
      const uint32_t need_w = __ballot_sync(0xffffffffu, need);
      if (!hi) fac[sb * kHB + hl] = f;
      if (lane == 0) flags[sb * 4 + warp] = need_w != 0 ? 1 : 0;
      // P (fp32 in s) and this thread's half of row hl of P^T in the slot's
      // rope chunk: 32 tokens (bf16), 16-byte units swizzled by hl & 7
      float pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        s[t] = ((vm >> t) & 1u) ? ex2_ftz(fmaf(s[t], A.sl2, -m2)) : 0.f;
        pq[t & 3] += s[t];
      }
      l2 += (pq[0] + pq[1]) + (pq[2] + pq[3]);
      {
        const uint32_t prow = sbase + kSlotOff + sb * kStageB + 8 * kChunkB + hl * 128;
        const int u0 = hi ? 4 : 0;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                           prow + (((u0 + u) ^ (hl & 7)) << 4)),
                       "r"(pack_bf16(s[8 * u], s[8 * u + 1])),
                       "r"(pack_bf16(s[8 * u + 2], s[8 * u + 3])),
                       "r"(pack_bf16(s[8 * u + 4], s[8 * u + 5])),
                       "r"(pack_bf16(s[8 * u + 6], s[8 * u + 7]))
                       : "memory");
      }
      fence_proxy_async_smem();
      warp_arrive(bars + 8 * (B_P_FULL + sb));
      // every softmax warp's flags are stored once the stage's P is complete
      if (!wwait(bars + 8 * (B_P_FULL + sb), (n >> 1) & 1)) {
        dead = true;
        break;
      }
      const bool rs = (flags[sb * 4 + 0] | flags[sb * 4 + 1] | flags[sb * 4 + 2] |
                       flags[sb * 4 + 3]) != 0;
      // S of this buffer was read long ago, but the release waits until the
      // flags are read: the next writer of these flags (stage n + 2) needs
      // Q.K^T of stage n + 2, which needs this release
      warp_arrive(bars + 8 * (B_S_FREE + sb));
      if (rs) {
        if (!wwait(bars + 8 * B_RS_GO, rsc & 1)) {
          dead = true;
          break;
        }
        ++rsc;
        tc_fence_after();
        rescale(fac + sb * kHB);
        tc_fence_before();
        warp_arrive(bars + 8 * B_RS_DONE);
      }
      if (st_last(e)) {
        // the segment's O^T is complete (the P V warp's event on B_RS_GO):
        // write this head's LSE, publish 1 / l, and write the quarter's rows
        if (!wwait(bars + 8 * B_RS_GO, rsc & 1)) {
          dead = true;
          break;
        }
        ++rsc;
        const float lt = l2 + __shfl_xor_sync(0xffffffffu, l2, 16);
        const int r = r0 + st_seg(e);
        const int64_t orow = ((int64_t)r * A.B + b) * A.Hq + h0;   // row of head h0
        if (!hi) {
          invl[hl] = lt > 0.f ? 1.f / lt : 0.f;
          A.part_lse[orow + hl] = lt > 0.f ? (m2 + log2f(lt)) * kLn2 : -INFINITY;
        }
        warp_arrive(bars + 8 * B_IX);
        if (!wwait(bars + 8 * B_IX, ixc & 1)) {
          dead = true;
          break;
        }
        ++ixc;
        tc_fence_after();
        float inv[64];
#pragma unroll
        for (int h = 0; h < 64; ++h) inv[h] = invl[h];
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          const int d = 128 * mb + 32 * warp + lane;             // value column
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t o[32];
            tc_ld32(tmem + lane_off + kColO + 64 * mb + 32 * hh, o);
            tc_wait_ld(o);
            if (kL2Hints) {
              const uint64_t pol = policy_evict_last();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                st_f32_hint(A.part_o + (orow + 32 * hh + i) * 512 + d,
                            __uint_as_float(o[i]) * inv[32 * hh + i], pol);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                A.part_o[(orow + 32 * hh + i) * 512 + d] = __uint_as_float(o[i]) * inv[32 * hh + i];
            }
          }
        }
        tc_fence_before();
        warp_arrive(bars + 8 * B_DRAIN);
      }
    }
    if (dead && lane == 0) atomicAdd(errp, kStuck);
  }
  if (tid == 0 && nst == 0 && !mbar_wait(bars + 8 * B_Q_FULL, 0)) atomicAdd(errp, kStuck);
  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarpA) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kTmemCols);
  }
  if (A.fuse) {
    // every CTA of the cluster wrote its ranks' partials (release / acquire
    // at cluster scope); CTA grp merges (head, chunk) rows grp, grp + ngroups, ...
    cluster_sync();
    DensePartsL2 P;
    P.o = A.part_o;
    P.lse = A.part_lse;
    P.stride = (int64_t)A.B * A.Hq;
    if (A.dcp <= 8) {
      // one warp per head row (all four 128-value chunks): head rows grp,
      // grp + ngroups, ...
      for (int hh = grp + A.ngroups * warp; hh < kHB; hh += A.ngroups * (kSfaTcThreads / 32)) {
        const int64_t row = (int64_t)b * A.Hq + h0 + hh;
        merge_row_chunks<8, 4>(P, A.dcp, row, A.sink != nullptr, A.sink ? A.sink[h0 + hh] : 0.f,
                               A.out, A.out_dtype, row, A.out_lse);
      }
    } else {
      constexpr int kTasks = kHB * 4;                         // (head, 128-value chunk) rows
      for (int t = grp + A.ngroups * warp; t < kTasks; t += A.ngroups * (kSfaTcThreads / 32)) {
        const int hh = t >> 2, ch = t & 3;
        const int64_t row = (int64_t)b * A.Hq + h0 + hh;
        merge_chunk<16>(P, A.dcp, row, 512, ch, A.sink != nullptr, A.sink ? A.sink[h0 + hh] : 0.f,
                        A.out, A.out_dtype, row, A.out_lse);
      }
    }
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

int sfa_tc_ranks_per_cta(int dcp, int B, int hblocks) {
  // the fewest ranks per CTA for which the grid fits in one wave (one CTA
  // per SM); all of them when even that does not fit
  const int sms = num_sms();
  for (int rpc = 1; rpc < dcp; ++rpc)
    if ((int64_t)((dcp + rpc - 1) / rpc) * B * hblocks <= sms) return rpc;
  return dcp;
}

namespace {

int launch_sfa_tc_impl(const SfaTcArgs& A0, const void* q, int dcp, cudaStream_t s, bool pdl,
                       bool want_merge, const float* sink, void* out, int out_dtype,
                       float* out_lse, bool* merged) {
  SfaTcArgs A = A0;
  A.hblocks = A.Hq / kHB;
  A.dcp = dcp;
  A.rpc = sfa_tc_ranks_per_cta(dcp, A.B, A.hblocks);
  A.ngroups = (dcp + A.rpc - 1) / A.rpc;
  // a cluster of the ngroups CTAs of a request (portable size) merges in the kernel
  A.fuse = want_merge && A.ngroups <= 8 ? 1 : 0;
  A.sink = sink;
  A.out = out;
  A.out_dtype = out_dtype;
  A.out_lse = out_lse;
  if (merged) *merged = A.fuse != 0;
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
  const int grid = A.ngroups * A.B * A.hblocks;
  if (grid <= 0) return DCP_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kSfaTcThreads);
  cfg.dynamicSmemBytes = kSfaTcSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  int na = 1;
  if (A.fuse) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)A.ngroups;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sfa_tc_kernel, A);
  if (e != cudaSuccess) return launch_status_report(e);
  return launch_status();
}

}  // namespace

int launch_sfa_tc(const SfaTcArgs& A, const void* q, int dcp, cudaStream_t s, bool pdl) {
  return launch_sfa_tc_impl(A, q, dcp, s, pdl, false, nullptr, nullptr, 0, nullptr, nullptr);
}

int launch_sfa_tc_merged(const SfaTcArgs& A, const void* q, int dcp, cudaStream_t s, bool pdl,
                         const float* sink, void* out, int out_dtype, float* out_lse,
                         bool* merged) {
  return launch_sfa_tc_impl(A, q, dcp, s, pdl, true, sink, out, out_dtype, out_lse, merged);
}

}  // namespace dcp
