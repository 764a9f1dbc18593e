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
//    (items never cross a rank: each shard attends only its local KV, page
//    "Decode Context Parallel (DCP)", section "Decode").  Cluster k runs the
//    contiguous items of run k of the balanced-parts plan, so every cluster
//    gets the same number of tokens and consecutive items mostly share a
//    request (its Q stays loaded);
//  * a cluster of two CTAs per item.  The fp32 output tile 128 x 512 would
//    fill all of tensor memory, so CTA c keeps value columns [256c, 256c+256)
//    of every head.  The 576-wide reduction of Q K^T is split to match: CTA c
//    reduces over latent columns [256c, 256c+256) and rope columns
//    [512+32c, 544+32c);
//  * the softmax is split by heads: CTA c owns heads [64c, 64c+64).  Per
//    stage it receives the peer's fp32 partial scores of those heads (16 KB,
//    bulk copies), adds its own, runs the online softmax, and sends the bf16 P
//    rows of its heads (8 KB) plus each head's rescale factor and running
//    sums back with bulk copies.  Both CTAs then hold all 128 P
//    rows and run P V on their value half;
//  * a stage is 64 tokens: one tcgen05.mma instruction costs its issuing
//    thread about as long as an N=64 product takes the tensor core, so Q K^T
//    runs at N=64 (16 instructions per stage with Q from tensor memory, plus
//    2 for the rope half, whose Q part sits in shared memory);
//  * tensor memory: O half (256 columns) | Q part (128) | two fp32 score
//    buffers of 64 columns.  Shared memory: a 4-deep ring of 36 KB stages
//    (64 tokens x 288 columns), a 16 KB receive slot for the peer's partial
//    scores, a 16 KB staging buffer for the partial scores this CTA sends
//    (each is refilled once the peer has read the previous stage, early in
//    its softmax), two 16 KB P tiles (128 rows x 64 bf16, the A operand of
//    P V), the (factor, sum) side arrays and the rope half of Q;
//  * warps: 0 issues TMA (no separate L2 prefetch: with the 4-deep ring it
//    only added traffic and issue time, 1.92 -> 1.84 ms without it), 1
//    issues Q K^T, 2 issues P V.  Warps 3-10 each sit
//    on the tensor-memory lane quarter warp % 4.  On the quarters of the own
//    heads, two warps run the softmax of each row, one per 32-column half
//    (the two half-row maxima meet in shared memory).  On the quarters of
//    the peer's heads, warps 3-6 ship the partial scores and warps 7-10
//    receive the peer's P: they apply the peer's rescale factors to those
//    rows of O and write those rows' output.  P V waits for them only in the
//    rare stages with a rescale; it reads the 64 factors itself.  Each
//    receiver releases the peer's P slot (a remote arrival) once it has read
//    the side entries.  Shipping stages the scores in
//    shared memory and sends them with bulk copies: 16-byte remote stores
//    would fill the SM's memory-instruction path, which the softmax's
//    shared-memory loads and exp2 instructions also use;
//  * barrier discipline: a barrier that several warps arrive on either has
//    each of them wait for the phase they arrived at, or is split by stage
//    parity so that no warp can arrive for phase n + 1 before phase n has
//    completed; every parity wait is for a phase at most one ahead of the
//    last one that waiter observed;
//  * the output is rescaled only when the running maximum grows by more
//    than 8 (log2 units), so P stays <= 256 and the rare rescale waits for
//    the in-flight P V.
// Every mbarrier wait is bounded; a timed-out wait adds 1<<20 to the error
// counter and that role stops waiting, so the kernel always terminates.
#include <stdlib.h>
#include <string.h>

#include "dcp_mla_tc.cuh"
#include "dcp_ptx.cuh"

namespace dcp {

struct MlaTcArgs {
  CUtensorMap kvmap[DCP_MAX_RANKS];    // [num_blocks*bs rows][576] bf16, box 64 x 64, 128 B swizzle
  CUtensorMap ropemap[DCP_MAX_RANKS];  // same matrix, box 32 x 64, 64 B swizzle
  const uint16_t* q;                   // [B][128][576] bf16
  int B, bs, dcp;
  float sl2;
  const int32_t* bt;
  int max_vb;
  int64_t bt_rank_stride;
  int64_t num_blocks;
  int32_t* err;
};

constexpr int kHeads = 128;
constexpr int kOwn = 64;                               // heads whose softmax a CTA runs
constexpr int kDk = 576;
constexpr int kDvHalf = 256;
constexpr int kSt = 64;                                // tokens per stage
constexpr int kNs = 4;                                 // KV stages in flight
constexpr int kChunkBytes = kSt * 128;                 // 8 KB: 64 tokens x 64 columns
constexpr int kRopeTileBytes = kSt * 64;               // 4 KB: 64 tokens x 32 rope columns
constexpr int kStageBytes = 4 * kChunkBytes + kRopeTileBytes;  // 36 KB
constexpr int kXsPlane = kOwn * 128;                   // 8 KB: 32 fp32 columns of the own rows
constexpr int kXsBytes = 2 * kXsPlane;                 // 16 KB of the peer's partial scores
constexpr int kPtBlock = kHeads * 64;                  // 8 KB: P for 32 tokens, 64-byte rows
constexpr int kPtBytes = 2 * kPtBlock;                 // 16 KB: P, 128 rows x 64 bf16
constexpr int kSideBytes = 2 * kOwn * 8;               // (factor, half-row sum) per half and own row
constexpr int kPMsgBytes = kOwn * 128 + kSideBytes;    // what the peer's softmax sends per stage
constexpr int kQRopeBytes = kHeads * 64;               // 8 KB: this CTA's rope half of Q
constexpr int kKvOff = 0;
constexpr int kXsOff = kKvOff + kNs * kStageBytes;     // 144 KB
constexpr int kStgOff = kXsOff + kXsBytes;             // 160 KB: my partial scores, staged
constexpr int kPtOff = kStgOff + kXsBytes;             // 176 KB
constexpr int kQRopeOff = kPtOff + 2 * kPtBytes;       // 208 KB
constexpr int kSideOwnOff = kQRopeOff + kQRopeBytes;   // 216 KB
constexpr int kSideRecvOff = kSideOwnOff + 2 * kSideBytes;
constexpr int kMxOff = kSideRecvOff + 2 * kSideBytes;  // half-row maxima, [sb][half][row]
constexpr int kBarOff = kMxOff + 3 * 2 * kOwn * 4;      // 221.5 KB
constexpr int kNumBars = 29;
constexpr int kMlaSmem = 1024 + kBarOff + kNumBars * 8 + 16;
constexpr int kFirstRowWarp = 3;
constexpr int kMlaThreads = 32 * (kFirstRowWarp + 8);  // 352
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384;
constexpr float kRescaleThreshold = 8.f;
constexpr int kStuckMla = 1 << 20;

static_assert(kColQ + 4 * 32 <= kColS && kColS + 2 * kSt <= kTmemCols, "tensor memory overflow");
static_assert(kMlaSmem <= 227 * 1024, "shared memory overflow");
static_assert(kNs <= 4, "four barrier slots per ring role");
static_assert(kStageBytes % 1024 == 0 && kXsOff % 1024 == 0 && kPtOff % 1024 == 0 &&
                  kQRopeOff % 1024 == 0,
              "swizzle atoms need 1 KB alignment");
static_assert(kSideOwnOff % 16 == 0 && kSideRecvOff % 16 == 0, "bulk copies need 16 B alignment");

// barrier slots
enum : int {
  B_KV_FULL = 0,    // +stage (kNs)
  B_KV_EMPTY = 4,   // +stage (kNs)
  B_S_FULL = 8,     // +score buffer
  B_S_FREE = 10,    // +score buffer: the softmax and shipper warps have read it
  B_P_FULL = 12,    // +stage parity: all 128 P rows of a stage are in place.  Split by
                    // parity because its arrivals come from two roles, and no role can
                    // reach stage g + 2 before the P V of stage g has consumed phase g
  B_X_FULL = 14,    // the peer's partial scores landed in my receive slot (per stage)
  B_XS_FREE = 16,   // the peer's softmax has read my partial scores (remote arrivals, per stage)
  B_PT_FREE = 18,   // +tile: the P V of both CTAs that read P tile sb completed.  Every
                    // role that waits on tile sb's phase for stage g has observed its
                    // phase for stage g - 2, so a parity wait never aliases
  B_P_RECV = 20,    // +tile: the peer's P rows and side pairs landed
  B_Q_FULL = 22,
  B_Q_EMPTY = 23,
  B_O_FULL = 24,
  B_O_FREE = 25,
  B_RS_DONE = 28,   // the receivers applied the peer's rescale factors (rescale stages only)
  B_MX = 26         // +own quarter: both halves of its rows stored their maxima (per stage,
                    // plus one phase per item for the row sums)
};

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kSt, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kDvHalf, false, true);

__device__ __forceinline__ int arrivals(int i) {
  if (i == B_S_FREE || i == B_S_FREE + 1 || i == B_O_FREE) return 6;
  if (i == B_P_FULL || i == B_P_FULL + 1 || i == B_Q_FULL || i == B_XS_FREE) return 4;
  // the P V of both CTAs (commits) and the peer's two receiver warps (remote)
  if (i == B_PT_FREE || i == B_PT_FREE + 1) return 4;
  if (i == B_MX || i == B_MX + 1 || i == B_RS_DONE) return 2;
  return 1;
}

// Eleven warps put three on some SM sub-partitions (16K registers each), so a
// thread may hold at most 168 registers.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMlaThreads, 1)
mla_tc_kernel(const __grid_constant__ MlaTcArgs A, Plan plan) {
  griddep_launch_dependents();   // the next call's first kernel may start its launch
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();          // 0 or 1: which halves this CTA owns
  const uint32_t peer = crank ^ 1u;
  const int cl = blockIdx.x >> 1;
  const int i0 = plan.pfirst[cl], i1 = plan.pfirst[cl + 1];
  int32_t* errp = A.err ? A.err : plan.hdr + 3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bars + 8 * i, arrivals(i));
    // the receive slot of stage 0 and the P tiles of stages 0 and 1 expect
    // the peer's bytes
    mbar_arrive_expect_tx(bars + 8 * B_X_FULL, kXsBytes);
    for (int i = 0; i < 2; ++i) mbar_arrive_expect_tx(bars + 8 * (B_P_RECV + i), kPMsgBytes);
    fence_mbar_init();
    for (int r = 0; r < A.dcp; ++r) {
      prefetch_tmap(&A.kvmap[r]);
      prefetch_tmap(&A.ropemap[r]);
    }
  }
  if (warp == 1) {
    tc_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // block-table entry of stage j of an item, as loaded (-1 beyond the
  // table).  Entries are fetched stages ahead of use and only then widened,
  // so no instruction waits on the load right after issuing it.
  auto bt_raw = [&](int b, int r, int p0, int j) -> int32_t {
    const int vb = (p0 + j * kSt) / A.bs;
    return vb < A.max_vb ? __ldg(A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb + vb) : -1;
  };
  auto usable = [&](int32_t raw) -> bool { return raw >= 0 && (int64_t)raw < A.num_blocks; };
  // row of the KV matrix holding local position p0 + j*kSt (raw usable)
  auto stage_row = [&](int32_t raw, int p0, int j) -> int {
    const int p = p0 + j * kSt;
    return (int)((int64_t)raw * A.bs + (p - (p / A.bs) * A.bs));
  };
  // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform
  auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, par));
  };
  auto cwait = [&](uint32_t bar, uint32_t par) -> bool {
    return __all_sync(0xffffffffu, mbar_wait_cluster(bar, par));
  };
  auto cwait2 = [&](uint32_t a, uint32_t pa, uint32_t b, uint32_t pb) -> bool {
    return __all_sync(0xffffffffu, mbar_wait2_cluster(a, pa, b, pb));
  };
  auto warp_arrive = [&](uint32_t bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int xlat = 256 * (int)crank, xrope = 512 + 32 * (int)crank;
      uint32_t g = 0;
      bool dead = false;
      for (int it = i0; it < i1 && !dead; ++it) {
        const int4 d = plan.item[it];
        const int b = d.x, r = d.y & 255, p0 = d.z, p1 = d.w;
        const int nst = (p1 - p0 + kSt - 1) / kSt;
        // block-table entries of stages j and j + 1 (the next one is loaded a
        // stage ahead of its use)
        int32_t raw0 = nst > 0 ? bt_raw(b, r, p0, 0) : -1, raw1 = nst > 1 ? bt_raw(b, r, p0, 1) : -1;
        for (int j = 0; j < nst; ++j, ++g) {
          const uint32_t st = g % kNs, u = g / kNs;
          if (!mbar_wait(bars + 8 * (B_KV_EMPTY + st), (u & 1) ^ 1)) {
            dead = true;
            break;
          }
          const uint32_t full = bars + 8 * (B_KV_FULL + st);
          if (usable(raw0)) {
            const int row = stage_row(raw0, p0, j);
            mbar_arrive_expect_tx(full, kStageBytes);
            const uint32_t dst = sbase + kKvOff + st * kStageBytes;
            for (int c = 0; c < 4; ++c)
              tma_load_2d_hint(dst + c * kChunkBytes, &A.kvmap[r], xlat + 64 * c, row, full, pol);
            tma_load_2d_hint(dst + 4 * kChunkBytes, &A.ropemap[r], xrope, row, full, pol);
          } else {
            if (crank == 0) count_error(A.err);
            mbar_arrive(full);
          }
          raw0 = raw1;
          raw1 = j + 2 < nst ? bt_raw(b, r, p0, j + 2) : -1;
        }
      }
      if (dead) atomicAdd(errp, kStuckMla);
    }
  } else if (warp == 1) {
    // ---------------- Q K^T issuer ----------------
    if (lane == 0) {
      uint32_t g = 0, qv = 0;
      int prev_b = -1;
      bool dead = false;
      const uint64_t qrope_a = sdesc_sw64(sbase + kQRopeOff, 512);
      for (int it = i0; it < i1 && !dead; ++it) {
        const int4 d = plan.item[it];
        const int b = d.x;
        const int nst = (d.w - d.z + kSt - 1) / kSt;
        const bool q_last = it + 1 >= i1 || plan.item[it + 1].x != b;
        if (b != prev_b) {
          if (!mbar_wait(bars + 8 * B_Q_FULL, qv & 1)) {
            dead = true;
            break;
          }
          ++qv;
          prev_b = b;
        }
        for (int j = 0; j < nst; ++j) {
          const uint32_t gs = g + j;
          const uint32_t st = gs % kNs, u = gs / kNs, sb = gs & 1, us = gs >> 1;
          if (!mbar_wait2_cluster(bars + 8 * (B_KV_FULL + st), u & 1, bars + 8 * (B_S_FREE + sb),
                                  (us & 1) ^ 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
          const uint32_t d_s = tmem + kColS + sb * kSt;
          const uint32_t kv = sbase + kKvOff + st * kStageBytes;
          const uint64_t b0 = sdesc_sw128(kv, 0, 1024);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_ts(d_s, tmem + kColQ + c * 32 + kk * 8,
                        b0 + (uint64_t)((c * kChunkBytes + kk * 32) >> 4), kIdescQK,
                        (c | kk) != 0);
          const uint64_t br = sdesc_sw64(kv + 4 * kChunkBytes, 512);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            tc_mma_ss(d_s, qrope_a + (uint64_t)((kk * 32) >> 4), br + (uint64_t)((kk * 32) >> 4),
                      kIdescQK, 1u);
          tc_commit(bars + 8 * (B_S_FULL + sb));
          if (q_last && j == nst - 1) tc_commit(bars + 8 * B_Q_EMPTY);  // last reader of this Q
        }
        if (dead) break;
        if (nst == 0 && q_last) tc_commit(bars + 8 * B_Q_EMPTY);
        g += nst;
      }
      if (dead) atomicAdd(errp, kStuckMla);
    }
  } else if (warp == 2) {
    // ---------------- P V issuer ----------------
    // The whole warp waits; lane 0 issues.  P V of a stage needs this CTA's
    // P rows (P_FULL, the four softmax warps) and the peer's (P_RECV, its bulk
    // copies).  Only when the peer rescaled one of its rows does it also wait
    // for the receivers to apply the rescale here (B_RS_DONE); the receivers
    // and this warp count those stages from the same factors.
    const uint32_t fside = sbase + kSideRecvOff + lane * 8;   // rows lane, lane + 32 (half 0)
    uint32_t g = 0, k = 0, rsc = 0;
    bool dead = false;
    for (int it = i0; it < i1 && !dead; ++it, ++k) {
      const int4 d = plan.item[it];
      const int nst = (d.w - d.z + kSt - 1) / kSt;
      for (int j = 0; j < nst; ++j) {
        const uint32_t gs = g + j, st = gs % kNs, sb = gs & 1, us = gs >> 1;
        if (!cwait2(bars + 8 * (B_P_FULL + sb), us & 1, bars + 8 * (B_P_RECV + sb), us & 1) ||
            (j == 0 && !wwait(bars + 8 * B_O_FREE, (k & 1) ^ 1))) {
          dead = true;
          break;
        }
        float f0, f1;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(f0) : "r"(fside + sb * kSideBytes));
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(f1) : "r"(fside + sb * kSideBytes + 256));
        if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) {
          if (!wwait(bars + 8 * B_RS_DONE, rsc & 1)) {
            dead = true;
            break;
          }
          ++rsc;
        }
        tc_fence_after();
        if (lane == 0) {
          // V = this CTA's four value chunks, the MN-major B operand: 64-column
          // atoms kChunkBytes apart, 8-token groups 1024 B apart; k-step kk
          // starts 16 tokens further.  P (K-major A operand) is P tile sb: two
          // 32-token blocks of 64-byte rows (64-byte swizzle, 8-row groups
          // 512 B apart), so k-step kk reads block kk / 2 at byte 32 (kk % 2).
          const uint32_t v = sbase + kKvOff + st * kStageBytes;
          const uint32_t pt = sbase + kPtOff + sb * kPtBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc_sw128(v + kk * 16 * 128, kChunkBytes, 1024);
            const uint64_t pa = sdesc_sw64(pt + (kk >> 1) * kPtBlock + (kk & 1) * 32, 512);
            tc_mma_ss(tmem + kColO, pa, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bars + 8 * (B_KV_EMPTY + st));
          // P tile sb of both CTAs may be rewritten once both P V have read it
          tc_commit_multicast(bars + 8 * (B_PT_FREE + sb), (uint16_t)3u);
        }
        __syncwarp();
      }
      if (dead) break;
      g += nst;
      if (lane == 0) tc_commit(bars + 8 * B_O_FULL);
      __syncwarp();
    }
    if (dead && lane == 0) atomicAdd(errp, kStuckMla);
  } else {
    // ---------------- row warps: one tensor-memory lane (head) per thread ----------------
    const int q4 = warp & 3;                         // lane quarter = SM sub-partition
    const int head = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const bool own = (uint32_t)(q4 >> 1) == crank;   // my softmax heads
    const bool first_set = warp < kFirstRowWarp + 4;
    const int hp = (q4 & 1) * 32 + lane;             // row among the 64 heads of its owner
    const int role = own ? 0 : (first_set ? 1 : 2);  // softmax, ship, receive

    // Q row `head`: four 64-column latent chunks into tensor memory, the rope
    // half into shared memory; loaded by the softmax and shipper warps (all
    // four lane quarters) once the previous Q's last Q K^T has completed.
    auto load_q = [&](int b, uint32_t qv) -> bool {
      if (qv > 0 && !wwait(bars + 8 * B_Q_EMPTY, (qv - 1) & 1)) return false;
      tc_fence_after();
      const uint4* src = reinterpret_cast<const uint4*>(
          A.q + ((int64_t)b * kHeads + head) * kDk + (int64_t)crank * 256);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint4 x = __ldg(src + c * 8 + t);
          v[4 * t] = x.x;
          v[4 * t + 1] = x.y;
          v[4 * t + 2] = x.z;
          v[4 * t + 3] = x.w;
        }
        tc_st32(tmem + lane_off + kColQ + c * 32, v);
      }
      // rope half: 64-byte row `head` of a 64-byte-swizzled tile
      const uint4* rsrc = reinterpret_cast<const uint4*>(
          A.q + ((int64_t)b * kHeads + head) * kDk + 512 + 32 * (int64_t)crank);
      const uint32_t rrow = sbase + kQRopeOff + head * 64;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 x = __ldg(rsrc + u);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                         rrow + ((u ^ ((head >> 1) & 3)) << 4)),
                     "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_wait_st();
      tc_fence_before();
      warp_arrive(bars + 8 * B_Q_FULL);
      return true;
    };
    // multiply columns [c0, c0 + 32 nc) of row `head` of the O half by f
    // (after the in-flight P V)
    auto rescale_o = [&](float f, int c0, int nc) {
#pragma unroll 1
      for (int cc = 0; cc < nc; ++cc) {
        uint32_t o[32];
        const uint32_t ta = tmem + lane_off + kColO + c0 + cc * 32;
        tc_ld32(ta, o);
        tc_wait_ld(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
        tc_st32(ta, o);
      }
      tc_wait_st();
    };
    // columns [c0, c0 + 32 nc) of O half row `head`, / l -> item partial
    auto write_o = [&](int it, float l, int c0, int nc) {
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      float* dst =
          plan.o + ((int64_t)it * kHeads + head) * (2 * kDvHalf) + crank * kDvHalf + c0;
#pragma unroll 1
      for (int cc = 0; cc < nc; ++cc) {
        uint32_t o[32];
        tc_ld32(tmem + lane_off + kColO + c0 + cc * 32, o);
        tc_wait_ld(o);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
          if (any)
            w = make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                            __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
          *reinterpret_cast<float4*>(dst + cc * 32 + i) = w;
        }
      }
    };

    if (role == 1) {
      // ---------- shipper: partial scores of the peer's heads -> the peer ----------
      // Row hp of a receive slot is split over two 8 KB planes (columns
      // 0..31, 32..63), 128 bytes each, 16-byte units swizzled by hp & 7.
      // The rows are staged in the same layout in this CTA and sent with two
      // 4 KB bulk copies per warp: remote 16-byte stores would queue in the
      // SM's memory-instruction path that the softmax shares.
      const uint32_t srow = sbase + kStgOff + hp * 128;
      const uint32_t half_off = (uint32_t)(q4 & 1) * 4096;
      const uint32_t xs_peer = mapa_shared(sbase + kXsOff + half_off, peer);
      const uint32_t xfull_peer = mapa_shared(bars + 8 * B_X_FULL, peer);
      uint32_t g = 0, qv = 0;
      int prev_b = -1;
      bool dead = false;
      for (int it = i0; it < i1 && !dead; ++it) {
        const int4 d = plan.item[it];
        const int nst = (d.w - d.z + kSt - 1) / kSt;
        if (d.x != prev_b) {
          if (!load_q(d.x, qv)) {
            dead = true;
            break;
          }
          ++qv;
          prev_b = d.x;
        }
        for (int j = 0; j < nst; ++j) {
          const uint32_t gs = g + j, sb = gs & 1, us = gs >> 1;
          if (!wwait(bars + 8 * (B_S_FULL + sb), us & 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
          uint32_t s0[32], s1[32];
          tc_ld32(tmem + lane_off + kColS + sb * kSt, s0);
          tc_ld32(tmem + lane_off + kColS + sb * kSt + 32, s1);
          tc_wait_ld(s0);
          tc_wait_ld(s1);
          tc_fence_before();
          warp_arrive(bars + 8 * (B_S_FREE + sb));
          // the staging buffer and the peer's slot are free once the peer's
          // softmax read stage gs - 1 (which the copy from this buffer filled)
          if (!__all_sync(0xffffffffu,
                          mbar_wait_relaxed_cluster(bars + 8 * B_XS_FREE, (gs & 1) ^ 1))) {
            dead = true;
            break;
          }
          const uint32_t dst = srow;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const uint32_t pu = (uint32_t)((t ^ (hp & 7)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst + pu), "r"(s0[4 * t]),
                         "r"(s0[4 * t + 1]), "r"(s0[4 * t + 2]), "r"(s0[4 * t + 3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst + kXsPlane + pu),
                         "r"(s1[4 * t]), "r"(s1[4 * t + 1]), "r"(s1[4 * t + 2]),
                         "r"(s1[4 * t + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const uint32_t src = sbase + kStgOff + half_off;
            bulk_copy_cluster(xs_peer, src, 4096, xfull_peer);
            bulk_copy_cluster(xs_peer + kXsPlane, src + kXsPlane, 4096, xfull_peer);
          }
        }
        if (dead) break;
        g += nst;
      }
      if (dead && lane == 0) atomicAdd(errp, kStuckMla);
    } else if (role == 2) {
      // ---------- receiver: the peer's P rows for its heads ----------
      const uint32_t side = sbase + kSideRecvOff + hp * 8;
      const uint32_t fother = sbase + kSideRecvOff + (hp ^ 32) * 8;  // the other receiver's rows
      const uint32_t ptfree_peer = mapa_shared(bars + 8 * B_PT_FREE, peer);
      const bool armer = lane == 0 && (q4 & 1) == 0;
      uint32_t g = 0, k = 0;
      bool dead = false;
      for (int it = i0; it < i1 && !dead; ++it, ++k) {
        const int4 d = plan.item[it];
        const int nst = (d.w - d.z + kSt - 1) / kSt;
        float lr = 0.f;
        for (int j = 0; j < nst; ++j) {
          const uint32_t gj = g + j, sb = gj & 1, us = gj >> 1;
          // the peer's P rows of stage gj; and P tile sb's phase for stage gj - 2,
          // observed so that the rescale wait of stage gj + 1 cannot alias
          if (!cwait2(bars + 8 * (B_P_RECV + sb), us & 1, bars + 8 * (B_PT_FREE + sb),
                      (us & 1) ^ 1)) {
            dead = true;
            break;
          }
          // side entries: (f, half-row sum) of half 0 and of half 1, and the
          // other receiver's factors (the P V warp decides on all 64 rows)
          float f, l0, l1, fo;
          asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];"
                       : "=f"(f), "=f"(l0)
                       : "r"(side + sb * kSideBytes));
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(l1) : "r"(side + sb * kSideBytes + kOwn * 8 + 4));
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(fo) : "r"(fother + sb * kSideBytes));
          lr = l0 + l1;   // both halves carry the same factor
          // the tile's next phase (stage gj + 2) expects the peer's bytes again
          if (armer) mbar_arrive_expect_tx_relaxed(bars + 8 * (B_P_RECV + sb), kPMsgBytes);
          // the side entries are read: the peer may refill this slot (its P of
          // stage gj + 2).  The vote orders the remote arrival after the loads.
          {
            const uint32_t vote = __ballot_sync(0xffffffffu, f + l0 + l1 + fo > 0.f);
            if (lane == 0) mbar_arrive_remote_relaxed(ptfree_peer + 8 * sb, __uint_as_float(vote));
          }
          if (__any_sync(0xffffffffu, f != 1.f || fo != 1.f)) {
            // wait for the P V of stage gj - 1 (in both CTAs), rescale, and let
            // the P V of stage gj go
            if (!cwait(bars + 8 * (B_PT_FREE + ((gj - 1) & 1)), ((gj - 1) >> 1) & 1)) {
              dead = true;
              break;
            }
            tc_fence_after();
            rescale_o(f, 0, kDvHalf / 32);
            tc_fence_before();
            warp_arrive(bars + 8 * B_RS_DONE);
          }
        }
        if (dead) break;
        g += nst;
        if (!wwait(bars + 8 * B_O_FULL, k & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        write_o(it, lr, 0, kDvHalf / 32);
        tc_fence_before();
        warp_arrive(bars + 8 * B_O_FREE);
      }
      if (dead && lane == 0) atomicAdd(errp, kStuckMla);
    } else {
      // ---------- softmax of the own heads: one 32-column half of a row per thread ----------
      const int h = first_set ? 0 : 1;               // which half of the 64 columns
      const int qo = q4 & 1;                         // which own quarter
      const int stid = h * 64 + qo * 32 + lane;      // 0..127
      const bool lead = lane == 0;
      const bool armer = lead && h == 0 && qo == 0;
      const uint32_t xrow = sbase + kXsOff + h * kXsPlane + hp * 128;  // my half-row of the slot
      // my row of P block h (64-byte rows, 16-byte units swizzled by (row >> 1) & 3)
      const uint32_t prow = sbase + kPtOff + h * kPtBlock + head * 64;
      const uint32_t pswz = (uint32_t)((head >> 1) & 3);
      const uint32_t side = sbase + kSideOwnOff + (h * kOwn + hp) * 8;
      // half-row maxima: slots [stage parity][half][row]; slot 2 carries the row sums
      const uint32_t mx_mine = sbase + kMxOff + (h * kOwn + hp) * 4;
      const uint32_t mx_other = sbase + kMxOff + ((1 - h) * kOwn + hp) * 4;
      const uint32_t mxbar = bars + 8 * (B_MX + qo);
      const uint32_t xsfree_peer = mapa_shared(bars + 8 * B_XS_FREE, peer);
      const uint32_t precv_peer = mapa_shared(bars + 8 * B_P_RECV, peer);
      // this warp's 32 rows of P block h and its 32 side entries, in the peer
      const uint32_t pt_peer = mapa_shared(sbase + kPtOff + h * kPtBlock + q4 * 2048, peer);
      const uint32_t side_peer = mapa_shared(sbase + kSideRecvOff + (h * kOwn + qo * 32) * 8, peer);
      uint32_t g = 0, k = 0, qv = 0, mxc = 0;
      int prev_b = -1;
      bool dead = false;
      // bf16 P of my half-row relative to the maximum mb, and its sum
      // (the first form for a half-row whose 32 tokens are all valid, the
      // usual case; nv is the same across the warp)
      auto make_p_full = [&](const float (&sc)[32], float mb, uint32_t (&pk)[16]) -> float {
        float ls = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float pa = ex2_ftz(fmaf(sc[2 * e], A.sl2, -mb));
          const float pq = ex2_ftz(fmaf(sc[2 * e + 1], A.sl2, -mb));
          ls += pa + pq;
          pk[e] = pack_bf16(pa, pq);
        }
        return ls;
      };
      auto make_p = [&](const float (&sc)[32], int nv, float mb, uint32_t (&pk)[16]) -> float {
        float ls = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i = 2 * e;
          const float pa = i < nv ? ex2_ftz(fmaf(sc[i], A.sl2, -mb)) : 0.f;
          const float pq = i + 1 < nv ? ex2_ftz(fmaf(sc[i + 1], A.sl2, -mb)) : 0.f;
          ls += pa + pq;
          pk[e] = pack_bf16(pa, pq);
        }
        return ls;
      };
      for (int it = i0; it < i1 && !dead; ++it, ++k) {
        const int4 d = plan.item[it];
        const int b = d.x, r = d.y & 255, p0 = d.z, p1 = d.w;
        const int nst = (p1 - p0 + kSt - 1) / kSt;
        if (b != prev_b) {
          if (h == 0 && !load_q(b, qv)) {
            dead = true;
            break;
          }
          ++qv;
          prev_b = b;
        }
        float m = -INFINITY, lh = 0.f;
        // block-table entries, loaded three stages ahead of use
        int32_t ph[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ph[i] = i < nst ? bt_raw(b, r, p0, i) : -1;
        for (int j = 0; j < nst; ++j) {
          const uint32_t gj = g + j, sb = gj & 1, us = gj >> 1;
          const int32_t phj = ph[0];
          ph[0] = ph[1];
          ph[1] = ph[2];
          ph[2] = ph[3];
          if (j + 4 < nst) ph[3] = bt_raw(b, r, p0, j + 4);
          const int nvalid = usable(phj) ? min(kSt, p1 - (p0 + j * kSt)) : 0;
          const int nv = nvalid - 32 * h;            // valid columns of my half (may be <= 0)
          // full scores of my half of stage gj: this CTA's partial (tensor
          // memory) plus the peer's (receive slot), 32 columns
          if (!cwait2(bars + 8 * (B_S_FULL + sb), us & 1, bars + 8 * B_X_FULL, gj & 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
          float sc[32];
          {
            uint32_t s0[32];
            tc_ld32(tmem + lane_off + kColS + sb * kSt + 32 * h, s0);
            tc_wait_ld(s0);
            tc_fence_before();
            warp_arrive(bars + 8 * (B_S_FREE + sb));
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const uint32_t pu = (uint32_t)((t ^ (hp & 7)) << 4);
              uint32_t a0, a1, a2, a3;
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                           : "r"(xrow + pu));
              sc[4 * t + 0] = __uint_as_float(s0[4 * t + 0]) + __uint_as_float(a0);
              sc[4 * t + 1] = __uint_as_float(s0[4 * t + 1]) + __uint_as_float(a1);
              sc[4 * t + 2] = __uint_as_float(s0[4 * t + 2]) + __uint_as_float(a2);
              sc[4 * t + 3] = __uint_as_float(s0[4 * t + 3]) + __uint_as_float(a3);
            }
          }
          // the slot's next phase (stage gj + 1) expects the peer's 16 KB again
          if (armer) mbar_arrive_expect_tx_relaxed(bars + 8 * B_X_FULL, kXsBytes);
          // half-row maximum (raw scores; the scale is positive)
          float t16[16];
          if (nv >= 32) {
#pragma unroll
            for (int i = 0; i < 16; ++i) t16[i] = fmaxf(sc[2 * i], sc[2 * i + 1]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a = 2 * i < nv ? sc[2 * i] : -INFINITY;
              const float c = 2 * i + 1 < nv ? sc[2 * i + 1] : -INFINITY;
              t16[i] = fmaxf(a, c);
            }
          }
#pragma unroll
          for (int w = 8; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) t16[i] = fmaxf(t16[i], t16[i + w]);
          // every lane's slot reads are complete once the vote has all maxima:
          // the vote result orders the remote arrival after them
          {
            const uint32_t vote = __ballot_sync(0xffffffffu, t16[0] > 0.f);
            if (lead) mbar_arrive_remote_relaxed(xsfree_peer, __uint_as_float(vote));
          }
          // the row maximum: exchange the half-row maxima with the other half
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(mx_mine + sb * (2 * kOwn * 4)),
                       "f"(t16[0])
                       : "memory");
          warp_arrive(mxbar);
          // also P tile sb: free once the P V of stage gj - 2 completed in both CTAs
          if (!cwait2(mxbar, mxc & 1, bars + 8 * (B_PT_FREE + sb), (us & 1) ^ 1)) {
            dead = true;
            break;
          }
          ++mxc;
          float mo;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(mo) : "r"(mx_other + sb * (2 * kOwn * 4)));
          const float mx = fmaxf(t16[0], mo) * A.sl2;
          const bool grow = mx > m + kRescaleThreshold;
          const bool need = grow && j > 0 && m > -INFINITY;  // O already holds this row's sums
          float f = 1.f;
          if (__any_sync(0xffffffffu, need)) {
            // wait for the P V of stage gj - 1 (in both CTAs), then rescale my
            // half of the rows that need it
            if (!cwait(bars + 8 * (B_PT_FREE + ((gj - 1) & 1)), ((gj - 1) >> 1) & 1)) {
              dead = true;
              break;
            }
            tc_fence_after();
            if (need) f = exp2f(m - mx);
            rescale_o(f, h * (kDvHalf / 2), kDvHalf / 64);
          }
          if (grow) m = mx;
          uint32_t pk[16];
          const float mb = (m == -INFINITY) ? 0.f : m;
          const float ls = nv >= 32 ? make_p_full(sc, mb, pk) : make_p(sc, nv, mb, pk);
          lh = lh * f + ls;
          const uint32_t pr = prow + sb * kPtBytes;
#pragma unroll
          for (int t = 0; t < 4; ++t)
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(pr + ((t ^ pswz) << 4)),
                         "r"(pk[4 * t]), "r"(pk[4 * t + 1]), "r"(pk[4 * t + 2]), "r"(pk[4 * t + 3])
                         : "memory");
          asm volatile("st.shared.v2.f32 [%0], {%1,%2};" ::"r"(side + sb * kSideBytes), "f"(f),
                       "f"(lh)
                       : "memory");
          if (nvalid < kSt) {
            // rows past the end may hold anything: zero this CTA's V columns so 0 * x stays 0
            const uint32_t st = gj % kNs;
            if (!wwait(bars + 8 * (B_KV_FULL + st), (gj / kNs) & 1)) {
              dead = true;
              break;
            }
            const uint32_t v = sbase + kKvOff + st * kStageBytes;
            const int total = (kSt - nvalid) * 4 * 8;
            for (int i = stid; i < total; i += 2 * kOwn) {
              const int rr = nvalid + (i >> 5), ch = (i >> 3) & 3, part = i & 7;
              asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                               v + ch * kChunkBytes + rr * 128 + part * 16),
                           "r"(0u)
                           : "memory");
            }
          }
          fence_proxy_async_smem();   // P, the side values and zeroed V rows are read asynchronously
          __syncwarp();
          if (lead) {
            // my 32 rows of P block h and my side entries -> the same places in the peer
            bulk_copy_cluster(pt_peer + sb * kPtBytes,
                              sbase + kPtOff + sb * kPtBytes + h * kPtBlock + q4 * 2048, 2048,
                              precv_peer + 8 * sb);
            bulk_copy_cluster(side_peer + sb * kSideBytes,
                              sbase + kSideOwnOff + sb * kSideBytes + (h * kOwn + qo * 32) * 8, 256,
                              precv_peer + 8 * sb);
            mbar_arrive(bars + 8 * (B_P_FULL + sb));
          }
        }
        if (dead) break;
        g += nst;
        // the row sum: exchange the half-row sums through slot 2
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(mx_mine + 2 * (2 * kOwn * 4)), "f"(lh)
                     : "memory");
        warp_arrive(mxbar);
        // epilogue: my half of O / l -> item partial, LSE in natural log
        if (!wwait(mxbar, mxc & 1) || !wwait(bars + 8 * B_O_FULL, k & 1)) {
          dead = true;
          break;
        }
        ++mxc;
        float lo;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(lo) : "r"(mx_other + 2 * (2 * kOwn * 4)));
        const float l = h == 0 ? lh + lo : lo + lh;  // (half 0) + (half 1), as the peer adds them
        tc_fence_after();
        write_o(it, l, h * (kDvHalf / 2), kDvHalf / 64);
        if (h == 0)
          plan.lse[(int64_t)it * kHeads + head] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        tc_fence_before();
        warp_arrive(bars + 8 * B_O_FREE);
      }
      if (dead && lane == 0) atomicAdd(errp, kStuckMla);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kTmemCols);
  }
  __syncwarp();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
}

namespace {

int g_clusters[64] = {0};
bool g_attr_done[64] = {false};

// 2-D bf16 map over the latent rows with the given box width and swizzle.
bool encode_latent(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_cols,
                   CUtensorMapSwizzle swz) {
  auto enc = tensor_map_encoder();
  if (!enc || ((uintptr_t)base & 15) || rows == 0 || rows > (1ull << 32)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDk, rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDk * 2};
  cuuint32_t box[2] = {box_cols, (cuuint32_t)kSt};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

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

int mla_tc_clusters() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return num_sms() / 2 > 0 ? num_sms() / 2 : 1;
  if (!g_attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem);
    if (e != cudaSuccess) {
      launch_status_report(e);
      return -1;
    }
    g_attr_done[dev] = true;
  }
  if (g_clusters[dev] == 0) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(kMlaThreads, 1, 1);
    cfg.dynamicSmemBytes = kMlaSmem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mla_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    if (n > kMaxParts) n = kMaxParts;
    g_clusters[dev] = n > 0 ? n : 1;
  }
  return g_clusters[dev];
}

int launch_mla_tc(const dcp_layout_t& layout, const void* q, int B, int Hq, float scale,
                  const dcp_paged_kv_t& kv, const Plan& plan, int clusters, int32_t* err,
                  cudaStream_t s) {
  (void)Hq;
  if ((uintptr_t)q & 15) return DCP_EUNSUPPORTED;
  if (clusters < 1 || clusters > kMaxParts) return DCP_EINVAL;
  MlaTcArgs A;
  memset(&A, 0, sizeof(A));
  const uint64_t rows = (uint64_t)kv.num_blocks * layout.block_size;
  for (int r = 0; r < layout.dcp_size; ++r)
    if (!encode_latent(&A.kvmap[r], kv.k.ptr[r], rows > 0 ? rows : 1, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_latent(&A.ropemap[r], kv.k.ptr[r], rows > 0 ? rows : 1, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B))
      return DCP_ECUDA;
  A.q = static_cast<const uint16_t*>(q);
  A.B = B;
  A.bs = layout.block_size;
  A.dcp = layout.dcp_size;
  A.sl2 = scale * kLog2e;
  A.bt = kv.block_table;
  A.max_vb = kv.max_vblocks;
  A.bt_rank_stride = kv.bt_rank_stride;
  A.num_blocks = kv.num_blocks;
  A.err = err;
  mla_tc_kernel<<<2 * clusters, kMlaThreads, kMlaSmem, s>>>(A, plan);
  return launch_status();
}

}  // namespace dcp
