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
//  * a cluster of two CTAs per item.  The fp32 output tile 128 x 512 would
//    fill all of tensor memory, so CTA c keeps value columns [256c, 256c+256).
//    The 576-wide reduction of Q K^T is split the same way: CTA 0 reduces
//    over latent columns 0..255, CTA 1 over 256..575 (latent 256..511 plus
//    the 64 rope columns).  Each CTA therefore holds only its part of Q
//    (64 or 80 KB) and of every KV stage (16 or 20 KB of a 32-token stage),
//    which leaves room for five KV stages, and no MMA work is duplicated;
//  * the two fp32 partial score tiles (128 x 32) are exchanged through
//    distributed shared memory, one stage ahead of the softmax, and added
//    (IEEE addition commutes, so both CTAs hold bit-identical scores and take
//    identical softmax decisions);
//  * warp 0 issues TMA (Q once per request, KV stages through a 5-deep
//    ring), warp 1 issues tcgen05.mma (Q K^T runs three stages ahead of
//    P V), warps 2-5 run the online softmax (one head row per thread; scores
//    read from tensor memory, P written back to tensor memory as the A
//    operand of P V) and the epilogue.  The softmax threads push their
//    partial scores into the peer's shared memory with st.async, which
//    completes transaction bytes on the peer's mbarrier without a fence on
//    the sender; warp 6 arms this CTA's receive barrier for every stage and
//    warp 7 tells the peer when a receive slot may be reused;
//  * the output is rescaled only when the running maximum grows by more
//    than 8 (log2 units), so P stays <= 256 and the rare rescale waits for
//    the in-flight P V.
// Every mbarrier wait is bounded; a timed-out wait adds 1<<20 to the error
// counter and that role stops waiting, so the kernel always terminates.
#include <stdlib.h>
#include <string.h>

#include <type_traits>

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
constexpr int kSt = 32;                              // tokens per KV stage
constexpr int kNs = 5;                               // KV stages in flight
constexpr int kMaxCh = 5;                            // 64-column chunks per CTA (CTA 1)
constexpr int kQChunkBytes = kHeads * 128;           // 16 KB
constexpr int kKvChunkBytes = kSt * 128;             // 4 KB
constexpr int kKvStageBytes = kMaxCh * kKvChunkBytes;  // 20 KB
constexpr int kXSlotBytes = kHeads * kSt * 4;        // 16 KB of fp32 partial scores
constexpr int kKvOff = kMaxCh * kQChunkBytes;        // 80 KB
constexpr int kXOff = kKvOff + kNs * kKvStageBytes;  // 180 KB
constexpr int kBarOff = kXOff + 2 * kXSlotBytes;     // 212 KB
constexpr int kNumBars = 32;
constexpr int kMlaSmem = 1024 + kBarOff + kNumBars * 8 + 16;
constexpr int kMlaThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kNsb = 4;                            // score buffers in tensor memory
constexpr int kLookahead = 3;                      // Q K^T issued this many stages ahead of P V
constexpr uint32_t kColO = 0, kColS = 256, kColP = 256 + kNsb * kSt;
constexpr float kRescaleThreshold = 8.f;
constexpr int kStuckMla = 1 << 20;

// barrier slots
enum : int {
  B_KV_FULL = 0,    // +stage (kNs)
  B_KV_EMPTY = 5,   // +stage (kNs)
  B_S_FULL = 10,    // +score buffer (kNsb)
  B_S_FREE = 14,    // +score buffer (kNsb)
  B_P_FULL = 18,    // +buffer
  B_PV_DONE = 20,   // +buffer
  B_X_FULL = 22,    // +slot: the peer's partial scores landed in my slot
  B_X_FREE = 24,    // +slot: the peer consumed what I wrote into its slot
  B_Q_FULL = 26,
  B_Q_EMPTY = 27,
  B_O_FULL = 28,
  B_O_FREE = 29,
  B_IB_DONE = 30   // +slot: my softmax threads finished reading the peer's scores
};

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kSt, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kDvHalf, false, true);

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMlaThreads, 1)
mla_tc_kernel(const __grid_constant__ MlaTcArgs A, Plan plan) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();          // 0 or 1: which half this CTA owns
  const uint32_t peer = crank ^ 1u;
  const int nch = crank == 0 ? 4 : 5;                // K^T chunks reduced here
  const int ch0 = crank == 0 ? 0 : 4;                // first global 64-column chunk
  const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int n_items = plan.hdr[0];
  int32_t* errp = A.err ? A.err : plan.hdr + 3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if ((i >= B_S_FREE && i < B_S_FREE + kNsb) || i == B_P_FULL || i == B_P_FULL + 1 ||
          i == B_O_FREE || i >= B_IB_DONE)
        cnt = 128;                                  // every softmax thread arrives
      mbar_init(bars + 8 * i, cnt);
    }
    fence_mbar_init();
    prefetch_tmap(&A.qmap);
    for (int r = 0; r < A.dcp; ++r) prefetch_tmap(&A.kvmap[r]);
  }
  if (warp == 1) {
    tc_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // block-table entry of stage j of an item (-1 beyond the table)
  auto bt_phys = [&](int b, int r, int p0, int j) -> int64_t {
    const int vb = (p0 + j * kSt) / A.bs;
    return vb < A.max_vb ? (int64_t)__ldg(A.bt + r * A.bt_rank_stride + (int64_t)b * A.max_vb + vb)
                         : (int64_t)-1;
  };
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
    for (int it = cl; it < n_items && !dead; it += ncl, ++k) {
      const int4 d = plan.item[it];
      const int b = d.x, r = d.y & 255, p0 = d.z, p1 = d.w;
      const int nst = (p1 - p0 + kSt - 1) / kSt;
      if (!mbar_wait(bars + 8 * B_Q_EMPTY, (k & 1) ^ 1)) {
        dead = true;
        break;
      }
      if (b != prev_b) {
        mbar_arrive_expect_tx(bars + 8 * B_Q_FULL, nch * kQChunkBytes);
        for (int c = 0; c < nch; ++c)
          tma_load_2d(sbase + c * kQChunkBytes, &A.qmap, 64 * (ch0 + c), b * kHeads,
                      bars + 8 * B_Q_FULL);
        prev_b = b;
      } else {
        mbar_arrive(bars + 8 * B_Q_FULL);
      }
      for (int j = 0; j < nst; ++j, ++g) {
        const uint32_t st = g % kNs, u = g / kNs;
        if (!mbar_wait(bars + 8 * (B_KV_EMPTY + st), (u & 1) ^ 1)) {
          dead = true;
          break;
        }
        const uint32_t full = bars + 8 * (B_KV_FULL + st);
        int row;
        if (stage_row(b, r, p0, j, row)) {
          mbar_arrive_expect_tx(full, nch * kKvChunkBytes);
          const uint32_t dst = sbase + kKvOff + st * kKvStageBytes;
          for (int c = 0; c < nch; ++c)
            tma_load_2d(dst + c * kKvChunkBytes, &A.kvmap[r], 64 * (ch0 + c), row, full);
        } else {
          if (crank == 0) count_error(A.err);
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
    auto qk_issue = [&](auto nch_c, uint32_t d_s, uint32_t kv) {
      constexpr int NCH = decltype(nch_c)::value;
      const uint64_t a0 = sdesc_sw128(sbase, 0, 1024);
      const uint64_t b0 = sdesc_sw128(kv, 0, 1024);
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_ss(d_s, a0 + (uint64_t)((c * kQChunkBytes + kk * 32) >> 4),
                    b0 + (uint64_t)((c * kKvChunkBytes + kk * 32) >> 4), kIdescQK, (c | kk) != 0);
    };
    auto qk = [&](uint32_t gs) -> bool {
      const uint32_t st = gs % kNs, u = gs / kNs, sb = gs % kNsb, us = gs / kNsb;
      if (!mbar_wait(bars + 8 * (B_KV_FULL + st), u & 1)) return false;
      if (!mbar_wait(bars + 8 * (B_S_FREE + sb), (us & 1) ^ 1)) return false;
      tc_fence_after();
      const uint32_t d_s = tmem + kColS + sb * kSt;
      const uint32_t kv = sbase + kKvOff + st * kKvStageBytes;
      if (nch == 4)
        qk_issue(std::integral_constant<int, 4>{}, d_s, kv);
      else
        qk_issue(std::integral_constant<int, 5>{}, d_s, kv);
      tc_commit(bars + 8 * (B_S_FULL + sb));
      return true;
    };
    auto pv = [&](uint32_t gs, bool first) -> bool {
      const uint32_t st = gs % kNs, pb = gs & 1, up = gs >> 1;
      if (!mbar_wait(bars + 8 * (B_P_FULL + pb), up & 1)) return false;
      if (first && !mbar_wait(bars + 8 * B_O_FREE, (k & 1) ^ 1)) return false;
      tc_fence_after();
      // V = this CTA's four value chunks, the MN-major B operand: 64-column
      // atoms kKvChunkBytes apart, 8-token groups 1024 B apart; the second
      // k-step starts 16 tokens in.
      const uint32_t v = sbase + kKvOff + st * kKvStageBytes;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint64_t bd = sdesc_sw128(v + kk * 16 * 128, kKvChunkBytes, 1024);
        tc_mma_ts(d_o, tmem + kColP + pb * 16 + kk * 8, bd, kIdescPV, (!first || kk) ? 1u : 0u);
      }
      tc_commit(bars + 8 * (B_KV_EMPTY + st));
      tc_commit(bars + 8 * (B_PV_DONE + pb));
      return true;
    };
    for (int it = cl; it < n_items && !dead; it += ncl, ++k) {
      const int4 d = plan.item[it];
      const int nst = (d.w - d.z + kSt - 1) / kSt;
      if (!mbar_wait(bars + 8 * B_Q_FULL, k & 1)) {
        dead = true;
        break;
      }
      tc_fence_after();
      for (int j = 0; j < kLookahead && j < nst; ++j)
        if (!qk(g + j)) {
          dead = true;
          break;
        }
      for (int j = 0; j < nst && !dead; ++j) {
        if (!pv(g + j, j == 0)) {
          dead = true;
          break;
        }
        if (j + kLookahead < nst && !qk(g + j + kLookahead)) {
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
  } else if (warp >= 6) {
    // ---------------- exchange helpers ----------------
    // warp 6: arm X_FULL of each stage with the 16 KB the peer will st.async
    //         into this CTA (after the slot's previous phase completed)
    // warp 7: I consumed the peer's scores -> arrive on the peer's X_FREE
    if (lane == 0) {
      const uint32_t free_remote = mapa_shared(bars + 8 * B_X_FREE, peer);
      uint32_t g = 0;
      bool dead = false;
      for (int it = cl; it < n_items && !dead; it += ncl) {
        const int4 d = plan.item[it];
        const int nst = (d.w - d.z + kSt - 1) / kSt;
        for (int j = 0; j < nst; ++j, ++g) {
          const uint32_t xs = g & 1, ux = g >> 1;
          if (warp == 6) {
            if (ux > 0 && !mbar_wait(bars + 8 * (B_X_FULL + xs), (ux - 1) & 1)) {
              dead = true;
              break;
            }
            mbar_arrive_expect_tx(bars + 8 * (B_X_FULL + xs), kXSlotBytes);
          } else {
            if (!mbar_wait(bars + 8 * (B_IB_DONE + xs), ux & 1)) {
              dead = true;
              break;
            }
            mbar_arrive_remote(free_remote + 8 * xs);
          }
        }
      }
      if (dead) atomicAdd(errp, kStuckMla);
    }
  } else if (warp >= 2) {
    // ---------------- softmax + epilogue (one head row per thread) ----------------
    const int q4 = warp & 3;                 // tensor-memory lane quarter of this warp
    const int head = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int tid = threadIdx.x - 64;        // 0..127
    const uint32_t xrow = sbase + kXOff + head * 128;      // my row of my exchange slots
    const uint32_t xrow_peer = mapa_shared(xrow, peer);    // my row of the peer's slots
    const uint32_t xfull_peer = mapa_shared(bars + 8 * B_X_FULL, peer);
    uint32_t g = 0, k = 0;
    bool dead = false;
    // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform
    auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par));
    };
    auto wwait_cl = [&](uint32_t bar, uint32_t par) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_cluster(bar, par));
    };
    // read this CTA's partial scores of stage gs and ship them to the peer
    auto send = [&](uint32_t gs, uint32_t (&mine)[32]) -> bool {
      const uint32_t sb = gs % kNsb, us = gs / kNsb, xs = gs & 1, ux = gs >> 1;
      if (!wwait(bars + 8 * (B_S_FULL + sb), us & 1)) return false;
      tc_fence_after();
      tc_ld32(tmem + lane_off + kColS + sb * kSt, mine);
      tc_wait_ld(mine);
      tc_fence_before();
      mbar_arrive(bars + 8 * (B_S_FREE + sb));
      // the peer must have consumed what I put in its slot two stages ago
      if (!wwait_cl(bars + 8 * (B_X_FREE + xs), (ux & 1) ^ 1)) return false;
      const uint32_t dst = xrow_peer + xs * kXSlotBytes;
      const uint32_t bar = xfull_peer + 8 * xs;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        st_async_v4(dst + ((i ^ (head & 7)) << 4), mine[4 * i], mine[4 * i + 1], mine[4 * i + 2],
                    mine[4 * i + 3], bar);
      return true;
    };
    // add the peer's partial scores of stage gs to mine
    auto recv = [&](uint32_t gs, const uint32_t (&mine)[32], float (&sc)[32]) -> bool {
      const uint32_t xs = gs & 1, ux = gs >> 1;
      if (!wwait_cl(bars + 8 * (B_X_FULL + xs), ux & 1)) return false;
      const uint32_t src = xrow + xs * kXSlotBytes;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t a, bq, c, d;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(a), "=r"(bq), "=r"(c), "=r"(d)
                     : "r"(src + ((i ^ (head & 7)) << 4)));
        sc[4 * i + 0] = __uint_as_float(mine[4 * i + 0]) + __uint_as_float(a);
        sc[4 * i + 1] = __uint_as_float(mine[4 * i + 1]) + __uint_as_float(bq);
        sc[4 * i + 2] = __uint_as_float(mine[4 * i + 2]) + __uint_as_float(c);
        sc[4 * i + 3] = __uint_as_float(mine[4 * i + 3]) + __uint_as_float(d);
      }
      mbar_arrive(bars + 8 * (B_IB_DONE + xs));  // warp 7 frees the slot on the peer
      return true;
    };
    for (int it = cl; it < n_items && !dead; it += ncl, ++k) {
      const int4 d = plan.item[it];
      const int b = d.x, r = d.y & 255, p0 = d.z, p1 = d.w;
      const int nst = (p1 - p0 + kSt - 1) / kSt;
      float m = -INFINITY, l = 0.f;
      // block-table entries of the current and next stage, loaded ahead of use
      int64_t ph_cur = bt_phys(b, r, p0, 0);
      int64_t ph_next = nst > 1 ? bt_phys(b, r, p0, 1) : 0;
      uint32_t cur[32];
      if (!send(g, cur)) {
        dead = true;
        break;
      }
      for (int j = 0; j < nst; ++j) {
        const uint32_t gj = g + j, pb = gj & 1, up = gj >> 1;
        uint32_t nxt[32];
        if (j + 1 < nst && !send(gj + 1, nxt)) {
          dead = true;
          break;
        }
        float sc[32];
        if (!recv(gj, cur, sc)) {
          dead = true;
          break;
        }
        const int nvalid = (ph_cur >= 0 && ph_cur < A.num_blocks) ? min(kSt, p1 - (p0 + j * kSt)) : 0;
        ph_cur = ph_next;
        if (j + 2 < nst) ph_next = bt_phys(b, r, p0, j + 2);  // consumed two stages later
        float x[32];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = i < nvalid ? sc[i] * A.sl2 : -INFINITY;
          mx = fmaxf(mx, x[i]);
        }
        const bool grow = mx > m + kRescaleThreshold;
        const bool need = grow && j > 0 && l > 0.f;  // O already holds this row's sums
        if (__any_sync(0xffffffffu, need)) {
          // wait for the in-flight P V, then rescale the rows that need it
          const uint32_t gp = gj - 1;
          if (!wwait(bars + 8 * (B_PV_DONE + (gp & 1)), (gp >> 1) & 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
          const float f = need ? exp2f(m - mx) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < kDvHalf / 32; ++cc) {
            uint32_t o[32];
            tc_ld32(tmem + lane_off + kColO + cc * 32, o);
            tc_wait_ld(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tc_st32(tmem + lane_off + kColO + cc * 32, o);
          }
          tc_wait_st();
          l *= f;
        }
        if (grow) m = mx;
        const float mb = (m == -INFINITY) ? 0.f : m;
        uint32_t pk[16];
        float ls = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float pa = ex2_ftz(x[2 * i] - mb), pq = ex2_ftz(x[2 * i + 1] - mb);
          ls += pa + pq;
          pk[i] = pack_bf16(pa, pq);
        }
        l += ls;
        // P buffer pb is free once the P V of two stages ago completed
        if (!wwait(bars + 8 * (B_PV_DONE + pb), (up & 1) ^ 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        tc_st16(tmem + lane_off + kColP + pb * 16, pk);
        tc_wait_st();
        if (nvalid < kSt) {
          // rows past the end may hold anything: zero this CTA's V columns so 0 * x stays 0
          const uint32_t v = sbase + kKvOff + (gj % kNs) * kKvStageBytes;
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
        mbar_arrive(bars + 8 * (B_P_FULL + pb));
#pragma unroll
        for (int i = 0; i < 32; ++i) cur[i] = nxt[i];
      }
      if (dead) break;
      g += nst;
      // epilogue: O / l -> item partial, LSE in natural log
      if (!wwait(bars + 8 * B_O_FULL, k & 1)) {
        dead = true;
        break;
      }
      tc_fence_after();
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      float* dst = plan.o + ((int64_t)it * kHeads + head) * (2 * kDvHalf) + crank * kDvHalf;
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
      if (crank == 0)
        plan.lse[(int64_t)it * kHeads + head] = any ? (m + log2f(l)) * kLn2 : -INFINITY;
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
  __syncwarp();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
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
  static int max_clusters[64] = {0};
  if (dev >= 0 && dev < 64 && max_clusters[dev] == 0) {
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
    max_clusters[dev] = n;
  }
  const int clusters = (dev >= 0 && dev < 64) ? max_clusters[dev] : num_sms() / 2;
  mla_tc_kernel<<<2 * (clusters > 0 ? clusters : 1), kMlaThreads, kMlaSmem, s>>>(A, plan);
  return launch_status();
}

}  // namespace dcp
