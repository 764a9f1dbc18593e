// Tensor-core SFA decode partials: per (request, rank), sparse attention of
// all query heads over the selected tokens that rank owns, MLA-shaped latent
// rows (576 bf16: key = whole row, value = first 512 entries).
//
// Page "Decode Context Parallel (DCP)", section "GLM-5.2 SFA DCP replicated
// indexer": the global top-k indices from the replicated indexer are
// remapped to local KV indices before SFA runs; each rank attends only the
// selected tokens it stores, and the per-rank results are merged by LSE
// (with the sink applied once, page "DeepSeek V4.1 context parallelism",
// section "Decode computation").
//
// One CTA per (rank, request, 64 query heads).  The CTA first builds the
// list of its selected slots in top-k order (remapping global indices itself
// in the fused call), then streams 16-token tiles of the gathered latent
// rows into a four-deep ring with cp.async (16-byte pieces; rows padded to
// 1168 bytes so ldmatrix is bank-conflict free without a swizzle).  Eight
// warps = four groups of 16 heads x two halves: the two
// warps of a group split the 576-wide Q.K^T reduction (18 k-steps each, two
// accumulator chains), add their partial scores through shared memory (IEEE
// addition commutes, so both hold identical scores and take identical
// softmax decisions), then each computes P.V for its half of the 512 value
// columns on mma.sync (bf16 in, fp32 accumulate).
#include "dcp_generic.cuh"
#include "dcp_ptx.cuh"
#include "dcp_sfa_mma.cuh"

namespace dcp {

constexpr int kSfaCompute = 8;                       // compute warps
constexpr int kSfaThreads = kSfaCompute * 32;
constexpr int kSfaHeadsPerCta = 64;                  // 4 groups of 16
constexpr int kRow = 576;                            // latent row (bf16)
constexpr int kRowBytes = kRow * 2;                  // 1152
constexpr int kPitch = kRowBytes + 16;               // padded smem row
constexpr int kTileTok = 16;
constexpr int kNbuf = 4;
constexpr int kQOff = 0;
constexpr int kRingOff = kSfaHeadsPerCta * kPitch;                // 74752
constexpr int kTileBytes = kTileTok * kPitch;                     // 18688
constexpr int kXOff = kRingOff + kNbuf * kTileBytes;              // 112128
constexpr int kXBytes = kSfaCompute * 32 * 8 * 4;                 // 8192
constexpr int kSelOff = kXOff + kXBytes;
constexpr int kMaxSel = 4096;                                     // selected tokens per (b, r)
constexpr int kBarOffS = kSelOff + kMaxSel * 4;
constexpr int kSfaSmem = kBarOffS + 16;

// Owner rank and in-block offset of global token x (< 2^31): the layout
// formulas in 32-bit arithmetic.
__device__ __forceinline__ void place_token32(int x, const Layout& L, int& rank, int& vb,
                                              int& loc) {
  const int vbs = L.bs * L.dcp;
  vb = x / vbs;
  const int off = x - vb * vbs;
  const int lbi = off / L.I;
  rank = lbi % L.dcp;
  loc = (lbi / L.dcp) * L.I + off % L.I;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void st_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
}

__global__ void __launch_bounds__(kSfaThreads, 1)
sfa_mma_kernel(SfaMmaArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  const uint32_t sbase = smem_u32(smem);
  float* xs = reinterpret_cast<float*>(smem + kXOff);
  int32_t* sel = reinterpret_cast<int32_t*>(smem + kSelOff);
  int32_t* s_cnt = reinterpret_cast<int32_t*>(smem + kBarOffS);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x / (A.B * A.hblocks);
  const int rem = blockIdx.x % (A.B * A.hblocks);
  const int b = rem / A.hblocks, h0 = (rem % A.hblocks) * kSfaHeadsPerCta;
  const int nh = min(kSfaHeadsPerCta, A.Hq - h0);
  const __nv_bfloat16* pool = (const __nv_bfloat16*)A.pool.ptr[r];
  const int64_t num_slots = A.num_blocks * A.bs;
  int32_t* errp = A.err;

  // Q of this CTA's heads: 16 threads per row, 16-byte pieces (rows beyond Hq are zero)
  for (int row = tid >> 4; row < kSfaHeadsPerCta; row += kSfaThreads / 16) {
    const uint32_t dst = sbase + kQOff + row * kPitch;
    const __nv_bfloat16* src = A.q + ((int64_t)b * A.Hq + h0 + row) * kRow;
    for (int pc = tid & 15; pc < kRowBytes / 16; pc += 16) {
      if (row < nh)
        cp_async16(dst + pc * 16, src + pc * 8);
      else
        st_zero16(dst + pc * 16);
    }
  }
  cp_async_commit();

  // ---- this rank's selected slots, in top-k order ----
  // Each thread owns a contiguous run of up to kPer entries; every global
  // load of the run is issued before any result is used.
  {
    constexpr int kPer = 16;
    static_assert(kPer * kSfaThreads >= kMaxSel, "selection runs must cover kMaxSel");
    const int per = (A.K + kSfaThreads - 1) / kSfaThreads;
    const int k0 = min(A.K, tid * per), k1 = min(A.K, k0 + per);
    int64_t slot[kPer];
    uint32_t own = 0;
    if (A.topk == nullptr) {
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
    } else {
      const int len = __ldg(A.seq_lens + b);
      int gi[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int k = k0 + i;
        gi[i] = k < k1 ? __ldg(A.topk + (int64_t)b * A.K + k) : -1;
      }
      int loc[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        int rk, vb;
        loc[i] = 0;
        slot[i] = -1;
        if (gi[i] >= 0 && gi[i] < len) {
          place_token32(gi[i], A.L, rk, vb, loc[i]);
          if (rk == r) {
            own |= 1u << i;
            slot[i] = vb < A.max_vb ? (int64_t)__ldg(A.bt + r * A.bt_rank_stride +
                                                     (int64_t)b * A.max_vb + vb)
                                    : (int64_t)-1;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (own >> i & 1)
          slot[i] = (slot[i] >= 0 && slot[i] < A.num_blocks) ? slot[i] * A.bs + loc[i] : -2;
    }
    const int mine = __popc(own);
    __shared__ int wsum[kSfaCompute + 1];
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
    if (tid == kSfaThreads - 1) *s_cnt = base + mine;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (own >> i & 1) {
        int64_t sl = slot[i];
        if (sl < 0 || sl >= num_slots) {
          if (h0 == 0) count_error(errp);
          sl = -1;  // unusable slot: attended as a masked token
        }
        if (base < kMaxSel) sel[base] = (int32_t)sl;
        ++base;
      }
    }
  }
  __syncthreads();
  const int n_sel = min(*s_cnt, kMaxSel);
  const int ntiles = (n_sel + kTileTok - 1) / kTileTok;

  // tile j -> ring buffer j % kNbuf: 16 threads per row, 16-byte pieces;
  // rows past the end or with an unusable slot are zero (their scores are
  // masked and their values add 0).  Always commits one group.
  auto load_tile = [&](int j) {
    if (j < ntiles) {
      const uint32_t dst0 = sbase + kRingOff + (j % kNbuf) * kTileBytes;
      const int row = tid >> 4, t = j * kTileTok + row;
      const int sl = t < n_sel ? sel[t] : -1;
      const uint32_t dst = dst0 + row * kPitch;
      const __nv_bfloat16* src = pool + (int64_t)(sl < 0 ? 0 : sl) * kRow;
      for (int pc = tid & 15; pc < kRowBytes / 16; pc += 16) {
        if (sl >= 0)
          cp_async16(dst + pc * 16, src + pc * 8);
        else
          st_zero16(dst + pc * 16);
      }
    }
    cp_async_commit();
  };
  for (int j = 0; j < kNbuf - 1; ++j) load_tile(j);

  // ---------------- compute warps ----------------
  const int hg = warp >> 1, part = warp & 1;
  const int r0 = lane >> 2, cq = 2 * (lane & 3), mi = lane >> 3;
  const int arow = hg * 16 + (lane & 7) + 8 * (mi & 1);  // Q row this lane addresses (ldmatrix)
  const int krow = (mi >> 1) * 8 + (lane & 7);            // token row for K fragments
  const int vrow = (mi & 1) * 8 + (lane & 7);             // token row for V fragments
  float* xmine = xs + ((hg * 2 + part) * 32 + lane) * 8;
  const float* xpeer = xs + ((hg * 2 + (part ^ 1)) * 32 + lane) * 8;
  const uint32_t qrow = sbase + kQOff + arow * kPitch;
  float o[32][4];
#pragma unroll
  for (int n = 0; n < 32; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int j = 0; j < ntiles; ++j) {
    cp_async_wait<kNbuf - 2>();  // Q and tile j have landed (one group per tile)
    __syncthreads();
    const uint32_t tile = sbase + kRingOff + (j % kNbuf) * kTileBytes;
    const int t0 = j * kTileTok, nvalid = min(kTileTok, n_sel - t0);
    // partial S (16 heads x 16 tokens) over this warp's 18 k-steps: two chains
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < 18; ++kk) {
      const int ks = part * 18 + kk;
      uint32_t b0, b1, b2, b3;
      uint32_t a[4];
      ldsm_x4(qrow + (2 * ks + (mi >> 1)) * 16, a[0], a[1], a[2], a[3]);
      ldsm_x4(tile + krow * kPitch + (2 * ks + (mi & 1)) * 16, b0, b1, b2, b3);
      mma_bf16_16816(s[0], a, b0, b1);
      mma_bf16_16816(s[1], a, b2, b3);
    }
    // exchange partial scores with the other warp of the head group
    *reinterpret_cast<float4*>(xmine) = make_float4(s[0][0], s[0][1], s[0][2], s[0][3]);
    *reinterpret_cast<float4*>(xmine + 4) = make_float4(s[1][0], s[1][1], s[1][2], s[1][3]);
    asm volatile("bar.sync %0, 64;" ::"r"(1 + hg) : "memory");
    {
      const float4 pa = *reinterpret_cast<const float4*>(xpeer);
      const float4 pb = *reinterpret_cast<const float4*>(xpeer + 4);
      s[0][0] += pa.x; s[0][1] += pa.y; s[0][2] += pa.z; s[0][3] += pa.w;
      s[1][0] += pb.x; s[1][1] += pb.y; s[1][2] += pb.z; s[1][3] += pb.w;
    }
    asm volatile("bar.sync %0, 64;" ::"r"(1 + hg) : "memory");  // slot reusable next tile
    // online softmax (base 2): rows r0 (c0,c1) and r0+8 (c2,c3)
    float x[2][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = nt * 8 + cq + (e & 1);
        const bool ok = col < nvalid && sel[t0 + col] >= 0;
        x[nt][e] = ok ? s[nt][e] * A.sl2 : -INFINITY;
        if (e < 2)
          mx0 = fmaxf(mx0, x[nt][e]);
        else
          mx1 = fmaxf(mx1, x[nt][e]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float b0s = mn0 == -INFINITY ? 0.f : mn0, b1s = mn1 == -INFINITY ? 0.f : mn1;
    if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
      const float a0 = ex2_ftz(m0 - b0s), a1 = ex2_ftz(m1 - b1s);
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        o[n][0] *= a0;
        o[n][1] *= a0;
        o[n][2] *= a1;
        o[n][3] *= a1;
      }
      m0 = mn0;
      m1 = mn1;
    }
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = ex2_ftz(x[nt][0] - b0s);
      p[nt][1] = ex2_ftz(x[nt][1] - b0s);
      p[nt][2] = ex2_ftz(x[nt][2] - b1s);
      p[nt][3] = ex2_ftz(x[nt][3] - b1s);
      l0 += p[nt][0] + p[nt][1];
      l1 += p[nt][2] + p[nt][3];
    }
    uint32_t pa4[4];
    pa4[0] = pack_bf16(p[0][0], p[0][1]);
    pa4[1] = pack_bf16(p[0][2], p[0][3]);
    pa4[2] = pack_bf16(p[1][0], p[1][1]);
    pa4[3] = pack_bf16(p[1][2], p[1][3]);
    // O += P V over this warp's 256 value columns (16-B pieces 32*part .. +31)
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      uint32_t b0, b1, b2, b3;
      const int c16 = part * 32 + 2 * jj + (mi >> 1);
      ldsm_x4_t(tile + vrow * kPitch + c16 * 16, b0, b1, b2, b3);
      mma_bf16_16816(o[2 * jj], pa4, b0, b1);
      mma_bf16_16816(o[2 * jj + 1], pa4, b2, b3);
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
    load_tile(j + kNbuf - 1);
  }
  cp_async_wait<0>();  // nothing left in flight

  // ---- per-rank partial: o = O / l, lse (natural log) ----
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int ha = h0 + hg * 16 + r0, hb = ha + 8;
  const float ia = l0 > 0.f ? 1.f / l0 : 0.f, ib = l1 > 0.f ? 1.f / l1 : 0.f;
  const int64_t rowa = ((int64_t)r * A.B + b) * A.Hq + ha;
  const int64_t rowb = rowa + 8;
#pragma unroll
  for (int n = 0; n < 32; ++n) {
    const int col = part * 256 + n * 8 + cq;
    if (ha < A.Hq)
      *reinterpret_cast<float2*>(A.part_o + rowa * 512 + col) =
          make_float2(o[n][0] * ia, o[n][1] * ia);
    if (hb < A.Hq)
      *reinterpret_cast<float2*>(A.part_o + rowb * 512 + col) =
          make_float2(o[n][2] * ib, o[n][3] * ib);
  }
  if (part == 0 && (lane & 3) == 0) {
    if (ha < A.Hq) A.part_lse[rowa] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
    if (hb < A.Hq) A.part_lse[rowb] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
  }
}

bool sfa_mma_supported(int Hq, int dk, int dv, dcp_dtype_t dtype, int K) {
  return dtype == DCP_BF16 && dk == kRow && dv == 512 && Hq % 16 == 0 && K <= kMaxSel;
}

int launch_sfa_mma(const SfaMmaArgs& A0, cudaStream_t s) {
  SfaMmaArgs A = A0;
  A.hblocks = (A.Hq + kSfaHeadsPerCta - 1) / kSfaHeadsPerCta;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(sfa_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSfaSmem + 128) != cudaSuccess)
      return DCP_ECUDA;
    attr_done[dev] = true;
  }
  const int grid = A.dcp * A.B * A.hblocks;
  if (grid <= 0) return DCP_OK;
  sfa_mma_kernel<<<grid, kSfaThreads, kSfaSmem + 128, s>>>(A);
  return launch_status();
}

}  // namespace dcp
