// fa_fwd.cu -- forward attention kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// One CTA owns two 128-row query tiles ("slots") that share every key/value
// tile it streams: either two query heads of one KV group at the same rows
// (grouped heads: K/V tiles are fetched once per KV head for both), or two
// consecutive row blocks of one head.  Per key/value tile j:
//
//   S_t = Q_t K_j^T          tcgen05.mma, A and B from shared memory, fp32 in TMEM
//   softmax warps of slot t  tcgen05.ld S_t (one TMEM lane = one query row = one
//                            thread), mask, row max, conditional rescale of O_t,
//                            p = 2^(s*c - m*c), row sum, P_t -> bf16 into the
//                            TMEM columns of S_t
//   O_t += P_t V_j           tcgen05.mma, A (P) from TMEM, B (V) from shared memory
//
// The two slots ping-pong: while the softmax warps of one slot work, the
// tensor core runs the other slot's MMAs.  The S x S matrix never leaves
// TMEM/registers; O is divided by l once at the end and the per-row
// logsumexp is written beside it.
//
// Method: "Flash Attention" history page 1.2 (running max, denominator and
// rescaled output), 1.3 (tiles discarded on chip), 2.1 (query-sequence
// parallelism, fully masked causal tiles skipped), 2.3 (asynchronous MMA and
// skipping the rescale while the running max does not grow); FlashAttention_01
// page, online-softmax derivation (m, l, u; mask before the max; empty rows).
//
// Warp roles (320 threads): warps 0-3 softmax of slot 0, warps 4-7 softmax of
// slot 1 (a warp may only touch TMEM lanes 32*(warp%4) .. +31, which are the
// rows it owns), warp 8 TMA producer, warp 9 MMA issuer and TMEM owner.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;

// wait-site ids reported in the status word
enum : unsigned int {
  kSiteQ = 1, kSiteKFree, kSiteVFree, kSiteKFull, kSiteVFull, kSitePFull, kSiteSFull,
  kSiteOFull, kSiteDrain
};

template <int D>
struct FwdSmem {
  static constexpr int NB = D / 64;               // 64-wide (128-byte) column blocks per row
  static constexpr int NS = (D == 128) ? 2 : 3;   // K and V pipeline depth
  static constexpr int kBox = kTileM * 64;        // elements per 128-row x 64-col box
  __nv_bfloat16 q[2][NB][kBox];
  __nv_bfloat16 k[NS][NB][kBox];
  __nv_bfloat16 v[NS][NB][kBox];
  uint64_t bar_q;
  uint64_t k_full[NS], v_full[NS];
  // kv_free[i % NS] completes a phase when every MMA of issue round i has
  // finished: round i reads K tile i and V tile i - 1, so it frees K stage
  // i % NS and V stage (i - 1) % NS (one commit per round instead of two).
  uint64_t kv_free[NS];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain;  // MMA teardown after an abort
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
constexpr size_t fwd_smem_bytes() {
  return sizeof(FwdSmem<D>) + 1024;  // + alignment slack
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Fast-path bound on a row's fp32 tile sum: every weight stays below 2^64,
// so P, l and O (at most 2^64 per tile per key block) stay far from fp32
// overflow while the running max is left as it is.
constexpr float kFastLimit = 18446744073709551616.0f;  // 2^64

// Scores of keys outside [klo, khi) become -inf (weight 0).
template <int FIRST, int COUNT>
__device__ __forceinline__ void mask_scores(uint32_t (&sr)[kTileN], int c0, int klo, int khi) {
#pragma unroll
  for (int jj = FIRST; jj < FIRST + COUNT; ++jj) {
    const int key = c0 + jj;
    if (key < klo || key >= khi) sr[jj] = 0xff800000u;
  }
}

// Scores of keys whose visibility bit is clear become -inf; bit jj of the
// 128-bit word group kb stands for key c0 + jj.
template <int FIRST, int COUNT>
__device__ __forceinline__ void mask_key_bits(uint32_t (&sr)[kTileN], uint4 kb) {
  const uint32_t w[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
  for (int jj = FIRST; jj < FIRST + COUNT; ++jj)
    if (!((w[jj >> 5] >> (jj & 31)) & 1u)) sr[jj] = 0xff800000u;
}

// Weights 2^(s*c - mc) of the 64 scores sr[64*HALF, +64) (nmc2 holds -mc
// twice), rounded to bf16 pairs and stored to TMEM columns [32*HALF, +32)
// from t_p.  sum2 gathers the fp32 weights (for l); sr_lo/sr_hi gather the
// rounded ones (for lr).  With DROP, the stored words of dropped weights are
// cleared after the sums (l, lr and the LSE stay those of the undropped
// softmax); key4 is the tile's first key / 4, row and bh the Philox counter's
// query row and query head.
template <int HALF, bool DROP>
__device__ __forceinline__ void softmax_half(const uint32_t (&sr)[kTileN], uint64_t c2,
                                             uint64_t nmc2, uint32_t t_p, uint64_t (&sum2)[4],
                                             float (&sr_lo)[4], float (&sr_hi)[4],
                                             const DropoutArgs& drop, uint32_t key4, uint32_t row,
                                             uint32_t bh) {
  uint32_t keep4 = 0;
  uint32_t pk[kTileN / 4];
#pragma unroll
  for (int jq = 0; jq < kTileN / 4; ++jq) {
    const int jj = HALF * (kTileN / 4) + jq;
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * jj]), __uint_as_float(sr[2 * jj + 1])), c2,
                     nmc2),
              x0, x1);
    const float p0 = ex2_approx(x0);
    const float p1 = ex2_approx(x1);
    pk[jq] = pack_bf16x2(p0, p1);
    sum2[jq & 3] = f2_add(sum2[jq & 3], f2_pack(p0, p1));
    add_bf16x2_f32(sr_lo[jq & 3], sr_hi[jq & 3], pk[jq]);
    if (DROP) {
      if ((jq & 1) == 0) keep4 = dropout_keep4(drop, key4 + HALF * 16 + jq / 2, row, bh);
      const uint32_t kb = keep4 >> (2 * (jq & 1));
      pk[jq] &= ((kb & 1u) ? 0x0000ffffu : 0u) | ((kb & 2u) ? 0xffff0000u : 0u);
    }
  }
  tmem_st32(t_p + HALF * 32, pk);
}

__device__ __forceinline__ float sum_f2x4(const uint64_t (&v)[4]) {
  float a, b;
  f2_unpack(f2_add(f2_add(v[0], v[1]), f2_add(v[2], v[3])), a, b);
  return a + b;
}

// Kernel modes: the plain path carries no mask or dropout code at all.
enum : int { kModePlain = 0, kModeKeyBits = 1, kModeDropout = 2 };

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using Smem = FwdSmem<D>;
  constexpr bool DROP = MODE == kModeDropout;
  constexpr bool BITS = MODE != kModePlain;  // key visibility bits may be present
  constexpr int NB = Smem::NB;
  constexpr int NS = Smem::NS;
  constexpr uint32_t kBoxBytes = Smem::kBox * 2;
  extern __shared__ unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: heavy (late) row blocks are launched first -------------
  const int L = blockIdx.x;
  const int rbu = p.n_rbu - 1 - L / p.units_per_rbu;
  const int u = L % p.units_per_rbu;
  int b, h0, h1, r0, r1;
  if (p.pack_heads) {
    const int hpairs = p.Hq >> 1;
    b = u / hpairs;
    h0 = 2 * (u % hpairs);
    h1 = h0 + 1;
    r0 = r1 = rbu * kTileM;
  } else {
    b = u / p.Hq;
    h0 = h1 = u % p.Hq;
    r0 = rbu * 2 * kTileM;
    r1 = r0 + kTileM;
  }
  // This unit's rows: logical rows [0, sq) start at packed row qb of tensor
  // batch bz.  Keys [klo, kend) are in the K/V tensor's own row coordinates.
  int sq = p.Sq, qb = 0, bz = b, klo, kend, off;
  if (p.cu_q) {  // packed ragged: b is the sequence
    qb = max(0, min(p.cu_q[b], p.Sq));
    sq = max(0, min(p.cu_q[b + 1], p.Sq) - qb);
    klo = max(0, min(p.cu_k[b], p.Sk));
    kend = max(klo, min(p.cu_k[b + 1], p.Sk));
    off = kend - sq;  // bottom-right causal alignment within the sequence
    bz = 0;
  } else {
    klo = p.k_start ? p.k_start[b] : 0;
    kend = p.k_end ? p.k_end[b] : p.Sk;
    klo = max(0, min(klo, p.Sk));
    kend = max(0, min(kend, p.Sk));
    off = p.Sk - p.Sq;  // bottom-right causal alignment
  }
  if (r0 >= sq) return;  // row block past the end of its sequence (whole CTA)
  const bool active1 = r1 < sq;
  const int hk = h0 / p.group;
  const uint32_t* kbits = p.key_bits ? p.key_bits + static_cast<size_t>(bz) * p.mask_words : nullptr;
  int khi = kend;
  if (p.causal) {
    const int last_row = min((active1 ? r1 : r0) + kTileM - 1, sq - 1);
    khi = min(khi, last_row + off + 1);
  }
  int j0 = 0, n_tiles = 0;
  if (khi > klo) {
    j0 = klo / kTileN;
    n_tiles = (khi + kTileN - 1) / kTileN - j0;
  }

  if (threadIdx.x == 0) {
    mbar_init(&s.bar_q, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.kv_free[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s.s_full[t], 1);
      mbar_init(&s.p_full[t], 4);  // one arrival per softmax warp
      mbar_init(&s.o_full[t], 1);
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;
  if (warp == 8) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      const uint64_t keep = policy_evict_last();
      mbar_arrive_expect_tx(&s.bar_q, (active1 ? 2 : 1) * NB * kBoxBytes);
      for (int cb = 0; cb < NB; ++cb) {
        tma_load_3d(s.q[0][cb], &tq, &s.bar_q, cb * 64, qb + r0, bz * p.Hq + h0);
        if (active1) tma_load_3d(s.q[1][cb], &tq, &s.bar_q, cb * 64, qb + r1, bz * p.Hq + h1);
      }
      const int zkv = bz * p.Hkv + hk;
      int k_issued = 0, v_issued = 0;  // tiles whose loads were issued
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % NS;
        const int use = j / NS;
        const int c0 = (j0 + j) * kTileN;
        // K tile j reuses the stage of K tile j - NS, read in round j - NS
        if (use > 0 && !mbar_wait(&s.kv_free[st], (use - 1) & 1, abort_flag, kSiteKFree)) break;
        mbar_arrive_expect_tx(&s.k_full[st], NB * kBoxBytes);
        for (int cb = 0; cb < NB; ++cb)
          tma_load_3d_hint(s.k[st][cb], &tk, &s.k_full[st], cb * 64, c0, zkv, keep);
        k_issued = j + 1;
        // V tile j reuses the stage of V tile j - NS, read in round j - NS + 1
        if (use > 0) {
          const int r = j - NS + 1;
          if (!mbar_wait(&s.kv_free[r % NS], (r / NS) & 1, abort_flag, kSiteVFree)) break;
        }
        mbar_arrive_expect_tx(&s.v_full[st], NB * kBoxBytes);
        for (int cb = 0; cb < NB; ++cb)
          tma_load_3d_hint(s.v[st][cb], &tv, &s.v_full[st], cb * 64, c0, zkv, keep);
        v_issued = j + 1;
      }
      if (*abort_flag) {
        // let every issued copy land before shared memory is released
        mbar_drain(&s.bar_q, 0, kSiteDrain);
        for (int j = max(0, k_issued - NS); j < k_issued; ++j)
          mbar_drain(&s.k_full[j % NS], (j / NS) & 1, kSiteDrain);
        for (int j = max(0, v_issued - NS); j < v_issued; ++j)
          mbar_drain(&s.v_full[j % NS], (j / NS) & 1, kSiteDrain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------- MMA issuer --
    // The whole warp runs this loop (warp-uniform control flow and operands);
    // one elected lane issues each MMA and commit.
    if (n_tiles > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kTileM, kTileN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kTileM, D, false, true);
      const int nslots = active1 ? 2 : 1;
      // Descriptors are built once; each MMA only adds a compile-time offset.
      constexpr uint32_t kStage = NB * kBoxBytes;  // bytes per K (or V) stage
      const uint64_t qd0 = smem_desc_sw128(smem_u32(s.q[0][0]), 16, 1024);
      const uint64_t qd1 = smem_desc_sw128(smem_u32(s.q[1][0]), 16, 1024);
      const uint64_t kd0 = smem_desc_sw128(smem_u32(s.k[0][0]), 16, 1024);
      const uint64_t vd0 = smem_desc_sw128(smem_u32(s.v[0][0]), NB > 1 ? kBoxBytes : 16u, 1024);
      bool ok = mbar_wait_warp(&s.bar_q, 0, abort_flag, kSiteQ);
      tc_fence_after();
      for (int j = 0; ok && j <= n_tiles; ++j) {
        // K and V arrive by TMA: the mbarrier wait alone orders those shared
        // memory writes before the MMAs (both sides are async-proxy accesses).
        // Only P, written by other threads' tcgen05.st, needs the tcgen05 fence.
        if (j < n_tiles && !mbar_wait_warp(&s.k_full[j % NS], (j / NS) & 1, abort_flag, kSiteKFull))
          break;
        const uint64_t kd = desc_add(kd0, static_cast<uint32_t>(j % NS) * kStage);
        const uint64_t vd = desc_add(vd0, static_cast<uint32_t>((j + NS - 1) % NS) * kStage);
        for (int t = 0; t < nslots; ++t) {
          const uint32_t t_s = tmem + t * kTileN;
          if (j > 0) {
            // O_t += P_t(j-1) V_{j-1}; P_t lives in the last 64 columns of S_t
            if (!mbar_wait_warp(&s.p_full[t], (j - 1) & 1, abort_flag, kSitePFull)) {
              ok = false;
              break;
            }
            const int vs = (j - 1) % NS;
            if (t == 0 && !mbar_wait_warp(&s.v_full[vs], ((j - 1) / NS) & 1, abort_flag, kSiteVFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t t_o = tmem + 2 * kTileN + t * D;
            const uint32_t t_p = t_s + kTileN / 2;
            mma_ts_warp(t_o, t_p, vd, idesc_pv, j > 1 ? 1u : 0u);
#pragma unroll
            for (int kk = 1; kk < kTileN / 16; ++kk)
              mma_ts_warp(t_o, t_p + kk * 8, desc_add(vd, kk * 16 * 128), idesc_pv, 1u);
          }
          if (j < n_tiles) {
            // S_t = Q_t K_j^T
            const uint64_t qd = t ? qd1 : qd0;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
              mma_ss_warp(t_s, desc_add(qd, off), desc_add(kd, off), idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit_warp(&s.s_full[t]);
          } else {
            mma_commit_warp(&s.o_full[t]);
          }
        }
        if (!ok) break;
        if (j < n_tiles) mma_commit_warp(&s.kv_free[j % NS]);
      }
      if (warp_aborted(abort_flag)) {
        // every MMA issued so far must finish before TMEM is released
        mma_commit_warp(&s.drain);
        mbar_drain(&s.drain, 0, kSiteDrain);
      }
    }
  } else {
    // ---------------------------------------------------- softmax warps --
    const int t = warp >> 2;
    const int row_in_tile = (warp & 3) * 32 + lane;
    const int i = (t == 0 ? r0 : r1) + row_in_tile;
    const int h = (t == 0) ? h0 : h1;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + t * kTileN + lane_off;
    const uint32_t t_o = tmem + 2 * kTileN + t * D + lane_off;
    const uint32_t t_p = t_s + kTileN / 2;  // P: bf16 pairs in S columns [64, 128)
    const uint32_t bh = static_cast<uint32_t>(bz * p.Hq + h);  // dropout counter word 2
    const float c = p.scale_log2;
    // keys visible to this row: [klo, khi_row)
    int khi_row = kend;
    if (p.causal) khi_row = min(khi_row, i + off + 1);
    float m = neg_inf();  // running max of raw scores (unscaled)
    float l = 0.f;        // running denominator, relative to 2^(m*c)
    float lr = 0.f;       // same, over the bf16-rounded weights
    bool ok = (t == 0) || active1;
    if (ok && n_tiles > 0) {
      for (int j = 0; j < n_tiles; ++j) {
        if (!mbar_wait_warp(&s.s_full[t], j & 1, abort_flag, kSiteSFull)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[kTileN];
#pragma unroll
        for (int cc = 0; cc < kTileN / 32; ++cc)
          tmem_ld32(t_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
        tmem_wait_ld();
        const int c0 = (j0 + j) * kTileN;
        const uint32_t key4 = static_cast<uint32_t>(c0) >> 2;  // dropout counter word 0
        const bool need_mask = (c0 < klo) || (c0 + kTileN > khi_row);
        const bool masked_tile = __any_sync(0xffffffffu, need_mask);
        if (masked_tile) mask_scores<0, kTileN>(sr, c0, klo, khi_row);
        // key visibility bits of this tile (the same 128 bits for every row)
        uint4 kb = make_uint4(~0u, ~0u, ~0u, ~0u);
        if (BITS && kbits) kb = __ldg(reinterpret_cast<const uint4*>(kbits + c0 / 32));
        const bool bit_masked = BITS && (kb.x & kb.y & kb.z & kb.w) != ~0u;
        if (bit_masked) mask_key_bits<0, kTileN>(sr, kb);
        // Fast path: weights relative to the running max as it stands.  The
        // max only keeps the weights finite, and the fp32 tile sum (needed for
        // l anyway) bounds every weight of the row, so the tile is checked
        // after the fact.  A row that has no max yet, or whose tile sum
        // reaches kFastLimit (or is not finite), sends the warp to the exact
        // path, which finds the tile max, rescales and recomputes.
        bool exact = __any_sync(0xffffffffu, m == neg_inf());
        const uint64_t c2 = f2_pack(c, c);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
        float sr_lo[4] = {0.f, 0.f, 0.f, 0.f}, sr_hi[4] = {0.f, 0.f, 0.f, 0.f};
        if (!exact) {
          const float mc = m * c;
          const uint64_t nmc2 = f2_pack(-mc, -mc);
          softmax_half<0, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, p.drop, key4, i, bh);
          softmax_half<1, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, p.drop, key4, i, bh);
          const float ts = sum_f2x4(sum2);
          exact = __any_sync(0xffffffffu, !(ts < kFastLimit));
          if (!exact) {
            l += ts;
            lr += (sr_lo[0] + sr_lo[1]) + (sr_lo[2] + sr_lo[3]) +
                  ((sr_hi[0] + sr_hi[1]) + (sr_hi[2] + sr_hi[3]));
          }
        }
        bool grow = false;
        float alpha = 1.f;
        if (exact) {
          // S columns [0, 64) are still in TMEM (P goes to [64, 128)); the
          // scores of [64, 128) are still in registers.
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            tmem_ld32(t_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
          tmem_wait_ld();
          tmem_wait_st();  // fast-path P stores land before they are rewritten
          if (masked_tile) mask_scores<0, kTileN / 2>(sr, c0, klo, khi_row);
          if (bit_masked) mask_key_bits<0, kTileN / 2>(sr, kb);
          // row max: 8 independent chains of 3-input max
          float mx8[8];
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2)
            mx8[q2] = fmaxf(__uint_as_float(sr[q2]), __uint_as_float(sr[q2 + 8]));
#pragma unroll
          for (int jj = 16; jj < kTileN; jj += 16)
#pragma unroll
            for (int q2 = 0; q2 < 8; ++q2)
              mx8[q2] = max3f(mx8[q2], __uint_as_float(sr[jj + q2]), __uint_as_float(sr[jj + 8 + q2]));
          const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                                 fmaxf(mx8[6], mx8[7]));
          const float m_new = fmaxf(m, mx);
          // A row's first visible key always sets its max (also when c = 0,
          // where (m_new - m) * c would be inf * 0); nothing is accumulated
          // yet, so the rescale factor is 0.  Later the max moves only when it
          // grows by more than the threshold.
          const bool first = (m == neg_inf()) && (m_new != neg_inf());
          grow = first || (m_new - m) * c > p.rescale_log2;
          alpha = first ? 0.f : (grow ? ex2_approx((m - m_new) * c) : 1.f);
          if (grow) {
            l *= alpha;
            lr *= alpha;
            m = m_new;
          }
          const float mc = (m == neg_inf()) ? 0.f : m * c;
          const uint64_t nmc2 = f2_pack(-mc, -mc);
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {
            sum2[q2] = 0ull;
            sr_lo[q2] = 0.f;
            sr_hi[q2] = 0.f;
          }
          softmax_half<0, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, p.drop, key4, i, bh);
          softmax_half<1, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, p.drop, key4, i, bh);
          l += sum_f2x4(sum2);
          lr += (sr_lo[0] + sr_lo[1]) + (sr_lo[2] + sr_lo[3]) +
                ((sr_hi[0] + sr_hi[1]) + (sr_hi[2] + sr_hi[3]));
        }
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // O_t is quiescent here: PV_t(j-1) completed before S_t(j) was
          // signalled, and PV_t(j) is issued only after p_full below.
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(t_o + cc * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int q2 = 0; q2 < 32; ++q2)
              orr[q2] = __float_as_uint(__uint_as_float(orr[q2]) * alpha);
            tmem_st32(t_o + cc * 32, orr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[t]);
      }
      if (ok) ok = mbar_wait_warp(&s.o_full[t], 0, abort_flag, kSiteOFull);
      tc_fence_after();
    }
    // ---- epilogue: O = u / l, LSE = m*scale + ln l ---------------------
    if (((t == 0) || active1) && ok && !warp_aborted(abort_flag)) {
      const bool live = l > 0.f;
      const float inv = live ? (DROP ? p.drop.scale : 1.f) / lr : 0.f;
      const bool in_range = i < sq;
      const size_t row = (static_cast<size_t>(bz) * p.Hq + h) * p.Sq + qb + i;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + row * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t orr[32];
        if (n_tiles > 0) {
          tmem_ld32(t_o + cc * 32, orr);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int q2 = 0; q2 < 32; ++q2) orr[q2] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int q2 = 0; q2 < 16; ++q2)
          pk[q2] = pack_bf16x2(__uint_as_float(orr[2 * q2]) * inv,
                               __uint_as_float(orr[2 * q2 + 1]) * inv);
        if (in_range) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2)
            dst[q2] = make_uint4(pk[4 * q2], pk[4 * q2 + 1], pk[4 * q2 + 2], pk[4 * q2 + 3]);
        }
      }
      if (in_range && p.lse) p.lse[row] = live ? fmaf(m, p.scale, logf(l)) : neg_inf();
    }
  }

  // ---- teardown ----------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int MODE>
cudaError_t launch_fwd_dd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdParams& p, cudaStream_t stream) {
  constexpr size_t smem = fwd_smem_bytes<D>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const unsigned int grid = static_cast<unsigned int>(p.n_rbu) * p.units_per_rbu;
  hook_before(stream);
  fa_fwd_kernel<D, MODE><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  hook_after(stream);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t stream) {
  if (p.drop.thr != 0) return launch_fwd_dd<D, kModeDropout>(tq, tk, tv, p, stream);
  if (p.key_bits) return launch_fwd_dd<D, kModeKeyBits>(tq, tk, tv, p, stream);
  return launch_fwd_dd<D, kModePlain>(tq, tk, tv, p, stream);
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch_fwd_d<128>(tq, tk, tv, p, stream);
  return launch_fwd_d<64>(tq, tk, tv, p, stream);
}

unsigned int read_fwd_status(bool clear) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_status, sizeof v);
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof z);
  }
  return v;
}

}  // namespace fa
