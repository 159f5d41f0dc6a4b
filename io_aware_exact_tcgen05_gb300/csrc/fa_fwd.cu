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
//
// The kernel is persistent: one CTA per SM walks a fixed sequence of work
// units (the heavy-first list, taken in alternating directions block by
// block so heavy and light units pair up).  Barrier phases run on across
// units; the next unit's Q is loaded once the current unit's last S product
// has read Q, its first S products overlap the current epilogue, and its
// first PV into O waits only until the epilogue has read O.
#include <algorithm>

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
  static constexpr int NS = FwdTiles<D>::kKvStages;  // K and V pipeline depth
  static constexpr int kBox = kTileM * 64;        // elements per 128-row x 64-col box
  __nv_bfloat16 q[2][NB][kBox];
  __nv_bfloat16 k[NS][NB][kBox];
  __nv_bfloat16 v[NS][NB][kBox];
  uint64_t bar_q;
  uint64_t q_free;             // the unit's last S product has read Q
  uint64_t k_full[NS], v_full[NS];
  // kv_free[g % NS] completes a phase when the round issuing S of tile g
  // (g counts tiles across the CTA's units) has finished.  That round also
  // finishes PV of tile g - 1, whether it belongs to the same unit or closes
  // the previous one (a commit covers every earlier MMA), so it frees K
  // stage g % NS and V stage (g - 1) % NS: one commit per tile.
  uint64_t kv_free[NS];
  uint64_t o_empty[2];          // the slot's softmax warps have read O
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
// softmax); bit jj of keep[jj / 32] says whether key jj of the tile is kept.
template <int HALF, bool DROP>
__device__ __forceinline__ void softmax_half(const uint32_t (&sr)[kTileN], uint64_t c2,
                                             uint64_t nmc2, uint32_t t_p, uint64_t (&sum2)[4],
                                             float (&sr_lo)[4], float (&sr_hi)[4],
                                             const uint32_t (&keep)[4]) {
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
      const int kj = HALF * (kTileN / 2) + 2 * jq;  // the pair's first key in the tile
      const uint32_t kb = keep[kj >> 5] >> (kj & 31);
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

// One work unit: two 128-row query tiles ("slots") and the key tiles they
// see.  Units are numbered heavy (late) row blocks first; every role of a
// CTA walks the same unit sequence, so their barrier phases stay in step.
struct Unit {
  int b, h0, h1, r0, r1;
  int sq, qb, bz;        // logical rows [0, sq) from packed row qb of tensor batch bz
  int klo, kend, off;    // visible key interval and bottom-right causal offset
  int hk, j0, n_tiles;
  bool rows, active1;    // rows: slot 0 has rows at all
};

__device__ __forceinline__ Unit unit_at(const FwdParams& p, int U) {
  Unit u;
  const int rbu = p.n_rbu - 1 - U / p.units_per_rbu;
  const int w = U % p.units_per_rbu;
  if (p.pack_heads) {
    const int hpairs = p.Hq >> 1;
    u.b = w / hpairs;
    u.h0 = 2 * (w % hpairs);
    u.h1 = u.h0 + 1;
    u.r0 = u.r1 = rbu * kTileM;
  } else {
    u.b = w / p.Hq;
    u.h0 = u.h1 = w % p.Hq;
    u.r0 = rbu * 2 * kTileM;
    u.r1 = u.r0 + kTileM;
  }
  u.sq = p.Sq;
  u.qb = 0;
  u.bz = u.b;
  if (p.cu_q) {  // packed ragged: b is the sequence
    u.qb = max(0, min(p.cu_q[u.b], p.Sq));
    u.sq = max(0, min(p.cu_q[u.b + 1], p.Sq) - u.qb);
    u.klo = max(0, min(p.cu_k[u.b], p.Sk));
    u.kend = max(u.klo, min(p.cu_k[u.b + 1], p.Sk));
    u.off = u.kend - u.sq;  // bottom-right causal alignment within the sequence
    u.bz = 0;
  } else {
    u.klo = p.k_start ? p.k_start[u.b] : 0;
    u.kend = p.k_end ? p.k_end[u.b] : p.Sk;
    u.klo = max(0, min(u.klo, p.Sk));
    u.kend = max(0, min(u.kend, p.Sk));
    u.off = p.Sk - p.Sq;  // bottom-right causal alignment
  }
  u.rows = u.r0 < u.sq;
  u.active1 = u.r1 < u.sq;
  u.hk = u.h0 / p.group;
  int khi = u.kend;
  if (p.causal) {
    const int last_row = min((u.active1 ? u.r1 : u.r0) + kTileM - 1, u.sq - 1);
    khi = min(khi, last_row + u.off + 1);
  }
  u.j0 = 0;
  u.n_tiles = 0;
  if (u.rows && khi > u.klo) {
    u.j0 = u.klo / kTileN;
    u.n_tiles = (khi + kTileN - 1) / kTileN - u.j0;
  }
  return u;
}

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
  const int n_units = p.n_rbu * p.units_per_rbu;
  // The k-th unit of this CTA: units run heavy to light, so blocks of
  // gridDim.x units are walked alternately forwards and backwards (the
  // heaviest unit of one block pairs with the lightest of the next).
  auto unit_index = [&](int k) {
    const int G = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    return k * G + ((k & 1) ? (G - 1 - c) : c);
  };

  if (threadIdx.x == 0) {
    mbar_init(&s.bar_q, 1);
    mbar_init(&s.q_free, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.kv_free[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s.s_full[t], 1);
      mbar_init(&s.p_full[t], 4);   // one arrival per softmax warp
      mbar_init(&s.o_full[t], 1);
      mbar_init(&s.o_empty[t], 4);  // the slot's softmax warps have read O
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
    // K/V stages follow a tile counter g that runs across the CTA's units;
    // the next unit's Q is loaded once the previous unit's last S product
    // has read Q (q_free).
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      const uint64_t keep = policy_evict_last();
      int g = 0, uq = 0;               // tiles and Q loads issued so far
      int k_issued = 0, v_issued = 0;  // (global tile counts, for the abort drain)
      bool ok = true;
      for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
        const int U = unit_index(k);
        if (U >= n_units) continue;
        const Unit un = unit_at(p, U);
        if (un.n_tiles == 0) continue;
        if (uq > 0 && !mbar_wait(&s.q_free, (uq - 1) & 1, abort_flag, kSiteQ)) break;
        mbar_arrive_expect_tx(&s.bar_q, (un.active1 ? 2 : 1) * NB * kBoxBytes);
        for (int cb = 0; cb < NB; ++cb) {
          tma_load_3d(s.q[0][cb], &tq, &s.bar_q, cb * 64, un.qb + un.r0, un.bz * p.Hq + un.h0);
          if (un.active1)
            tma_load_3d(s.q[1][cb], &tq, &s.bar_q, cb * 64, un.qb + un.r1, un.bz * p.Hq + un.h1);
        }
        ++uq;
        const int zkv = un.bz * p.Hkv + un.hk;
        for (int j = 0; j < un.n_tiles; ++j, ++g) {
          const int st = g % NS;
          const int use = g / NS;
          const int c0 = (un.j0 + j) * kTileN;
          // stage st last held tile g - NS: its K was freed in round g - NS,
          // its V in round g - NS + 1
          if (use > 0 && !mbar_wait(&s.kv_free[st], (use - 1) & 1, abort_flag, kSiteKFree)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.k_full[st], NB * kBoxBytes);
          for (int cb = 0; cb < NB; ++cb)
            tma_load_3d_hint(s.k[st][cb], &tk, &s.k_full[st], cb * 64, c0, zkv, keep);
          k_issued = g + 1;
          if (use > 0) {
            const int r = g - NS + 1;
            if (!mbar_wait(&s.kv_free[r % NS], (r / NS) & 1, abort_flag, kSiteVFree)) {
              ok = false;
              break;
            }
          }
          mbar_arrive_expect_tx(&s.v_full[st], NB * kBoxBytes);
          for (int cb = 0; cb < NB; ++cb)
            tma_load_3d_hint(s.v[st][cb], &tv, &s.v_full[st], cb * 64, c0, zkv, keep);
          v_issued = g + 1;
        }
      }
      if (*abort_flag) {
        // let every issued copy land before shared memory is released
        if (uq > 0) mbar_drain(&s.bar_q, (uq - 1) & 1, kSiteDrain);
        for (int j = max(0, k_issued - NS); j < k_issued; ++j)
          mbar_drain(&s.k_full[j % NS], (j / NS) & 1, kSiteDrain);
        for (int j = max(0, v_issued - NS); j < v_issued; ++j)
          mbar_drain(&s.v_full[j % NS], (j / NS) & 1, kSiteDrain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------- MMA issuer --
    // The whole warp runs this loop (warp-uniform control flow and operands);
    // one elected lane issues each MMA and commit.  Per unit, round j issues
    // PV_t(j-1) and S_t(j) for each active slot.  A unit's first S products
    // run while the softmax warps still finish the previous unit's epilogue;
    // its first PV into O_t waits until they have read O_t (o_empty).
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kTileM, kTileN, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kTileM, D, false, true);
    constexpr uint32_t kStage = NB * kBoxBytes;  // bytes per K (or V) stage
    const uint64_t qd0 = smem_desc_sw128(smem_u32(s.q[0][0]), 16, 1024);
    const uint64_t qd1 = smem_desc_sw128(smem_u32(s.q[1][0]), 16, 1024);
    const uint64_t kd0 = smem_desc_sw128(smem_u32(s.k[0][0]), 16, 1024);
    const uint64_t vd0 = smem_desc_sw128(smem_u32(s.v[0][0]), NB > 1 ? kBoxBytes : 16u, 1024);
    int g = 0, uq = 0;
    int ts[2] = {0, 0}, us[2] = {0, 0};  // per slot: tiles and units so far
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
      const int U = unit_index(k);
      if (U >= n_units) continue;
      const Unit un = unit_at(p, U);
      if (un.n_tiles == 0) continue;
      const int n = un.n_tiles;
      const int nslots = un.active1 ? 2 : 1;
      if (!mbar_wait_warp(&s.bar_q, uq & 1, abort_flag, kSiteQ)) break;
      ++uq;
      for (int j = 0; ok && j <= n; ++j) {
        // K and V arrive by TMA: the mbarrier wait alone orders those shared
        // memory writes before the MMAs (both sides are async-proxy accesses).
        // Only P, written by other threads' tcgen05.st, needs the tcgen05 fence.
        const int gk = g + j, gv = g + j - 1;  // this round's K tile, V tile
        if (j < n && !mbar_wait_warp(&s.k_full[gk % NS], (gk / NS) & 1, abort_flag, kSiteKFull)) {
          ok = false;
          break;
        }
        const uint64_t kd = desc_add(kd0, static_cast<uint32_t>(gk % NS) * kStage);
        const uint64_t vd = desc_add(vd0, static_cast<uint32_t>(((gv % NS) + NS) % NS) * kStage);
        for (int t = 0; t < nslots; ++t) {
          const uint32_t t_s = tmem + t * kTileN;
          if (j > 0) {
            // O_t += P_t(j-1) V_{j-1}; P_t lives in the last 64 columns of S_t
            if (!mbar_wait_warp(&s.p_full[t], (ts[t] + j - 1) & 1, abort_flag, kSitePFull) ||
                (t == 0 &&
                 !mbar_wait_warp(&s.v_full[gv % NS], (gv / NS) & 1, abort_flag, kSiteVFull)) ||
                (j == 1 && us[t] > 0 &&
                 !mbar_wait_warp(&s.o_empty[t], (us[t] - 1) & 1, abort_flag, kSiteOFull))) {
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
          if (j < n) {
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
        if (j < n) mma_commit_warp(&s.kv_free[gk % NS]);
        if (j == n - 1) mma_commit_warp(&s.q_free);  // the unit's last S has read Q
      }
      g += n;
      for (int t = 0; t < nslots; ++t) {
        ts[t] += n;
        ++us[t];
      }
    }
    if (warp_aborted(abort_flag)) {
      // every MMA issued so far must finish before TMEM is released
      mma_commit_warp(&s.drain);
      mbar_drain(&s.drain, 0, kSiteDrain);
    }
  } else {
    // ---------------------------------------------------- softmax warps --
    const int t = warp >> 2;
    const int row_in_tile = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + t * kTileN + lane_off;
    const uint32_t t_o = tmem + 2 * kTileN + t * D + lane_off;
    const uint32_t t_p = t_s + kTileN / 2;  // P: bf16 pairs in S columns [64, 128)
    const float c = p.scale_log2;
    int ts = 0, us = 0;  // this slot's tiles and units so far
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
      const int U = unit_index(k);
      if (U >= n_units) continue;
      const Unit un = unit_at(p, U);
      if (!un.rows || (t == 1 && !un.active1)) continue;
      const int n_tiles = un.n_tiles, j0 = un.j0, klo = un.klo, kend = un.kend;
      const int sq = un.sq, qb = un.qb, bz = un.bz;
      const int i = (t == 0 ? un.r0 : un.r1) + row_in_tile;
      const int h = (t == 0) ? un.h0 : un.h1;
      const uint32_t bh = static_cast<uint32_t>(bz * p.Hq + h);  // dropout counter word 2
      const uint32_t* kbits =
          p.key_bits ? p.key_bits + static_cast<size_t>(bz) * p.mask_words : nullptr;
      // keys visible to this row: [klo, khi_row)
      int khi_row = kend;
      if (p.causal) khi_row = min(khi_row, i + un.off + 1);
      float m = neg_inf();  // running max of raw scores (unscaled)
      float l = 0.f;        // running denominator, relative to 2^(m*c)
      float lr = 0.f;       // same, over the bf16-rounded weights
      // Dropout keep bits of this row for one key tile (bit jj of word jj / 32
      // = key jj of the tile kept).  They are computed one tile ahead, after
      // the row's P has been released and while the warp waits for the next
      // S, so the Philox rounds stay off the S -> P path.
      uint32_t keep[4] = {~0u, ~0u, ~0u, ~0u};
      auto keep_bits = [&](int jt) {
        const uint32_t k8 = static_cast<uint32_t>((j0 + jt) * kTileN) >> 3;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t word = 0;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            word |= dropout_keep8(p.drop, k8 + 4 * w + g, static_cast<uint32_t>(i), bh) << (8 * g);
          keep[w] = word;
        }
      };
      if (DROP && n_tiles > 0) keep_bits(0);
      for (int j = 0; j < n_tiles; ++j) {
        if (!mbar_wait_warp(&s.s_full[t], (ts + j) & 1, abort_flag, kSiteSFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kTileN];
#pragma unroll
        for (int cc = 0; cc < kTileN / 32; ++cc)
          tmem_ld32(t_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
        tmem_wait_ld();
        const int c0 = (j0 + j) * kTileN;
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
          softmax_half<0, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, keep);
          softmax_half<1, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, keep);
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
          // grows by more than the threshold.  The difference m_new - m is
          // formed only once m is finite: a row that still sees no key keeps
          // m = -inf and never evaluates -inf - (-inf).
          const bool first = (m == neg_inf()) && (m_new != neg_inf());
          grow = first || (m != neg_inf() && (m_new - m) * c > p.rescale_log2);
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
          softmax_half<0, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, keep);
          softmax_half<1, DROP>(sr, c2, nmc2, t_p, sum2, sr_lo, sr_hi, keep);
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
        if (DROP && j + 1 < n_tiles) keep_bits(j + 1);
      }
      if (!ok) break;
      if (n_tiles > 0) {
        if (!mbar_wait_warp(&s.o_full[t], us & 1, abort_flag, kSiteOFull)) break;
        tc_fence_after();
      }
      if (warp_aborted(abort_flag)) break;
      // ---- epilogue: O = u / lr, LSE = m*scale + ln l ----------------------
      {
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
      if (n_tiles > 0) {
        // O_t has been read: the next unit's first PV may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.o_empty[t]);
        ts += n_tiles;
        ++us;
      }
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
  // The shared-memory limit is a per-device attribute of the kernel: it is
  // set on every call, for whichever device is current (no process-wide
  // state, so several devices, threads and device resets need no care).
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (shared memory allows one), each walking the
  // heavy-first unit list with stride gridDim.x
  int dev = 0, n_sm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // Packed ragged batches keep one unit per CTA: their unit costs vary with
  // the sequence lengths, which only the hardware's dynamic CTA scheduling
  // balances (with gridDim.x = units every CTA's sequence is just its own unit).
  const long long units = static_cast<long long>(p.n_rbu) * p.units_per_rbu;
  const unsigned int grid =
      static_cast<unsigned int>(p.cu_q ? units : std::min<long long>(units, n_sm));
  hook_before(stream);
  fa_fwd_kernel<D, MODE><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  hook_after(stream);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t stream) {
  if (p.drop.on) return launch_fwd_dd<D, kModeDropout>(tq, tk, tv, p, stream);
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
