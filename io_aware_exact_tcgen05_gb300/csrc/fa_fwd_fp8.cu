// fa_fwd_fp8.cu -- forward attention with FP8 (e4m3) inputs for sm_103a.
//
// The bf16 forward's schedule (two 128-row query slots per CTA, ping-ponged;
// a TMA producer warp, an MMA warp and eight softmax warps) with 8-bit
// operands on the tensor core ("Flash Attention" history page 2.2: FP8 in
// FA3; both matrix products run in FP8, accumulation in fp32):
//
//   S_t = Q_t K_j^T     tcgen05.mma kind::f8f6f4, e4m3 A (Q) and B (K) from
//                       shared memory, fp32 in TMEM; K = 32 per instruction
//   P_t                 softmax warps: weights as in the bf16 forward, rounded
//                       to e4m3 (saturating at 448) and written row by row to
//                       shared memory in the MMA's K-major 128-byte-swizzled
//                       layout
//   O_t += P_t V_j      tcgen05.mma kind::f8f6f4, A = P (shared), B = V^T
//                       (shared; V is passed transposed, [d, Sk] per head, so
//                       that both operands of both products are K-major)
//
// Dequantisation is folded into the arithmetic: the score scale becomes
// scale * q_descale * k_descale, and O is multiplied by v_descale once in the
// epilogue.  Weights are kept below 448 (e4m3's largest finite value): the
// fast path accepts a tile only while the row's fp32 weight sum stays below
// it, and the exact path rescales once the max grows by more than 2^1, so
// that later tiles of the row pass that bound again.  O is
// divided by the sum of the *rounded* weights (what the PV product used), l
// (fp32, unrounded) gives the LSE.
//
// Method: as fa_fwd.cu ("Flash Attention" history page 1.2, 1.3, 2.1, 2.3;
// FlashAttention_01 page, online-softmax derivation and masking rule).
#include <algorithm>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr int kD = 128;                   // head dimension (bytes per fp8 row)
constexpr int kNS = Fp8Tiles::kKvStages;  // K and V^T pipeline depth
constexpr uint32_t kTile = 128 * 128;     // bytes of one 128 x 128 e4m3 tile

enum : unsigned int {
  kSiteQ = 1, kSiteKFree, kSiteVFree, kSiteKFull, kSiteVFull, kSitePFull, kSiteSFull,
  kSiteOFull, kSiteDrain
};

struct Fp8Smem {
  uint8_t q[2][kTile];      // Q_t, rows = query rows, 128 bytes (= d) per row
  uint8_t k[kNS][kTile];    // K_j, rows = keys
  uint8_t vt[kNS][kTile];   // V_j^T, rows = head dimension, 128 keys per row
  uint64_t bar_q;
  uint64_t q_free;          // the unit's last S product has read Q
  uint64_t k_full[kNS], v_full[kNS];
  uint64_t kv_free[kNS];    // round g (tiles counted across units) read K tile g and V tile g - 1
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t o_empty[2];      // the slot's softmax warps have read O
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void mask_scores(uint32_t (&sr)[kTileN], int first, int count, int c0,
                                            int klo, int khi) {
#pragma unroll
  for (int jj = 0; jj < kTileN; ++jj) {
    if (jj < first || jj >= first + count) continue;
    const int key = c0 + jj;
    if (key < klo || key >= khi) sr[jj] = 0xff800000u;
  }
}

// Weights 2^(s*c - mc) of the tile's 128 scores (nmc2 holds -mc twice),
// rounded to e4m3 and stored as the row's 128 bytes of P in TMEM (32
// columns from t_p, four keys per column, key 4w + b in byte b of column w);
// sum2 gathers the fp32 weights (l), sr_lo/sr_hi the rounded ones (lr).
__device__ __forceinline__ void softmax_tile_fp8(const uint32_t (&sr)[kTileN], uint64_t c2,
                                                 uint64_t nmc2, uint32_t t_p,
                                                 uint64_t (&sum2)[4], float (&sr_lo)[4],
                                                 float (&sr_hi)[4]) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {  // 64 keys, 16 columns per store
    uint32_t w[16];
#pragma unroll
    for (int q4 = 0; q4 < 16; ++q4) {  // 4 keys per 32-bit word
      uint16_t h[2];
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        const int jj = hf * 64 + q4 * 4 + pr * 2;
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[jj]), __uint_as_float(sr[jj + 1])), c2, nmc2),
                  x0, x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        h[pr] = pack_e4m3x2(p0, p1);
        const int a = (q4 * 2 + pr) & 3;
        sum2[a] = f2_add(sum2[a], f2_pack(p0, p1));
        add_e4m3x2_f32(sr_lo[a], sr_hi[a], h[pr]);
      }
      w[q4] = static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16);
    }
    tmem_st16(t_p + hf * 16, w);
  }
}

__device__ __forceinline__ float sum_f2x4(const uint64_t (&v)[4]) {
  float a, b;
  f2_unpack(f2_add(f2_add(v[0], v[1]), f2_add(v[2], v[3])), a, b);
  return a + b;
}

// One work unit: two 128-row query tiles (slots) and the key tiles they see,
// numbered heavy (late) row blocks first, as in the bf16 forward.
struct Fp8Unit {
  int b, h0, h1, r0, r1;
  bool active1;
  int hk, klo, kend, off, j0, n_tiles;
};

__device__ __forceinline__ Fp8Unit fp8_unit_at(const Fp8FwdParams& p, int U) {
  Fp8Unit u;
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
  u.active1 = u.r1 < p.Sq;
  u.hk = u.h0 / p.group;
  u.klo = p.k_start ? p.k_start[u.b] : 0;
  u.kend = p.k_end ? p.k_end[u.b] : p.Sk;
  u.klo = max(0, min(u.klo, p.Sk));
  u.kend = max(0, min(u.kend, p.Sk));
  u.off = p.Sk - p.Sq;  // bottom-right causal alignment
  int khi = u.kend;
  if (p.causal) {
    const int last_row = min((u.active1 ? u.r1 : u.r0) + kTileM - 1, p.Sq - 1);
    khi = min(khi, last_row + u.off + 1);
  }
  u.j0 = 0;
  u.n_tiles = 0;
  if (khi > u.klo) {
    u.j0 = u.klo / kTileN;
    u.n_tiles = (khi + kTileN - 1) / kTileN - u.j0;
  }
  return u;
}

// Persistent, like the bf16 forward: one CTA per SM walks the heavy-first
// unit list in alternating directions block by block.  Barrier phases run on
// across units: the next unit's Q is loaded once the current unit's last S
// product has read Q (q_free), K/V stages and their release commits count
// tiles across units, and the next unit's first PV into O_t waits only until
// the softmax warps have read O_t in the epilogue (o_empty).
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tvt, const Fp8FwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  Fp8Smem& s = *reinterpret_cast<Fp8Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_units = p.n_rbu * p.units_per_rbu;
  auto unit_index = [&](int k) {
    const int G = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    return k * G + ((k & 1) ? (G - 1 - c) : c);
  };

  if (threadIdx.x == 0) {
    mbar_init(&s.bar_q, 1);
    mbar_init(&s.q_free, 1);
    for (int i = 0; i < kNS; ++i) {
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
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tvt);
      const uint64_t keep = policy_evict_last();
      int g = 0, uq = 0, k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
        const int U = unit_index(k);
        if (U >= n_units) continue;
        const Fp8Unit un = fp8_unit_at(p, U);
        if (un.n_tiles == 0) continue;
        if (uq > 0 && !mbar_wait(&s.q_free, (uq - 1) & 1, abort_flag, kSiteQ)) break;
        mbar_arrive_expect_tx(&s.bar_q, (un.active1 ? 2 : 1) * kTile);
        tma_load_3d(s.q[0], &tq, &s.bar_q, 0, un.r0, un.b * p.Hq + un.h0);
        if (un.active1) tma_load_3d(s.q[1], &tq, &s.bar_q, 0, un.r1, un.b * p.Hq + un.h1);
        ++uq;
        const int zkv = un.b * p.Hkv + un.hk;
        for (int j = 0; j < un.n_tiles; ++j, ++g) {
          const int st = g % kNS;
          const int use = g / kNS;
          const int c0 = (un.j0 + j) * kTileN;
          // stage st last held tile g - NS: its K was freed in round g - NS,
          // its V^T in round g - NS + 1
          if (use > 0 && !mbar_wait(&s.kv_free[st], (use - 1) & 1, abort_flag, kSiteKFree)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.k_full[st], kTile);
          tma_load_3d_hint(s.k[st], &tk, &s.k_full[st], 0, c0, zkv, keep);
          k_issued = g + 1;
          if (use > 0) {
            const int r = g - kNS + 1;
            if (!mbar_wait(&s.kv_free[r % kNS], (r / kNS) & 1, abort_flag, kSiteVFree)) {
              ok = false;
              break;
            }
          }
          // V^T tile: keys [c0, c0 + 128) of every head-dimension row
          mbar_arrive_expect_tx(&s.v_full[st], kTile);
          tma_load_3d_hint(s.vt[st], &tvt, &s.v_full[st], c0, 0, zkv, keep);
          v_issued = g + 1;
        }
      }
      if (*abort_flag) {
        if (uq > 0) mbar_drain(&s.bar_q, (uq - 1) & 1, kSiteDrain);
        for (int j = max(0, k_issued - kNS); j < k_issued; ++j)
          mbar_drain(&s.k_full[j % kNS], (j / kNS) & 1, kSiteDrain);
        for (int j = max(0, v_issued - kNS); j < v_issued; ++j)
          mbar_drain(&s.v_full[j % kNS], (j / kNS) & 1, kSiteDrain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------- MMA issuer --
    // Per unit, round j issues PV_t(j-1) and S_t(j) for each active slot.
    constexpr uint32_t idesc = idesc_e4m3_f32(kTileM, kTileN);  // N = keys or d, both 128
    const uint64_t qd0 = smem_desc_sw128(smem_u32(s.q[0]), 16, 1024);
    const uint64_t qd1 = smem_desc_sw128(smem_u32(s.q[1]), 16, 1024);
    const uint64_t kd0 = smem_desc_sw128(smem_u32(s.k[0]), 16, 1024);
    const uint64_t vd0 = smem_desc_sw128(smem_u32(s.vt[0]), 16, 1024);
    int g = 0, uq = 0;
    int ts[2] = {0, 0}, us[2] = {0, 0};  // per slot: tiles and units so far
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
      const int U = unit_index(k);
      if (U >= n_units) continue;
      const Fp8Unit un = fp8_unit_at(p, U);
      if (un.n_tiles == 0) continue;
      const int n = un.n_tiles;
      const int nslots = un.active1 ? 2 : 1;
      if (!mbar_wait_warp(&s.bar_q, uq & 1, abort_flag, kSiteQ)) break;
      ++uq;
      for (int j = 0; ok && j <= n; ++j) {
        const int gk = g + j, gv = g + j - 1;  // this round's K tile, V tile
        if (j < n && !mbar_wait_warp(&s.k_full[gk % kNS], (gk / kNS) & 1, abort_flag, kSiteKFull)) {
          ok = false;
          break;
        }
        const uint64_t kd = desc_add(kd0, static_cast<uint32_t>(gk % kNS) * kTile);
        const uint64_t vd = desc_add(vd0, static_cast<uint32_t>(((gv % kNS) + kNS) % kNS) * kTile);
        for (int t = 0; t < nslots; ++t) {
          const uint32_t t_s = tmem + t * kTileN;
          if (j > 0) {
            // O_t += P_t(j-1) V_{j-1}: P from TMEM (the softmax warps' stores
            // ordered before p_full by the tcgen05 fences), V^T from TMA
            if (!mbar_wait_warp(&s.p_full[t], (ts[t] + j - 1) & 1, abort_flag, kSitePFull) ||
                (t == 0 &&
                 !mbar_wait_warp(&s.v_full[gv % kNS], (gv / kNS) & 1, abort_flag, kSiteVFull)) ||
                (j == 1 && us[t] > 0 &&
                 !mbar_wait_warp(&s.o_empty[t], (us[t] - 1) & 1, abort_flag, kSiteOFull))) {
              ok = false;
              break;
            }
            tc_fence_after();  // the softmax warps' TMEM reads of S_t come first
            const uint32_t t_o = tmem + 2 * kTileN + t * kD;
            const uint32_t t_p = t_s + kTileN - kTileN / 4;
#pragma unroll
            for (int kk = 0; kk < kTileN / 32; ++kk)
              mma_ts_warp_f8(t_o, t_p + kk * 8, desc_add(vd, kk * 32), idesc,
                             (j > 1 || kk > 0) ? 1u : 0u);
          }
          if (j < n) {
            const uint64_t qd = t ? qd1 : qd0;
#pragma unroll
            for (int kk = 0; kk < kD / 32; ++kk)
              mma_ss_warp_f8(t_s, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc,
                             kk > 0 ? 1u : 0u);
            mma_commit_warp(&s.s_full[t]);
          } else {
            mma_commit_warp(&s.o_full[t]);
          }
        }
        if (!ok) break;
        if (j < n) mma_commit_warp(&s.kv_free[gk % kNS]);
        if (j == n - 1) mma_commit_warp(&s.q_free);  // the unit's last S has read Q
      }
      g += n;
      for (int t = 0; t < nslots; ++t) {
        ts[t] += n;
        ++us[t];
      }
    }
    if (warp_aborted(abort_flag)) {
      mma_commit_warp(&s.drain);
      mbar_drain(&s.drain, 0, kSiteDrain);
    }
  } else {
    // ---------------------------------------------------- softmax warps --
    const int t = warp >> 2;
    const int row_in_tile = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + t * kTileN + lane_off;
    const uint32_t t_o = tmem + 2 * kTileN + t * kD + lane_off;
    // this row's 128 bytes of P: 8-row swizzle atoms of 1024 bytes
    const uint32_t t_p = t_s + kTileN - kTileN / 4;
    const float c = p.scale_log2;
    int ts = 0, us = 0;  // this slot's tiles and units so far
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
      const int U = unit_index(k);
      if (U >= n_units) continue;
      const Fp8Unit un = fp8_unit_at(p, U);
      if (t == 1 && !un.active1) continue;
      const int n_tiles = un.n_tiles, j0 = un.j0, klo = un.klo, kend = un.kend;
      const int i = (t == 0 ? un.r0 : un.r1) + row_in_tile;
      const int h = (t == 0) ? un.h0 : un.h1;
      int khi_row = kend;
      if (p.causal) khi_row = min(khi_row, i + un.off + 1);
      float m = neg_inf();
      float l = 0.f;   // fp32 weights
      float lr = 0.f;  // e4m3-rounded weights
      for (int j = 0; j < n_tiles; ++j) {
        if (!mbar_wait_warp(&s.s_full[t], (ts + j) & 1, abort_flag, kSiteSFull)) { ok = false; break; }
        tc_fence_after();
        // The reducing TMEM load returns each 32-column chunk's max with the
        // scores; a tile that needs masking takes its max after the mask.
        uint32_t sr[kTileN];
        float cmx[kTileN / 32];
#pragma unroll
        for (int cc = 0; cc < kTileN / 32; ++cc)
          tmem_ld32_max(t_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]), cmx[cc]);
        tmem_wait_ld();
        const int c0 = (j0 + j) * kTileN;
        const bool need_mask = (c0 < klo) || (c0 + kTileN > khi_row);
        // Row max of the tile, then the lazily moved running max: m moves to
        // the new max only when that grows by more than 2^rescale_log2 (= 2^8),
        // so every weight 2^(s*c - m*c) stays at most 256, inside e4m3's range
        // (448).  A row's first visible key always sets m; the difference
        // m_new - m is formed only once m is finite (no -inf - (-inf)).
        float mx = fmaxf(fmaxf(cmx[0], cmx[1]), fmaxf(cmx[2], cmx[3]));
        if (__any_sync(0xffffffffu, need_mask)) {
          mask_scores(sr, 0, kTileN, c0, klo, khi_row);
          float mx8[8];
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2)
            mx8[q2] = fmaxf(__uint_as_float(sr[q2]), __uint_as_float(sr[q2 + 8]));
#pragma unroll
          for (int jj = 16; jj < kTileN; jj += 16)
#pragma unroll
            for (int q2 = 0; q2 < 8; ++q2)
              mx8[q2] = max3f(mx8[q2], __uint_as_float(sr[jj + q2]), __uint_as_float(sr[jj + 8 + q2]));
          mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                     fmaxf(mx8[6], mx8[7]));
        }
        const float m_new = fmaxf(m, mx);
        const bool first = (m == neg_inf()) && (m_new != neg_inf());
        const bool grow = first || (m != neg_inf() && (m_new - m) * c > p.rescale_log2);
        const float alpha = first ? 0.f : (grow ? ex2_approx((m - m_new) * c) : 1.f);
        if (grow) {
          l *= alpha;
          lr *= alpha;
          m = m_new;
        }
        const float mc = (m == neg_inf()) ? 0.f : m * c;
        const uint64_t c2 = f2_pack(c, c);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
        float sr_lo[4] = {0.f, 0.f, 0.f, 0.f}, sr_hi[4] = {0.f, 0.f, 0.f, 0.f};
        softmax_tile_fp8(sr, c2, f2_pack(-mc, -mc), t_p, sum2, sr_lo, sr_hi);
        l += sum_f2x4(sum2);
        lr += (sr_lo[0] + sr_lo[1]) + (sr_lo[2] + sr_lo[3]) +
              ((sr_hi[0] + sr_hi[1]) + (sr_hi[2] + sr_hi[3]));
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // O_t is quiescent: PV_t(j-1) completed before S_t(j) was signalled
#pragma unroll
          for (int cc = 0; cc < kD / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(t_o + cc * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int q2 = 0; q2 < 32; ++q2)
              orr[q2] = __float_as_uint(__uint_as_float(orr[q2]) * alpha);
            tmem_st32(t_o + cc * 32, orr);
          }
          tmem_wait_st();
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[t]);
      }
      if (!ok) break;
      if (n_tiles > 0) {
        if (!mbar_wait_warp(&s.o_full[t], us & 1, abort_flag, kSiteOFull)) break;
        tc_fence_after();
      }
      if (warp_aborted(abort_flag)) break;
      // ---- epilogue: O = v_descale * u / lr, LSE = m * scale_qk + ln l -----
      {
        const bool live = l > 0.f;
        const float inv = live ? p.v_descale / lr : 0.f;
        const bool in_range = i < p.Sq;
        const size_t row = (static_cast<size_t>(un.b) * p.Hq + h) * p.Sq + i;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + row * kD;
#pragma unroll 1
        for (int cc = 0; cc < kD / 32; ++cc) {
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
        if (in_range && p.lse) p.lse[row] = live ? fmaf(m, p.scale_qk, logf(l)) : neg_inf();
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

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const Fp8FwdParams& p, cudaStream_t stream) {
  constexpr size_t smem = sizeof(Fp8Smem) + 1024;
  // per-device kernel attribute: set on every call for the current device
  const cudaError_t e = cudaFuncSetAttribute(fa_fwd_fp8_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM over the heavy-first unit list
  int dev = 0, n_sm = 0;
  cudaError_t e2 = cudaGetDevice(&dev);
  if (e2 == cudaSuccess) e2 = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e2 != cudaSuccess) return e2;
  const long long units = static_cast<long long>(p.n_rbu) * p.units_per_rbu;
  const unsigned int grid = static_cast<unsigned int>(std::min<long long>(units, n_sm));
  hook_before(stream);
  fa_fwd_fp8_kernel<<<grid, kThreads, smem, stream>>>(tq, tk, tvt, p);
  hook_after(stream);
  return cudaGetLastError();
}

unsigned int read_fwd_fp8_status(bool clear) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_status, sizeof v);
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof z);
  }
  return v;
}

}  // namespace fa
