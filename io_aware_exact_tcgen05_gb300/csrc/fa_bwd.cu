// fa_bwd.cu -- backward attention by recomputation for sm_103a.
//
//   1. fa_bwd_pre:   D_i = rowsum(dO_i * O_i) (fp32) and dQacc = 0
//   2. fa_bwd_main:  work units of (128-key tile, KV head, batch row).  K and
//                    V stay in shared memory; a unit walks every query head of
//                    the group and every 128-row query tile that can see its
//                    keys.  Per query tile i (all five contractions on tcgen05):
//        S^T  = K Q^T            (keys x queries, fp32 in TMEM)
//        dP^T = V dO^T           (keys x queries, fp32 in TMEM)
//        P^T  = exp(scale*S^T - LSE) on visible entries, 0 elsewhere
//               -> bf16 back into the S^T columns           [compute warps]
//        dV  += P^T dO           (A = P^T from TMEM)
//        dS^T = P^T * (dP^T - D) -> bf16 into shared memory [compute warps]
//        dQ   = dS K             (A = dS from shared memory, into the dP^T
//                                 columns, which the compute warps have read)
//        dK  += dS^T Q           (A = the same shared dS^T rows, K-major)
//        dQacc += dQ             TMEM -> registers -> 32 KB of staging in
//                                shared memory -> TMA reduce-add into the fp32
//                                accumulator                 [drain warps]
//      At the end dK (times scale) and dV leave TMEM as bf16.  With grouped
//      heads dK/dV already hold the sum over the group's query heads.
//   3. fa_bwd_convert: dQ = bf16(scale * dQacc)
//
// Issue order per tile: dP^T(i), dV(i), S^T(i+1), dQ(i), dK(i).
//   * S^T(i+1) follows dV(i), which has read P^T(i) from the S^T columns, so
//     P(i+1) is computed while dQ(i), dK(i) and dP^T(i+1) run.
//   * dQ(i) goes before dK(i): dK reads dS^T from shared memory, not from
//     TMEM, so dQ may overwrite the dP^T columns as soon as every compute
//     warp has loaded dP^T(i).  The drain of dQ(i) then overlaps dK(i).
//   * dP^T(i+1) waits for the drain to have read dQ(i) out of TMEM; this
//     loop (dQ -> drain -> dP^T -> dS -> dQ) sets the pace.
// Q is double-buffered (S^T(i+1) is issued before dK(i) has read Q(i)); dO
// has one buffer, refilled as soon as dV(i) has read it, which leaves dK(i),
// dQ(i) and S^T(i+1) to cover the load.  The dQ staging is separate from
// both, so refilling a Q/dO buffer never waits for a reduce-add.
//
// Method: FlashAttention_01 page, "why the backward can recompute" (rebuild P
// from the saved per-row logsumexp; dV and dP first, then dS from the softmax
// Jacobian, then dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d)) and the chain-rule
// section (masked probabilities and their score gradients are 0); the same
// mask, statistics and scale as the forward.
//
// The main kernel is persistent: one CTA per SM walks a fixed list of units,
// heavy first and in alternating directions block by block.  The list is
// key-tile-major inside groups of (batch row, KV head) pairs, sized by the
// launcher so that a group's dQ accumulators and Q/dO tiles stay in L2 once
// all of them would not.  Per-tile barrier phases run on across units; the
// next unit's K/V load waits for the current unit's last MMA (kv_empty) and
// its first dV/dK products for the epilogue's TMEM reads (dkv_empty), so a
// unit's drain and epilogue overlap the next unit's first tiles.  The
// producer prefetches each tile's Q and dO into L2 while it waits for the
// tile's stage.
//
// Warp roles (448 threads): warps 0-7 compute (one key row = one TMEM lane per
// thread; warps w and w+4 share the lanes of group w and split the 128 query
// columns, so P and dS need no cross-warp exchange), warps 8-11 drain dQ (one
// query row per thread, 8 KB of staging each), warp 12 TMA producer, warp 13
// MMA issuer and TMEM owner.
#include <algorithm>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

// Warp roles: 0-7 compute (lane group warp&3, query-column half warp>>2),
// 8-11 dQ drain, 12 TMA producer, 13 MMA issuer and TMEM owner.
constexpr int kThreads = 448;
constexpr int kWarpProducer = 12;
constexpr int kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;


enum : unsigned int {
  kSiteKV = 1, kSiteQFull, kSiteQEmpty, kSiteS, kSiteP, kSiteDP, kSiteDS, kSiteDQFull,
  kSiteDQEmpty, kSiteDKV, kSiteDrain, kSiteAlign, kSiteStat, kSiteDOFull, kSiteDOEmpty
};

template <int D>
struct BwdSmem {
  static constexpr int kQStages = BwdTiles<D>::kQStages;
  static constexpr int NB = D / 64;
  static constexpr int kBox = kTileM * 64;
  __nv_bfloat16 k[NB][kBox];
  __nv_bfloat16 v[NB][kBox];
  __nv_bfloat16 q[kQStages][NB][kBox];
  __nv_bfloat16 dout[NB][kBox];     // one buffer: dO(i+1) loads while dK/dQ(i) and S^T(i+1) run
  __nv_bfloat16 ds[2][kBox];        // dS^T rows = keys, two 64-query blocks, 128B swizzle
  float dq_stage[4][2][32 * 32];    // per drain warp: two 32x32 fp32 boxes, 128B swizzle
  float nlse2[2][kTileM];           // -LSE * log2(e), -inf for rows without keys
  float ndelta[2][kTileM];          // -D_i; both double-buffered by tile parity
  uint64_t stat_ready[2];
  uint64_t kv_full;
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t do_full, do_empty;
  uint64_t s_full, p_full, dp_full, ds_full, dq_full, dq_empty, dkv_full, drain;
  uint64_t kv_empty, dkv_empty;  // hand-over between consecutive units
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// One work unit: a 128-key tile of one KV head of one batch row (or packed
// sequence), walked against every query tile of the group's heads that sees
// it.  Numbered key tile major, so under the causal rule the heaviest (tile
// 0) come first.  Queries: logical rows [0, sq) from packed row qb of tensor
// batch bz; keys [c0, c0 + 128) and the visible interval [klo, kend) are in
// the K/V tensor's row coordinates, and keys at or past kseq belong to
// another sequence (never stored).
struct BwdUnit {
  int b, hk, sq, qb, bz, klo, kend, kseq, off, c0, qt_lo, n_qt, n_it;
  bool exists;  // the key tile lies inside its sequence
};

__device__ __forceinline__ BwdUnit bwd_unit_at(const BwdParams& p, int U) {
  BwdUnit u;
  // Units run key-tile-major (heavy causal key tiles first) inside groups of
  // unit_group (batch or sequence, KV head) pairs, group after group.
  const int BH = p.grid_b * p.Hkv;
  const int per_group = p.n_kt * p.unit_group;
  const int grp = U / per_group;
  const int first = grp * p.unit_group;
  const int cnt = min(p.unit_group, BH - first);
  const int r = U - grp * per_group;
  const int kt = r / cnt;
  const int bh = first + r % cnt;
  u.b = bh / p.Hkv;
  u.hk = bh % p.Hkv;
  u.sq = p.Sq;
  u.qb = 0;
  u.bz = u.b;
  if (p.cu_q) {  // packed ragged: b is the sequence
    u.qb = max(0, min(p.cu_q[u.b], p.Sq));
    u.sq = max(0, min(p.cu_q[u.b + 1], p.Sq) - u.qb);
    u.klo = max(0, min(p.cu_k[u.b], p.Sk));
    u.kend = max(u.klo, min(p.cu_k[u.b + 1], p.Sk));
    u.kseq = u.kend;
    u.off = u.kend - u.sq;
    u.c0 = u.klo + kt * kTileN;
    u.bz = 0;
  } else {
    u.klo = p.k_start ? p.k_start[u.b] : 0;
    u.kend = p.k_end ? p.k_end[u.b] : p.Sk;
    u.klo = max(0, min(u.klo, p.Sk));
    u.kend = max(0, min(u.kend, p.Sk));
    u.kseq = p.Sk;
    u.off = p.Sk - p.Sq;
    u.c0 = kt * kTileN;
  }
  u.exists = u.c0 < u.kseq;
  const int n_qt_all = (u.sq + kTileM - 1) / kTileM;
  u.qt_lo = 0;
  if (p.causal) u.qt_lo = max(0, u.c0 - u.off) / kTileM;  // first query row that sees key c0
  const bool keys_live = u.exists && (u.c0 < u.kend) && (u.c0 + kTileN > u.klo) &&
                         (!p.causal || u.c0 - u.off < u.sq);
  u.n_qt = keys_live ? max(0, n_qt_all - u.qt_lo) : 0;
  u.n_it = u.n_qt * p.group;
  return u;
}

// ------------------------------------------------------------ preprocess --
// D/8 lanes per row (8 bf16 each): D_i = sum_c dO_ic O_ic; the row of dQacc is zeroed.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre(const BwdParams p, long long rows) {
  constexpr int LPR = D / 8;
  const long long row = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) / LPR;
  const int x = threadIdx.x % LPR;
  float acc = 0.f;
  if (row < rows) {
    const uint4 o = *reinterpret_cast<const uint4*>(
        reinterpret_cast<const __nv_bfloat16*>(p.o) + row * D + x * 8);
    const uint4 g = *reinterpret_cast<const uint4*>(
        reinterpret_cast<const __nv_bfloat16*>(p.dout) + row * D + x * 8);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(ow[e] << 16), __uint_as_float(gw[e] << 16), acc);
      acc = fmaf(__uint_as_float(ow[e] & 0xffff0000u), __uint_as_float(gw[e] & 0xffff0000u), acc);
    }
    float4* z = reinterpret_cast<float4*>(p.dq_acc + row * D + x * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (row < rows && x == 0) p.delta[row] = acc;
}

// --------------------------------------------------------------- convert --
__global__ void __launch_bounds__(256) fa_bwd_convert(const BwdParams p, long long n4) {
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= n4) return;
  const float4 a = reinterpret_cast<const float4*>(p.dq_acc)[i];
  uint2 out;
  out.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
  out.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
  reinterpret_cast<uint2*>(p.dq)[i] = out;
}

// ------------------------------------------------------------------ main --
template <int D, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_main(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                const __grid_constant__ CUtensorMap tdq, const BwdParams p) {
  using Smem = BwdSmem<D>;
  constexpr int NB = Smem::NB;
  constexpr uint32_t kBoxBytes = Smem::kBox * 2;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // 128B-swizzle atoms need 1024B alignment
    if (threadIdx.x == 0) raise_status(2u, kSiteAlign);
    return;
  }

  const int n_units = p.n_kt * p.grid_b * p.Hkv;
  // The k-th unit of this CTA (units run heavy to light: key tile 0 first
  // under the causal rule); blocks of gridDim.x units are walked alternately
  // forwards and backwards so heavy and light units pair up.
  auto unit_index = [&](int k) {
    const int G = static_cast<int>(gridDim.x);
    const int cb = static_cast<int>(blockIdx.x);
    return k * G + ((k & 1) ? (G - 1 - cb) : cb);
  };

  if (threadIdx.x == 0) {
    mbar_init(&s.kv_full, 1);
    for (int i = 0; i < Smem::kQStages; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1);  // MMA commit after the tile's last product
    }
    mbar_init(&s.do_full, 1);
    mbar_init(&s.do_empty, 1);  // MMA commit after dV
    mbar_init(&s.s_full, 1);
    mbar_init(&s.p_full, 8);  // one arrival per compute warp
    mbar_init(&s.dp_full, 1);
    mbar_init(&s.ds_full, 8);
    mbar_init(&s.dq_full, 1);
    mbar_init(&s.dq_empty, 4);  // one arrival per drain warp
    mbar_init(&s.dkv_full, 1);
    mbar_init(&s.kv_empty, 1);   // the unit's last MMA has read K and V
    mbar_init(&s.dkv_empty, 8);  // the compute warps have read dK and dV
    mbar_init(&s.drain, 1);
    mbar_init(&s.stat_ready[0], 4);
    mbar_init(&s.stat_ready[1], 4);
    s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  // P^T (bf16) of query half hf sits in S^T columns [64 hf, 64 hf + 32):
  // inside the columns that half's own warps read, so neither half
  // overwrites scores the other still needs.
  const uint32_t t_S = tmem;              // S^T, then P^T
  const uint32_t t_dP = tmem + kTileN;    // dP^T, then dQ
  const uint32_t t_dV = tmem + 2 * kTileN;
  const uint32_t t_dK = tmem + 2 * kTileN + D;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------ TMA producer --
    // Q/dO stages follow an iteration counter that runs across the CTA's
    // units; a unit's K/V load waits until the previous unit's last MMA has
    // read K and V (kv_empty).
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      int ig = 0, uk = 0;  // iterations and K/V loads issued so far
      int issued = 0, do_issued = 0;
      bool ok = true;
      for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
        const int U = unit_index(k);
        if (U >= n_units) continue;
        const BwdUnit un = bwd_unit_at(p, U);
        if (!un.exists || un.n_it == 0) continue;
        if (uk > 0 && !mbar_wait(&s.kv_empty, (uk - 1) & 1, abort_flag, kSiteKV)) break;
        const int zkv = un.bz * p.Hkv + un.hk;
        mbar_arrive_expect_tx(&s.kv_full, 2 * NB * kBoxBytes);
        for (int cb = 0; cb < NB; ++cb) {
          tma_load_3d(s.k[cb], &tk, &s.kv_full, cb * 64, un.c0, zkv);
          tma_load_3d(s.v[cb], &tv, &s.kv_full, cb * 64, un.c0, zkv);
        }
        ++uk;
        for (int it = 0; it < un.n_it; ++it, ++ig) {
          const int st = ig % Smem::kQStages;
          const int use = ig / Smem::kQStages;
          const int g = it / un.n_qt;
          const int q0 = (un.qt_lo + it % un.n_qt) * kTileM;
          const int zq = un.bz * p.Hq + un.hk * p.group + g;
          // The stage frees only once the dQ reduce staged in it has been
          // read (about a tile's time): meanwhile pull this tile's Q and dO
          // into L2, so that the load below does not wait on DRAM.
          for (int cb = 0; cb < NB; ++cb) {
            tma_prefetch_l2_3d(&tq, cb * 64, un.qb + q0, zq);
            tma_prefetch_l2_3d(&tdo, cb * 64, un.qb + q0, zq);
          }
          if (use > 0 && !mbar_wait(&s.q_empty[st], (use - 1) & 1, abort_flag, kSiteQEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.q_full[st], NB * kBoxBytes);
          for (int cb = 0; cb < NB; ++cb)
            tma_load_3d(s.q[st][cb], &tq, &s.q_full[st], cb * 64, un.qb + q0, zq);
          issued = ig + 1;
          // dO has one buffer, free once dV of the previous tile has read it
          if (ig > 0 && !mbar_wait(&s.do_empty, (ig - 1) & 1, abort_flag, kSiteDOEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.do_full, NB * kBoxBytes);
          for (int cb = 0; cb < NB; ++cb)
            tma_load_3d(s.dout[cb], &tdo, &s.do_full, cb * 64, un.qb + q0, zq);
          do_issued = ig + 1;
        }
      }
      if (*abort_flag) {
        if (uk > 0) mbar_drain(&s.kv_full, (uk - 1) & 1, kSiteDrain);
        for (int i = max(0, issued - Smem::kQStages); i < issued; ++i)
          mbar_drain(&s.q_full[i % Smem::kQStages], (i / Smem::kQStages) & 1, kSiteDrain);
        if (do_issued > 0) mbar_drain(&s.do_full, (do_issued - 1) & 1, kSiteDrain);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------- MMA issuer --
    // The whole warp runs this loop (warp-uniform control flow and operands);
    // one elected lane issues each MMA and commit.  Per-tile barrier phases
    // follow the iteration counter ig, which runs across the CTA's units; a
    // unit's first dV/dK products (which overwrite the accumulators) wait
    // until the previous unit's epilogue has read them (dkv_empty).
    {
      constexpr uint32_t id_kq = idesc_bf16_f32(kTileN, kTileM, false, false);  // S^T, dP^T
      constexpr uint32_t id_acc = idesc_bf16_f32(kTileN, D, false, true);       // dV, dK
      constexpr uint32_t id_dq = idesc_bf16_f32(kTileM, D, true, true);         // dQ
      // Descriptors are built once; each MMA adds a compile-time offset.
      constexpr uint32_t kStage = NB * kBoxBytes;
      constexpr uint32_t kLbo = NB > 1 ? kBoxBytes : 16u;  // next 64-wide d block
      const uint64_t k_kmaj = smem_desc_sw128(smem_u32(s.k[0]), 16, 1024);
      const uint64_t v_kmaj = smem_desc_sw128(smem_u32(s.v[0]), 16, 1024);
      const uint64_t k_mn = smem_desc_sw128(smem_u32(s.k[0]), kLbo, 1024);
      const uint64_t q_kmaj0 = smem_desc_sw128(smem_u32(s.q[0][0]), 16, 1024);
      const uint64_t o_kmaj0 = smem_desc_sw128(smem_u32(s.dout[0]), 16, 1024);
      const uint64_t q_mn0 = smem_desc_sw128(smem_u32(s.q[0][0]), kLbo, 1024);
      const uint64_t o_mn0 = smem_desc_sw128(smem_u32(s.dout[0]), kLbo, 1024);
      const uint64_t ds_mn = smem_desc_sw128(smem_u32(s.ds[0]), kBoxBytes, 1024);
      const uint64_t ds_kmaj = smem_desc_sw128(smem_u32(s.ds[0]), 16, 1024);
      int ig = 0, uk = 0;
      bool ok = true;
      for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
        const int U = unit_index(k);
        if (U >= n_units) continue;
        const BwdUnit un = bwd_unit_at(p, U);
        if (!un.exists || un.n_it == 0) continue;
        if (!mbar_wait_warp(&s.kv_full, uk & 1, abort_flag, kSiteKV)) break;
        for (int it = 0; ok && it < un.n_it; ++it, ++ig) {
          const int st = ig % Smem::kQStages;
          const uint32_t so = static_cast<uint32_t>(st) * kStage;
          // Q and dO arrive by TMA (the mbarrier wait orders them before the
          // MMAs); the S^T columns this overwrites were last touched by other
          // threads before p_full of the previous tile, whose fence covers them.
          if (it == 0) {
            if (!mbar_wait_warp(&s.q_full[st], (ig / Smem::kQStages) & 1, abort_flag, kSiteQFull)) {
              ok = false;
              break;
            }
            // S^T = K Q^T  (A = K rows, B = Q rows, both K-major over d)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
              mma_ss_warp(t_S, desc_add(k_kmaj, off), desc_add(q_kmaj0, so + off), id_kq, kk > 0 ? 1u : 0u);
            }
            mma_commit_warp(&s.s_full);
          }
          // dP^T = V dO^T; its columns held dQ of the previous tile
          if (ig > 0 && !mbar_wait_warp(&s.dq_empty, (ig - 1) & 1, abort_flag, kSiteDQEmpty)) {
            ok = false;
            break;
          }
          if (!mbar_wait_warp(&s.do_full, ig & 1, abort_flag, kSiteDOFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss_warp(t_dP, desc_add(v_kmaj, off), desc_add(o_kmaj0, off), id_kq, kk > 0 ? 1u : 0u);
          }
          mma_commit_warp(&s.dp_full);
          // dV += P^T dO  (A = P^T in TMEM; B = dO rows, MN-major over d)
          if (!mbar_wait_warp(&s.p_full, ig & 1, abort_flag, kSiteP) ||
              (it == 0 && uk > 0 &&
               !mbar_wait_warp(&s.dkv_empty, (uk - 1) & 1, abort_flag, kSiteDKV))) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_ts_warp(t_dV, t_S, o_mn0, id_acc, it > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < kTileM / 16; ++kk)
            mma_ts_warp(t_dV, t_S + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(o_mn0, kk * 2048),
                   id_acc, 1u);
          mma_commit_warp(&s.do_empty);  // dO has been read: the next tile's may load
          // next tile's S^T now: the pipe runs dV before it, so P^T has been read
          if (it + 1 < un.n_it) {
            const int st1 = (ig + 1) % Smem::kQStages;
            const uint32_t so1 = static_cast<uint32_t>(st1) * kStage;
            if (!mbar_wait_warp(&s.q_full[st1], ((ig + 1) / Smem::kQStages) & 1, abort_flag, kSiteQFull)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
              mma_ss_warp(t_S, desc_add(k_kmaj, off), desc_add(q_kmaj0, so1 + off), id_kq, kk > 0 ? 1u : 0u);
            }
            mma_commit_warp(&s.s_full);
          }
          // dS is complete in shared memory and dP^T has been read into registers
          if (!mbar_wait_warp(&s.ds_full, ig & 1, abort_flag, kSiteDS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dQ = dS K  (A = dS: shared rows = keys, queries contiguous -> MN-major;
          //             B = K rows, d contiguous -> MN-major), into the dP^T columns.
          // Issued before dK so that the drain of dQ overlaps dK.
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            mma_ss_warp(t_dP, desc_add(ds_mn, kk * 2048), desc_add(k_mn, kk * 2048), id_dq,
                   kk > 0 ? 1u : 0u);
          mma_commit_warp(&s.dq_full);
          // dK += dS^T Q  (A = dS^T: the same shared rows = keys, queries contiguous
          //               -> K-major; B = Q rows, MN-major over d)
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss_warp(t_dK, desc_add(ds_kmaj, off), desc_add(q_mn0, so + kk * 2048), id_acc,
                        (it > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_warp(&s.q_empty[st]);
        }
        if (!ok) break;
        mma_commit_warp(&s.dkv_full);
        mma_commit_warp(&s.kv_empty);  // the unit's last MMA has read K and V
        ++uk;
      }
      if (warp_aborted(abort_flag)) {
        mma_commit_warp(&s.drain);
        mbar_drain(&s.drain, 0, kSiteDrain);
      }
    }
  } else if (warp < 8) {
    // ---------------------------------------------------- compute warps --
    const int grp = warp & 3;           // TMEM lane group
    const int hf = warp >> 2;           // query columns [64 hf, 64 hf + 64)
    const int row = grp * 32 + lane;    // key row in the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(grp * 32) << 16;
    const float c = p.scale_log2;
    const uint32_t ds_base = smem_u32(s.ds[0]);
    // dropout: the eight lanes of keys 8a..8a+7 share a Philox counter per
    // query (the key tile starts on a multiple of 8 keys); lane (l & 7) of the
    // group draws query t = l & 7 of each block of 8, and eight ballots (one
    // per key of the group) hand every lane its own key's bits
    const uint32_t grp8 = static_cast<uint32_t>(lane & ~7);
    const uint32_t kix = static_cast<uint32_t>(lane & 7);  // this lane's key in its group
    int ig = 0, uk = 0;  // iterations and units with work, across the CTA's units
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
      const int U = unit_index(k);
      if (U >= n_units) continue;
      const BwdUnit un = bwd_unit_at(p, U);
      if (!un.exists) continue;
      const int c0 = un.c0, klo = un.klo, kend = un.kend, kseq = un.kseq, sq = un.sq;
      const int qb = un.qb, bz = un.bz, off = un.off, qt_lo = un.qt_lo, n_qt = un.n_qt;
      const int n_it = un.n_it, hk = un.hk;
      const int key = c0 + row;
      bool key_in = key >= klo && key < kend;
      if (p.key_bits && key_in) {
        const uint32_t w = __ldg(p.key_bits + static_cast<size_t>(bz) * p.mask_words + key / 32);
        key_in = (w >> (key & 31)) & 1u;
      }
      const uint32_t key8 = static_cast<uint32_t>(key) >> 3;
      for (int it = 0; it < n_it; ++it) {
        const int gi = ig + it;  // this iteration's index across units (barrier phases)
        const int g = it / n_qt;
        const int q0 = (qt_lo + it % n_qt) * kTileM;
        const int h = hk * p.group + g;
        // Row statistics of this query tile, staged by the hf = 0 warps in the
        // buffer of this tile's parity.  A buffer is rewritten two tiles later,
        // after every compute warp has signalled dS of the tile that read it
        // (S^T of the next tile is issued only after that).
        const int sb = gi & 1;
        if (hf == 0) {
          // stored negated so that p = 2^(s*c + nl) and dP - D = dP + nd are one
          // packed FMA / add per pair; rows without keys get nl = -inf (p = 0)
          const int qi = q0 + row;
          float nl = neg_inf(), nd = 0.f;
          if (qi < sq) {
            const size_t ri = (static_cast<size_t>(bz) * p.Hq + h) * p.Sq + qb + qi;
            const float lse = p.lse[ri];
            nl = (lse == neg_inf()) ? neg_inf() : -lse * 1.4426950408889634f;
            nd = -p.delta[ri];
          }
          s.nlse2[sb][row] = nl;
          s.ndelta[sb][row] = nd;
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.stat_ready[sb]);
        }
        if (!mbar_wait_warp(&s.stat_ready[sb], (gi >> 1) & 1, abort_flag, kSiteStat)) { ok = false; break; }
        const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(s.nlse2[sb]);
        const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(s.ndelta[sb]);
        const uint64_t c2 = f2_pack(c, c);
        // visible queries of this key row: q >= key - off (causal), key in [klo, kend)
        const int qmin = p.causal ? key - off : -0x7fffffff;
        const bool need_mask = !key_in || (p.causal && q0 + hf * 64 < qmin);
        if (!mbar_wait_warp(&s.s_full, gi & 1, abort_flag, kSiteS)) { ok = false; break; }
        tc_fence_after();
        uint32_t pk[32];  // this half's P^T, bf16 pairs
        uint32_t keepw[2] = {~0u, ~0u};  // dropout: bit q = query hf*64 + 32 cc + q kept
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sr[32];
          tmem_ld32(t_S + lane_off + hf * 64 + cc * 32, sr);
          if (DROP) {
            const uint32_t bh = static_cast<uint32_t>(bz * p.Hq + h);
            uint32_t kw = 0;
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              const uint32_t qi = static_cast<uint32_t>(q0 + hf * 64 + cc * 32 + g8 * 8) + kix;
              const uint32_t k8 = dropout_keep8(p.drop, key8, qi, bh);
              // bit L of bt[t]: key 8 (L / 8) + t kept for the query lane L drew
              uint32_t bt[8];
#pragma unroll
              for (int t = 0; t < 8; ++t) bt[t] = __ballot_sync(0xffffffffu, (k8 >> t) & 1u);
              const uint32_t s0 = (kix & 1) ? bt[1] : bt[0];
              const uint32_t s1 = (kix & 1) ? bt[3] : bt[2];
              const uint32_t s2 = (kix & 1) ? bt[5] : bt[4];
              const uint32_t s3 = (kix & 1) ? bt[7] : bt[6];
              const uint32_t sel = (kix & 4) ? ((kix & 2) ? s3 : s2) : ((kix & 2) ? s1 : s0);
              kw |= ((sel >> grp8) & 0xFFu) << (8 * g8);
            }
            keepw[cc] = kw;
          }
          tmem_wait_ld();
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int qa = hf * 64 + cc * 32 + 2 * e;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), c2,
                             nl2[qa >> 1]),
                      x0, x1);
            float p0 = ex2_approx(x0);
            float p1 = ex2_approx(x1);
            if (need_mask) {
              if (!key_in || q0 + qa < qmin) p0 = 0.f;
              if (!key_in || q0 + qa + 1 < qmin) p1 = 0.f;
            }
            pk[cc * 16 + e] = pack_bf16x2(p0, p1);
            pw[e] = pk[cc * 16 + e];
            if (DROP) {
              const uint32_t kb = keepw[cc] >> (2 * e);
              pw[e] &= ((kb & 1u) ? 0x0000ffffu : 0u) | ((kb & 2u) ? 0xffff0000u : 0u);
            }
          }
          // P columns [64 hf + 16 cc, +16) hold scores this warp already loaded
          tmem_st16(t_S + lane_off + hf * 64 + cc * 16, pw);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full);
        // dS^T = P^T * (dP^T - D)
        if (!mbar_wait_warp(&s.dp_full, gi & 1, abort_flag, kSiteDP)) { ok = false; break; }
        tc_fence_after();
        const uint32_t blk = ds_base + hf * (kTileN * 128) + row * 128;  // query block hf
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t dr[32];
          tmem_ld32(t_dP + lane_off + hf * 64 + cc * 32, dr);
          tmem_wait_ld();
          uint32_t dw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int qa = hf * 64 + cc * 32 + 2 * e;
            uint64_t dp2;
            if (DROP) {  // dP of the dropped weights: keep / (1 - p) * <dO, v>
              const uint32_t kb = keepw[cc] >> (2 * e);
              dp2 = f2_fma(f2_pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])),
                           f2_pack((kb & 1u) ? p.drop.scale : 0.f, (kb & 2u) ? p.drop.scale : 0.f),
                           nd2[qa >> 1]);
            } else {
              dp2 = f2_add(f2_pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])),
                           nd2[qa >> 1]);
            }
            float d0, d1;
            f2_unpack(f2_mul(bf16x2_to_f2(pk[cc * 16 + e]), dp2), d0, d1);
            dw[e] = pack_bf16x2(d0, d1);
          }
          // dS^T to shared memory only: 32 queries = four 16-byte chunks of query block hf
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t chunk = static_cast<uint32_t>((cc * 4 + ch) ^ (row & 7));
            st_shared_v4(blk + chunk * 16, dw[4 * ch], dw[4 * ch + 1], dw[4 * ch + 2], dw[4 * ch + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.ds_full);
      }
      // ---- epilogue: dK = scale * acc, dV = acc for head-dim columns
      //      [D/2 hf, D/2 hf + D/2)  (zeros when no query sees the keys)
      if (!ok) break;
      if (n_it > 0 && !mbar_wait_warp(&s.dkv_full, uk & 1, abort_flag, kSiteDKV)) break;
      tc_fence_after();
      if (warp_aborted(abort_flag)) break;
      // warp-uniform: the TMEM loads below are warp-collective, only the stores
      // depend on the lane's key
      {
        const bool store = key < kseq;
        const size_t kr = (static_cast<size_t>(bz) * p.Hkv + hk) * p.Sk + key;
        __nv_bfloat16* dkrow = reinterpret_cast<__nv_bfloat16*>(p.dk) + kr * D;
        __nv_bfloat16* dvrow = reinterpret_cast<__nv_bfloat16*>(p.dv) + kr * D;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          const uint32_t src = (pass == 0) ? t_dK : t_dV;
          const float mul = (pass == 0) ? p.scale : (DROP ? p.drop.scale : 1.f);
          __nv_bfloat16* dst = (pass == 0) ? dkrow : dvrow;
#pragma unroll
          for (int c2i = 0; c2i < D / 64; ++c2i) {
            const int cc = hf * (D / 64) + c2i;  // 32-column chunk of the head dimension
            uint32_t r[32];
            if (n_it > 0) {
              tmem_ld32(src + lane_off + cc * 32, r);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = 0u;
            }
            uint32_t pw[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pw[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
            if (store) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                d4[e] = make_uint4(pw[4 * e], pw[4 * e + 1], pw[4 * e + 2], pw[4 * e + 3]);
            }
          }
        }
      }
      if (n_it > 0) {
        // dK and dV have been read: the next unit's first products may overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.dkv_empty);
        ig += n_it;
        ++uk;
      }
    }
  } else if (warp < 12) {
    // --------------------------------------------- dQ drain (warps 8-11) --
    // Each warp moves its 32 query rows of dQ from TMEM to global memory with
    // TMA reduce-adds through its own 8 KB of staging (two 32x32 fp32 boxes,
    // 128-byte swizzle).  With d = 128 the row is staged in two halves: the
    // first 64 columns go to shared memory and the last 64 are held in
    // registers, so TMEM is released after one pass; the second half waits
    // only for the first half's reduces to have read the staging.
    const int wq = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    unsigned char* region = reinterpret_cast<unsigned char*>(&s.dq_stage[wq][0][0]);
    const uint32_t region_u32 = smem_u32(region);
    auto stage_64 = [&](const uint32_t (&r0)[32], const uint32_t (&r1)[32]) {
      const uint32_t b0 = region_u32 + lane * 128, b1 = region_u32 + 4096 + lane * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        st_shared_v4(b0 + ((ch ^ (lane & 7)) * 16), r0[4 * ch], r0[4 * ch + 1], r0[4 * ch + 2], r0[4 * ch + 3]);
        st_shared_v4(b1 + ((ch ^ (lane & 7)) * 16), r1[4 * ch], r1[4 * ch + 1], r1[4 * ch + 2], r1[4 * ch + 3]);
      }
    };
    int ig = 0;  // iterations across the CTA's units (barrier phases)
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_units; ++k) {
      const int U = unit_index(k);
      if (U >= n_units) continue;
      const BwdUnit un = bwd_unit_at(p, U);
      if (!un.exists || un.n_it == 0) continue;
      for (int it = 0; it < un.n_it; ++it, ++ig) {
        const int g = it / un.n_qt;
        const int q0 = (un.qt_lo + it % un.n_qt) * kTileM;
        const int h = un.hk * p.group + g;
        const int row = un.qb + q0 + wq * 32;
        const int zz = un.bz * p.Hq + h;
        if (!mbar_wait_warp(&s.dq_full, ig & 1, abort_flag, kSiteDQFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(t_dP + lane_off, r0);
        tmem_ld32(t_dP + lane_off + 32, r1);
        tmem_wait_ld();
        // the previous tile's reduces must have read the staging (waiting at
        // the end of that tile instead measured slower)
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        stage_64(r0, r1);
        if constexpr (D == 128) {
          tmem_ld32(t_dP + lane_off + 64, r0);
          tmem_ld32(t_dP + lane_off + 96, r1);
          tmem_wait_ld();
        }
        // dQ is out of TMEM: dP^T of the next tile may reuse the columns
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.dq_empty);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tdq, region, 0, row, zz);
          tma_reduce_add_3d(&tdq, region + 4096, 32, row, zz);
          bulk_commit_group();
        }
        if constexpr (D == 128) {
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          stage_64(r0, r1);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tdq, region, 64, row, zz);
            tma_reduce_add_3d(&tdq, region + 4096, 96, row, zz);
            bulk_commit_group();
          }
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait0();  // reduces complete before the CTA leaves
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                         cudaStream_t stream) {
  constexpr size_t smem = sizeof(BwdSmem<D>);
  static_assert(smem <= 232448, "backward shared memory exceeds the per-CTA limit");
  const bool drop = p.drop.on != 0;
  // per-device kernel attribute: set on every call for the current device
  cudaError_t e = cudaFuncSetAttribute(drop ? fa_bwd_main<D, true> : fa_bwd_main<D, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
  const long long pre_threads = rows * (D / 8);
  fa_bwd_pre<D><<<static_cast<unsigned int>((pre_threads + 255) / 256), 256, 0, stream>>>(p, rows);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (shared memory allows one) over the unit list
  int dev = 0, n_sm = 0, l2_bytes = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess) return e;
  const long long l2 = std::max(1LL << 20, static_cast<long long>(l2_bytes));
  const long long units = static_cast<long long>(p.n_kt) * p.grid_b * p.Hkv;
  const unsigned int grid = static_cast<unsigned int>(std::min<long long>(units, n_sm));
  // Pairs per group.  A pair's dQ accumulators and Q/dO tiles take 8 bytes
  // per row and head-dim column of each of its query heads.  While all pairs
  // together stay within about twice L2 they form one group (the plain
  // key-tile-major walk, best balanced).  Beyond that L2 thrashes: a group
  // then holds about half of L2's worth of pairs, but at least three waves of
  // units so the walk's pairing of heavy and light units stays balanced, and
  // it is rounded to whole batch rows (or to a divisor of the KV heads), so
  // that the units of a group share one sequence length.
  BwdParams pu = p;
  {
    const long long pairs = static_cast<long long>(p.grid_b) * p.Hkv;
    const long long rows = p.cu_q ? static_cast<long long>(p.n_kt) * kTileN : p.Sq;
    const long long per_pair = std::max(1LL, 8LL * rows * D * p.group);
    long long g = pairs;
    if (per_pair > (2 * l2) / std::max(1LL, pairs)) {  // pairs * per_pair, without overflow
      const long long fit = std::max(1LL, (l2 / 2) / per_pair);
      const long long waves = (3LL * n_sm + p.n_kt - 1) / std::max(1, p.n_kt);
      const long long t = std::max(fit, waves);
      if (t >= p.Hkv) {
        g = static_cast<long long>(p.Hkv) * ((t + p.Hkv / 2) / p.Hkv);
      } else {
        g = 1;
        for (long long dv = t; dv >= 1; --dv)
          if (p.Hkv % dv == 0) {
            g = dv;
            break;
          }
      }
      g = std::min(pairs, std::max(1LL, g));
    }
    pu.unit_group = static_cast<int>(g);
  }
  if (grid > 0) {  // packed sequences that all lack keys: dQ stays zero
    hook_before(stream);
    if (drop)
      fa_bwd_main<D, true><<<grid, kThreads, smem, stream>>>(tq, tk, tv, tdo, tdq, pu);
    else
      fa_bwd_main<D, false><<<grid, kThreads, smem, stream>>>(tq, tk, tv, tdo, tdq, pu);
    hook_after(stream);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long long n4 = rows * D / 4;
  fa_bwd_convert<<<static_cast<unsigned int>((n4 + 255) / 256), 256, 0, stream>>>(p, n4);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                       cudaStream_t stream) {
  if (d == 128) return launch_bwd_d<128>(tq, tk, tv, tdo, tdq, p, stream);
  return launch_bwd_d<64>(tq, tk, tv, tdo, tdq, p, stream);
}

unsigned int read_bwd_status(bool clear) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_status, sizeof v);
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof z);
  }
  return v;
}

}  // namespace fa
