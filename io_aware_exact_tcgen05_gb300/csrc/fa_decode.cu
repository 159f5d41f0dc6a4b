// fa_decode.cu -- single-query (Sq = 1) attention over a ragged, padded KV
// cache: split-KV partial kernel plus a logsumexp merge.
//
// Decode reads every cached key and value once and does about 4 flops per
// byte, so it is bound by HBM bandwidth, not by the tensor cores: it runs on
// the CUDA cores with the bytes staged through shared memory by 1-D bulk
// async copies (cp.async.bulk) in a 3-deep mbarrier ring.
//
// Partial kernel: one CTA per (split, KV head, batch row) streams keys
// [split*chunk, min((split+1)*chunk, seqlen)) of that KV head once and serves
// all the query heads that read it (grouped heads).  Each of the 8 compute
// warps takes 16 keys of every 128-key stage; a key row (d bf16) is spread over
// d/8 lanes (8 values each), so one warp instruction covers 32*8/d keys.  The
// per-key dot products with every query head are reduced across those lanes
// with a transpose-reduce (each exchange halves the heads a lane carries), then
// the online-softmax state (running max m, denominator l, unnormalised output)
// is updated per head.  Splits past the sequence end exit at once.
//
// Merge kernel: per (b, query head), LSE = log sum_s exp(LSE_s) and
// O = sum_s exp(LSE_s - LSE) O_s over the non-empty splits -- the rescale rule
// of the online softmax ("Flash Attention" history page 1.2) applied to
// whole per-chunk states.  Empty rows (seqlen 0) give O = 0, LSE = -inf.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;  // + 1 producer warp
constexpr int kStageKeys = DecodeTiles::kStageKeys;
constexpr int kStages = DecodeTiles::kStages;
constexpr int kMaxHeadsPerCta = 8;

enum : unsigned int { kSiteFull = 1, kSiteEmpty = 2, kSiteDrain = 3 };

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int D>
struct DecodeSmem {
  __nv_bfloat16 k[kStages][kStageKeys * D];
  __nv_bfloat16 v[kStages][kStageKeys * D];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort_flag;
};

// Reduce per-lane partial sums a[0..HG) across the LPK lanes of one key so that
// afterwards lane x (x = lane % LPK) holds the full sum for head head_of(x).
// Each exchange step with heads left > 1 halves the set of heads a lane keeps.
template <int HG, int LPK>
__device__ __forceinline__ float transpose_reduce(float (&a)[HG], int lane) {
  float cur[HG];
#pragma unroll
  for (int h = 0; h < HG; ++h) cur[h] = a[h];
  int n = HG;
#pragma unroll
  for (int o = LPK / 2; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool upper = (lane & o) != 0;
      const int half = n / 2;
#pragma unroll
      for (int h = 0; h < HG / 2; ++h) {
        if (h < half) {
          const float send = upper ? cur[h] : cur[h + half];
          const float keep = upper ? cur[h + half] : cur[h];
          cur[h] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      n = half;
    } else {
      cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], o);
    }
  }
  return cur[0];
}

// Head index held by lane x after transpose_reduce<HG, LPK>.
template <int HG, int LPK>
__device__ __forceinline__ int head_of(int x) {
  int h = 0, n = HG;
#pragma unroll
  for (int o = LPK / 2; o >= 1; o >>= 1) {
    if (n > 1) {
      n >>= 1;
      if (x & o) h += n;
    }
  }
  return h;
}

// First lane (within a key's LPK lanes) that holds head h.
template <int HG, int LPK>
__device__ __forceinline__ int lane_of_head(int h) {
  int x = 0, n = HG;
#pragma unroll
  for (int o = LPK / 2; o >= 1; o >>= 1) {
    if (n > 1) {
      n >>= 1;
      if (h >= n) {
        x |= o;
        h -= n;
      }
    }
  }
  return x;
}

template <int D, int HG>
__global__ void __launch_bounds__(kThreads, 1)
    fa_decode_partial(const DecodeParams p, int heads_per_cta) {
  constexpr int LPK = D / 8;          // lanes per key row (8 bf16 = 16 bytes per lane)
  constexpr int KPR = 32 / LPK;       // keys per warp instruction ("round")
  constexpr int KPW = kStageKeys / kComputeWarps;  // keys per warp per stage
  constexpr int ROUNDS = KPW / KPR;
  extern __shared__ unsigned char smem_raw[];
  DecodeSmem<D>& s = *reinterpret_cast<DecodeSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) +
                                                        127) & ~uintptr_t(127));
  const int split = blockIdx.x;
  const int hk = blockIdx.y / ((p.group + heads_per_cta - 1) / heads_per_cta);
  const int hsub = blockIdx.y % ((p.group + heads_per_cta - 1) / heads_per_cta);
  const int b = blockIdx.z;
  int seqlen = p.seqlens[b];
  seqlen = max(0, min(seqlen, p.Sk_max));
  const int key_begin = split * p.chunk;
  if (key_begin >= seqlen) return;  // empty split: the merge skips it
  const int n_keys = min(p.chunk, seqlen - key_begin);
  const int n_stages = (n_keys + kStageKeys - 1) / kStageKeys;
  const int hq0 = hk * p.group + hsub * heads_per_cta;
  const int n_heads = min(heads_per_cta, p.group - hsub * heads_per_cta);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kComputeWarps);
    }
    s.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &s.abort_flag;
  const size_t kv_row0 = (static_cast<size_t>(b) * p.Hkv + hk) * p.Sk_max + key_begin;

  // per-warp softmax states for the CTA-level merge; the per-warp outputs reuse
  // the K stage buffers once every stage has been consumed
  __shared__ float red_m[kComputeWarps][kMaxHeadsPerCta];
  __shared__ float red_l[kComputeWarps][kMaxHeadsPerCta];
  static_assert(sizeof(float) * kComputeWarps * HG * D <= sizeof(s.k), "merge area");
  float (*red_o)[HG][D] = reinterpret_cast<float (*)[HG][D]>(&s.k[0][0]);

  if (warp == kComputeWarps) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const __nv_bfloat16* kbase = reinterpret_cast<const __nv_bfloat16*>(p.k) + kv_row0 * D;
      const __nv_bfloat16* vbase = reinterpret_cast<const __nv_bfloat16*>(p.v) + kv_row0 * D;
      int issued = 0;
      for (int st = 0; st < n_stages; ++st) {
        const int slot = st % kStages;
        const int use = st / kStages;
        if (use > 0 && !mbar_wait(&s.empty[slot], (use - 1) & 1, abort_flag, kSiteEmpty)) break;
        const int nk = min(kStageKeys, n_keys - st * kStageKeys);
        const uint32_t bytes = static_cast<uint32_t>(nk) * D * 2;
        mbar_arrive_expect_tx(&s.full[slot], 2 * bytes);
        bulk_load(s.k[slot], kbase + static_cast<size_t>(st) * kStageKeys * D, bytes,
                  &s.full[slot]);
        bulk_load(s.v[slot], vbase + static_cast<size_t>(st) * kStageKeys * D, bytes,
                  &s.full[slot]);
        issued = st + 1;
      }
      if (*abort_flag)
        for (int st = max(0, issued - kStages); st < issued; ++st)
          mbar_drain(&s.full[st % kStages], (st / kStages) & 1, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------- compute --
    const int x = lane % LPK;          // this lane's 8-wide slice of d
    const int kr = lane / LPK;         // key within a round
    const int my_head = head_of<HG, LPK>(x);
    const float c = p.scale_log2;
    // query slices (fp32) for every head this CTA serves; padding heads are 0
    // query slices and output accumulators as fp32 pairs for the f32x2 FMA pipe;
    // padding heads get q = 0
    uint64_t qv2[HG][4];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      if (h < n_heads) {
        const uint4 w = *reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(p.q) +
            (static_cast<size_t>(b) * p.Hq + hq0 + h) * D + x * 8);
        qv2[h][0] = bf16x2_to_f2(w.x);
        qv2[h][1] = bf16x2_to_f2(w.y);
        qv2[h][2] = bf16x2_to_f2(w.z);
        qv2[h][3] = bf16x2_to_f2(w.w);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) qv2[h][e] = 0ull;
      }
    }
    uint64_t acc2[HG][4];
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2[h][e] = 0ull;
    float m = neg_inf();  // running max (raw score) of my_head over this warp's keys
    float l = 0.f;

    for (int st = 0; st < n_stages; ++st) {
      const int slot = st % kStages;
      if (!mbar_wait_warp(&s.full[slot], (st / kStages) & 1, abort_flag, kSiteFull)) break;
      const int stage_keys = min(kStageKeys, n_keys - st * kStageKeys);
      float sc[ROUNDS];
      uint4 vraw[ROUNDS];
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        const int key = warp * KPW + r * KPR + kr;
        const bool valid = key < stage_keys;
        uint4 kw = make_uint4(0u, 0u, 0u, 0u);
        vraw[r] = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
          kw = *reinterpret_cast<const uint4*>(&s.k[slot][key * D + x * 8]);
          vraw[r] = *reinterpret_cast<const uint4*>(&s.v[slot][key * D + x * 8]);
        }
        const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w};
        uint64_t part2[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) part2[h] = 0ull;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint64_t k2 = bf16x2_to_f2(kk[e]);
#pragma unroll
          for (int h = 0; h < HG; ++h) part2[h] = f2_fma(qv2[h][e], k2, part2[h]);
        }
        float part[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          float lo, hi;
          f2_unpack(part2[h], lo, hi);
          part[h] = lo + hi;
        }
        const float sfull = transpose_reduce<HG, LPK>(part, lane);
        sc[r] = valid ? sfull : neg_inf();
      }
      // ---- online softmax over this stage's keys, per head ----
      float mx = neg_inf();
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) mx = fmaxf(mx, sc[r]);
#pragma unroll
      for (int o = LPK; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m, mx);
      // the first finite max is always taken (also when c = 0); before it
      // nothing is accumulated, so its rescale factor is 0.  m_new - m is
      // formed only once m is finite, so -inf - (-inf) is never evaluated.
      const bool first = (m == neg_inf()) && (m_new != neg_inf());
      const bool grow = first || (m != neg_inf() && (m_new - m) * c > 0.f);
      if (__any_sync(0xffffffffu, grow)) {
        const float alpha = first ? 0.f : (grow ? ex2_approx((m - m_new) * c) : 1.f);
        l *= alpha;
        if (grow) m = m_new;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float ah = __shfl_sync(0xffffffffu, alpha, lane_of_head<HG, LPK>(h));
          const uint64_t ah2 = f2_pack(ah, ah);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[h][e] = f2_mul(acc2[h][e], ah2);
        }
      }
      const float mc = (m == neg_inf()) ? 0.f : m * c;
      float pr[ROUNDS];
      float lsum = 0.f;
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        pr[r] = ex2_approx(fmaf(sc[r], c, -mc));
        lsum += pr[r];
      }
#pragma unroll
      for (int o = LPK; o < 32; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
      l += lsum;
      // ---- O_h += p_h(key) * v(key) ----
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        const uint64_t v2[4] = {bf16x2_to_f2(vraw[r].x), bf16x2_to_f2(vraw[r].y),
                                bf16x2_to_f2(vraw[r].z), bf16x2_to_f2(vraw[r].w)};
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float ph =
              __shfl_sync(0xffffffffu, pr[r], (lane & ~(LPK - 1)) + lane_of_head<HG, LPK>(h));
          const uint64_t ph2 = f2_pack(ph, ph);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[h][e] = f2_fma(ph2, v2[e], acc2[h][e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[slot]);
    }
    float acc[HG][8];
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) f2_unpack(acc2[h][e], acc[h][2 * e], acc[h][2 * e + 1]);
    // ---- fold the key groups of the warp (lanes with equal x) ----
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1)
#pragma unroll
      for (int h = 0; h < HG; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
    __syncthreads();  // (A) every warp is done reading the stage buffers
    if (lane < LPK && !*abort_flag) {
#pragma unroll
      for (int h = 0; h < HG; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) red_o[warp][h][x * 8 + e] = acc[h][e];
      if (x == lane_of_head<HG, LPK>(my_head)) {
        red_m[warp][my_head] = m;
        red_l[warp][my_head] = l;
      }
    }
  }
  if (warp == kComputeWarps) __syncthreads();  // (A) for the producer warp
  __syncthreads();
  if (*abort_flag) return;
  // the merge kernel may launch now (it waits for this grid's completion)
  griddep_launch_dependents();
  // ---- merge the warps' states, write this split's normalised partial ----
  for (int idx = threadIdx.x; idx < n_heads * D; idx += kThreads) {
    const int h = idx / D;
    const int e = idx % D;
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, red_m[w][h]);
    float L = 0.f, o = 0.f;
    if (M != neg_inf()) {
      const float Mc = M * p.scale_log2;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) {
        const float mw = red_m[w][h];
        const float wt = (mw == neg_inf()) ? 0.f : ex2_approx(fmaf(mw, p.scale_log2, -Mc));
        L = fmaf(wt, red_l[w][h], L);
        o = fmaf(wt, red_o[w][h][e], o);
      }
    }
    const size_t pi = (static_cast<size_t>(b) * p.Hq + hq0 + h) * p.n_split + split;
    p.part_o[pi * D + e] = (L > 0.f) ? o / L : 0.f;
    if (e == 0)
      p.part_lse[pi] = (L > 0.f) ? (M * p.scale_log2 + __log2f(L)) : neg_inf();  // log2 units
  }
}

// One CTA per (b, query head), one thread per output element.
template <int D>
__global__ void __launch_bounds__(D) fa_decode_merge(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int e = threadIdx.x;
  int seqlen = p.seqlens[b];
  seqlen = max(0, min(seqlen, p.Sk_max));
  const int n_valid = min(p.n_split, (seqlen + p.chunk - 1) / p.chunk);
  const float* lse2 = p.part_lse + static_cast<size_t>(bh) * p.n_split;
  const float* po = p.part_o + static_cast<size_t>(bh) * p.n_split * D;
  griddep_wait();  // the partial kernel's results are complete and visible
  float M = neg_inf();
  for (int sidx = 0; sidx < n_valid; ++sidx) M = fmaxf(M, lse2[sidx]);
  float wsum = 0.f, o = 0.f;
  if (M != neg_inf()) {
    for (int sidx = 0; sidx < n_valid; ++sidx) {
      const float ls = lse2[sidx];
      const float w = (ls == neg_inf()) ? 0.f : ex2_approx(ls - M);
      wsum += w;
      o = fmaf(w, po[static_cast<size_t>(sidx) * D + e], o);
    }
  }
  const bool live = wsum > 0.f;
  reinterpret_cast<__nv_bfloat16*>(p.o)[static_cast<size_t>(bh) * D + e] =
      __float2bfloat16_rn(live ? o / wsum : 0.f);
  if (p.lse && e == 0)
    p.lse[bh] = live ? (M + __log2f(wsum)) * 0.69314718055994530942f : neg_inf();
}

template <int D, int HG>
cudaError_t launch_partial(const DecodeParams& p, int heads_per_cta, cudaStream_t stream) {
  const size_t smem = sizeof(DecodeSmem<D>) + 128;
  // per-device kernel attribute: set on every call for the current device
  cudaError_t e = cudaFuncSetAttribute(fa_decode_partial<D, HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int n_hsub = (p.group + heads_per_cta - 1) / heads_per_cta;
  dim3 grid(p.n_split, p.Hkv * n_hsub, p.B);
  hook_before(stream);
  fa_decode_partial<D, HG><<<grid, kThreads, smem, stream>>>(p, heads_per_cta);
  hook_after(stream);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, cudaStream_t stream) {
  const int heads = min(p.group, kMaxHeadsPerCta);
  cudaError_t e;
  if (heads <= 1) e = launch_partial<D, 1>(p, 1, stream);
  else if (heads <= 2) e = launch_partial<D, 2>(p, 2, stream);
  else if (heads <= 4) e = launch_partial<D, 4>(p, 4, stream);
  else e = launch_partial<D, 8>(p, 8, stream);
  if (e != cudaSuccess) return e;
  // The merge is launched as a programmatic dependent of the partial kernel,
  // so its launch overlaps the partial kernel's tail; it waits for the
  // partial results on the device (griddep_wait).
  return launch_dependent(fa_decode_merge<D>, static_cast<unsigned int>(p.B * p.Hq), D, 0, stream,
                          p);
}

}  // namespace

void decode_plan(int B, int Hq, int Hkv, int Sk_max, int* chunk, int* n_split) {
  (void)B;
  (void)Hq;
  (void)Hkv;
  // 4096 keys (2 MiB of K+V at d=128) per CTA: long streams per CTA amortise
  // the start-up and the per-split merge (measured on GB300: 512-key chunks
  // reached 4.1 TB/s, 4096-key chunks 6.1 TB/s); short caches use smaller
  // chunks so that a row still spreads over several CTAs.  Multiple of the
  // 128-key stage.
  int c = DecodeTiles::kMaxChunk;
  while (c > kStageKeys && Sk_max <= 4 * c) c >>= 1;
  *chunk = c;
  *n_split = (Sk_max + c - 1) / c;
}

cudaError_t launch_decode(int d, const DecodeParams& p, cudaStream_t stream) {
  if (d == 128) return launch_decode_d<128>(p, stream);
  return launch_decode_d<64>(p, stream);
}

unsigned int read_decode_status(bool clear) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_status, sizeof v);
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof z);
  }
  return v;
}

}  // namespace fa
