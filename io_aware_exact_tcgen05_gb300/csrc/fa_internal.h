// fa_internal.h -- parameter blocks and launch entry points shared between
// the C-ABI layer (fa_api.cu) and the kernel translation units.  Host-side
// only declarations plus plain structs; no device code.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace fa {

// One-shot profiling events armed by fa_profile_next_launch (per host thread):
// the launch helpers record `start` right before and `stop` right after the
// main kernel of the next call, then clear them.
struct ProfileHook {
  cudaEvent_t start = nullptr;
  cudaEvent_t stop = nullptr;
};
ProfileHook& profile_hook();
inline void hook_before(cudaStream_t s) {
  if (profile_hook().start) cudaEventRecord(profile_hook().start, s);
}
inline void hook_after(cudaStream_t s) {
  if (profile_hook().stop) cudaEventRecord(profile_hook().stop, s);
  profile_hook() = ProfileHook{};
}

// Launch `kernel` as a programmatic dependent of the previous kernel in the
// stream: its launch overlaps that kernel's tail.  A kernel launched this
// way calls griddep_wait() before it touches memory the previous kernel may
// still use.  (Used for the decode merge; on the forward and backward
// kernels it measured -2% to +0.3%.)
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Tile-size and pipeline table.  Every tile shape, pipeline depth and split
// length of the kernels is read from here, per head dimension and kernel;
// each value is the one measured fastest on GB300 among the alternatives
// that fit the 227 KB of shared memory per CTA (and 512 TMEM columns).
// ---------------------------------------------------------------------------

// Rows of one query tile and keys of one key/value tile in the tensor-core
// kernels (one tcgen05.mma M=128 accumulator; 128 TMEM lanes).  Two query
// tiles ("slots") share each K/V tile in the forward: two S tiles and two O
// accumulators fill the 512 TMEM columns at d = 128.
constexpr int kTileM = 128;
constexpr int kTileN = 128;

// bf16 forward: K/V pipeline depth (stages of one 128-key K tile and V tile).
template <int D> struct FwdTiles;
template <> struct FwdTiles<128> { static constexpr int kKvStages = 2; };  // 3 needs 256 KB
template <> struct FwdTiles<64> { static constexpr int kKvStages = 3; };

// Backward main kernel: Q tile buffers (S^T(i+1) is issued before dK(i) has
// read Q(i), so two are needed); dO has one buffer.
template <int D> struct BwdTiles { static constexpr int kQStages = 2; };

// FP8 forward (d = 128): K / V^T pipeline depth.
struct Fp8Tiles { static constexpr int kKvStages = 4; };

// Decode: keys per pipeline stage, stages per CTA, and the longest split a
// CTA streams (shorter caches use shorter splits, see decode_plan).
struct DecodeTiles {
  static constexpr int kStageKeys = 128;
  static constexpr int kStages = 3;
  static constexpr int kMaxChunk = 4096;
};

// Dropout on the attention weights (see fa_philox.cuh for the mapping).
struct DropoutArgs {
  uint32_t thr_hi;   // floor(p * 2^16) << 16: the 16-bit threshold in the high half
  uint32_t seed_lo;
  uint32_t seed_hi;
  uint32_t offset;
  float scale;       // 2^16 / (2^16 - floor(p * 2^16)): 1 / the keep probability
  uint32_t on;       // p > 0
};

struct FwdParams {
  void* o;             // bf16 [B,Hq,Sq,d]
  float* lse;          // fp32 [B,Hq,Sq] or nullptr
  const int32_t* k_start;
  const int32_t* k_end;
  // Packed ragged sequences (B = 1, Sq/Sk = packed totals): sequence s owns
  // rows [cu_q[s], cu_q[s+1]) and keys [cu_k[s], cu_k[s+1]); the grid's batch
  // index is the sequence.  nullptr for the batched layout.
  const int32_t* cu_q;
  const int32_t* cu_k;
  // Optional key visibility bits: bit (j & 31) of word [row * mask_words + j / 32],
  // row = batch row (or 0 for packed keys); nullptr = every key visible.
  const uint32_t* key_bits;
  int mask_words;
  DropoutArgs drop;    // on == 0: no dropout
  int B, Hq, Hkv, Sq, Sk;
  int group;           // Hq / Hkv
  int pack_heads;      // 1: a CTA's two query tiles are two heads of one KV group
  int n_rbu;           // row-block units per (b, head unit)
  int units_per_rbu;   // (b, head unit) pairs
  int causal;
  float scale;         // natural-log softmax scale
  float scale_log2;    // scale * log2(e)
  float rescale_log2;  // skip the O rescale unless the max grows by more than this (log2 units)
};

// Launch the forward kernel for head dimension d (64 or 128).
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream);
unsigned int read_fwd_status(bool clear);

// FP8 (e4m3) forward: the batched layout, key interval, causal rule and GQA
// of FwdParams; Q, K and V^T are e4m3 with per-tensor dequantisation factors.
struct Fp8FwdParams {
  void* o;             // bf16 [B,Hq,Sq,128]
  float* lse;          // fp32 [B,Hq,Sq] or nullptr
  const int32_t* k_start;
  const int32_t* k_end;
  int B, Hq, Hkv, Sq, Sk;
  int group;
  int pack_heads;
  int n_rbu;
  int units_per_rbu;
  int causal;
  float scale_qk;      // scale * q_descale * k_descale (natural log units)
  float scale_log2;    // scale_qk * log2(e), kept >= 2^-126
  float rescale_log2;
  float v_descale;
};

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const Fp8FwdParams& p, cudaStream_t stream);
unsigned int read_fwd_fp8_status(bool clear);

// Self-test of the bounded waits (fa_selftest.cu): result[0], result[1] are
// set to 1 when the two waits report failure.
cudaError_t launch_selftest_wait(unsigned int* result, cudaStream_t stream);
unsigned int read_selftest_status(bool clear);

struct DecodeParams {
  const void* q;        // bf16 [B,Hq,1,d]
  const void* k;        // bf16 [B,Hkv,Sk_max,d]
  const void* v;
  void* o;              // bf16 [B,Hq,1,d]
  float* lse;           // fp32 [B,Hq] or nullptr
  const int32_t* seqlens;
  float* part_o;        // fp32 [B,Hq,n_split,d]
  float* part_lse;      // fp32 [B,Hq,n_split]
  int B, Hq, Hkv, Sk_max, group;
  int chunk;            // keys per split
  int n_split;
  float scale_log2;
};

cudaError_t launch_decode(int d, const DecodeParams& p, cudaStream_t stream);
unsigned int read_decode_status(bool clear);
void decode_plan(int B, int Hq, int Hkv, int Sk_max, int* chunk, int* n_split);

struct BwdParams {
  const void* q;        // bf16 [B,Hq,Sq,d]
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;     // fp32 [B,Hq,Sq]
  void* dq;             // bf16 out
  void* dk;
  void* dv;
  float* dq_acc;        // fp32 [B,Hq,Sq,d] workspace
  float* delta;         // fp32 [B,Hq,Sq] workspace: D_i
  const int32_t* k_start;
  const int32_t* k_end;
  const int32_t* cu_q;     // packed ragged sequences, as in FwdParams (nullptr: batched)
  const int32_t* cu_k;
  const uint32_t* key_bits;  // optional key visibility bits, as in FwdParams
  int mask_words;
  DropoutArgs drop;          // the forward's dropout (on == 0: none)
  int grid_b;  // units along the grid's batch axis: B, or the sequence count when packed
  int n_kt;    // key tiles per unit: ceil(Sk / 128), or ceil(longest sequence's keys / 128)
  int unit_group;  // (batch or sequence, KV head) pairs walked together (set by the launcher)
  int B, Hq, Hkv, Sq, Sk, group;
  int causal;
  float scale;
  float scale_log2;
};

// bits[r][words] = packed (mask[r][Sk] != 0), zero past Sk.
cudaError_t launch_pack_key_mask(const uint8_t* mask, uint32_t* bits, int rows, int Sk, int words,
                                 cudaStream_t stream);

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                       const BwdParams& p,
                       cudaStream_t stream);
unsigned int read_bwd_status(bool clear);

}  // namespace fa
