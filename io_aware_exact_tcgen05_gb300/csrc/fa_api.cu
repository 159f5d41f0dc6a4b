// fa_api.cu -- the extern "C" boundary of libfa.so (declared in include/fa.h):
// argument validation, TMA tensor-map encoding, workspace carving and kernel
// launch.  No device memory is allocated here; no device memory is read on the
// host (the calls stay asynchronous and capturable).
#include <cfloat>
#include <cmath>
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
ProfileHook& profile_hook() {
  static thread_local ProfileHook h;
  return h;
}
}  // namespace fa

namespace {

thread_local char g_detail[256] = "";

}  // namespace

namespace fa {
// Lets other translation units report a detail through fa_last_error_detail.
void set_error_detail(const char* text) { snprintf(g_detail, sizeof g_detail, "%s", text); }
}  // namespace fa

namespace {

fa_status fail(fa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof g_detail, fmt, ap);
  va_end(ap);
  return s;
}

fa_status ok() {
  g_detail[0] = '\0';
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device check: the kernels are built for sm_103a only.
fa_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  static int cached_major[64], cached_minor[64];
  static bool cached[64];
  if (dev < 0 || dev >= 64) return fail(FA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  if (!cached[dev]) {
    int ma = 0, mi = 0;
    cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev);
    cached_major[dev] = ma;
    cached_minor[dev] = mi;
    cached[dev] = true;
  }
  if (cached_major[dev] != 10 || cached_minor[dev] != 3)
    return fail(FA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, cached_major[dev], cached_minor[dev]);
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [heads, rows, d] bf16 tensor, 128-row x 64-column boxes, 128-byte swizzle;
// rows past the end of a head read as zero.
fa_status make_map(CUtensorMap* map, const void* base, long heads, long rows, int d) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(fa::kTileM), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FA_OK;
}

// [heads, rows, cols] 8-bit tensor, 128-row x 128-column (128-byte) boxes,
// 128-byte swizzle; out-of-range rows and columns read as zero.
fa_status make_map_u8(CUtensorMap* map, const void* base, long heads, long rows, long cols) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols),
                           static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (u8) failed (%d)", (int)r);
  return FA_OK;
}

// [heads, rows, d] fp32 tensor (the backward's dQ accumulator), 32-row x
// 32-column boxes (128 bytes wide), 128-byte swizzle; used as the target of
// TMA reduce-add, which skips rows past the end of a head.
fa_status make_map_acc(CUtensorMap* map, void* base, long heads, long rows, int d) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                           static_cast<cuuint64_t>(d) * 4 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (fp32) failed (%d)", (int)r);
  return FA_OK;
}

// Base-2 scale c = scale * log2(e) the kernels multiply scores by.  It is
// kept >= 2^-126 so that a masked score (-inf) still gives -inf * c = -inf
// (weight 0) when the caller's scale is 0; finite scores then give s * c far
// below fp32 resolution, i.e. the exactly uniform weights of scale 0.
float scale_log2_of(float scale) {
  const float c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  return std::max(c, FLT_MIN);
}

fa_status check_sizes(int B, int Hq, int Hkv, int Sq, int Sk, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1)
    return fail(FA_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d Hq=%d Hkv=%d Sq=%d Sk=%d)", B, Hq,
                Hkv, Sq, Sk);
  if (Hq % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "Hq (%d) %% Hkv (%d) != 0", Hq, Hkv);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension %d (want 64 or 128)", d);
  // TMA coordinates are int32 and the head count is a tensor-map extent
  const long long rows_q = 1LL * B * Hq * Sq, rows_k = 1LL * B * Hkv * Sk;
  if (rows_q >= (1LL << 31) || rows_k >= (1LL << 31))
    return fail(FA_ERR_INVALID_ARG, "tensor too large for 32-bit row indices");
  return FA_OK;
}

fa_status check_ptr(const void* p, const char* name, bool nullable = false) {
  if (!p) return nullable ? FA_OK : fail(FA_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(FA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return FA_OK;
}

fa_status check_i32(const void* p, const char* name) {
  if (p && (reinterpret_cast<uintptr_t>(p) & 3u))
    return fail(FA_ERR_INVALID_ARG, "%s is not 4-byte aligned", name);
  return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

#define FA_TRY(expr)                 \
  do {                               \
    fa_status _s = (expr);           \
    if (_s != FA_OK) return _s;      \
  } while (0)

// Where a launch's rows and keys come from: the batched layout (grid batch
// = B, optional per-batch key interval) or packed ragged sequences.
struct SeqLayout {
  int grid_b;          // B, or the sequence count
  int longest_q;       // rows of the longest unit (Sq, or max_seqlen_q)
  int longest_k;       // keys of the longest unit (Sk, or max_seqlen_k)
  const int32_t* k_start;
  const int32_t* k_end;
  const int32_t* cu_q;
  const int32_t* cu_k;
};

fa_status varlen_layout(const int32_t* cu_q, const int32_t* cu_k, int nseq, int max_q, int max_k,
                        int total_q, int total_k, SeqLayout* lay) {
  if (!cu_q || !cu_k) return fail(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k are required");
  FA_TRY(check_i32(cu_q, "cu_seqlens_q"));
  FA_TRY(check_i32(cu_k, "cu_seqlens_k"));
  if (nseq < 1) return fail(FA_ERR_INVALID_ARG, "nseq (%d) must be >= 1", nseq);
  if (max_q < 1 || max_k < 0 || max_q > total_q || max_k > total_k)
    return fail(FA_ERR_INVALID_ARG,
                "max_seqlen_q=%d max_seqlen_k=%d must lie in [1, total_q=%d] and [0, total_k=%d]",
                max_q, max_k, total_q, total_k);
  lay->grid_b = nseq;
  lay->longest_q = max_q;
  lay->longest_k = max_k;
  lay->cu_q = cu_q;
  lay->cu_k = cu_k;
  return FA_OK;
}

fa_status check_key_bits(const uint32_t* bits) {
  if (bits && !aligned16(bits))
    return fail(FA_ERR_INVALID_ARG, "key_mask_bits is not 16-byte aligned");
  return FA_OK;
}

// Dropout arguments from the caller's probability, seed and offset: keep a
// weight iff its 16-bit Philox draw is >= thr = floor(p * 2^16) (computed in
// double, the same integer threshold the reference computation uses); kept
// weights are scaled by 2^16 / (2^16 - thr), the reciprocal of the keep
// probability, so the dropped output is unbiased.
fa_status make_dropout(float p_drop, unsigned long long seed, unsigned int offset,
                       fa::DropoutArgs* out) {
  if (!(p_drop >= 0.f && p_drop < 1.f))
    return fail(FA_ERR_INVALID_ARG, "dropout_p (%g) must lie in [0, 1)", (double)p_drop);
  fa::DropoutArgs dr{};
  const uint32_t thr = static_cast<uint32_t>(std::floor(static_cast<double>(p_drop) * 65536.0));
  dr.thr_hi = thr << 16;
  dr.on = p_drop > 0.f ? 1u : 0u;
  dr.seed_lo = static_cast<uint32_t>(seed & 0xffffffffull);
  dr.seed_hi = static_cast<uint32_t>(seed >> 32);
  dr.offset = offset;
  dr.scale = static_cast<float>(65536.0 / (65536.0 - static_cast<double>(thr)));
  *out = dr;
  return FA_OK;
}

const fa::DropoutArgs kNoDropout{0u, 0u, 0u, 0u, 1.f, 0u};

fa_status fwd_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                     const SeqLayout& lay, const uint32_t* key_bits, const fa::DropoutArgs& drop,
                     cudaStream_t stream) {
  FA_TRY(check_ptr(q, "q"));
  FA_TRY(check_ptr(k, "k"));
  FA_TRY(check_ptr(v, "v"));
  FA_TRY(check_ptr(o, "o"));
  FA_TRY(check_ptr(lse, "lse", true));
  FA_TRY(check_key_bits(key_bits));
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(FA_ERR_INVALID_ARG, "scale (%g) must be finite and >= 0", (double)scale);
  FA_TRY(check_device());

  CUtensorMap tq, tk, tv;
  FA_TRY(make_map(&tq, q, 1L * B * Hq, Sq, d));
  FA_TRY(make_map(&tk, k, 1L * B * Hkv, Sk, d));
  FA_TRY(make_map(&tv, v, 1L * B * Hkv, Sk, d));

  fa::FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.k_start = lay.k_start;
  p.k_end = lay.k_end;
  p.cu_q = lay.cu_q;
  p.cu_k = lay.cu_k;
  p.key_bits = key_bits;
  p.mask_words = static_cast<int>(fa_key_mask_words(Sk));
  p.drop = drop;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.group = Hq / Hkv;
  p.pack_heads = (p.group % 2 == 0) ? 1 : 0;
  const int n_rb = (lay.longest_q + fa::kTileM - 1) / fa::kTileM;
  if (p.pack_heads) {
    p.n_rbu = n_rb;
    p.units_per_rbu = lay.grid_b * (Hq / 2);
  } else {
    p.n_rbu = (n_rb + 1) / 2;
    p.units_per_rbu = lay.grid_b * Hq;
  }
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale_log2_of(scale);
  p.rescale_log2 = 8.0f;
  if (1LL * p.n_rbu * p.units_per_rbu >= (1LL << 31))
    return fail(FA_ERR_INVALID_ARG, "grid too large");
  cudaError_t e = fa::launch_fwd(d, tq, tk, tv, p, stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "fa_fwd launch: %s", cudaGetErrorString(e));
  return ok();
}

fa_status bwd_launch(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                     int Sq, int Sk, int d, int causal, float scale, const SeqLayout& lay,
                     const uint32_t* key_bits, const fa::DropoutArgs& drop, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_ptr(q, "q"));
  FA_TRY(check_ptr(k, "k"));
  FA_TRY(check_ptr(v, "v"));
  FA_TRY(check_ptr(o, "o"));
  FA_TRY(check_ptr(dout, "dout"));
  FA_TRY(check_ptr(lse, "lse"));
  FA_TRY(check_ptr(dq, "dq"));
  FA_TRY(check_ptr(dk, "dk"));
  FA_TRY(check_ptr(dv, "dv"));
  FA_TRY(check_key_bits(key_bits));
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(FA_ERR_INVALID_ARG, "scale (%g) must be finite and >= 0", (double)scale);
  const size_t need = fa_bwd_workspace_size(B, Hq, Sq, d);
  if (!workspace || workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "backward workspace needs %zu bytes, got %zu", need,
                workspace ? workspace_bytes : size_t(0));
  FA_TRY(check_ptr(workspace, "workspace"));
  FA_TRY(check_device());

  CUtensorMap tq, tk, tv, tdo;
  FA_TRY(make_map(&tq, q, 1L * B * Hq, Sq, d));
  FA_TRY(make_map(&tk, k, 1L * B * Hkv, Sk, d));
  FA_TRY(make_map(&tv, v, 1L * B * Hkv, Sk, d));
  FA_TRY(make_map(&tdo, dout, 1L * B * Hq, Sq, d));

  fa::BwdParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  const size_t rows = static_cast<size_t>(B) * Hq * Sq;
  p.dq_acc = static_cast<float*>(workspace);
  p.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                     align256(rows * d * sizeof(float)));
  p.k_start = lay.k_start;
  p.k_end = lay.k_end;
  p.cu_q = lay.cu_q;
  p.cu_k = lay.cu_k;
  p.key_bits = key_bits;
  p.mask_words = static_cast<int>(fa_key_mask_words(Sk));
  p.drop = drop;
  p.grid_b = lay.grid_b;
  p.n_kt = (lay.longest_k + fa::kTileN - 1) / fa::kTileN;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.group = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale_log2_of(scale);
  if (1LL * p.n_kt * p.grid_b * Hkv >= (1LL << 31))
    return fail(FA_ERR_INVALID_ARG, "grid too large");
  CUtensorMap tdq;
  FA_TRY(make_map_acc(&tdq, p.dq_acc, 1L * B * Hq, Sq, d));
  cudaError_t e = fa::launch_bwd(d, tq, tk, tv, tdo, tdq, p, stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "fa_bwd launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int Sq, int Sk, int d, int causal, float scale,
                 const int32_t* k_start, const int32_t* k_end, cudaStream_t stream) {
  return fa_fwd_masked(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, k_start, k_end,
                       nullptr, stream);
}

fa_status fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                        const int32_t* k_start, const int32_t* k_end,
                        const uint32_t* key_mask_bits, cudaStream_t stream) {
  FA_TRY(check_sizes(B, Hq, Hkv, Sq, Sk, d));
  FA_TRY(check_i32(k_start, "k_start"));
  FA_TRY(check_i32(k_end, "k_end"));
  SeqLayout lay{};
  lay.grid_b = B;
  lay.longest_q = Sq;
  lay.longest_k = Sk;
  lay.k_start = k_start;
  lay.k_end = k_end;
  return fwd_launch(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, lay, key_mask_bits,
                    kNoDropout, stream);
}

fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                         const int32_t* k_start, const int32_t* k_end,
                         const uint32_t* key_mask_bits, float dropout_p,
                         unsigned long long seed, unsigned int offset, cudaStream_t stream) {
  FA_TRY(check_sizes(B, Hq, Hkv, Sq, Sk, d));
  FA_TRY(check_i32(k_start, "k_start"));
  FA_TRY(check_i32(k_end, "k_end"));
  fa::DropoutArgs dr{};
  FA_TRY(make_dropout(dropout_p, seed, offset, &dr));
  SeqLayout lay{};
  lay.grid_b = B;
  lay.longest_q = Sq;
  lay.longest_k = Sk;
  lay.k_start = k_start;
  lay.k_end = k_end;
  return fwd_launch(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, lay, key_mask_bits,
                    dr, stream);
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, int causal, float scale, const uint32_t* key_mask_bits,
                        cudaStream_t stream) {
  FA_TRY(check_sizes(1, Hq, Hkv, total_q, total_k, d));
  SeqLayout lay{};
  FA_TRY(varlen_layout(cu_seqlens_q, cu_seqlens_k, nseq, max_seqlen_q, max_seqlen_k, total_q,
                       total_k, &lay));
  return fwd_launch(q, k, v, o, lse, 1, Hq, Hkv, total_q, total_k, d, causal, scale, lay,
                    key_mask_bits, kNoDropout, stream);
}

size_t fa_decode_workspace_size(int B, int Hq, int Sk_max, int d) {
  if (B < 1 || Hq < 1 || Sk_max < 1 || d < 1) return 0;
  int chunk = 0, n_split = 0;
  fa::decode_plan(B, Hq, 1, Sk_max, &chunk, &n_split);
  const size_t rows = static_cast<size_t>(B) * Hq * n_split;
  return align256(rows * d * sizeof(float)) + align256(rows * sizeof(float));
}

fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    const int32_t* seqlens_k, int B, int Hq, int Hkv, int Sk_max, int d,
                    float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_sizes(B, Hq, Hkv, 1, Sk_max, d));
  FA_TRY(check_ptr(q, "q"));
  FA_TRY(check_ptr(k_cache, "k_cache"));
  FA_TRY(check_ptr(v_cache, "v_cache"));
  FA_TRY(check_ptr(o, "o"));
  FA_TRY(check_ptr(lse, "lse", true));
  if (!seqlens_k) return fail(FA_ERR_INVALID_ARG, "seqlens_k is NULL");
  FA_TRY(check_i32(seqlens_k, "seqlens_k"));
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(FA_ERR_INVALID_ARG, "scale (%g) must be finite and >= 0", (double)scale);
  const size_t need = fa_decode_workspace_size(B, Hq, Sk_max, d);
  if (!workspace || workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "decode workspace needs %zu bytes, got %zu", need,
                workspace ? workspace_bytes : size_t(0));
  FA_TRY(check_ptr(workspace, "workspace"));
  FA_TRY(check_device());

  fa::DecodeParams p{};
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.o = o;
  p.lse = lse;
  p.seqlens = seqlens_k;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sk_max = Sk_max;
  p.group = Hq / Hkv;
  fa::decode_plan(B, Hq, Hkv, Sk_max, &p.chunk, &p.n_split);
  const size_t rows = static_cast<size_t>(B) * Hq * p.n_split;
  p.part_o = static_cast<float*>(workspace);
  p.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        align256(rows * d * sizeof(float)));
  p.scale_log2 = scale_log2_of(scale);
  if (p.n_split > 65535 * 64 || 1LL * B > 65535)
    return fail(FA_ERR_INVALID_ARG, "decode grid too large");
  cudaError_t e = fa::launch_decode(d, p, stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "fa_decode launch: %s", cudaGetErrorString(e));
  return ok();
}

size_t fa_bwd_workspace_size(int B, int Hq, int Sq, int d) {
  if (B < 1 || Hq < 1 || Sq < 1 || d < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * Sq;
  return align256(rows * d * sizeof(float)) + align256(rows * sizeof(float));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
                 int Sk, int d, int causal, float scale, const int32_t* k_start,
                 const int32_t* k_end, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
  return fa_bwd_masked(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
                       k_start, k_end, nullptr, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_masked(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                        const int32_t* k_start, const int32_t* k_end,
                        const uint32_t* key_mask_bits, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  FA_TRY(check_sizes(B, Hq, Hkv, Sq, Sk, d));
  FA_TRY(check_i32(k_start, "k_start"));
  FA_TRY(check_i32(k_end, "k_end"));
  SeqLayout lay{};
  lay.grid_b = B;
  lay.longest_q = Sq;
  lay.longest_k = Sk;
  lay.k_start = k_start;
  lay.k_end = k_end;
  return bwd_launch(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale, lay,
                    key_mask_bits, kNoDropout, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                         const int32_t* k_start, const int32_t* k_end,
                         const uint32_t* key_mask_bits, float dropout_p,
                         unsigned long long seed, unsigned int offset, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_sizes(B, Hq, Hkv, Sq, Sk, d));
  FA_TRY(check_i32(k_start, "k_start"));
  FA_TRY(check_i32(k_end, "k_end"));
  fa::DropoutArgs dr{};
  FA_TRY(make_dropout(dropout_p, seed, offset, &dr));
  SeqLayout lay{};
  lay.grid_b = B;
  lay.longest_q = Sq;
  lay.longest_k = Sk;
  lay.k_start = k_start;
  lay.k_end = k_end;
  return bwd_launch(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale, lay,
                    key_mask_bits, dr, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, int causal, float scale, const uint32_t* key_mask_bits,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  FA_TRY(check_sizes(1, Hq, Hkv, total_q, total_k, d));
  SeqLayout lay{};
  FA_TRY(varlen_layout(cu_seqlens_q, cu_seqlens_k, nseq, max_seqlen_q, max_seqlen_k, total_q,
                       total_k, &lay));
  return bwd_launch(q, k, v, o, dout, lse, dq, dk, dv, 1, Hq, Hkv, total_q, total_k, d, causal,
                    scale, lay, key_mask_bits, kNoDropout, workspace, workspace_bytes, stream);
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                     float q_descale, float k_descale, float v_descale, const int32_t* k_start,
                     const int32_t* k_end, cudaStream_t stream) {
  FA_TRY(check_sizes(B, Hq, Hkv, Sq, Sk, d));
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "fa_fwd_fp8 supports d = 128 only (got %d)", d);
  if (Sk % 16 != 0)
    return fail(FA_ERR_INVALID_ARG, "fa_fwd_fp8 needs Sk %% 16 == 0 (rows of V^T are Sk bytes)");
  FA_TRY(check_ptr(q, "q"));
  FA_TRY(check_ptr(k, "k"));
  FA_TRY(check_ptr(vt, "vt"));
  FA_TRY(check_ptr(o, "o"));
  FA_TRY(check_ptr(lse, "lse", true));
  FA_TRY(check_i32(k_start, "k_start"));
  FA_TRY(check_i32(k_end, "k_end"));
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(FA_ERR_INVALID_ARG, "scale (%g) must be finite and >= 0", (double)scale);
  for (float ds : {q_descale, k_descale, v_descale})
    if (!std::isfinite(ds) || !(ds > 0.f))
      return fail(FA_ERR_INVALID_ARG, "descale factors must be finite and > 0");
  FA_TRY(check_device());
  CUtensorMap tq, tk, tvt;
  FA_TRY(make_map_u8(&tq, q, 1L * B * Hq, Sq, d));
  FA_TRY(make_map_u8(&tk, k, 1L * B * Hkv, Sk, d));
  FA_TRY(make_map_u8(&tvt, vt, 1L * B * Hkv, d, Sk));  // [d rows, Sk columns] per head
  fa::Fp8FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.k_start = k_start;
  p.k_end = k_end;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.group = Hq / Hkv;
  p.pack_heads = (p.group % 2 == 0) ? 1 : 0;
  const int n_rb = (Sq + fa::kTileM - 1) / fa::kTileM;
  p.n_rbu = p.pack_heads ? n_rb : (n_rb + 1) / 2;
  p.units_per_rbu = p.pack_heads ? B * (Hq / 2) : B * Hq;
  p.causal = causal ? 1 : 0;
  const double qk = static_cast<double>(scale) * q_descale * k_descale;
  p.scale_qk = static_cast<float>(qk);
  p.scale_log2 = scale_log2_of(static_cast<float>(qk));
  // e4m3 tops out at 448: the running max moves once the tile max exceeds
  // it by more than 2^8, so every weight stays <= 256
  p.rescale_log2 = 8.0f;
  p.v_descale = v_descale;
  if (1LL * p.n_rbu * p.units_per_rbu >= (1LL << 31))
    return fail(FA_ERR_INVALID_ARG, "grid too large");
  cudaError_t e = fa::launch_fwd_fp8(tq, tk, tvt, p, stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "fa_fwd_fp8 launch: %s", cudaGetErrorString(e));
  return ok();
}

size_t fa_key_mask_words(int Sk) {
  if (Sk < 1) return 0;
  return static_cast<size_t>((Sk + fa::kTileN - 1) / fa::kTileN) * (fa::kTileN / 32);
}

fa_status fa_pack_key_mask(const uint8_t* mask, uint32_t* bits, int rows, int Sk,
                           cudaStream_t stream) {
  if (rows < 1 || Sk < 1)
    return fail(FA_ERR_INVALID_ARG, "fa_pack_key_mask: rows=%d Sk=%d must be >= 1", rows, Sk);
  if (!mask) return fail(FA_ERR_INVALID_ARG, "fa_pack_key_mask: mask is NULL");
  FA_TRY(check_ptr(bits, "bits"));
  const size_t words = fa_key_mask_words(Sk);
  if (static_cast<double>(rows) * words * 32 >= 2147483648.0)
    return fail(FA_ERR_INVALID_ARG, "fa_pack_key_mask: mask too large");
  FA_TRY(check_device());
  cudaError_t e = fa::launch_pack_key_mask(mask, bits, rows, Sk, static_cast<int>(words), stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "fa_pack_key_mask launch: %s", cudaGetErrorString(e));
  return ok();
}

fa_status fa_device_status(unsigned int* code_out, int clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
  const unsigned int w = fa::read_fwd_status(clear != 0) | fa::read_decode_status(clear != 0) |
                         fa::read_bwd_status(clear != 0) | fa::read_fwd_fp8_status(clear != 0) |
                         fa::read_selftest_status(clear != 0);
  if (code_out) *code_out = w;
  if (w != 0) return fail(FA_ERR_TIMEOUT, "device status word 0x%08x", w);
  return ok();
}

fa_status fa_selftest_wait_timeout(unsigned int* result, cudaStream_t stream) {
  FA_TRY(check_ptr(result, "result"));
  FA_TRY(check_device());
  const cudaError_t e = fa::launch_selftest_wait(result, stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return ok();
}

fa_status fa_profile_next_launch(cudaEvent_t start, cudaEvent_t stop) {
  if ((start == nullptr) != (stop == nullptr))
    return fail(FA_ERR_INVALID_ARG, "pass both events or neither");
  fa::profile_hook().start = start;
  fa::profile_hook().stop = stop;
  return ok();
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device pipeline wait timed out";
  }
  return "unknown status";
}

const char* fa_last_error_detail(void) { return g_detail; }

const char* fa_version(void) { return "io_aware_exact_tcgen05_gb300 0.1 (sm_103a)"; }

}  // extern "C"
