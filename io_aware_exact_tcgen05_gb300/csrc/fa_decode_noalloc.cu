// fa_decode_noalloc.cu -- fa_decode for callers that cannot allocate device
// memory themselves.
//
// fa_decode needs a scratch workspace for its per-split partial results.  Some
// callers cannot provide one: their interface carries only the input and
// output buffers (a fixed plugin or operator signature has no workspace
// slot), or allocation is not available to them where they run (a host
// framework that owns every byte of device memory through its own pool, or a
// latency-critical loop that cannot pay for cudaMalloc and its implicit
// device synchronisation).  This entry point serves them from a fixed scratch
// array that lives in this file, so nothing is allocated at call time.
//
// The array is a module-scope __device__ variable: every GPU on which this
// module is loaded holds its kDecodeScratchBytes until the process exits.  In
// host code the array's name only stands in for the device symbol, so its
// device address is looked up with cudaGetSymbolAddress, with the device
// current, on the first call on each device.  The address is kept together
// with the identity of the CUDA context it belongs to; if that context is
// replaced (cudaDeviceReset, or another context made current), the next call
// sees a different identity and repeats the look-up, so a stale address is
// never passed to a kernel.
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {
void set_error_detail(const char* text);  // defined beside fa_last_error_detail
}

namespace {

constexpr size_t kDecodeScratchBytes = FA_DECODE_NOALLOC_MAX_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; holds whatever the last call left there.
static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

struct ScratchEntry {
  unsigned long long ctx_id = 0;  // CUDA context the address belongs to (0: none yet)
  void* ptr = nullptr;
};

std::mutex g_setup_mutex;
ScratchEntry g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Driver entry points for the context identity (no link-time libcuda).
bool driver_fns(CtxGetCurrentFn* cur, CtxGetIdFn* id) {
  static CtxGetCurrentFn f_cur = nullptr;
  static CtxGetIdFn f_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_cur = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  *cur = f_cur;
  *id = f_id;
  return f_cur && f_id;
}

// Identity of the context current on this thread, or 0 if none is current yet.
cudaError_t current_context_id(unsigned long long* out) {
  CtxGetCurrentFn cur;
  CtxGetIdFn id;
  *out = 0;
  if (!driver_fns(&cur, &id)) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (cur(&ctx) != CUDA_SUCCESS) return cudaErrorNotSupported;
  if (!ctx) return cudaSuccess;
  return id(ctx, out) == CUDA_SUCCESS ? cudaSuccess : cudaErrorNotSupported;
}

// Device address of the scratch array in the current device's context,
// looked up once per device (and again whenever that context has changed).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx_id = 0;
  e = current_context_id(&ctx_id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchEntry& ent = g_scratch[dev];
  if (ctx_id == 0 || ent.ctx_id != ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // also makes the context current
    if (e != cudaSuccess) return e;
    e = current_context_id(&ctx_id);
    if (e != cudaSuccess) return e;
    ent.ctx_id = ctx_id;
    ent.ptr = p;
  }
  *out = ent.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" {

fa_status fa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o,
                            float* lse, const int32_t* seqlens_k, int B, int Hq, int Hkv,
                            int Sk_max, int d, float scale, cudaStream_t stream) {
  char msg[256];
  const size_t need = fa_decode_workspace_size(B, Hq, Sk_max, d);
  if (need > kDecodeScratchBytes) {
    snprintf(msg, sizeof msg,
             "fa_decode_noalloc: this problem needs %zu bytes of scratch, the built-in "
             "scratch holds %zu; use fa_decode with a caller workspace",
             need, kDecodeScratchBytes);
    fa::set_error_detail(msg);
    return FA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "fa_decode_noalloc: scratch set-up failed: %s",
             cudaGetErrorString(e));
    fa::set_error_detail(msg);
    return FA_ERR_CUDA;
  }
  // Every split slot the merge reads is written by the partial kernel of the
  // same call first, so the scratch needs no clearing between calls.
  return fa_decode(q, k_cache, v_cache, o, lse, seqlens_k, B, Hq, Hkv, Sk_max, d, scale, scratch,
                   kDecodeScratchBytes, stream);
}

}  // extern "C"
