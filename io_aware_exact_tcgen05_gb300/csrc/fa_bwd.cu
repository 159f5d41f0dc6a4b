// fa_bwd.cu -- backward attention kernels (placeholder until the tcgen05
// backward lands; returns cudaErrorNotYetImplemented).
#include <cuda_runtime.h>
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
cudaError_t launch_bwd(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, const BwdParams&, cudaStream_t) {
  return cudaErrorNotYetImplemented;
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
