// fa_mask.cu -- pack a per-key boolean mask (one byte per key) into the
// visibility bit words the attention kernels read (32 keys per word, 4 words
// per 128-key tile, bits past Sk left clear).
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace fa {
namespace {

// One warp per 32-key word: lane t tests key 32*w + t and the ballot is the word.
__global__ void fa_pack_key_mask_kernel(const uint8_t* __restrict__ mask, uint32_t* __restrict__ bits,
                                        int rows, int Sk, int words) {
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_id >= static_cast<long long>(rows) * words) return;  // warp-uniform
  const int r = static_cast<int>(warp_id / words);
  const int w = static_cast<int>(warp_id % words);
  const int j = w * 32 + lane;
  const bool vis = j < Sk && mask[static_cast<size_t>(r) * Sk + j] != 0;
  const uint32_t word = __ballot_sync(0xffffffffu, vis);
  if (lane == 0) bits[static_cast<size_t>(r) * words + w] = word;
}

}  // namespace

cudaError_t launch_pack_key_mask(const uint8_t* mask, uint32_t* bits, int rows, int Sk, int words,
                                 cudaStream_t stream) {
  const long long threads = static_cast<long long>(rows) * words * 32;
  const unsigned int grid = static_cast<unsigned int>((threads + 255) / 256);
  fa_pack_key_mask_kernel<<<grid, 256, 0, stream>>>(mask, bits, rows, Sk, words);
  return cudaGetLastError();
}

}  // namespace fa
