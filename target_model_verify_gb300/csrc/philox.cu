// The library's uniforms written out, so another implementation of
// Philox4x32-10 can be compared with them value for value.
#include "kernels.h"

namespace specdec {
namespace {

__global__ void philox_uniforms_kernel(uint64_t seed, int B, int n_pos, int purpose,
                                       float* out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * n_pos) return;
  const int b = idx / n_pos, i = idx - b * n_pos;
  out[idx] = purpose == 0 ? accept_uniform(seed, b, i) : sample_uniform(seed, b, i);
}

}  // namespace

cudaError_t launch_philox_uniforms(uint64_t seed, int B, int n_pos, int purpose, float* out,
                                   cudaStream_t stream) {
  const int n = B * n_pos;
  philox_uniforms_kernel<<<(n + 255) / 256, 256, 0, stream>>>(seed, B, n_pos, purpose, out);
  return cudaGetLastError();
}

}  // namespace specdec
