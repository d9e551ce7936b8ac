// Host -> device staging for the host entry point. When the step's host
// buffers are pinned and mapped into the GPU's address space (on
// Grace-Blackwell the GPU reaches them over NVLink-C2C), one kernel gathers
// the step's inputs from host memory into the workspace instead of one
// copy-engine transfer per buffer (the results are stored straight into the
// caller's mapped output buffers by the kernels that produce them).
#include "kernels.h"

namespace specdec {
namespace {

// Copy of `n` units of type T per segment, grid-stride, four units in
// flight per thread.
template <typename T>
__device__ __forceinline__ void copy_units(const T* __restrict__ src, T* __restrict__ dst,
                                           long long n) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const T a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

__global__ void __launch_bounds__(256) stage_in_kernel(const StageInLaunch S) {
  // The LM-head kernel that follows may set itself up meanwhile; it reads
  // global memory only after this grid has completed.
  grid_launch_dependents();
  for (int s = 0; s < S.nseg; ++s) {
    const HostSeg g = S.seg[s];
    const long long body = g.bytes / g.unit;
    if (g.unit == 16)
      copy_units(reinterpret_cast<const uint4*>(g.src), reinterpret_cast<uint4*>(g.dst), body);
    else if (g.unit == 4)
      copy_units(reinterpret_cast<const uint32_t*>(g.src), reinterpret_cast<uint32_t*>(g.dst), body);
    else
      copy_units(reinterpret_cast<const uint8_t*>(g.src), reinterpret_cast<uint8_t*>(g.dst), body);
    if (blockIdx.x == 0 && threadIdx.x == 0)   // the bytes after the last whole unit
      for (long long i = body * g.unit; i < g.bytes; ++i)
        static_cast<uint8_t*>(g.dst)[i] = static_cast<const uint8_t*>(g.src)[i];
  }
}

}  // namespace

cudaError_t launch_stage_in(const StageInLaunch& S, int num_sms, cudaStream_t stream) {
  long long units = 0;
  for (int s = 0; s < S.nseg; ++s) units += S.seg[s].bytes / S.seg[s].unit;
  long long blocks = (units + 4 * 256 - 1) / (4 * 256);
  const long long cap = 2ll * (num_sms > 0 ? num_sms : 1);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  stage_in_kernel<<<(unsigned)blocks, 256, 0, stream>>>(S);
  return cudaGetLastError();
}

}  // namespace specdec
