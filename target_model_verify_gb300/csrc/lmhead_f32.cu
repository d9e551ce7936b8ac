// LM-head scoring for fp32 inputs on the CUDA cores.
//
// The same contraction and fused epilogue as the tensor-core kernel, for
// the fp32 dtype (small heads, where the step is bound by launch latency
// rather than by the weight read). One CTA per (128-row vocabulary tile,
// 16 token rows); the k dimension is staged through shared memory in
// slices of 32 with coalesced loads, and each thread accumulates the 16
// logits of its vocabulary row in fp32 FMAs.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kKSlice = 32;

__global__ void __launch_bounds__(128)
    lmhead_f32_kernel(const float* __restrict__ H, const float* __restrict__ W, int d,
                      const EpiParams ep, int* status) {
  grid_dependency_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *(volatile int*)status = SPECDEC_OK;
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < ep.n_counters; i += blockDim.x) ep.counters[i] = 0;
  __shared__ float ws[kKSlice][kBlockV + 1];
  __shared__ float hs[16][kKSlice];
  __shared__ RedSlot red[64];
  const int vt = blockIdx.x;
  const int m0 = blockIdx.y * 16;
  const int tid = threadIdx.x;
  const int v = vt * kBlockV + tid;
  float acc[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) acc[n] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kKSlice) {
    for (int e = tid; e < kBlockV * kKSlice; e += 128) {
      const int r = e / kKSlice, kk = e % kKSlice;
      const int vv = vt * kBlockV + r, k = k0 + kk;
      ws[kk][r] = (vv < ep.V && k < d) ? W[(size_t)vv * d + k] : 0.f;
    }
    for (int e = tid; e < 16 * kKSlice; e += 128) {
      const int n = e / kKSlice, kk = e % kKSlice;
      const int m = m0 + n, k = k0 + kk;
      hs[n][kk] = (m < ep.M && k < d) ? H[(size_t)m * d + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKSlice; ++kk) {
      const float w = ws[kk][tid];
#pragma unroll
      for (int n = 0; n < 16; ++n) acc[n] = fmaf(w, hs[n][kk], acc[n]);
    }
    __syncthreads();
  }
  float zq[16];
  prefetch_draft16<float>(zq, m0, v, ep);
  epilogue_chunk16<float>(acc, zq, m0, v, vt, tid >> 5, tid & 31, tid, red, ep, 1);
}

}  // namespace

cudaError_t launch_lmhead_f32(const float* hidden, const float* W, int d, const EpiParams& ep,
                              int* status, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((ep.V + kBlockV - 1) / kBlockV, (ep.M + 15) / 16);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lmhead_f32_kernel, hidden, W, d, ep, status);
}

}  // namespace specdec
