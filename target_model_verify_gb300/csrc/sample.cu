// Replacement and bonus draw (sampling mode).
//
// "推测解码" (world.lapla.si/zh/specdec), section 通过的规则: a rejected guess
// is replaced by a token drawn from max(0, p - q), renormalised -- tokens
// the small model under-guessed are topped up, over-guessed ones never come
// back. Section 留下对的，换掉错的: if every guess passes, the position after
// them is drawn from p.
//
// The draw inverts the prefix sum C of the weights w in token-ID order at
// t = u * S (S the total): the token is the smallest v with C_v > t. Grid =
// (V chunks of 4096, B). Each CTA sums its chunk's weights, reading the
// chunk as four coalesced 1024-token sweeps (16-byte logit loads, 8-byte
// draft-logit loads, all issued before the arithmetic). The last CTA of a
// sequence to finish (atomic ticket, no waiting) forms the prefix of the
// chunk sums with one warp, finds the chunk holding t, rescans that chunk in
// token order (16 contiguous tokens per thread) and writes the token.
// With many sequences (more than kSampleOneKernelItems (sequence, chunk)
// pairs) the sums come from a kernel without tickets and one CTA per
// sequence draws in a second kernel: the fence and atomic that the ticket
// needs kept every summing CTA resident past its loads (measured: 79 ->
// 74 us for accept and draw at batch 256, 35 -> 34 us at batch 64).
#include "accept.cuh"
#include "sample.cuh"

namespace specdec {
namespace {
using namespace sampling;

// Small batch: grid (chunks, B). Each CTA sums one chunk; the last CTA of a
// sequence to finish (atomic ticket, no waiting) draws.
template <typename DL>
__global__ void __launch_bounds__(kSampleThreads, 6) sample_kernel(const SampleLaunch L) {
  __shared__ DrawSmem sm;
  __shared__ int s_last;

  const int b = blockIdx.y;
  const int chunk = blockIdx.x;
  if (L.prefetch && threadIdx.x < 2 * (L.gamma + 1)) {
    // Small batch: the row is not known yet, but every candidate row's chunk
    // was written by the LM-head kernel, which finished before the
    // acceptance kernel began; pull them into L2 while that kernel runs.
    const int r = threadIdx.x >> 1;
    const int v0 = chunk * kChunkV;
    const int n = min(kChunkV, L.V - v0);
    if (threadIdx.x & 1) {
      if (r < L.gamma)
        bulk_prefetch_l2(static_cast<const __nv_bfloat16*>(L.dl) + ((size_t)b * L.gamma + r) * L.V + v0,
                         (uint32_t)n * 2u);
    } else {
      bulk_prefetch_l2(L.z + ((size_t)b * (L.gamma + 1) + r) * L.V + v0, (uint32_t)n * 4u);
    }
  }
  grid_dependency_wait();      // the acceptance kernel's selection is complete
  const SelectedRow sr = L.sel[b];
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const DL* qr = sr.residual ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                             : nullptr;
  const float total =
      chunk_total<DL>(zr, qr, sr, sr.residual != 0, L.c, L.V, L.vec != 0, chunk, sm.red);
  if (threadIdx.x == 0) {
    L.chunk_sums[(size_t)b * L.nchunks + chunk] = total;
    __threadfence();
    const int ticket = atomicAdd(&L.counters[b], 1);
    s_last = ticket == L.nchunks - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  draw_sequence<DL>(L, b, sr, zr, qr, sm);
}

// Small batch, acceptance fused in: grid (chunks, B). Every CTA folds its
// sequence's records and takes the acceptance decision itself (the same
// records in the same order, so every CTA of a sequence decides alike; the
// chunk-0 CTA writes the kept prefix, n_accepted and the status), then sums
// its chunk of the selected row, and the last CTA of the sequence to finish
// (atomic ticket; the LM-head kernel zeroed the tickets) draws. One kernel
// boundary fewer than acceptance kernel + sampler.
template <typename DL>
__global__ void __launch_bounds__(kSampleThreads) accept_sample_kernel(const AcceptLaunch A,
                                                                       const SampleLaunch L) {
  __shared__ DrawSmem sm;
  __shared__ AcceptSmem asm_;
  __shared__ int s_last;

  const int b = blockIdx.y;
  const int chunk = blockIdx.x;
  if (L.prefetch && threadIdx.x < 2 * (L.gamma + 1)) {
    // The row is not known yet, but every candidate row's chunk was written
    // by the LM-head kernel: pull them into L2 while the records fold.
    const int r = threadIdx.x >> 1;
    const int v0 = chunk * kChunkV;
    const int n = min(kChunkV, L.V - v0);
    if (threadIdx.x & 1) {
      if (r < L.gamma)
        bulk_prefetch_l2(static_cast<const __nv_bfloat16*>(L.dl) + ((size_t)b * L.gamma + r) * L.V + v0,
                         (uint32_t)n * 2u);
    } else {
      bulk_prefetch_l2(L.z + ((size_t)b * (L.gamma + 1) + r) * L.V + v0, (uint32_t)n * 4u);
    }
  }
  grid_dependency_wait();      // the LM-head kernel's records are complete
  if (b == 0 && chunk == 0 && threadIdx.x == 0) *A.calls += 1;   // the LM head of this call is done
  accept_fold<DL>(A, b, asm_);
  __syncthreads();
  if (threadIdx.x < 32) accept_decide<DL>(A, b, asm_, chunk == 0);
  __syncthreads();
  const SelectedRow sr = asm_.sr;
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const DL* qr = sr.residual ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                             : nullptr;
  const float total =
      chunk_total<DL>(zr, qr, sr, sr.residual != 0, L.c, L.V, L.vec != 0, chunk, sm.red);
  if (threadIdx.x == 0) {
    L.chunk_sums[(size_t)b * L.nchunks + chunk] = total;
    __threadfence();
    const int ticket = atomicAdd(&L.counters[b], 1);
    s_last = ticket == L.nchunks - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  draw_sequence<DL>(L, b, sr, zr, qr, sm);
}

// Many sequences: the same chunk sums without tickets (each CTA writes its
// sum and leaves, so no CTA stays resident through a fence and an atomic),
// then one CTA per sequence draws in a second kernel.
template <typename DL>
__global__ void __launch_bounds__(kSampleThreads, 6) sample_sums_kernel(const SampleLaunch L) {
  __shared__ float red[kSampleThreads / 32];
  const int b = blockIdx.y;
  const int chunk = blockIdx.x;
  // No early trigger of the draw kernel: its CTAs would sit on SMs the
  // chunk sums need (measured slower at batch 64 and 256).
  grid_dependency_wait();      // the acceptance kernel's selection is complete
  const SelectedRow sr = L.sel[b];
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const DL* qr = sr.residual ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                             : nullptr;
  const float total =
      chunk_total<DL>(zr, qr, sr, sr.residual != 0, L.c, L.V, L.vec != 0, chunk, red);
  if (threadIdx.x == 0) L.chunk_sums[(size_t)b * L.nchunks + chunk] = total;
}

template <typename DL>
__global__ void __launch_bounds__(kSampleThreads) sample_draw_kernel(const SampleLaunch L) {
  __shared__ DrawSmem sm;
  const int b = blockIdx.x;
  grid_dependency_wait();      // every chunk sum is written
  const SelectedRow sr = L.sel[b];
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const DL* qr = sr.residual ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                             : nullptr;
  draw_sequence<DL>(L, b, sr, zr, qr, sm);
}

}  // namespace

namespace {
SampleLaunch prepare_sample(const SampleLaunch& L0) {
  SampleLaunch L = L0;
  const uintptr_t dl_align = L.dl_bf16 ? 8 : 16;
  L.vec = (L.V % kVec == 0 && ((uintptr_t)L.z & 15u) == 0 &&
           ((uintptr_t)L.dl & (dl_align - 1)) == 0)
              ? 1
              : 0;
  // Bulk prefetches need 16-byte aligned rows of both arrays (bf16 draft
  // logits: V % 8 == 0); only worth it while the rows are few.
  L.prefetch = (L.dl_bf16 && L.B <= 16 && L.V % 8 == 0 && ((uintptr_t)L.z & 15u) == 0 &&
                ((uintptr_t)L.dl & 15u) == 0)
                   ? 1
                   : 0;
  return L;
}
}  // namespace

bool fused_accept_sample(int B, int nchunks) {
  return (long long)B * nchunks <= kFusedAcceptItems;
}

cudaError_t launch_accept_sample(const AcceptLaunch& A, const SampleLaunch& L0,
                                 cudaStream_t stream) {
  const SampleLaunch L = prepare_sample(L0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.nchunks, L.B);
  cfg.blockDim = dim3(kSampleThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.dl_bf16) return cudaLaunchKernelEx(&cfg, accept_sample_kernel<__nv_bfloat16>, A, L);
  return cudaLaunchKernelEx(&cfg, accept_sample_kernel<float>, A, L);
}

cudaError_t launch_sample(const SampleLaunch& L0, cudaStream_t stream) {
  const SampleLaunch L = prepare_sample(L0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.nchunks, L.B);
  cfg.blockDim = dim3(kSampleThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((long long)L.B * L.nchunks <= kSampleOneKernelItems) {
    if (L.dl_bf16) return cudaLaunchKernelEx(&cfg, sample_kernel<__nv_bfloat16>, L);
    return cudaLaunchKernelEx(&cfg, sample_kernel<float>, L);
  }
  cudaError_t e = L.dl_bf16 ? cudaLaunchKernelEx(&cfg, sample_sums_kernel<__nv_bfloat16>, L)
                            : cudaLaunchKernelEx(&cfg, sample_sums_kernel<float>, L);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(L.B);
  if (L.dl_bf16) return cudaLaunchKernelEx(&cfg, sample_draw_kernel<__nv_bfloat16>, L);
  return cudaLaunchKernelEx(&cfg, sample_draw_kernel<float>, L);
}

}  // namespace specdec
