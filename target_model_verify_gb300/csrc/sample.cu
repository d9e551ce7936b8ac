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
// (V chunks of 4096, B). Each CTA sums its chunk's weights; the last CTA of
// a sequence to finish (atomic ticket, no waiting) scans the chunk sums in
// order, finds the chunk holding t, rescans that chunk and writes the token.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kPer = kChunkV / kSampleThreads;   // 16 tokens per thread
constexpr int kMaxChunks = kMaxVocab / kChunkV;

template <typename DL>
__device__ __forceinline__ void chunk_weights(const float* __restrict__ zr,
                                              const DL* __restrict__ qr, const SelectedRow& sr,
                                              bool residual, float c, int V, int v0,
                                              float (&w)[kPer]) {
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int v = v0 + k;
    float x = 0.f;
    if (v < V) {
      const float p = exp2f((zr[v] - sr.mp) * c - sr.lsp);
      if (residual) {
        const float qv = exp2f((load_logit(qr, (size_t)v) - sr.mq) * c - sr.lsq);
        x = fmaxf(0.f, p - qv);
      } else {
        x = p;
      }
    }
    w[k] = x;
  }
}

// Block sum in a fixed order: per-thread sequential, then warp shuffles,
// then the 8 warp sums in order.
__device__ __forceinline__ float block_sum(float x, float* red) {
  x = warp_sum(x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < kSampleThreads / 32; ++i) t += red[i];
  return t;
}

template <typename DL>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleLaunch L) {
  __shared__ float red[kSampleThreads / 32];
  __shared__ float wscan[kSampleThreads / 32];
  __shared__ float s_cs[kMaxChunks];
  __shared__ int s_last;
  __shared__ int s_tok;
  __shared__ int s_lastpos;
  __shared__ int s_chunk;
  __shared__ float s_before, s_t;
  __shared__ int s_residual;

  const int b = blockIdx.y;
  const int chunk = blockIdx.x;
  grid_dependency_wait();      // the acceptance kernel's selection is complete
  const SelectedRow sr = L.sel[b];
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const DL* qr = sr.residual ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                             : nullptr;
  const int tid = threadIdx.x;

  float w[kPer];
  chunk_weights<DL>(zr, qr, sr, sr.residual != 0, L.c, L.V, chunk * kChunkV + tid * kPer, w);
  float ts = 0.f;
#pragma unroll
  for (int k = 0; k < kPer; ++k) ts += w[k];
  const float total = block_sum(ts, red);
  if (tid == 0) {
    L.chunk_sums[(size_t)b * L.nchunks + chunk] = total;
    __threadfence();
    const int ticket = atomicAdd(&L.counters[b], 1);
    s_last = ticket == L.nchunks - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of sequence b: locate the chunk holding t = u * S ----
  const float u = sample_uniform(L.seed, b, sr.j);
  for (int k = tid; k < L.nchunks; k += kSampleThreads)
    s_cs[k] = __ldcg(L.chunk_sums + (size_t)b * L.nchunks + k);
  __syncthreads();
  if (tid == 0) {
    float S = 0.f;
    for (int k = 0; k < L.nchunks; ++k) S += s_cs[k];
    s_residual = sr.residual;
    if (sr.residual && !(S > 0.f)) s_residual = 0;   // p == q to rounding: draw from p
    s_t = u * S;
  }
  __syncthreads();
  if (s_residual != sr.residual) {
    // Fallback: recompute every chunk sum with w = p.
    for (int k = 0; k < L.nchunks; ++k) {
      float wk[kPer];
      chunk_weights<DL>(zr, qr, sr, false, L.c, L.V, k * kChunkV + tid * kPer, wk);
      float t2 = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) t2 += wk[e];
      const float tot = block_sum(t2, red);
      if (tid == 0) s_cs[k] = tot;
    }
    __syncthreads();
    if (tid == 0) {
      float S = 0.f;
      for (int k = 0; k < L.nchunks; ++k) S += s_cs[k];
      s_t = u * S;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const float* cs = s_cs;
    const float t = s_t;
    float acc = 0.f;
    int found = -1, last_pos = 0;
    float before = 0.f;
    for (int k = 0; k < L.nchunks; ++k) {
      const float nxt = acc + cs[k];
      if (cs[k] > 0.f) last_pos = k;
      if (found < 0 && nxt > t) {
        found = k;
        before = acc;
      }
      acc = nxt;
    }
    if (found < 0) {   // t rounded up to S: the last chunk with weight
      found = last_pos;
      before = acc - cs[last_pos];
    }
    s_chunk = found;
    s_before = before;
    s_tok = 0x7fffffff;
    s_lastpos = -1;
  }
  __syncthreads();

  // ---- rescan the chosen chunk in token order ----
  const int v0 = s_chunk * kChunkV + tid * kPer;
  chunk_weights<DL>(zr, qr, sr, s_residual != 0, L.c, L.V, v0, w);
  ts = 0.f;
#pragma unroll
  for (int k = 0; k < kPer; ++k) ts += w[k];
  const int warp = tid >> 5, lane = tid & 31;
  float incl = ts;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  if (lane == 31) wscan[warp] = incl;
  __syncthreads();
  float wbefore = 0.f;
  for (int i = 0; i < warp; ++i) wbefore += wscan[i];
  float run = s_before + (wbefore + excl);
  const float t = s_t;
  int cand = 0x7fffffff, lastp = -1;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    run += w[k];
    if (w[k] > 0.f) lastp = v0 + k;
    if (cand == 0x7fffffff && w[k] > 0.f && run > t) cand = v0 + k;
  }
  if (cand != 0x7fffffff) atomicMin(&s_tok, cand);
  if (lastp >= 0) atomicMax(&s_lastpos, lastp);
  __syncthreads();
  if (tid == 0) {
    int tok = s_tok;
    if (tok == 0x7fffffff) tok = s_lastpos;   // t beyond the rescanned total (rounding)
    L.out_tokens[b * g1 + sr.j] = tok;
  }
}

}  // namespace

cudaError_t launch_sample(const SampleLaunch& L, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.nchunks, L.B);
  cfg.blockDim = dim3(kSampleThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.dl_bf16) return cudaLaunchKernelEx(&cfg, sample_kernel<__nv_bfloat16>, L);
  return cudaLaunchKernelEx(&cfg, sample_kernel<float>, L);
}

}  // namespace specdec
