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

namespace specdec {
namespace {

constexpr int kVec = 4;                              // tokens per load
constexpr int kSweep = kSampleThreads * kVec;        // 1024 tokens per sweep
constexpr int kSweeps = kChunkV / kSweep;            // 4 sweeps per chunk
constexpr int kPer = kChunkV / kSampleThreads;       // 16 tokens per thread
constexpr int kMaxChunks = kMaxVocab / kChunkV;
static_assert(kSweeps * kVec == kPer, "chunk layout");

struct Raw4 {
  float4 z;
  float q[kVec];
};

// Logits and draft logits of tokens v .. v+3 (v a multiple of 4); tokens at
// or past V read as weight-free (-inf logit for p, nothing for q).
template <typename DL>
__device__ __forceinline__ Raw4 load4(const float* __restrict__ zr, const DL* __restrict__ qr,
                                      int v, int V, bool vec, bool residual) {
  Raw4 r;
  if (vec && v < V) {   // V % 4 == 0: the whole group is in range
    r.z = __ldg(reinterpret_cast<const float4*>(zr + v));
    if (residual) {
      if constexpr (sizeof(DL) == 2) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(qr + v));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        r.q[0] = a.x; r.q[1] = a.y; r.q[2] = b.x; r.q[3] = b.y;
      } else {
        const float4 f = __ldg(reinterpret_cast<const float4*>(qr + v));
        r.q[0] = f.x; r.q[1] = f.y; r.q[2] = f.z; r.q[3] = f.w;
      }
    }
    return r;
  }
  float zz[kVec];
#pragma unroll
  for (int e = 0; e < kVec; ++e) {
    const bool in = v + e < V;
    zz[e] = in ? zr[v + e] : -INFINITY;
    r.q[e] = (in && residual) ? load_logit(qr, (size_t)(v + e)) : 0.f;
  }
  r.z = make_float4(zz[0], zz[1], zz[2], zz[3]);
  return r;
}

// w = max(0, p - q) (residual) or p, for the four tokens of a group.
__device__ __forceinline__ void weights4(const Raw4& r, const SelectedRow& sr, bool residual,
                                         float c, float* w) {
  const float zz[kVec] = {r.z.x, r.z.y, r.z.z, r.z.w};
#pragma unroll
  for (int e = 0; e < kVec; ++e) {
    const float p = exp2f((zz[e] - sr.mp) * c - sr.lsp);
    if (residual) {
      const float qv = exp2f((r.q[e] - sr.mq) * c - sr.lsq);
      w[e] = fmaxf(0.f, p - qv);
    } else {
      w[e] = p;
    }
  }
}

// Sum of one chunk's weights: four coalesced sweeps, thread-sequential,
// then warp shuffles, then the 8 warp sums in order. Every thread returns
// the chunk total.
template <typename DL>
__device__ __forceinline__ float chunk_total(const float* zr, const DL* qr, const SelectedRow& sr,
                                             bool residual, float c, int V, bool vec, int chunk,
                                             float* red) {
  const int v0 = chunk * kChunkV + threadIdx.x * kVec;
  Raw4 raw[kSweeps];
#pragma unroll
  for (int k = 0; k < kSweeps; ++k) raw[k] = load4<DL>(zr, qr, v0 + k * kSweep, V, vec, residual);
  float ts = 0.f;
#pragma unroll
  for (int k = 0; k < kSweeps; ++k) {
    float w[kVec];
    weights4(raw[k], sr, residual, c, w);
#pragma unroll
    for (int e = 0; e < kVec; ++e) ts += w[e];
  }
  ts = warp_sum(ts);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = ts;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < kSampleThreads / 32; ++i) t += red[i];
  return t;
}

// Warp 0: inclusive prefix of the chunk sums in chunk order (groups of 32,
// shuffle scan, carried total), and the last chunk holding weight.
__device__ __forceinline__ void prefix_chunks(const float* cs, float* pre, int n, int* last_pos) {
  const int lane = threadIdx.x & 31;
  float carry = 0.f;
  int lp = -1;
  for (int g = 0; g < n; g += 32) {
    const int k = g + lane;
    const float x = k < n ? cs[k] : 0.f;
    float incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (k < n) pre[k] = carry + incl;
    const unsigned pos = __ballot_sync(0xffffffffu, k < n && x > 0.f);
    if (pos) lp = g + 31 - __clz(pos);
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) *last_pos = lp;
}

// Shared memory of the draw (the last step of a sequence, one CTA).
struct DrawSmem {
  float red[kSampleThreads / 32];
  float wscan[kSampleThreads / 32];
  float s_cs[kMaxChunks];
  float s_pre[kMaxChunks];
  int s_tok, s_lastpos, s_lastchunk, s_chunk, s_residual;
  float s_before, s_t;
};

// The draw of sequence b with the whole CTA, once every chunk sum of its
// row is in L.chunk_sums: prefix of the chunk sums, the chunk holding
// t = u * S, a rescan of that chunk in token order, the token.
template <typename DL>
__device__ __forceinline__ void draw_sequence(const SampleLaunch& L, int b, const SelectedRow& sr,
                                              const float* zr, const DL* qr, DrawSmem& sm) {
  float* red = sm.red;
  float* wscan = sm.wscan;
  float* s_cs = sm.s_cs;
  float* s_pre = sm.s_pre;
  int& s_tok = sm.s_tok;
  int& s_lastpos = sm.s_lastpos;
  int& s_lastchunk = sm.s_lastchunk;
  int& s_chunk = sm.s_chunk;
  int& s_residual = sm.s_residual;
  float& s_before = sm.s_before;
  float& s_t = sm.s_t;
  const bool vec = L.vec != 0;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g1 = L.gamma + 1;
  // ---- last CTA of sequence b: locate the chunk holding t = u * S ----
  const float u = sample_uniform(L.seed, b, sr.j);
  for (int k = tid; k < L.nchunks; k += kSampleThreads)
    s_cs[k] = __ldcg(L.chunk_sums + (size_t)b * L.nchunks + k);
  __syncthreads();
  if (warp == 0) prefix_chunks(s_cs, s_pre, L.nchunks, &s_lastchunk);
  __syncthreads();
  bool residual = sr.residual != 0;
  if (residual && !(s_pre[L.nchunks - 1] > 0.f)) {
    // p == q to rounding: draw from p. Recompute every chunk sum with w = p.
    residual = false;
    for (int k = 0; k < L.nchunks; ++k) {
      const float tot = chunk_total<DL>(zr, qr, sr, false, L.c, L.V, vec, k, red);
      if (tid == 0) s_cs[k] = tot;
    }
    __syncthreads();
    if (warp == 0) prefix_chunks(s_cs, s_pre, L.nchunks, &s_lastchunk);
    __syncthreads();
  }
  if (warp == 0) {
    const float t = u * s_pre[L.nchunks - 1];
    int found = -1;
    for (int g = 0; g < L.nchunks && found < 0; g += 32) {
      const int k = g + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, k < L.nchunks && s_pre[k] > t);
      if (hit) found = g + __ffs(hit) - 1;
    }
    if (found < 0) found = s_lastchunk;   // t rounded up to S: the last chunk with weight
    if (found < 0) found = 0;             // no weight at all (cannot happen for w = p)
    if (lane == 0) {
      s_chunk = found;
      s_before = found > 0 ? s_pre[found - 1] : 0.f;
      s_t = t;
      s_tok = 0x7fffffff;
      s_lastpos = -1;
      s_residual = residual;
    }
  }
  __syncthreads();

  // ---- rescan the chosen chunk in token order: 16 contiguous tokens per thread ----
  const int v0 = s_chunk * kChunkV + tid * kPer;
  float w[kPer];
#pragma unroll
  for (int k = 0; k < kPer / kVec; ++k) {
    const Raw4 r = load4<DL>(zr, qr, v0 + k * kVec, L.V, vec, s_residual != 0);
    weights4(r, sr, s_residual != 0, L.c, w + k * kVec);
  }
  float ts = 0.f;
#pragma unroll
  for (int k = 0; k < kPer; ++k) ts += w[k];
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
