// Device pieces of the residual / bonus draw shared by the draw kernels of
// the single-GPU step (sample.cu) and of the vocabulary-parallel step
// (shard.cu): token loads, weights, chunk sums, the prefix over chunks and
// the find-and-rescan at a position t. See sample.cu for the method.
#pragma once

#include "kernels.h"

namespace specdec {
namespace sampling {


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

// The whole CTA, with the prefix of the row's chunk sums in sm.s_pre (and
// sm.s_lastchunk set): find the chunk holding t, rescan it in token order
// and return the smallest token v with C_v > t (column within the row; the
// last weighted token when rounding puts t past the rescanned total).
// Valid in thread 0.
template <typename DL>
__device__ __forceinline__ int draw_at(const SampleLaunch& L, const SelectedRow& sr,
                                       const float* zr, const DL* qr, bool residual, float t,
                                       DrawSmem& sm) {
  const bool vec = L.vec != 0;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int found = -1;
    for (int g = 0; g < L.nchunks && found < 0; g += 32) {
      const int k = g + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, k < L.nchunks && sm.s_pre[k] > t);
      if (hit) found = g + __ffs(hit) - 1;
    }
    if (found < 0) found = sm.s_lastchunk;   // t rounded up to S: the last chunk with weight
    if (found < 0) found = 0;                // no weight at all (cannot happen for w = p)
    if (lane == 0) {
      sm.s_chunk = found;
      sm.s_before = found > 0 ? sm.s_pre[found - 1] : 0.f;
      sm.s_t = t;
      sm.s_tok = 0x7fffffff;
      sm.s_lastpos = -1;
      sm.s_residual = residual;
    }
  }
  __syncthreads();

  // ---- rescan the chosen chunk in token order: 16 contiguous tokens per thread ----
  const int v0 = sm.s_chunk * kChunkV + tid * kPer;
  float w[kPer];
#pragma unroll
  for (int k = 0; k < kPer / kVec; ++k) {
    const Raw4 r = load4<DL>(zr, qr, v0 + k * kVec, L.V, vec, sm.s_residual != 0);
    weights4(r, sr, sm.s_residual != 0, L.c, w + k * kVec);
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
  if (lane == 31) sm.wscan[warp] = incl;
  __syncthreads();
  float wbefore = 0.f;
  for (int i = 0; i < warp; ++i) wbefore += sm.wscan[i];
  float run = sm.s_before + (wbefore + excl);
  const float tt = sm.s_t;
  int cand = 0x7fffffff, lastp = -1;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    run += w[k];
    if (w[k] > 0.f) lastp = v0 + k;
    if (cand == 0x7fffffff && w[k] > 0.f && run > tt) cand = v0 + k;
  }
  if (cand != 0x7fffffff) atomicMin(&sm.s_tok, cand);
  if (lastp >= 0) atomicMax(&sm.s_lastpos, lastp);
  __syncthreads();
  int tok = sm.s_tok;
  if (tok == 0x7fffffff) tok = sm.s_lastpos;   // t beyond the rescanned total (rounding)
  return tok;
}

// The draw of sequence b with the whole CTA, once every chunk sum of its
// row is in L.chunk_sums: prefix of the chunk sums, the chunk holding
// t = u * S, a rescan of that chunk in token order, the token.
template <typename DL>
__device__ __forceinline__ void draw_sequence(const SampleLaunch& L, int b, const SelectedRow& sr,
                                              const float* zr, const DL* qr, DrawSmem& sm) {
  const bool vec = L.vec != 0;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int g1 = L.gamma + 1;
  const float u = sample_uniform(L.seed, b, sr.j);
  for (int k = tid; k < L.nchunks; k += kSampleThreads)
    sm.s_cs[k] = __ldcg(L.chunk_sums + (size_t)b * L.nchunks + k);
  __syncthreads();
  if (warp == 0) prefix_chunks(sm.s_cs, sm.s_pre, L.nchunks, &sm.s_lastchunk);
  __syncthreads();
  bool residual = sr.residual != 0;
  if (residual && !(sm.s_pre[L.nchunks - 1] > 0.f)) {
    // p == q to rounding: draw from p. Recompute every chunk sum with w = p.
    residual = false;
    for (int k = 0; k < L.nchunks; ++k) {
      const float tot = chunk_total<DL>(zr, qr, sr, false, L.c, L.V, vec, k, sm.red);
      if (tid == 0) sm.s_cs[k] = tot;
    }
    __syncthreads();
    if (warp == 0) prefix_chunks(sm.s_cs, sm.s_pre, L.nchunks, &sm.s_lastchunk);
    __syncthreads();
  }
  const float t = u * sm.s_pre[L.nchunks - 1];
  const int tok = draw_at<DL>(L, sr, zr, qr, residual, t, sm);
  if (tid == 0) L.out_tokens[b * g1 + sr.j] = tok;
}

}  // namespace sampling
}  // namespace specdec
