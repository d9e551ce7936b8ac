// The vocabulary-parallel verify step: one shard of the vocabulary per GPU.
//
// "推测解码" (world.lapla.si/zh/specdec), section 几段话一起写: the weight
// read is the step's cost, so a tensor-parallel target model splits W_lm by
// vocabulary rows and each GPU reads only its slice. The acceptance rule
// ("推测解码", section 通过的规则) needs the full-vocabulary normalisers of p
// and q, the two logits of every guessed token, and, for the draw, the
// prefix of max(0, p - q) over the whole vocabulary. Per step:
//
//   score   (each GPU)  LM head on its slice; one record per row: (max,
//                       sum exp2) of p and q, the argmax (global token ID),
//                       and the guessed tokens' logits where this slice
//                       holds them.
//   exchange 1          the caller all-gathers the records (rank order).
//   accept  (each GPU)  folds the G records of every row in one fixed order,
//                       so every GPU holds the same normalisers and the same
//                       acceptance decisions; writes the kept prefix and
//                       n_accepted (greedy mode: the whole result); then
//                       sums this slice's residual weights max(0, p - q)
//                       (and p, for the rare p == q fallback) of the row the
//                       draw uses.
//   exchange 2          the caller all-gathers the (residual, p) sums.
//   draw    (each GPU)  every GPU forms the same prefix over slices and
//                       t = u * S; the GPU whose slice holds t draws its
//                       token, the others write -1.
//   exchange 3          the caller reduces the tokens with max.
#include "accept.cuh"
#include "sample.cuh"

namespace specdec {
namespace {

using namespace sampling;

constexpr int kFoldThreads = 512;
constexpr int kAccThreads = 256;
static_assert(kAccThreads == kSampleThreads, "the fused kernel sums chunks with the sampler's layout");

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct ShardPtrs {
  ShardRec* P;
  ShardQRec* Q;
  ShardXRec* X;
};
__host__ __device__ inline ShardPtrs shard_ptrs(void* base, int B, int gamma) {
  char* c = static_cast<char*>(base);
  const size_t M = (size_t)B * (gamma + 1), N = (size_t)B * gamma;
  ShardPtrs p;
  p.P = reinterpret_cast<ShardRec*>(c);
  p.Q = reinterpret_cast<ShardQRec*>(c + align256(M * sizeof(ShardRec)));
  p.X = reinterpret_cast<ShardXRec*>(c + align256(M * sizeof(ShardRec)) +
                                     align256(N * sizeof(ShardQRec)));
  return p;
}

// One CTA per sequence: fold this slice's partial records into one record
// per row (the acceptance kernel's fold, run on the slice).
template <typename DL>
__global__ void __launch_bounds__(kFoldThreads) shard_fold_kernel(const AcceptLaunch a,
                                                                  void* records) {
  __shared__ AcceptSmem sm;
  const int b = blockIdx.x;
  grid_dependency_wait();      // the slice's LM-head records are complete
  if (b == 0 && threadIdx.x == 0) *a.calls += 1;   // the LM head of this call is done
  accept_fold<DL>(a, b, sm);
  __syncthreads();
  const int gamma = a.gamma, g1 = gamma + 1;
  const bool sample = a.mode == SPECDEC_SAMPLE;
  const ShardPtrs rp = shard_ptrs(records, gridDim.x, gamma);
  for (int r = threadIdx.x; r < g1; r += blockDim.x) {
    const int ai = sm.ai[r];
    // sampling keeps no argmax; greedy keeps (value, global token ID)
    const bool has_ai = !sample && ai != 0x7fffffff;
    rp.P[b * g1 + r] = ShardRec{sample ? sm.pm[r] : -INFINITY, sample ? sm.ps[r] : 0.f,
                                sample ? -INFINITY : sm.am[r], has_ai ? ai + a.tok_offset : 0x7fffffff};
  }
  for (int i = threadIdx.x; i < gamma; i += blockDim.x) {
    const int xl = sm.x[i] - a.tok_offset;
    const int owned = xl >= 0 && xl < a.V;
    rp.Q[b * gamma + i] = ShardQRec{sample ? sm.qm[i] : -INFINITY, sample ? sm.qs[i] : 0.f};
    rp.X[b * gamma + i] =
        ShardXRec{owned && sample ? sm.zx[i] : 0.f, owned && sample ? sm.zqx[i] : 0.f, owned, 0};
  }
}

// Folds the G slices' records of sequence b in a fixed order (identical on
// every GPU), looks up the slice holding each guessed token, and takes the
// acceptance decision of the single-GPU step (accept_decide, warp 0) on the
// folded values; `outputs` writes the kept prefix, n_accepted and the
// status. All threads of the CTA (kAccThreads) enter.
template <typename DL>
__device__ __forceinline__ void shard_fold_decide(const AcceptLaunch& a, int b, AcceptSmem& sm,
                                                  const char* base, size_t record_bytes,
                                                  int n_shards, bool outputs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gamma = a.gamma, g1 = gamma + 1;
  const bool sample = a.mode == SPECDEC_SAMPLE;
  const int B = a.B;
  const int rows = g1 + (sample ? gamma : 0);
  for (int r = warp; r < rows; r += kAccThreads / 32) {
    float m = -INFINITY, s = 0.f, av = -INFINITY;
    int ai = 0x7fffffff;
    // lanes take shards lane, lane+32, ...; the warp merge then visits them
    // in a fixed order, identical on every GPU.
    for (int k = lane; k < n_shards; k += 32) {
      const ShardPtrs rp = shard_ptrs(const_cast<char*>(base) + (size_t)k * record_bytes, B, gamma);
      if (r < g1) {
        const ShardRec x = rp.P[b * g1 + r];
        softmax_merge(m, s, x.m, x.s, a.c);
        if (argmax_better(x.amax_v, x.amax_i, av, ai)) {
          av = x.amax_v;
          ai = x.amax_i;
        }
      } else {
        const ShardQRec x = rp.Q[b * gamma + (r - g1)];
        softmax_merge(m, s, x.m, x.s, a.c);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      softmax_merge(m, s, m2, s2, a.c);
    }
    warp_argmax(av, ai);
    if (lane == 0) {
      if (r < g1) {
        sm.pm[r] = m;
        sm.ps[r] = s;
        sm.am[r] = av;
        sm.ai[r] = ai;
      } else {
        sm.qm[r - g1] = m;
        sm.qs[r - g1] = s;
      }
    }
  }
  // The guessed tokens and the logits from the slice that holds each: a
  // warp per guess, its lanes reading the slices' flags side by side.
  for (int i = warp; i < gamma; i += kAccThreads / 32) {
    const int x = a.draft_tokens[b * gamma + i];
    int own = -1;
    float zx = 0.f, zqx = 0.f;
    for (int k0 = 0; k0 < n_shards && own < 0; k0 += 32) {
      const int k = k0 + lane;
      ShardXRec xr{0.f, 0.f, 0, 0};
      if (k < n_shards)
        xr = shard_ptrs(const_cast<char*>(base) + (size_t)k * record_bytes, B, gamma)
                 .X[b * gamma + i];
      const unsigned owned = __ballot_sync(0xffffffffu, xr.owned != 0);
      if (owned) {
        const int src = __ffs(owned) - 1;
        own = k0 + src;
        zx = __shfl_sync(0xffffffffu, xr.zx, src);
        zqx = __shfl_sync(0xffffffffu, xr.zqx, src);
      }
    }
    if (lane == 0) {
      // A token no slice holds is out of range for the whole step.
      sm.x[i] = own >= 0 ? x : -1;
      sm.zx[i] = zx;
      sm.zqx[i] = zqx;
    }
  }
  __syncthreads();
  if (warp == 0) accept_decide<DL>(a, b, sm, outputs);
  __syncthreads();
}

// One CTA per sequence: the decision (shard_fold_decide) and the selected
// row for the sums kernel.
template <typename DL>
__global__ void __launch_bounds__(kAccThreads) shard_accept_kernel(const AcceptLaunch a,
                                                                   const void* all_records,
                                                                   size_t record_bytes,
                                                                   int n_shards) {
  __shared__ AcceptSmem sm;
  const int b = blockIdx.x;
  grid_dependency_wait();
  shard_fold_decide<DL>(a, b, sm, static_cast<const char*>(all_records), record_bytes, n_shards,
                        true);
  if (threadIdx.x == 0 && a.mode == SPECDEC_SAMPLE) {
    a.sel[b] = sm.sr;
    a.counters[b] = 0;
  }
}

// Few sequences: decision and slice sums in one kernel, grid (slice chunks,
// B). Every CTA of a sequence folds the records and decides (chunk 0 writes
// the outputs), then sums its chunk's residual and p weights; the last CTA
// of the sequence (ticket on a counter the slice's LM-head kernel zeroed)
// adds the chunk sums in chunk order and writes the slice's pair.
template <typename DL>
__global__ void __launch_bounds__(kAccThreads) shard_accept_sums_kernel(const AcceptLaunch a,
                                                                        const SampleLaunch L,
                                                                        const void* all_records,
                                                                        size_t record_bytes,
                                                                        int n_shards, float* cs_p,
                                                                        float2* shard_sums) {
  __shared__ AcceptSmem sm;
  __shared__ float red[kSampleThreads / 32];
  __shared__ int s_last;
  const int b = blockIdx.y;
  const int chunk = blockIdx.x;
  grid_dependency_wait();
  shard_fold_decide<DL>(a, b, sm, static_cast<const char*>(all_records), record_bytes, n_shards,
                        chunk == 0);
  const SelectedRow sr = sm.sr;
  if (chunk == 0 && threadIdx.x == 0) a.sel[b] = sr;
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  const bool residual = sr.residual != 0;
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const DL* qr = residual ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                          : nullptr;
  const bool vec = L.vec != 0;
  const float tp = chunk_total<DL>(zr, nullptr, sr, false, L.c, L.V, vec, chunk, red);
  const float tr = residual ? chunk_total<DL>(zr, qr, sr, true, L.c, L.V, vec, chunk, red) : tp;
  if (threadIdx.x == 0) {
    L.chunk_sums[(size_t)b * L.nchunks + chunk] = tr;
    cs_p[(size_t)b * L.nchunks + chunk] = tp;
    __threadfence();
    s_last = atomicAdd(&L.counters[b], 1) % L.nchunks == L.nchunks - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  float sres = 0.f, sp = 0.f;
  for (int k = 0; k < L.nchunks; ++k) {
    sres += __ldcg(L.chunk_sums + (size_t)b * L.nchunks + k);
    sp += __ldcg(cs_p + (size_t)b * L.nchunks + k);
  }
  shard_sums[b] = make_float2(sres, sp);
}

// Grid (slice chunks, B): the residual weights max(0, p - q) and the p
// weights of the row each sequence draws from, summed per chunk; the last
// CTA of a sequence (atomic ticket) adds the chunk sums in chunk order and
// writes the slice's pair (residual sum, p sum); for the bonus row the two
// are the same p sum.
template <typename DL>
__global__ void __launch_bounds__(kSampleThreads) shard_sums_kernel(const SampleLaunch L,
                                                                    float* cs_p,
                                                                    float2* shard_sums) {
  __shared__ float red[2][kSampleThreads / 32];
  __shared__ int s_last;
  const int b = blockIdx.y;
  const int chunk = blockIdx.x;
  grid_dependency_wait();      // the acceptance decisions are complete
  const SelectedRow sr = L.sel[b];
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const bool residual = sr.residual != 0;
  const DL* qr = residual ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                          : nullptr;
  const bool vec = L.vec != 0;
  const int v0 = chunk * kChunkV + threadIdx.x * kVec;
  Raw4 raw[kSweeps];
#pragma unroll
  for (int k = 0; k < kSweeps; ++k) raw[k] = load4<DL>(zr, qr, v0 + k * kSweep, L.V, vec, residual);
  float tr = 0.f, tp = 0.f;
#pragma unroll
  for (int k = 0; k < kSweeps; ++k) {
    float wr[kVec], wp[kVec];
    weights4(raw[k], sr, residual, L.c, wr);
    weights4(raw[k], sr, false, L.c, wp);
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      tr += wr[e];
      tp += wp[e];
    }
  }
  tr = warp_sum(tr);
  tp = warp_sum(tp);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][warp] = tr;
    red[1][warp] = tp;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f, c = 0.f;
    for (int i = 0; i < kSampleThreads / 32; ++i) {
      a += red[0][i];
      c += red[1][i];
    }
    L.chunk_sums[(size_t)b * L.nchunks + chunk] = a;
    cs_p[(size_t)b * L.nchunks + chunk] = c;
    __threadfence();
    s_last = atomicAdd(&L.counters[b], 1) == L.nchunks - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  float sres = 0.f, sp = 0.f;
  for (int k = 0; k < L.nchunks; ++k) {
    sres += __ldcg(L.chunk_sums + (size_t)b * L.nchunks + k);
    sp += __ldcg(cs_p + (size_t)b * L.nchunks + k);
  }
  shard_sums[b] = make_float2(residual ? sres : sp, sp);
}

// One CTA per sequence: the same prefix over slices on every GPU; the
// slice that holds t = u * S draws (token ID = its column + tok_offset),
// every other slice writes -1 at the drawn position.
template <typename DL>
__global__ void __launch_bounds__(kSampleThreads) shard_draw_kernel(const SampleLaunch L,
                                                                    const float* cs_p,
                                                                    const float2* all_sums,
                                                                    int n_shards, int shard,
                                                                    int tok_offset) {
  __shared__ DrawSmem sm;
  __shared__ int s_owner, s_res;
  __shared__ float s_tloc;
  const int b = blockIdx.x;
  grid_dependency_wait();
  const SelectedRow sr = L.sel[b];
  if (sr.j < 0) return;
  const int g1 = L.gamma + 1;
  if (threadIdx.x == 0) {
    float tres = 0.f;
    for (int k = 0; k < n_shards; ++k) tres += all_sums[(size_t)k * gridDim.x + b].x;
    // p == q to rounding (no residual mass anywhere): every slice draws from p.
    const bool res = sr.residual != 0 && tres > 0.f;
    float S = 0.f;
    for (int k = 0; k < n_shards; ++k) {
      const float2 v = all_sums[(size_t)k * gridDim.x + b];
      S += res ? v.x : v.y;
    }
    const float t = sample_uniform(L.seed, b, sr.j) * S;
    int owner = -1, last = -1;
    float before = 0.f, run = 0.f, before_last = 0.f;
    for (int k = 0; k < n_shards; ++k) {
      const float2 v = all_sums[(size_t)k * gridDim.x + b];
      const float w = res ? v.x : v.y;
      if (w > 0.f) {
        last = k;
        before_last = run;
      }
      if (owner < 0 && w > 0.f && run + w > t) {
        owner = k;
        before = run;
      }
      run += w;
    }
    if (owner < 0) {   // t rounded up to S: the last slice with weight
      owner = last;
      before = before_last;
    }
    s_owner = owner;
    s_res = res;
    s_tloc = t - before;
  }
  __syncthreads();
  if (s_owner != shard) {
    if (threadIdx.x == 0) L.out_tokens[b * g1 + sr.j] = -1;
    return;
  }
  const bool res = s_res != 0;
  const float* cs = res ? L.chunk_sums : cs_p;
  for (int k = threadIdx.x; k < L.nchunks; k += kSampleThreads)
    sm.s_cs[k] = __ldcg(cs + (size_t)b * L.nchunks + k);
  __syncthreads();
  if (threadIdx.x < 32) prefix_chunks(sm.s_cs, sm.s_pre, L.nchunks, &sm.s_lastchunk);
  __syncthreads();
  const float* zr = L.z + (size_t)(b * g1 + sr.j) * L.V;
  const DL* qr = res ? static_cast<const DL*>(L.dl) + ((size_t)b * L.gamma + sr.j) * L.V
                     : nullptr;
  const int tok = draw_at<DL>(L, sr, zr, qr, res, s_tloc, sm);
  if (threadIdx.x == 0) L.out_tokens[b * g1 + sr.j] = tok + tok_offset;
}

cudaLaunchConfig_t pdl_config(dim3 grid, int threads, cudaStream_t stream,
                              cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

size_t shard_record_bytes(int B, int gamma) {
  const size_t M = (size_t)B * (gamma + 1), N = (size_t)B * gamma;
  return align256(M * sizeof(ShardRec)) + align256(N * sizeof(ShardQRec)) +
         align256(N * sizeof(ShardXRec));
}

cudaError_t launch_shard_fold(const AcceptLaunch& A, void* records, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(A.B), kFoldThreads, stream, attr);
  return cudaLaunchKernelEx(&cfg, shard_fold_kernel<__nv_bfloat16>, A, records);
}

cudaError_t launch_shard_accept(const AcceptLaunch& A, const void* all_records,
                                size_t record_bytes, int n_shards, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(A.B), kAccThreads, stream, attr);
  return cudaLaunchKernelEx(&cfg, shard_accept_kernel<__nv_bfloat16>, A, all_records,
                            record_bytes, n_shards);
}

bool shard_fused_accept_sums(int B, int nchunks) {
  return (long long)B * nchunks <= kFusedAcceptItems;
}

cudaError_t launch_shard_accept_sums(const AcceptLaunch& A, const SampleLaunch& L0,
                                     const void* all_records, size_t record_bytes, int n_shards,
                                     float* cs_p, float2* shard_sums, cudaStream_t stream) {
  SampleLaunch L = L0;
  L.vec = (L.V % kVec == 0 && ((uintptr_t)L.z & 15u) == 0 && ((uintptr_t)L.dl & 7u) == 0) ? 1 : 0;
  L.prefetch = 0;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(L.nchunks, L.B), kAccThreads, stream, attr);
  return cudaLaunchKernelEx(&cfg, shard_accept_sums_kernel<__nv_bfloat16>, A, L, all_records,
                            record_bytes, n_shards, cs_p, shard_sums);
}

cudaError_t launch_shard_sums(const SampleLaunch& L0, float* cs_p, float2* shard_sums,
                              cudaStream_t stream) {
  SampleLaunch L = L0;
  L.vec = (L.V % kVec == 0 && ((uintptr_t)L.z & 15u) == 0 && ((uintptr_t)L.dl & 7u) == 0) ? 1 : 0;
  L.prefetch = 0;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(L.nchunks, L.B), kSampleThreads, stream, attr);
  return cudaLaunchKernelEx(&cfg, shard_sums_kernel<__nv_bfloat16>, L, cs_p, shard_sums);
}

cudaError_t launch_shard_draw(const SampleLaunch& L0, const float* cs_p, const float2* all_sums,
                              int n_shards, int shard, int tok_offset, cudaStream_t stream) {
  SampleLaunch L = L0;
  L.vec = (L.V % kVec == 0 && ((uintptr_t)L.z & 15u) == 0 && ((uintptr_t)L.dl & 7u) == 0) ? 1 : 0;
  L.prefetch = 0;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(L.B), kSampleThreads, stream, attr);
  return cudaLaunchKernelEx(&cfg, shard_draw_kernel<__nv_bfloat16>, L, cs_p, all_sums, n_shards,
                            shard, tok_offset);
}

}  // namespace specdec
