// Acceptance test and first-reject scan, one CTA per sequence.
//
// "推测解码" (world.lapla.si/zh/specdec), section 通过的规则: with p the large
// model's and q the small model's probability of the guessed token, the
// guess is kept iff r <= p/q for a uniform r (so q <= p always keeps it).
// Section 留下对的，换掉错的: checking stops at the first guess that fails.
// Greedy mode (maxstudionews.com article 1664, the verify paragraph) keeps a
// guess iff it equals the large model's argmax.
//
// Each warp folds the per-tile partials of one row into (max, sum) -- the
// log-normaliser of z/T -- and the row's argmax; warp 0 then tests the
// gamma guesses in parallel and finds the first rejection with a ballot.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kThreads = 512;   // one warp per record row: up to 2*32+1 rows in one round
constexpr int kBatch = 8;

template <typename DL>
__global__ void __launch_bounds__(kThreads) accept_kernel(const AcceptLaunch a) {
  __shared__ float s_pm[SPECDEC_MAX_GAMMA + 1], s_ps[SPECDEC_MAX_GAMMA + 1];
  __shared__ float s_am[SPECDEC_MAX_GAMMA + 1];
  __shared__ int s_ai[SPECDEC_MAX_GAMMA + 1];
  __shared__ float s_qm[SPECDEC_MAX_GAMMA], s_qs[SPECDEC_MAX_GAMMA];

  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gamma = a.gamma, g1 = gamma + 1;
  const bool sample = a.mode == SPECDEC_SAMPLE;
  const int rows = g1 + (sample ? gamma : 0);

  grid_dependency_wait();      // the LM-head kernel's records are complete
  grid_launch_dependents();    // the sampler may start launching
  if (b == 0 && threadIdx.x == 0) *a.calls += 1;   // the LM head of this call is done

  // The drafted tokens' logits do not depend on the folds: warp 0 loads
  // them first, so their latency overlaps the record loads.
  __shared__ float s_zx[SPECDEC_MAX_GAMMA], s_zqx[SPECDEC_MAX_GAMMA];
  __shared__ int s_x[SPECDEC_MAX_GAMMA];
  if (warp == 0 && lane < gamma) {
    const int x = a.draft_tokens[b * gamma + lane];
    s_x[lane] = x;
    if (sample && x >= 0 && x < a.V) {
      const DL* dl = static_cast<const DL*>(a.dl);
      s_zx[lane] = a.z[(size_t)(b * g1 + lane) * a.V + x];
      s_zqx[lane] = load_logit(dl, ((size_t)b * gamma + lane) * a.V + x);
    }
  }

  for (int r = warp; r < rows; r += kThreads / 32) {
    float m = -INFINITY, s = 0.f;
    if (r < g1) {
      const PartialP* row = a.pp + (size_t)(b * g1 + r) * a.P;
      float av = -INFINITY;
      int ai = 0x7fffffff;
      // Records t = lane, lane+32, ... folded in that order; kBatch loads
      // are issued before their merges so they overlap in flight.
      for (int base = lane; base < a.P; base += 32 * kBatch) {
        PartialP x[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int t = base + 32 * u;
          x[u] = t < a.P ? row[t] : PartialP{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (sample) softmax_merge(m, s, x[u].m, x[u].s, a.c);
          if (argmax_better(x[u].amax_v, x[u].amax_i, av, ai)) {
            av = x[u].amax_v;
            ai = x[u].amax_i;
          }
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
        s_pm[r] = m;
        s_ps[r] = s;
        s_am[r] = av;
        s_ai[r] = ai;
      }
    } else {
      const int i = r - g1;
      const PartialQ* row = a.pq + ((size_t)b * gamma + i) * a.Pq;
      for (int base = lane; base < a.Pq; base += 32 * kBatch) {
        PartialQ x[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int t = base + 32 * u;
          x[u] = t < a.Pq ? row[t] : PartialQ{-INFINITY, 0.f};
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) softmax_merge(m, s, x[u].m, x[u].s, a.c);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        softmax_merge(m, s, m2, s2, a.c);
      }
      if (lane == 0) {
        s_qm[i] = m;
        s_qs[i] = s;
      }
    }
  }
  __syncthreads();
  if (warp != 0) return;

  const int prior = *(volatile int*)a.status;
  bool bad = false, rej = false;
  int x = -1;
  if (lane < gamma) {
    x = s_x[lane];
    if (x < 0 || x >= a.V) {
      bad = true;
    } else if (!sample) {
      rej = x != s_ai[lane];
    } else {
      const float zx = s_zx[lane];
      const float zqx = s_zqx[lane];
      const float px = exp2f((zx - s_pm[lane]) * a.c - log2f(s_ps[lane]));
      const float qx = exp2f((zqx - s_qm[lane]) * a.c - log2f(s_qs[lane]));
      const float r = accept_uniform(a.seed, b, lane);
      rej = !(r * qx <= px);
      if (a.p_x) a.p_x[b * gamma + lane] = px;
      if (a.q_x) a.q_x[b * gamma + lane] = qx;
    }
  }
  const unsigned bad_mask = __ballot_sync(0xffffffffu, bad);
  const unsigned rej_mask = __ballot_sync(0xffffffffu, rej);
  if (bad_mask && lane == 0) set_status(a.status, SPECDEC_ERR_TOKEN_RANGE);
  const bool failed = bad_mask != 0 || prior == SPECDEC_ERR_TIMEOUT;
  const int j = rej_mask ? __ffs(rej_mask) - 1 : gamma;

  for (int i = lane; i < g1; i += 32) {
    int t;
    if (failed) t = -1;
    else if (i < j) t = a.draft_tokens[b * gamma + i];
    else if (i == j) t = sample ? -1 : s_ai[j];   // sampling: written by the sampler
    else t = -1;
    a.out_tokens[b * g1 + i] = t;
    if (a.lse_p && sample) a.lse_p[b * g1 + i] = (s_pm[i] * a.c + log2f(s_ps[i])) * kLn2;
    if (a.argmax_out) a.argmax_out[b * g1 + i] = s_ai[i];
  }
  if (a.lse_q && sample)
    for (int i = lane; i < gamma; i += 32)
      a.lse_q[b * gamma + i] = (s_qm[i] * a.c + log2f(s_qs[i])) * kLn2;
  if (lane == 0) {
    a.n_accepted[b] = failed ? -1 : j;
    if (sample) {
      SelectedRow sr;
      sr.mp = s_pm[j];
      sr.lsp = log2f(s_ps[j]);
      sr.residual = j < gamma ? 1 : 0;
      sr.mq = j < gamma ? s_qm[j] : 0.f;
      sr.lsq = j < gamma ? log2f(s_qs[j]) : 0.f;
      sr.j = failed ? -1 : j;
      sr.pad[0] = sr.pad[1] = 0;
      a.sel[b] = sr;
      a.counters[b] = 0;
    }
  }
}

}  // namespace

cudaError_t launch_accept(const AcceptLaunch& L, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.B);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.dl_bf16) return cudaLaunchKernelEx(&cfg, accept_kernel<__nv_bfloat16>, L);
  return cudaLaunchKernelEx(&cfg, accept_kernel<float>, L);
}

}  // namespace specdec
