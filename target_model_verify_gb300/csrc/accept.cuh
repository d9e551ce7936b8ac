// Acceptance test and first-reject scan of one sequence, as device functions
// shared by the acceptance kernel and the small-batch fused draw kernel.
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
#pragma once

#include "kernels.h"

namespace specdec {

constexpr int kAcceptBatch = 8;   // record loads in flight per lane

struct AcceptSmem {
  float pm[SPECDEC_MAX_GAMMA + 1], ps[SPECDEC_MAX_GAMMA + 1];
  float am[SPECDEC_MAX_GAMMA + 1];
  int ai[SPECDEC_MAX_GAMMA + 1];
  float qm[SPECDEC_MAX_GAMMA], qs[SPECDEC_MAX_GAMMA];
  float zx[SPECDEC_MAX_GAMMA], zqx[SPECDEC_MAX_GAMMA];
  int x[SPECDEC_MAX_GAMMA];
  SelectedRow sr;
};

// Every warp of the CTA: fold the partial records of sequence b's gamma+1
// target rows and gamma draft rows (one warp per row at a time), after warp
// 0 has fetched the drafted tokens' two logits. Ends with the results in
// `sm` (the caller synchronises the CTA before reading them).
template <typename DL>
__device__ __forceinline__ void accept_fold(const AcceptLaunch& a, int b, AcceptSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int gamma = a.gamma, g1 = gamma + 1;
  const bool sample = a.mode == SPECDEC_SAMPLE;
  const int rows = g1 + (sample ? gamma : 0);
  // The drafted tokens' logits do not depend on the folds: warp 0 loads
  // them first, so their latency overlaps the record loads.
  if (warp == 0 && lane < gamma) {
    const int x = a.draft_tokens[b * gamma + lane];
    sm.x[lane] = x;
    const int xl = x - a.tok_offset;   // column of x in this (shard's) vocabulary
    if (sample && xl >= 0 && xl < a.V) {
      const DL* dl = static_cast<const DL*>(a.dl);
      sm.zx[lane] = a.z[(size_t)(b * g1 + lane) * a.V + xl];
      sm.zqx[lane] = load_logit(dl, ((size_t)b * gamma + lane) * a.V + xl);
    }
  }
  for (int r = warp; r < rows; r += nwarps) {
    float m = -INFINITY, s = 0.f;
    if (r < g1) {
      const PartialP* row = a.pp + (size_t)(b * g1 + r) * a.P;
      float av = -INFINITY;
      int ai = 0x7fffffff;
      // Records t = lane, lane+32, ... folded in that order; kAcceptBatch
      // loads are issued before their merges so they overlap in flight.
      for (int base = lane; base < a.P; base += 32 * kAcceptBatch) {
        PartialP x[kAcceptBatch];
#pragma unroll
        for (int u = 0; u < kAcceptBatch; ++u) {
          const int t = base + 32 * u;
          x[u] = t < a.P ? row[t] : PartialP{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
        }
#pragma unroll
        for (int u = 0; u < kAcceptBatch; ++u) {
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
        sm.pm[r] = m;
        sm.ps[r] = s;
        sm.am[r] = av;
        sm.ai[r] = ai;
      }
    } else {
      const int i = r - g1;
      const PartialQ* row = a.pq + ((size_t)b * gamma + i) * a.Pq;
      for (int base = lane; base < a.Pq; base += 32 * kAcceptBatch) {
        PartialQ x[kAcceptBatch];
#pragma unroll
        for (int u = 0; u < kAcceptBatch; ++u) {
          const int t = base + 32 * u;
          x[u] = t < a.Pq ? row[t] : PartialQ{-INFINITY, 0.f};
        }
#pragma unroll
        for (int u = 0; u < kAcceptBatch; ++u) softmax_merge(m, s, x[u].m, x[u].s, a.c);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        softmax_merge(m, s, m2, s2, a.c);
      }
      if (lane == 0) {
        sm.qm[i] = m;
        sm.qs[i] = s;
      }
    }
  }
}

// Warp 0, after accept_fold and a CTA barrier: test the gamma guesses in
// parallel, take the first rejection with a ballot, leave the draw's
// selection in sm.sr, and (when `outputs`) write the kept prefix,
// n_accepted, the status and the debug outputs.
template <typename DL>
__device__ __forceinline__ void accept_decide(const AcceptLaunch& a, int b, AcceptSmem& sm,
                                              bool outputs) {
  const int lane = threadIdx.x & 31;
  const int gamma = a.gamma, g1 = gamma + 1;
  const bool sample = a.mode == SPECDEC_SAMPLE;
  const int prior = *(volatile int*)a.status;
  bool bad = false, rej = false;
  int x = -1;
  if (lane < gamma) {
    x = sm.x[lane];
    if (x < 0 || x >= a.V) {
      bad = true;
    } else if (!sample) {
      rej = x != sm.ai[lane];
    } else {
      const float zx = sm.zx[lane];
      const float zqx = sm.zqx[lane];
      const float px = exp2f((zx - sm.pm[lane]) * a.c - log2f(sm.ps[lane]));
      const float qx = exp2f((zqx - sm.qm[lane]) * a.c - log2f(sm.qs[lane]));
      const float r = accept_uniform(a.seed, b, lane);
      rej = !(r * qx <= px);
      if (outputs && a.p_x) a.p_x[b * gamma + lane] = px;
      if (outputs && a.q_x) a.q_x[b * gamma + lane] = qx;
    }
  }
  const unsigned bad_mask = __ballot_sync(0xffffffffu, bad);
  const unsigned rej_mask = __ballot_sync(0xffffffffu, rej);
  const bool failed = bad_mask != 0 || prior == SPECDEC_ERR_TIMEOUT;
  const int j = rej_mask ? __ffs(rej_mask) - 1 : gamma;
  if (outputs) {
    if (bad_mask && lane == 0) set_status(a.status, SPECDEC_ERR_TOKEN_RANGE);
    for (int i = lane; i < g1; i += 32) {
      int t;
      if (failed) t = -1;
      else if (i < j) t = a.draft_tokens[b * gamma + i];
      else if (i == j) t = sample ? -1 : sm.ai[j];   // sampling: written by the draw
      else t = -1;
      a.out_tokens[b * g1 + i] = t;
      if (a.lse_p && sample) a.lse_p[b * g1 + i] = (sm.pm[i] * a.c + log2f(sm.ps[i])) * kLn2;
      if (a.argmax_out) a.argmax_out[b * g1 + i] = sm.ai[i];
    }
    if (a.lse_q && sample)
      for (int i = lane; i < gamma; i += 32)
        a.lse_q[b * gamma + i] = (sm.qm[i] * a.c + log2f(sm.qs[i])) * kLn2;
    if (lane == 0) a.n_accepted[b] = failed ? -1 : j;
  }
  if (lane == 0 && sample) {
    SelectedRow sr;
    sr.mp = sm.pm[j];
    sr.lsp = log2f(sm.ps[j]);
    sr.residual = j < gamma ? 1 : 0;
    sr.mq = j < gamma ? sm.qm[j] : 0.f;
    sr.lsq = j < gamma ? log2f(sm.qs[j]) : 0.f;
    sr.j = failed ? -1 : j;
    sr.pad[0] = sr.pad[1] = 0;
    sm.sr = sr;
  }
}

}  // namespace specdec
