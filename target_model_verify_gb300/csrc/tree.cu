// Tree verification: the acceptance rule at every fork of a token tree.
//
// "推测解码" (world.lapla.si/zh/specdec), section 不要第二个模型: guesses
// arranged as a tree are checked in one pass of the large model, and the
// same acceptance rule applied at every fork keeps the output distribution.
// The LM-head kernel has already scored every node (records and fp32 logits
// of row b*N + n) and reduced every node's draft logits (q records); this
// kernel walks each sequence's tree:
//
//   at node u, try its children in increasing index: keep child c iff
//   r_c * q_u(x_c) <= f(x_c), f = p_u at first and max(0, f - q_u) / S after
//   each rejection (S the residual's sum over the vocabulary); a kept child
//   becomes the node; otherwise draw one token from the last residual (or
//   from p_u) by inverting its prefix sum in token-ID order at t = u * S.
//
// Sampling: one cluster of kTreeCluster CTAs per sequence (kTreeClusterWide
// while every sequence's cluster of that size can run at once), each CTA
// owning a contiguous slice of the vocabulary. Every decision is computed identically
// by all CTAs of the cluster (same records, same values, sums exchanged
// through distributed shared memory and added in rank order), so their
// control flow never diverges and every cluster barrier is reached by all.
// Greedy: one CTA per sequence; the walk follows the child holding the
// target argmax.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kTC = 128;   // tokens per warp chunk: 32 lanes x 4
constexpr int kMaxSlice = (kMaxVocab + kTreeCluster - 1) / kTreeCluster + 4;
constexpr int kMaxChunks = (kMaxSlice + kTC - 1) / kTC;

struct NodeStats {
  float mp, lsp, mq, lsq;   // log2-domain normalisers: p(v) = exp2((z - mp) c - lsp)
  float av;                 // target argmax value and token
  int ai;
};

struct Shared {
  float chunk[kMaxChunks];  // weight sums of this CTA's 128-token chunks
  float pre[kMaxChunks];    // their inclusive prefix
  float S[SPECDEC_MAX_TREE_NODES + 1];   // residual sums S_1.. at the current node
  float Sinv[SPECDEC_MAX_TREE_NODES + 1];   // and their reciprocals
  NodeStats node[SPECDEC_MAX_TREE_NODES];   // every node's normalisers and argmax
  float cz[SPECDEC_MAX_TREE_NODES], cd[SPECDEC_MAX_TREE_NODES];   // child's logits at its parent
  float xv[2][kTreeClusterWide];   // cluster exchange slots, written by every CTA
  int xi[2][kTreeClusterWide];     // of the cluster (double buffered)
  float allv[kTreeClusterWide];
  int alli[kTreeClusterWide];
  float wm[kWarps], ws[kWarps], wav[kWarps];
  int wai[kWarps];
  int16_t first_child[SPECDEC_MAX_TREE_NODES], next_sibling[SPECDEC_MAX_TREE_NODES];
  int16_t parent[SPECDEC_MAX_TREE_NODES];
  int flag;
  int last_found;
};

constexpr int kFoldDepth = 8;   // record loads a lane keeps in flight while folding

// 2^x by the PTX approximate base-2 exponential (flushes subnormals; -inf
// gives 0): one instruction per weight in the vocabulary passes.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Every node's records folded, one half-warp per node (records
// lane-strided with kFoldDepth loads in flight per lane, then a butterfly
// over the 16 lanes): the node's target (max, sum) and argmax, and in
// sampling mode its draft (max, sum). All in a fixed order, so every CTA of
// a cluster gets the same values.
__device__ void fold_all_nodes(const TreeLaunch& L, int b, bool sample, Shared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane & 15;
  for (int n0 = 2 * warp; n0 < L.N; n0 += 2 * kWarps) {
    const int n = n0 + (lane >> 4);
    const bool valid = n < L.N;              // both halves run every shuffle below
    const size_t m = (size_t)b * L.N + (valid ? n : n0);
    float pm = -INFINITY, ps = 0.f, av = -INFINITY;
    int ai = 0x7fffffff;
    float qm = -INFINITY, qs = 0.f;
    const PartialP* row = L.pp + m * L.P;
    const PartialQ* qrow = L.pq + m * L.Pq;
    const int np = valid ? L.P : 0, nq = (valid && sample) ? L.Pq : 0;
    for (int t0 = hl; t0 < np || t0 < nq; t0 += 16 * kFoldDepth) {
      PartialP x[kFoldDepth];
      PartialQ y[kFoldDepth];
#pragma unroll
      for (int j = 0; j < kFoldDepth; ++j) {
        const int t = t0 + 16 * j;
        if (t < np) x[j] = row[t];
        if (t < nq) y[j] = qrow[t];
      }
#pragma unroll
      for (int j = 0; j < kFoldDepth; ++j) {
        const int t = t0 + 16 * j;
        if (t < np) {
          if (sample) softmax_merge(pm, ps, x[j].m, x[j].s, L.c);
          if (argmax_better(x[j].amax_v, x[j].amax_i, av, ai)) {
            av = x[j].amax_v;
            ai = x[j].amax_i;
          }
        }
        if (t < nq) softmax_merge(qm, qs, y[j].m, y[j].s, L.c);
      }
    }
#pragma unroll
    for (int o = 8; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, pm, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, ps, o);
      softmax_merge(pm, ps, m2, s2, L.c);
      const float qm2 = __shfl_xor_sync(0xffffffffu, qm, o);
      const float qs2 = __shfl_xor_sync(0xffffffffu, qs, o);
      softmax_merge(qm, qs, qm2, qs2, L.c);
      const float av2 = __shfl_xor_sync(0xffffffffu, av, o);
      const int ai2 = __shfl_xor_sync(0xffffffffu, ai, o);
      if (argmax_better(av2, ai2, av, ai)) {
        av = av2;
        ai = ai2;
      }
    }
    if (valid && hl == 0) {
      NodeStats st;
      st.mp = pm;
      st.lsp = log2f(ps);
      st.mq = qm;
      st.lsq = log2f(qs);
      st.av = av;
      st.ai = ai;
      sh.node[n] = st;
    }
  }
}

// Weight of level `lev` at one token: lev 0 -> p(v); lev k >= 1 ->
// max(0, f_{k-1}(v) - q(v)) with f_0 = p and f_j = max(0, f_{j-1} - q) / S_j
// (multiplied by the reciprocal, the same way in every pass and test).
__device__ __forceinline__ float weight(float z, float d, const NodeStats& st, float c, int lev,
                                        const float* Sinv) {
  const float p = ex2((z - st.mp) * c - st.lsp);
  if (lev == 0) return p;
  const float q = ex2((d - st.mq) * c - st.lsq);
  float f = p;
  for (int j = 1; j < lev; ++j) f = fmaxf(0.f, f - q) * Sinv[j];
  return fmaxf(0.f, f - q);
}

// Raw logits and draft logits of tokens v..v+3 of row m (v a multiple of
// 4); tokens at or past hi read as absent (-inf logit).
struct Raw4 {
  float4 z;
  uint2 d;
};
__device__ __forceinline__ Raw4 load4(const TreeLaunch& L, size_t m, int v, int hi, int lev) {
  const float* zr = L.z + m * (size_t)L.V;
  const __nv_bfloat16* dr = L.dl + m * (size_t)L.V;
  Raw4 r;
  r.d = make_uint2(0u, 0u);
  if (L.vec && v + 3 < hi) {
    r.z = __ldg(reinterpret_cast<const float4*>(zr + v));
    if (lev > 0) r.d = __ldg(reinterpret_cast<const uint2*>(dr + v));
    return r;
  }
  float zz[4];
  unsigned short dd[4] = {0, 0, 0, 0};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int x = v + e;
    zz[e] = x < hi ? zr[x] : -INFINITY;
    if (lev > 0 && x < hi) dd[e] = __bfloat16_as_ushort(dr[x]);
  }
  r.z = make_float4(zz[0], zz[1], zz[2], zz[3]);
  r.d = make_uint2((uint32_t)dd[0] | ((uint32_t)dd[1] << 16), (uint32_t)dd[2] | ((uint32_t)dd[3] << 16));
  return r;
}
__device__ __forceinline__ void weights_of(const Raw4& r, const NodeStats& st, float c, int lev,
                                           const float* S, float (&w)[4]) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.d.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.d.y));
  w[0] = weight(r.z.x, a.x, st, c, lev, S);
  w[1] = weight(r.z.y, a.y, st, c, lev, S);
  w[2] = weight(r.z.z, b.x, st, c, lev, S);
  w[3] = weight(r.z.w, b.y, st, c, lev, S);
}
// Four weights at tokens v..v+3 of row m (v a multiple of 4, inside the
// slice [.., hi)).
__device__ __forceinline__ void weights4(const TreeLaunch& L, size_t m, int v, int hi,
                                         const NodeStats& st, int lev, const float* S,
                                         float (&w)[4]) {
  weights_of(load4(L, m, v, hi, lev), st, L.c, lev, S, w);
}

// Chunk sums of this CTA's slice [lo, hi) at level `lev` (kept in
// sh.chunk for a draw); returns the slice total and sets sh.last_found. Each warp takes chunks
// warp, warp + 8, ...; with vector loads the loads of kBatch chunks are
// issued (predicated, straight-line) before any arithmetic, so they are in
// flight together.
constexpr int kBatch = 4;
__device__ float slice_pass(const TreeLaunch& L, size_t m, int lo, int hi, int lev,
                           const NodeStats& st, Shared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = (hi - lo + kTC - 1) / kTC;
  const float* zr = L.z + m * (size_t)L.V;
  const __nv_bfloat16* dr = L.dl + m * (size_t)L.V;
  const float c = L.c;
  if (L.vec) {
    // V % 4 == 0: a group of 4 starting below hi lies wholly inside it.
    for (int k0 = warp; k0 < nch; k0 += kWarps * kBatch) {
      float4 zv[kBatch];
      uint2 dv[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int v = lo + (k0 + j * kWarps) * kTC + 4 * lane;
        const bool in = v < hi;
        zv[j] = in ? __ldg(reinterpret_cast<const float4*>(zr + v))
                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        dv[j] = (in && lev > 0) ? __ldg(reinterpret_cast<const uint2*>(dr + v)) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        float w[4];
        weights_of(Raw4{zv[j], dv[j]}, st, c, lev, sh.Sinv, w);
        float s = (w[0] + w[1]) + (w[2] + w[3]);
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const int k = k0 + j * kWarps;
        if (lane == 0 && k < nch) sh.chunk[k] = s;
      }
    }
  } else {
    for (int k = warp; k < nch; k += kWarps) {
      float w[4];
      weights4(L, m, lo + k * kTC + 4 * lane, hi, st, lev, sh.Sinv, w);
      float s = (w[0] + w[1]) + (w[2] + w[3]);
#pragma unroll
      for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) sh.chunk[k] = s;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // The slice total (fixed order: lane-strided, then a butterfly) and the
    // last chunk holding weight (for a draw point rounded up to the total).
    float tot = 0.f;
    int lastc = -1;
    for (int k = lane; k < nch; k += 32) {
      const float x = sh.chunk[k];
      tot += x;
      if (x > 0.f) lastc = k;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      lastc = max(lastc, __shfl_xor_sync(0xffffffffu, lastc, o));
    }
    if (lane == 0) {
      sh.flag = __float_as_int(tot);
      sh.last_found = lastc;
    }
  }
  __syncthreads();
  return __int_as_float(sh.flag);
}

// Inclusive prefix of the slice's chunk sums in chunk order (warp 0 only),
// 32 chunks at a time with a carry, into sh.pre.
__device__ void chunk_prefix(int nch, Shared& sh) {
  const int lane = threadIdx.x & 31;
  float carry = 0.f;
  for (int g = 0; g < nch; g += 32) {
    const int k = g + lane;
    const float x = k < nch ? sh.chunk[k] : 0.f;
    float incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (k < nch) sh.pre[k] = carry + incl;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
}

// Every CTA of the cluster publishes (v, i); all get every CTA's pair in
// rank order. Each CTA stores its pair into every CTA's slot for it, so
// after the cluster barrier (release / acquire) all reads are local.
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
template <int kCW>
__device__ void exchange(float v, int i, int& par, Shared& sh) {
  const int rank = (int)cluster_ctarank();
  if (threadIdx.x < kCW) {
    st_cluster_f32(mapa_shared(smem_u32(&sh.xv[par][rank]), threadIdx.x), v);
    st_cluster_s32(mapa_shared(smem_u32(&sh.xi[par][rank]), threadIdx.x), i);
  }
  cluster_sync_all();
  if (threadIdx.x < kCW) {
    sh.allv[threadIdx.x] = sh.xv[par][threadIdx.x];
    sh.alli[threadIdx.x] = sh.xi[par][threadIdx.x];
  }
  __syncthreads();
  par ^= 1;
}

template <int kCW>
__global__ void __launch_bounds__(kThreads, 1) tree_walk_kernel(const TreeLaunch L) {
  __shared__ Shared sh;
  const bool sample = L.mode == SPECDEC_SAMPLE;
  const int rank = kCW > 1 ? (int)cluster_ctarank() : 0;
  const int b = blockIdx.x / kCW;
  const int N = L.N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // This CTA's vocabulary slice (multiple-of-4 boundaries).
  const int slice = ((L.V + kCW - 1) / kCW + 3) & ~3;
  const int lo = min(L.V, rank * slice);
  const int hi = min(L.V, lo + slice);

  for (int n = tid; n < N; n += kThreads) {
    sh.first_child[n] = L.first_child[n];
    sh.next_sibling[n] = L.next_sibling[n];
    sh.parent[n] = L.parent[n];
  }
  __syncthreads();
  grid_dependency_wait();   // the LM-head kernel's records, logits and q records are complete
  if (blockIdx.x == 0 && threadIdx.x == 0) *L.calls += 1;   // the LM head of this call is done
  const int prior = *(volatile int*)L.status;
  bool bad = false;
  for (int n = 1 + tid; n < N; n += kThreads) {
    const int x = L.tok[(size_t)b * N + n];
    if (x < 0 || x >= L.V) bad = true;
  }
  bad = __syncthreads_or(bad) != 0;
  if (bad || prior == SPECDEC_ERR_TIMEOUT) {
    if (rank == 0) {
      if (bad && tid == 0) set_status(L.status, SPECDEC_ERR_TOKEN_RANGE);
      for (int n = tid; n < N; n += kThreads) {
        L.out_tokens[(size_t)b * N + n] = -1;
        L.out_nodes[(size_t)b * N + n] = -1;
      }
      if (tid == 0) L.n_accepted[b] = -1;
    }
    if (kCW > 1) cluster_sync_all();
    return;
  }

  // Every node's statistics, and every child's target and draft logit at
  // its parent's row, before the walk: the walk itself then waits only for
  // vocabulary passes.
  // (The children's logits are requested first, so their loads overlap the
  // fold; N <= 128 < kThreads, one child per thread.)
  const int cc = 1 + tid;
  float czv = 0.f, cdv = 0.f;
  if (sample && cc < N) {
    const size_t mp = (size_t)b * N + sh.parent[cc];
    const int x = L.tok[(size_t)b * N + cc];
    czv = L.z[mp * (size_t)L.V + x];
    cdv = __bfloat162float(L.dl[mp * (size_t)L.V + x]);
  }
  fold_all_nodes(L, b, sample, sh);
  if (sample && cc < N) {
    sh.cz[cc] = czv;
    sh.cd[cc] = cdv;
  }
  __syncthreads();

  int par = 0;
  int u = 0, depth = 0;
  while (true) {
    const size_t m = (size_t)b * N + u;
    const NodeStats st = sh.node[u];
    if (!sample) {
      int match = -1;
      for (int c = sh.first_child[u]; c >= 0; c = sh.next_sibling[c])
        if (L.tok[(size_t)b * N + c] == st.ai) {
          match = c;
          break;
        }
      if (rank == 0 && tid == 0) L.out_tokens[(size_t)b * N + depth] = st.ai;
      if (match < 0) break;
      if (rank == 0 && tid == 0) L.out_nodes[(size_t)b * N + depth] = match;
      ++depth;
      u = match;
      continue;
    }

    // ---- sampling: children in order, residual after each rejection ----
    int nrej = 0, kept = -1;
    bool fallback = false;
    float last_total = 0.f;   // this CTA's share of the last residual's sum
    for (int c = sh.first_child[u]; c >= 0; c = sh.next_sibling[c]) {
      const float zx = sh.cz[c];
      const float dx = sh.cd[c];
      const float px = ex2((zx - st.mp) * L.c - st.lsp);
      const float qx = ex2((dx - st.mq) * L.c - st.lsq);
      float f = px;
      for (int j = 1; j <= nrej; ++j) f = fmaxf(0.f, f - qx) * sh.Sinv[j];
      const float r = accept_uniform(L.seed, b, c - 1);
      if (r * qx <= f) {
        kept = c;
        break;
      }
      // Rejected: S_{nrej+1} = sum of max(0, f_nrej - q) over the vocabulary.
      const float part = slice_pass(L, m, lo, hi, nrej + 1, st, sh);
      float S = part;
      if (kCW > 1) {
        exchange<kCW>(part, sh.last_found, par, sh);
        S = 0.f;
        for (int q = 0; q < kCW; ++q) S += sh.allv[q];
      }
      if (!(S > 0.f)) {   // rounding left no residual: draw from p_u
        fallback = true;
        break;
      }
      ++nrej;
      last_total = part;
      __syncthreads();
      if (tid == 0) {
        sh.S[nrej] = S;
        sh.Sinv[nrej] = 1.f / S;
      }
      __syncthreads();
    }
    if (kept >= 0) {
      if (rank == 0 && tid == 0) {
        L.out_tokens[(size_t)b * N + depth] = L.tok[(size_t)b * N + kept];
        L.out_nodes[(size_t)b * N + depth] = kept;
      }
      ++depth;
      u = kept;
      continue;
    }

    // ---- draw from the last residual (or p_u) ----
    // The last rejection pass computed exactly these weights: its chunk
    // sums and exchanged totals are reused. Otherwise (no child, or
    // the fallback) one pass over p_u.
    const int lev = fallback ? 0 : nrej;
    float total;
    if (lev > 0) {
      total = last_total;
    } else {
      total = slice_pass(L, m, lo, hi, 0, st, sh);
      if (kCW > 1) exchange<kCW>(total, sh.last_found, par, sh);
    }
    const int lastc = sh.last_found;
    float before = 0.f, S = total;
    int owner = rank;
    float t_all = 0.f;
    const float uu = sample_uniform(L.seed, b, depth);
    if (kCW > 1) {
      S = 0.f;
      for (int q = 0; q < kCW; ++q) S += sh.allv[q];
      t_all = uu * S;
      // The first CTA whose running total passes t; else the last with weight.
      float run = 0.f;
      owner = -1;
      int last_owner = -1;
      for (int q = 0; q < kCW; ++q) {
        if (owner < 0 && run + sh.allv[q] > t_all) {
          owner = q;
          before = run;
        }
        if (sh.alli[q] >= 0) last_owner = q;
        run += sh.allv[q];
      }
      if (owner < 0) {
        owner = last_owner < 0 ? 0 : last_owner;
        before = 3.0e38f;   // forces the last-weight token in the owner
      }
    } else {
      t_all = uu * S;
    }
    if (rank == owner) {
      const float t = before == 3.0e38f ? 3.0e38f : t_all - before;
      const int nch = (hi - lo + kTC - 1) / kTC;
      if (warp == 0) {
        chunk_prefix(nch, sh);
        int found = -1;
        for (int g = 0; g < nch && found < 0; g += 32) {
          const int k = g + lane;
          const unsigned hit = __ballot_sync(0xffffffffu, k < nch && sh.pre[k] > t);
          if (hit) found = g + __ffs(hit) - 1;
        }
        if (found < 0) found = lastc;   // t at or past the slice total: its last chunk with weight
        int tok = -1;
        if (found >= 0) {
          const float cb = found > 0 ? sh.pre[found - 1] : 0.f;
          float w[4];
          const int v0 = lo + found * kTC + 4 * lane;
          weights4(L, m, v0, hi, st, lev, sh.Sinv, w);
          const float ls = (w[0] + w[1]) + (w[2] + w[3]);
          float incl = ls;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          float run = cb + (incl - ls);
          int cand = 0x7fffffff, lastp = -1;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            run += w[e];
            if (w[e] > 0.f) lastp = v0 + e;
            if (cand == 0x7fffffff && w[e] > 0.f && run > t) cand = v0 + e;
          }
#pragma unroll
          for (int o = 16; o; o >>= 1) {
            cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
            lastp = max(lastp, __shfl_xor_sync(0xffffffffu, lastp, o));
          }
          tok = cand != 0x7fffffff ? cand : lastp;
        }
        if (lane == 0) L.out_tokens[(size_t)b * N + depth] = tok;
      }
    }
    break;
  }
  if (rank == 0) {
    for (int n = depth + 1 + tid; n < N; n += kThreads) L.out_tokens[(size_t)b * N + n] = -1;
    for (int n = depth + tid; n < N; n += kThreads) L.out_nodes[(size_t)b * N + n] = -1;
    if (tid == 0) L.n_accepted[b] = depth;
  }
  if (kCW > 1) cluster_sync_all();   // no CTA leaves while another may read its shared memory
}

}  // namespace

// How many clusters of kTreeClusterWide CTAs can run at once on this
// device (0 if the size is not available); cached per device.
int max_wide_clusters() {
  static int cache[64];
  static bool have[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!have[dev]) {
    int n = 0;
    bool refused = cudaFuncSetAttribute(tree_walk_kernel<kTreeClusterWide>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed,
                                        1) != cudaSuccess;
    if (!refused) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kTreeClusterWide);
      cfg.blockDim = dim3(kThreads);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kTreeClusterWide;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, tree_walk_kernel<kTreeClusterWide>, &cfg) !=
          cudaSuccess) {
        n = 0;
        refused = true;
      }
    }
    if (refused) cudaGetLastError();   // the size is not offered: clear that (non-sticky) error
    cache[dev] = n;
    have[dev] = true;
  }
  return cache[dev];
}

cudaError_t launch_tree_walk(const TreeLaunch& L, cudaStream_t stream) {
  const bool sample = L.mode == SPECDEC_SAMPLE;
  // Wider clusters halve every vocabulary pass, as long as every
  // sequence's cluster runs at once.
  const bool wide = sample && L.B <= max_wide_clusters();
  const int cw = sample ? (wide ? kTreeClusterWide : kTreeCluster) : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.B * cw);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cw;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (wide) return cudaLaunchKernelEx(&cfg, tree_walk_kernel<kTreeClusterWide>, L);
  if (sample) return cudaLaunchKernelEx(&cfg, tree_walk_kernel<kTreeCluster>, L);
  return cudaLaunchKernelEx(&cfg, tree_walk_kernel<1>, L);
}

}  // namespace specdec
