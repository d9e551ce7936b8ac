// The drafter's clustered LM head ("多詞元預測視覺化指南", section 高效嵌入器):
// score the hidden state against one embedding per token cluster, keep the
// top-k clusters, compute token logits for their members only, and draw the
// draft token from the softmax over those members.
//
// Four small kernels, each a programmatic dependent of the one before
// (three for one kept cluster and M <= 8: the member kernel then selects it):
//   cluster_logits   y[m, c] = h_m . E_c          one warp per cluster
//   top_clusters     the k largest y per row      one CTA per row
//   member_logits    z = h_m . W_r for kept rows  one kept row per warp
//   draw             argmax, or the inverse CDF of softmax(z / T) in token-ID
//                    order (members sorted by token ID in shared memory)
// Bytes: n_c * d * 2 (cluster table) + kept rows * d * 2 per row, against
// V * d * 2 for the full head; every kernel is latency-bound at these sizes.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerChunk = 16;   // hidden rows staged in shared memory at once
constexpr int kRowGroup = 8;        // hidden rows a warp dots with its cluster row together
constexpr int kRankPer = 1;         // members per thread when the draw orders them by counting
constexpr int kFuseRows = 8;        // rows up to which (one kept cluster) the member kernel selects it
constexpr int kMaxPieces = SPECDEC_CLUSTER_MAX_D / 256;   // 16-byte pieces of a row per lane
static_assert(kMaxPieces == 16, "cluster_logits instantiations cover d up to 4096");
constexpr int kMemberBlock = kWarps;   // member rows per CTA of member_logits: one per warp
constexpr int kDotDepth = 4;            // 16-byte loads a lane keeps in flight in warp_dot

// Dot product of one bf16 row of length d (16-byte aligned, d % 8 == 0)
// with hidden row hs (shared memory, bf16), reduced over the warp. Each lane
// issues kDotDepth loads before it consumes any, so one warp keeps
// 32 * kDotDepth * 16 bytes of the row in flight.
__device__ __forceinline__ float warp_dot(const __nv_bfloat16* __restrict__ row,
                                          const __nv_bfloat16* hs, int d) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int j0 = lane * 8; j0 < d; j0 += 256 * kDotDepth) {
    uint4 a[kDotDepth];
#pragma unroll
    for (int u = 0; u < kDotDepth; ++u) {
      const int j = j0 + u * 256;
      a[u] = j < d ? __ldg(reinterpret_cast<const uint4*>(row + j)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kDotDepth; ++u) {
      const int j = j0 + u * 256;
      if (j >= d) break;
      const uint4 b = *reinterpret_cast<const uint4*>(hs + j);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(pa[e]);
        const float2 y = __bfloat1622float2(pb[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
  }
  return warp_sum(acc);
}

// kPieces: 16-byte pieces per lane the instantiation holds (d <= kPieces * 256).
template <int kPieces>
__global__ void __launch_bounds__(kThreads) cluster_logits_kernel(const ClusterLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_h[];
  __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(smem_h);
  grid_launch_dependents();
  grid_dependency_wait();
  // The status word is cleared here, after the previous work on the stream
  // has finished; the later kernels of the chain only set it.
  if (blockIdx.x == 0 && threadIdx.x == 0) *L.status = SPECDEC_OK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kWarps + warp;
  // With kRowGroup rows or more, the warp's cluster embedding stays in
  // registers (16-byte piece k of the row at lane * 8 + k * 256) and hidden
  // rows are dotted with it kRowGroup at a time, so their reductions
  // overlap.
  const int npc = L.d / 256 + ((lane * 8) < (L.d % 256) ? 1 : 0);   // pieces this lane holds
  uint4 e[kPieces];
#pragma unroll
  for (int k = 0; k < kPieces; ++k)
    e[k] = (c < L.n_c && k < npc && L.M >= kRowGroup)
               ? __ldg(reinterpret_cast<const uint4*>(L.E + (size_t)c * L.d + lane * 8 + k * 256))
               : make_uint4(0u, 0u, 0u, 0u);
  for (int m0 = 0; m0 < L.M; m0 += kRowsPerChunk) {
    const int nm = min(kRowsPerChunk, L.M - m0);
    __syncthreads();
    for (int q = threadIdx.x; q < nm * L.d / 8; q += kThreads)
      reinterpret_cast<uint4*>(hs)[q] = __ldg(reinterpret_cast<const uint4*>(L.h + (size_t)m0 * L.d) + q);
    __syncthreads();
    if (c >= L.n_c) continue;
    if (L.M < kRowGroup) {   // few rows: one dot at a time, the row streamed from L2
      for (int m = 0; m < nm; ++m) {
        const float y = warp_dot(L.E + (size_t)c * L.d, hs + (size_t)m * L.d, L.d);
        if (lane == 0) L.y[(size_t)(m0 + m) * L.n_c + c] = y;
      }
      continue;
    }
    for (int g0 = 0; g0 < nm; g0 += kRowGroup) {
      float acc[kRowGroup];
#pragma unroll
      for (int j = 0; j < kRowGroup; ++j) acc[j] = 0.f;
#pragma unroll
      for (int k = 0; k < kPieces; ++k) {
        if (k >= npc) break;
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&e[k]);
#pragma unroll
        for (int j = 0; j < kRowGroup; ++j) {
          if (g0 + j >= nm) break;
          const uint4 b = *reinterpret_cast<const uint4*>(hs + (size_t)(g0 + j) * L.d + lane * 8 + k * 256);
          const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 x = __bfloat1622float2(pa[q]);
            const float2 y = __bfloat1622float2(pb[q]);
            acc[j] = fmaf(x.x, y.x, acc[j]);
            acc[j] = fmaf(x.y, y.y, acc[j]);
          }
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int j = 0; j < kRowGroup; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
      if (lane == 0)
#pragma unroll
        for (int j = 0; j < kRowGroup; ++j)
          if (g0 + j < nm) L.y[(size_t)(m0 + g0 + j) * L.n_c + c] = acc[j];
    }
  }
}

// The top_k largest cluster logits of row m (ties to the lower index) into
// sel, and the kept members' offsets and first table rows into off
// [top_k + 1] and row0 (all shared). With `publish`, the kept clusters and
// offsets also go to global memory for the later kernels, and a kept
// cluster larger than max_cluster is reported. Every thread of the CTA
// calls it.
__device__ __forceinline__ void select_clusters(const ClusterLaunch& L, int m, bool publish,
                                                int* sel, int* off, int* row0, float* s_v,
                                                int* s_i) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* y = L.y + (size_t)m * L.n_c;
  for (int k = 0; k < L.top_k; ++k) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int c = threadIdx.x; c < L.n_c; c += kThreads) {
      bool taken = false;
      for (int j = 0; j < k; ++j) taken |= sel[j] == c;
      const float v = y[c];
      if (!taken && argmax_better(v, c, bv, bi)) {
        bv = v;
        bi = c;
      }
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      s_v[warp] = bv;
      s_i[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kWarps; ++w)
        if (argmax_better(s_v[w], s_i[w], bv, bi)) {
          bv = s_v[w];
          bi = s_i[w];
        }
      sel[k] = bi;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int o = 0;
    bool bad = false;
    for (int k = 0; k < L.top_k; ++k) {
      const int c = sel[k];
      const int r0 = L.starts[c];
      const int n = L.starts[c + 1] - r0;
      bad |= n < 0 || n > L.max_cluster;
      off[k] = o;
      row0[k] = r0;
      if (publish) {
        L.clusters[(size_t)m * L.top_k + k] = c;
        L.offs[(size_t)m * (L.top_k + 1) + k] = o;
      }
      o += max(0, min(n, L.max_cluster));
    }
    off[L.top_k] = o;
    if (publish) {
      L.offs[(size_t)m * (L.top_k + 1) + L.top_k] = o;
      if (bad) set_status(L.status, SPECDEC_ERR_INVALID_ARG);
    }
  }
  __syncthreads();
}

// The kept clusters of row m and their members' table rows, in kept order,
// so the member kernel reads each row with one load (it replaces them by
// token IDs).
__global__ void __launch_bounds__(kThreads) top_clusters_kernel(const ClusterLaunch L) {
  __shared__ float s_v[kWarps];
  __shared__ int s_i[kWarps];
  __shared__ int s_sel[SPECDEC_CLUSTER_MAX_TOP_K];
  __shared__ int s_off[SPECDEC_CLUSTER_MAX_TOP_K + 1], s_row0[SPECDEC_CLUSTER_MAX_TOP_K];
  grid_launch_dependents();
  grid_dependency_wait();
  const int m = blockIdx.x;
  select_clusters(L, m, true, s_sel, s_off, s_row0, s_v, s_i);
  for (int k = 0; k < L.top_k; ++k)
    for (int i = s_off[k] + threadIdx.x; i < s_off[k + 1]; i += kThreads)
      L.ids[(size_t)m * L.max_members + i] = s_row0[k] + (i - s_off[k]);
}

// Logits of kept member rows: CTA (block, m) takes members
// [8 * block, 8 * block + 8) of row m's kept list, one per warp; each
// member's table row comes from ids[m, i], which then takes its token ID.
__global__ void __launch_bounds__(kThreads) member_logits_kernel(const ClusterLaunch L) {
  __shared__ __align__(16) __nv_bfloat16 hs[SPECDEC_CLUSTER_MAX_D];
  grid_launch_dependents();
  grid_dependency_wait();
  const int m = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* offs = L.offs + (size_t)m * (L.top_k + 1);
  const int total = offs[L.top_k];
  const int i0 = blockIdx.x * kMemberBlock;
  if (i0 >= total) return;
  for (int e = threadIdx.x; e < L.d / 8; e += kThreads)
    reinterpret_cast<uint4*>(hs)[e] = __ldg(reinterpret_cast<const uint4*>(L.h + (size_t)m * L.d) + e);
  __syncthreads();
  for (int i = i0 + warp; i < min(total, i0 + kMemberBlock); i += kWarps) {
    const int r = L.ids[(size_t)m * L.max_members + i];   // table row (written by top_clusters)
    if (r < 0 || r >= L.V) {   // starts outside the table: report, read nothing
      if (lane == 0) set_status(L.status, SPECDEC_ERR_INVALID_ARG);
      continue;
    }
    const float z = warp_dot(L.W + (size_t)r * L.d, hs, L.d);
    if (lane == 0) {
      const int id = L.token_of_row[r];
      L.z[(size_t)m * L.max_members + i] = z;
      L.ids[(size_t)m * L.max_members + i] = id;
      if (L.logits_out != nullptr && id >= 0 && id < L.V) L.logits_out[(size_t)m * L.V + id] = z;
    }
  }
}

// One kept cluster and at most kFuseRows rows: the member kernel selects
// the cluster itself (every CTA of row m the same way; CTA 0 of the row
// publishes it), saving the top-k kernel and its launch.
__global__ void __launch_bounds__(kThreads) member_logits_fused_kernel(const ClusterLaunch L) {
  __shared__ __align__(16) __nv_bfloat16 hs[SPECDEC_CLUSTER_MAX_D];
  __shared__ float s_v[kWarps];
  __shared__ int s_i[kWarps];
  __shared__ int s_sel[SPECDEC_CLUSTER_MAX_TOP_K];
  __shared__ int s_off[SPECDEC_CLUSTER_MAX_TOP_K + 1], s_row0[SPECDEC_CLUSTER_MAX_TOP_K];
  grid_launch_dependents();
  grid_dependency_wait();
  const int m = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < L.d / 8; e += kThreads)
    reinterpret_cast<uint4*>(hs)[e] = __ldg(reinterpret_cast<const uint4*>(L.h + (size_t)m * L.d) + e);
  select_clusters(L, m, blockIdx.x == 0, s_sel, s_off, s_row0, s_v, s_i);   // ends with a barrier
  const int total = s_off[L.top_k];
  const int i0 = blockIdx.x * kMemberBlock;
  for (int i = i0 + warp; i < min(total, i0 + kMemberBlock); i += kWarps) {
    int k = 0;
    while (k + 1 < L.top_k && s_off[k + 1] <= i) ++k;
    const int r = s_row0[k] + (i - s_off[k]);
    if (r < 0 || r >= L.V) {   // starts outside the table: report, read nothing
      if (lane == 0) set_status(L.status, SPECDEC_ERR_INVALID_ARG);
      continue;
    }
    const float z = warp_dot(L.W + (size_t)r * L.d, hs, L.d);
    if (lane == 0) {
      const int id = L.token_of_row[r];
      L.z[(size_t)m * L.max_members + i] = z;
      L.ids[(size_t)m * L.max_members + i] = id;
      if (L.logits_out != nullptr && id >= 0 && id < L.V) L.logits_out[(size_t)m * L.V + id] = z;
    }
  }
}

// Draft token of row m: members put in token-ID order in shared memory (by
// counting ranks up to 256 members, else a bitonic sort), then the greedy
// argmax or the inverse CDF of softmax(z / T).
__global__ void __launch_bounds__(kThreads) draw_kernel(const ClusterLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_d[];
  int* sid = reinterpret_cast<int*>(smem_d);
  float* sz = reinterpret_cast<float*>(sid + L.sort_n);
  __shared__ float s_red[kWarps];
  __shared__ int s_redi[kWarps];
  __shared__ int s_tok, s_last;
  grid_dependency_wait();
  const int m = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = L.offs[(size_t)m * (L.top_k + 1) + L.top_k];
  const int n = L.sort_n;   // power of two >= max_members
  if (total <= kRankPer * kThreads) {
    // Up to kRankPer member(s) per thread: a member's place in token-ID order
    // is the number of members before it (lower ID, or equal ID and lower
    // index), counted against all IDs staged in shared memory (the z area
    // holds them).
    int* sin = reinterpret_cast<int*>(sz);
    int my_id[kRankPer], rank[kRankPer];
    float my_z[kRankPer];
#pragma unroll
    for (int u = 0; u < kRankPer; ++u) {
      const int t = threadIdx.x + u * kThreads;
      my_id[u] = t < total ? L.ids[(size_t)m * L.max_members + t] : 0;
      my_z[u] = t < total ? L.z[(size_t)m * L.max_members + t] : 0.f;
      rank[u] = 0;
      if (t < total) sin[t] = my_id[u];
    }
    __syncthreads();
    for (int j = 0; j < total; ++j) {
      const int o = sin[j];
#pragma unroll
      for (int u = 0; u < kRankPer; ++u) {
        const int t = threadIdx.x + u * kThreads;
        rank[u] += (o < my_id[u] || (o == my_id[u] && j < t)) ? 1 : 0;
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kRankPer; ++u) {
      const int t = threadIdx.x + u * kThreads;
      if (t < total) {
        sid[rank[u]] = my_id[u];
        sz[rank[u]] = my_z[u];
      }
    }
    __syncthreads();
  } else {
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const bool in = i < total;
    sid[i] = in ? L.ids[(size_t)m * L.max_members + i] : 0x7fffffff;
    sz[i] = in ? L.z[(size_t)m * L.max_members + i] : -INFINITY;
  }
  __syncthreads();
  // bitonic sort by token ID (ascending)
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          if ((sid[i] > sid[j]) == up) {
            const int ti = sid[i];
            sid[i] = sid[j];
            sid[j] = ti;
            const float tz = sz[i];
            sz[i] = sz[j];
            sz[j] = tz;
          }
        }
      }
      __syncthreads();
    }
  }
  // max logit (and its lowest token ID: members are in token-ID order)
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < total; i += kThreads)
    if (argmax_better(sz[i], sid[i], bv, bi)) {
      bv = sz[i];
      bi = sid[i];
    }
  warp_argmax(bv, bi);
  if (lane == 0) {
    s_red[warp] = bv;
    s_redi[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kWarps; ++w)
      if (argmax_better(s_red[w], s_redi[w], bv, bi)) {
        bv = s_red[w];
        bi = s_redi[w];
      }
    s_red[0] = bv;
    s_redi[0] = bi;
  }
  __syncthreads();
  const float zmax = s_red[0];
  if (!L.sample) {
    if (threadIdx.x == 0) L.tokens[m] = total > 0 ? s_redi[0] : -1;
    return;
  }
  // Weights exp2((z - zmax) c) in token-ID order; the draw inverts their
  // prefix sum at u * S: contiguous segments per thread, a block scan of the
  // segment sums, then the first weighted token whose running sum passes t.
  for (int i = threadIdx.x; i < total; i += kThreads) sz[i] = exp2f((sz[i] - zmax) * L.c);
  __syncthreads();
  const int per = (total + kThreads - 1) / kThreads;
  const int a = min(total, threadIdx.x * per), e = min(total, a + per);
  float ts = 0.f;
  for (int i = a; i < e; ++i) ts += sz[i];
  float incl = ts;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_red[warp] = incl;
  if (threadIdx.x == 0) {
    s_tok = 0x7fffffff;
    s_last = -1;
  }
  __syncthreads();
  float before = 0.f, S = 0.f;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += s_red[w];
    S += s_red[w];
  }
  const float t = draft_uniform(L.seed, m, L.position) * S;
  float run = before + (incl - ts);
  int cand = 0x7fffffff, lastp = -1;
  for (int i = a; i < e; ++i) {
    run += sz[i];
    if (sz[i] > 0.f) lastp = sid[i];
    if (cand == 0x7fffffff && sz[i] > 0.f && run > t) cand = sid[i];
  }
  if (cand != 0x7fffffff) atomicMin(&s_tok, cand);
  if (lastp >= 0) atomicMax(&s_last, lastp);
  __syncthreads();
  if (threadIdx.x == 0) L.tokens[m] = s_tok != 0x7fffffff ? s_tok : s_last;   // t rounded past S
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, const ClusterLaunch& L,
                       cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<ClusterLaunch*>(&L)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_cluster_head(const ClusterLaunch& L, cudaStream_t stream) {
  const size_t smem1 = (size_t)kRowsPerChunk * L.d * 2;
  const size_t smem4 = (size_t)L.sort_n * 8;
  static int set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !set[dev]) {
    e = cudaFuncSetAttribute(cluster_logits_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRowsPerChunk * SPECDEC_CLUSTER_MAX_D * 2);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(cluster_logits_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRowsPerChunk * SPECDEC_CLUSTER_MAX_D * 2);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(draw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SPECDEC_CLUSTER_MAX_MEMBERS * 8);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) set[dev] = 1;
  }
  const void* logits_fn = L.d <= 8 * 256 ? (const void*)cluster_logits_kernel<8>
                                         : (const void*)cluster_logits_kernel<16>;
  e = launch_pdl(logits_fn, dim3((L.n_c + kWarps - 1) / kWarps),
                 dim3(kThreads), smem1, L, stream);
  if (e != cudaSuccess) return e;
  const dim3 member_grid((L.max_members + kMemberBlock - 1) / kMemberBlock, L.M);
  if (L.top_k == 1 && L.M <= kFuseRows) {
    e = launch_pdl((const void*)member_logits_fused_kernel, member_grid, dim3(kThreads), 0, L,
                   stream);
  } else {
    e = launch_pdl((const void*)top_clusters_kernel, dim3(L.M), dim3(kThreads), 0, L, stream);
    if (e != cudaSuccess) return e;
    e = launch_pdl((const void*)member_logits_kernel, member_grid, dim3(kThreads), 0, L, stream);
  }
  if (e != cudaSuccess) return e;
  return launch_pdl((const void*)draw_kernel, dim3(L.M), dim3(kThreads), smem4, L, stream);
}

}  // namespace specdec
