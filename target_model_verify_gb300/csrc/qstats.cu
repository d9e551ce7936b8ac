// Softmax statistics of the draft logits (q), as a standalone stream.
//
// "推测解码" (world.lapla.si/zh/specdec), section 通过的规则: q is the small
// model's probability, softmax(draft_logits / T). Its normaliser does not
// depend on the target, so with many draft rows it is computed here, before
// the LM-head kernel, at full streaming bandwidth: one warp per draft row
// and 8192-column chunk, 16-byte loads (8 bf16) with 8 in flight per lane.
// Each (row, chunk) leaves one (max, sum exp2((x - max) * c)) record.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kThreads = 128;     // 4 warps = 4 draft rows per CTA
constexpr int kCols = kQChunk;    // columns per record
constexpr int kInFlight = 8;      // 16-byte loads per lane in flight

__device__ __forceinline__ void fold8(float& m, float& s, const uint4& u, float c) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
  float x[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    x[2 * k] = f.x;
    x[2 * k + 1] = f.y;
  }
  float mx = x[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) mx = fmaxf(mx, x[k]);
  const float mm = fmaxf(m, mx);
  if (mm == -INFINITY) return;   // nothing seen yet: (m, s) stays (-inf, 0)
  float acc = m == -INFINITY ? 0.f : s * exp2f((m - mm) * c);
#pragma unroll
  for (int k = 0; k < 8; ++k) acc += exp2f((x[k] - mm) * c);
  m = mm;
  s = acc;
}

__global__ void __launch_bounds__(kThreads) qstats_kernel(const __nv_bfloat16* __restrict__ dl,
                                                          int n_rows, int V, float c,
                                                          PartialQ* __restrict__ pq, int Pq,
                                                          int vec_ok) {
  grid_dependency_wait();   // programmatic dependent launch: inputs are ready after this
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * (kThreads / 32) + warp;
  if (r >= n_rows) return;
  const int chunk = blockIdx.y;
  const int c0 = chunk * kCols;
  const int c1 = min(V, c0 + kCols);
  const __nv_bfloat16* row = dl + (size_t)r * V;
  float m = -INFINITY, s = 0.f;
  if (vec_ok) {
    // Whole 8-element groups in [c0, c1); V % 8 == 0 and a 16-byte aligned base.
    const uint4* base = reinterpret_cast<const uint4*>(row + c0);
    const int n8 = (c1 - c0) / 8;
    for (int t0 = lane; t0 < n8; t0 += 32 * kInFlight) {
      uint4 u[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int t = t0 + 32 * k;
        u[k] = t < n8 ? __ldcs(base + t) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) fold8(m, s, u[k], c);
    }
  } else {
    for (int v = c0 + lane; v < c1; v += 32) {
      const float x = __bfloat162float(row[v]);
      const float mm = fmaxf(m, x);
      if (mm == -INFINITY) continue;
      s = (m == -INFINITY ? 0.f : s * exp2f((m - mm) * c)) + exp2f((x - mm) * c);
      m = mm;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    osm_merge(m, s, m2, s2, c);
  }
  if (lane == 0) pq[(size_t)r * Pq + chunk] = PartialQ{m, s};
}

}  // namespace

cudaError_t launch_qstats(const __nv_bfloat16* dl, int n_rows, int V, float c, PartialQ* pq,
                          cudaStream_t stream) {
  const int n_chunks = (V + kCols - 1) / kCols;
  const int vec_ok = (V % 8 == 0 && ((uintptr_t)dl & 15u) == 0) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n_rows + kThreads / 32 - 1) / (kThreads / 32), n_chunks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qstats_kernel, dl, n_rows, V, c, pq, n_chunks, vec_ok);
}

}  // namespace specdec
