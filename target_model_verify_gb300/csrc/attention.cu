// Verify-step attention: the gamma + 1 new positions of every sequence over
// its KV cache, for one layer.
//
// "推测解码" (world.lapla.si/zh/specdec), section 几段话一起写: each sequence
// has its own KV cache that every step must read; at batch 64 with 4,096
// cached tokens that read outweighs the weights. New position i of sequence
// b (at P = seq_len - n_new + i) attends to cache rows 0..P; query head h
// reads KV head h / G (grouped-query attention).
//
// Bound: HBM (K and V are read once; about 20 flop per byte at G = 4,
// n_new = 5), so the contractions run on the warp-level tensor-core MMA
// (mma.sync m16n8k16, bf16 in, fp32 accumulate), which keeps pace with the
// memory stream; the K/V blocks move with cp.async into swizzled shared
// memory, double-buffered. Split-KV ("flash decoding"): CTA (split, kv head,
// b) takes one contiguous key range for all R = n_new * G query rows of that
// KV head; each m16 row tile has two warps, one per half of every 64-key
// block; online softmax in registers (log2 domain); partials (max, sum,
// unnormalised output) merged across splits by a second kernel.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kD = 128;            // head dimension
constexpr int kBlk = 64;           // keys per block (two warp halves of 32)
constexpr int kRowBytes = kD * 2;  // one key / query row in shared memory
constexpr int kStages = 3;         // K/V blocks in flight per CTA

// Byte offset of 16-byte chunk c of row r in a swizzled [rows][128] bf16 tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Issue the cp.async copies of key block [j0, j0 + 64) of K and V (rows at
// or past Lmax are zero-filled without reading).
__device__ __forceinline__ void load_block(const AttnLaunch& A, int b, int hkv, int j0,
                                           uint32_t ks, uint32_t vs) {
  const size_t row_stride = (size_t)A.Hkv * kD;   // elements between consecutive keys
  for (int e = threadIdx.x; e < kBlk * 16; e += blockDim.x) {
    const int r = e >> 4, c = e & 15;
    const int j = j0 + r;
    const bool ok = j < A.Lmax;
    const size_t off = ((size_t)b * A.Lmax + (ok ? j : 0)) * row_stride + (size_t)hkv * kD + c * 8;
    cp_async16(ks + swz(r, c), A.k + off, ok);
    cp_async16(vs + swz(r, c), A.v + off, ok);
  }
}

__global__ void __launch_bounds__(256) attn_split_kernel(const AttnLaunch A) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = warp >> 1;          // m16 row tile
  const int kh = warp & 1;           // which 32 keys of each block
  const int g = lane >> 2, t = lane & 3;
  const int G = A.Hq / A.Hkv;
  const int R = A.n_new * G;
  // shared memory: Q [64 rows], then kStages stages of K [64] and V [64]
  const uint32_t qs = smem_u32(smem);
  const uint32_t stage0 = qs + 64 * kRowBytes;
  auto kst = [&](int s) { return stage0 + (uint32_t)s * 2u * kBlk * kRowBytes; };
  auto vst = [&](int s) { return kst(s) + (uint32_t)kBlk * kRowBytes; };

  grid_dependency_wait();
  const int L = A.seq_lens[b];
  const bool bad = L < A.n_new || L > A.Lmax;
  if (bad) {
    if (split == 0 && hkv == 0 && threadIdx.x == 0) set_status(A.status, SPECDEC_ERR_INVALID_ARG);
  }
  const int j_begin = split * A.split_len;
  const int j_end = bad ? j_begin : min(L, j_begin + A.split_len);

  // Q rows r = i * G + gq (query i, head hkv * G + gq); rows >= R are zero.
  for (int e = threadIdx.x; e < 64 * 16; e += blockDim.x) {
    const int r = e >> 4, c = e & 15;
    const bool ok = r < R;
    const int i = ok ? r / G : 0, gq = ok ? r % G : 0;
    const size_t off = (((size_t)b * A.n_new + i) * A.Hq + (size_t)hkv * G + gq) * kD + c * 8;
    cp_async16(qs + swz(r, c), A.q + off, ok);
  }
  // Q and the first kStages - 1 blocks, one commit group each.
#pragma unroll
  for (int p = 0; p < kStages - 1; ++p) {
    const int jp = j_begin + p * kBlk;
    if (jp < j_end) load_block(A, b, hkv, jp, kst(p), vst(p));
    cp_async_commit();
  }

  float m_run[2] = {-INFINITY, -INFINITY};   // rows g and g + 8 of this tile (log2 units)
  float l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  uint32_t qf[8][4];
  bool q_loaded = false;
  const int row0 = mt * 16 + g;              // tile rows of this thread: row0, row0 + 8
  const int qi0 = row0 < R ? row0 / G : 0;
  const int qi1 = row0 + 8 < R ? (row0 + 8) / G : 0;
  const int vis0 = L - A.n_new + qi0;        // last visible key of each row
  const int vis1 = L - A.n_new + qi1;

  int s = 0;
  for (int j0 = j_begin; j0 < j_end; j0 += kBlk) {
    {
      const int jn = j0 + (kStages - 1) * kBlk;
      const int sn = (s + kStages - 1) % kStages;
      if (jn < j_end) load_block(A, b, hkv, jn, kst(sn), vst(sn));
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();
    if (!q_loaded) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        ldsm_x4(qs + swz(mt * 16 + (lane & 15), ks * 2 + (lane >> 4)), qf[ks]);
      q_loaded = true;
    }
    // S = Q K^T for this warp's 32 keys: 4 tiles of 8
    float sc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
    const uint32_t kb = kst(s), vb = vst(s);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t r[4];
        const int key = kh * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(kb + swz(key, ks * 2 + ((lane >> 3) & 1)), r);
        mma16816(sc[2 * np], qf[ks], r[0], r[1]);
        mma16816(sc[2 * np + 1], qf[ks], r[2], r[3]);
      }
    }
    // scale, mask, online softmax (rows g and g + 8)
    float bmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + kh * 32 + n * 8 + 2 * t + (e & 1);
        const int vis = e < 2 ? vis0 : vis1;
        const float x = (j <= vis && j < j_end) ? sc[n][e] * A.scale_log2 : -INFINITY;
        sc[n][e] = x;
        bmax[e >> 1] = fmaxf(bmax[e >> 1], x);
      }
    float alpha[2], m_use[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      bmax[h] = fmaxf(bmax[h], __shfl_xor_sync(0xffffffffu, bmax[h], 1));
      bmax[h] = fmaxf(bmax[h], __shfl_xor_sync(0xffffffffu, bmax[h], 2));
      const float m_new = fmaxf(m_run[h], bmax[h]);
      m_use[h] = m_new == -INFINITY ? 0.f : m_new;   // nothing visible yet
      alpha[h] = exp2f(m_run[h] - m_use[h]);          // m_run = -inf gives 0
      m_run[h] = m_new;
      l_run[h] *= alpha[h];
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    uint32_t pa[2][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const float p0 = exp2f(sc[n][0] - m_use[0]), p1 = exp2f(sc[n][1] - m_use[0]);
      const float p2 = exp2f(sc[n][2] - m_use[1]), p3 = exp2f(sc[n][3] - m_use[1]);
      l_run[0] += p0 + p1;
      l_run[1] += p2 + p3;
      pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
      pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    // O += P V over this warp's 32 keys (2 steps of 16) and 128 dims (16 tiles)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t r[4];
        const int key = kh * 32 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        ldsm_x4_t(vb + swz(key, dp * 2 + (lane >> 4)), r);
        mma16816(o[2 * dp], pa[kk], r[0], r[1]);
        mma16816(o[2 * dp + 1], pa[kk], r[2], r[3]);
      }
    }
    __syncthreads();   // this stage is refilled kStages - 1 blocks later
    s = (s + 1) % kStages;
  }
  cp_async_wait<0>();
  __syncthreads();

  // Row sums across the quad, then merge the two key-half warps of a tile
  // through shared memory (the stage buffers are free now).
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  float* xo = reinterpret_cast<float*>(smem + 64 * kRowBytes) + mt * (16 * kD + 32);
  float* xm = xo + 16 * kD;
  float* xl = xm + 16;
  if (kh == 1) {
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      xo[g * kD + n * 8 + 2 * t] = o[n][0];
      xo[g * kD + n * 8 + 2 * t + 1] = o[n][1];
      xo[(g + 8) * kD + n * 8 + 2 * t] = o[n][2];
      xo[(g + 8) * kD + n * 8 + 2 * t + 1] = o[n][3];
    }
    if (t == 0) {
      xm[g] = m_run[0];
      xm[g + 8] = m_run[1];
      xl[g] = l_run[0];
      xl[g + 8] = l_run[1];
    }
  }
  __syncthreads();
  if (kh == 1) return;
  float w_self[2], w_other[2], m_tot[2], l_tot[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float mo = xm[g + 8 * h], lo = xl[g + 8 * h];
    const float M = fmaxf(m_run[h], mo);
    const float Mu = M == -INFINITY ? 0.f : M;
    w_self[h] = exp2f(m_run[h] - Mu);
    w_other[h] = exp2f(mo - Mu);
    m_tot[h] = M;
    l_tot[h] = l_run[h] * w_self[h] + lo * w_other[h];
  }
  const int rows[2] = {row0, row0 + 8};
  if (A.n_splits == 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rows[h];
      if (r >= R) continue;
      const int i = r / G, gq = r % G;
      float* dst = A.out + (((size_t)b * A.n_new + i) * A.Hq + (size_t)hkv * G + gq) * kD;
      const float inv = l_tot[h] > 0.f ? 1.f / l_tot[h] : 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const float a0 = o[n][2 * h] * w_self[h] + xo[(g + 8 * h) * kD + n * 8 + 2 * t] * w_other[h];
        const float a1 =
            o[n][2 * h + 1] * w_self[h] + xo[(g + 8 * h) * kD + n * 8 + 2 * t + 1] * w_other[h];
        *reinterpret_cast<float2*>(dst + n * 8 + 2 * t) = make_float2(a0 * inv, a1 * inv);
      }
    }
    return;
  }
  // Partial of this split: (max, sum) per row and the unnormalised output.
  const size_t base = (((size_t)b * A.Hkv + hkv) * A.n_splits + split) * 64;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = rows[h];
    if (r >= R) continue;
    float* po = A.part_o + (base + r) * kD;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const float a0 = o[n][2 * h] * w_self[h] + xo[(g + 8 * h) * kD + n * 8 + 2 * t] * w_other[h];
      const float a1 =
          o[n][2 * h + 1] * w_self[h] + xo[(g + 8 * h) * kD + n * 8 + 2 * t + 1] * w_other[h];
      *reinterpret_cast<float2*>(po + n * 8 + 2 * t) = make_float2(a0, a1);
    }
    if (t == 0) {
      A.part_m[base + r] = m_tot[h];
      A.part_l[base + r] = l_tot[h];
    }
  }
}

// Merge the splits: one warp per (b, kv head, row), 4 dims per lane.
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnLaunch A) {
  grid_dependency_wait();
  const int G = A.Hq / A.Hkv;
  const int R = A.n_new * G;
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= (long long)A.B * A.Hkv * R) return;
  const int r = (int)(w % R);
  const int hkv = (int)((w / R) % A.Hkv);
  const int b = (int)(w / ((long long)R * A.Hkv));
  const size_t base = ((size_t)b * A.Hkv + hkv) * A.n_splits * 64;
  float M = -INFINITY;
  for (int s = 0; s < A.n_splits; ++s) M = fmaxf(M, A.part_m[base + (size_t)s * 64 + r]);
  const float Mu = M == -INFINITY ? 0.f : M;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  for (int s = 0; s < A.n_splits; ++s) {
    const size_t k = base + (size_t)s * 64 + r;
    const float wgt = exp2f(A.part_m[k] - Mu);
    l += A.part_l[k] * wgt;
    const float4 v = reinterpret_cast<const float4*>(A.part_o + k * kD)[lane];
    acc.x += v.x * wgt;
    acc.y += v.y * wgt;
    acc.z += v.z * wgt;
    acc.w += v.w * wgt;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int i = r / G, gq = r % G;
  float* dst = A.out + (((size_t)b * A.n_new + i) * A.Hq + (size_t)hkv * G + gq) * kD;
  reinterpret_cast<float4*>(dst)[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

}  // namespace

int attn_smem_bytes() { return 64 * kRowBytes + kStages * 2 * kBlk * kRowBytes; }

cudaError_t launch_attention(const AttnLaunch& A, cudaStream_t stream) {
  const int G = A.Hq / A.Hkv;
  const int n_mt = (A.n_new * G + 15) / 16;
  const int smem = attn_smem_bytes();
  static int smem_set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !smem_set[dev]) {
    e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) smem_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(A.n_splits, A.Hkv, A.B);
  cfg.blockDim = dim3(64 * n_mt);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_split_kernel, A);
  if (e != cudaSuccess || A.n_splits == 1) return e;
  const long long warps = (long long)A.B * A.Hkv * A.n_new * G;
  cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, A);
}

}  // namespace specdec
