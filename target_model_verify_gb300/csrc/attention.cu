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
// memory stream as long as few instructions surround it. Split-KV ("flash
// decoding"): CTA (split, kv head, b) takes one contiguous key range for all
// R = n_new * G query rows of that KV head. One producer thread moves each
// 64-key block of K and V with four TMA tensor copies (64 keys x 64 dims,
// 128-byte swizzle) into a ring of stages guarded by mbarriers; each m16
// row tile has two consumer warps, one per half of every block, whose
// ldmatrix addresses are fixed per thread up to the stage base. Online
// softmax in registers (log2 domain, the scale folded into the exponent,
// masks only on the blocks that need them, the output rescaled only when a
// row maximum moved); partials (max, sum, unnormalised output) are merged
// across splits by a second kernel.
#include "kernels.h"

namespace specdec {
namespace {

constexpr int kD = 128;                  // head dimension
constexpr int kBlk = 64;                 // keys per block (two warp halves of 32)
constexpr int kQRowBytes = kD * 2;       // one query row in shared memory
constexpr int kHalf = kBlk * 128;        // 64 keys x 64 dims of bf16: one TMA box, 8 KB
constexpr int kStageBytes = 4 * kHalf;   // K and V, two halves each: 32 KB
constexpr unsigned long long kAttnDrainNs = 1000000000ull;

// Byte offset of 16-byte chunk c of query row r in a swizzled [rows][256 B] tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * kQRowBytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
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
// 2^x by the PTX approximate base-2 exponential (flushes subnormals; -inf
// gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 4-D tiled TMA load completing on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tmap, uint32_t bar,
                                            int x, int y, int z, int w, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}
// Wait for copies already issued, with its own time limit (after a give-up).
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kAttnDrainNs) return false;
  return true;
}

// Shared memory (dynamic, aligned up to 1024 bytes here): n_stages stages
// of [K dims 0-63 | K dims 64-127 | V dims 0-63 | V dims 64-127], each part
// 64 keys x 128 bytes in the TMA 128-byte swizzle (16-byte chunk c of key
// row r at r * 128 + ((c ^ (r & 7)) << 4)); then the n_mt * 16 query rows;
// then the full and empty barriers of every stage and the give-up flag.
__global__ void __launch_bounds__(288) attn_split_kernel(const AttnLaunch A,
                                                        const __grid_constant__ CUtensorMap tmap_k,
                                                        const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = A.Hq / A.Hkv;
  const int R = A.n_new * G;
  const int n_mt = (R + 15) >> 4;
  const int n_cons = 2 * n_mt;             // consumer warps; warp n_cons is the producer
  const int S = A.n_stages;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t stage0 = (raw + 1023u) & ~1023u;
  const uint32_t qs = stage0 + (uint32_t)S * kStageBytes;
  const uint32_t bars = qs + (uint32_t)n_mt * 16 * kQRowBytes;
  auto full_bar = [&](int s) { return bars + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bars + 8u * (uint32_t)(S + s); };
  volatile int* abort = reinterpret_cast<volatile int*>(smem_raw + (bars - raw) + 16 * S);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), (uint32_t)n_cons);
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();
  const int L = A.seq_lens[b];
  const bool bad = L < A.n_new || L > A.Lmax;
  if (bad && split == 0 && hkv == 0 && threadIdx.x == 0) set_status(A.status, SPECDEC_ERR_INVALID_ARG);
  const int j_begin = split * A.split_len;
  const int j_end = bad ? j_begin : min(L, j_begin + A.split_len);

  // Q rows r = i * G + gq (query i, head hkv * G + gq); rows >= R are zero.
  for (int e = threadIdx.x; e < n_mt * 16 * 16; e += blockDim.x) {
    const int r = e >> 4, c = e & 15;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < R) {
      const int i = r / G, gq = r % G;
      val = __ldg(reinterpret_cast<const uint4*>(
          A.q + (((size_t)b * A.n_new + i) * A.Hq + (size_t)hkv * G + gq) * kD + c * 8));
    }
    st_shared_u4(qs + swz(r, c), val);
  }
  __syncthreads();

  // Consumer state (rows g and g + 8 of the warp's tile; log2 units once scaled).
  const int mt = warp >> 1, kh = warp & 1;
  const int g = lane >> 2, t = lane & 3;
  float m_run[2] = {-INFINITY, -INFINITY};   // raw score maxima (unscaled)
  float l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  uint32_t issued_mask = 0, issued_phase = 0;   // producer: stages with copies in flight

  if (warp == n_cons) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      for (int j0 = j_begin; j0 < j_end; j0 += kBlk) {
        if (!mbar_wait(empty_bar(s), ph ^ 1u, abort, A.status)) break;
        mbar_arrive_expect_tx(full_bar(s), (uint32_t)kStageBytes);
        const uint32_t st = stage0 + (uint32_t)s * kStageBytes;
        tma_load_4d(st, &tmap_k, full_bar(s), 0, hkv, j0, b, pol);
        tma_load_4d(st + kHalf, &tmap_k, full_bar(s), 64, hkv, j0, b, pol);
        tma_load_4d(st + 2 * kHalf, &tmap_v, full_bar(s), 0, hkv, j0, b, pol);
        tma_load_4d(st + 3 * kHalf, &tmap_v, full_bar(s), 64, hkv, j0, b, pol);
        issued_mask |= 1u << s;
        issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else {
    // ----------------------------------------------------------- consumers --
    uint32_t qf[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      ldsm_x4(qs + swz(mt * 16 + (lane & 15), ks * 2 + (lane >> 4)), qf[ks]);
    const int row0 = mt * 16 + g;
    const int qi0 = row0 < R ? row0 / G : 0;
    const int qi1 = row0 + 8 < R ? (row0 + 8) / G : 0;
    const int vis0 = L - A.n_new + qi0;      // last visible key of each row
    const int vis1 = L - A.n_new + qi1;
    const int open_end = min(j_end, L - A.n_new + 1);   // keys below it: visible to every row
    const float c = A.scale_log2;
    // Fixed parts of this thread's ldmatrix addresses. Every key row it
    // addresses is = lane (mod 8), so the swizzle term of 16-byte chunk 2a
    // (+1) is (a << 5) ^ y with y fixed per thread.
    const uint32_t krow = (uint32_t)((kh * 32 + (lane & 7) + ((lane >> 4) << 3)) * 128);
    const uint32_t vrow =
        (uint32_t)(2 * kHalf + (kh * 32 + (lane & 7) + (((lane >> 3) & 1) << 3)) * 128);
    const uint32_t yk = (uint32_t)(((((lane >> 3) & 1) ^ (lane & 7))) << 4);
    const uint32_t yv = (uint32_t)((((lane >> 4) ^ (lane & 7))) << 4);

    int s = 0;
    uint32_t ph = 0;
    for (int j0 = j_begin; j0 < j_end; j0 += kBlk) {
      if (!mbar_wait(full_bar(s), ph, abort, A.status)) break;
      const uint32_t sb = stage0 + (uint32_t)s * kStageBytes;
      // S = Q K^T for this warp's 32 keys: 4 tiles of 8 keys, k over 128 dims
      float sc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const uint32_t ka = sb + krow + (((uint32_t)a << 5) ^ yk);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t r[4];
            ldsm_x4(ka + (uint32_t)(hf * kHalf + np * 2048), r);
            mma16816(sc[2 * np], qf[hf * 4 + a], r[0], r[1]);
            mma16816(sc[2 * np + 1], qf[hf * 4 + a], r[2], r[3]);
          }
      }
      // causal window and range end, only where a block reaches past them
      if (j0 + kBlk > open_end) {
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = j0 + kh * 32 + n * 8 + 2 * t + (e & 1);
            const int vis = e < 2 ? vis0 : vis1;
            if (!(j <= vis && j < j_end)) sc[n][e] = -INFINITY;
          }
      }
      float bmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        bmax[0] = fmaxf(bmax[0], fmaxf(sc[n][0], sc[n][1]));
        bmax[1] = fmaxf(bmax[1], fmaxf(sc[n][2], sc[n][3]));
      }
      float alpha[2], mc[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        bmax[h] = fmaxf(bmax[h], __shfl_xor_sync(0xffffffffu, bmax[h], 1));
        bmax[h] = fmaxf(bmax[h], __shfl_xor_sync(0xffffffffu, bmax[h], 2));
        const float m_new = fmaxf(m_run[h], bmax[h]);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;   // nothing visible yet
        alpha[h] = ex2((m_run[h] - m_use) * c);                 // m_run = -inf gives 0
        m_run[h] = m_new;
        l_run[h] *= alpha[h];
        mc[h] = m_use * c;
      }
      if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][0] *= alpha[0];
          o[n][1] *= alpha[0];
          o[n][2] *= alpha[1];
          o[n][3] *= alpha[1];
        }
      }
      uint32_t pa[2][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const float p0 = ex2(fmaf(sc[n][0], c, -mc[0])), p1 = ex2(fmaf(sc[n][1], c, -mc[0]));
        const float p2 = ex2(fmaf(sc[n][2], c, -mc[1])), p3 = ex2(fmaf(sc[n][3], c, -mc[1]));
        l_run[0] += p0 + p1;
        l_run[1] += p2 + p3;
        pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
        pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
      }
      // O += P V over this warp's 32 keys (2 steps of 16) and 128 dims (16 tiles)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const uint32_t va = sb + vrow + (((uint32_t)a << 5) ^ yv);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            uint32_t r[4];
            ldsm_x4_t(va + (uint32_t)(hf * kHalf + kk * 2048), r);
            mma16816(o[2 * (hf * 4 + a)], pa[kk], r[0], r[1]);
            mma16816(o[2 * (hf * 4 + a) + 1], pa[kk], r[2], r[3]);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));   // the stage may be refilled
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
  }
  __syncthreads();   // every role has left its loop
  if (*abort) {
    // A wait gave up: let every copy already issued land before the CTA exits.
    if (warp == n_cons && lane == 0)
      for (int s = 0; s < S; ++s)
        if (issued_mask & (1u << s)) wait_drain(full_bar(s), (issued_phase >> s) & 1u);
    return;
  }
  if (warp >= n_cons) return;

  // Merge the two key-half warps of each tile through shared memory (the
  // stages are free: every issued copy was waited for).
  float* xo = reinterpret_cast<float*>(smem_raw + (stage0 - raw)) + mt * (16 * kD + 32);
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
  named_bar_sync(1, 32 * n_cons);
  if (kh == 1) return;
  const float c = A.scale_log2;
  float w_self[2], w_other[2], m_tot[2], l_tot[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float mo = xm[g + 8 * h], lo = xl[g + 8 * h];
    const float M = fmaxf(m_run[h], mo);
    const float Mu = M == -INFINITY ? 0.f : M;
    w_self[h] = ex2((m_run[h] - Mu) * c);
    w_other[h] = ex2((mo - Mu) * c);
    m_tot[h] = M * c;                        // partial maxima leave in log2 units
    l_tot[h] = l_run[h] * w_self[h] + lo * w_other[h];
  }
  const int row0 = mt * 16 + g;
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

// Merge the splits: one warp per (b, kv head, row). The lanes take the
// splits' (max, sum) pairs 32 at a time; then every lane sums its 4 output
// dims over the splits, several splits' loads in flight.
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
  const int n = A.n_splits;
  const size_t base = ((size_t)b * A.Hkv + hkv) * n * 64 + r;   // + 64 * split
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, A.part_m[base + (size_t)s * 64]);
  M = warp_max(M);
  const float Mu = M == -INFINITY ? 0.f : M;
  float l = 0.f;
  for (int s = lane; s < n; s += 32) {
    const size_t k = base + (size_t)s * 64;
    l += A.part_l[k] * exp2f(A.part_m[k] - Mu);
  }
  l = warp_sum(l);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = 0; s < n; ++s) {
    const size_t k = base + (size_t)s * 64;
    const float wgt = exp2f(A.part_m[k] - Mu);
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

int attn_n_stages(int B, int n_new, int Hq, int Hkv) {
  (void)B;
  (void)Hkv;
  const int n_mt = (n_new * (Hq / Hkv) + 15) / 16;
  // Three stages while two CTAs still fit on an SM (228 KB, 1 KB reserved per CTA).
  return 2 * (attn_smem_bytes(n_mt, 3) + 1024) <= 228 * 1024 ? 3 : 2;
}

int attn_smem_bytes(int n_mt, int n_stages) {
  return 1024 + n_stages * kStageBytes + n_mt * 16 * kQRowBytes + 2 * n_stages * 8 + 16;
}

cudaError_t launch_attention(const AttnLaunch& A, const CUtensorMap& tmap_k,
                             const CUtensorMap& tmap_v, cudaStream_t stream) {
  const int G = A.Hq / A.Hkv;
  const int n_mt = (A.n_new * G + 15) / 16;
  const int smem = attn_smem_bytes(n_mt, A.n_stages);
  static int smem_set[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !smem_set[dev]) {
    e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_smem_bytes(4, 3));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) smem_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(A.n_splits, A.Hkv, A.B);
  cfg.blockDim = dim3(64 * n_mt + 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_split_kernel, A, tmap_k, tmap_v);
  if (e != cudaSuccess || A.n_splits == 1) return e;
  const long long warps = (long long)A.B * A.Hkv * A.n_new * G;
  cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, A);
}

}  // namespace specdec
