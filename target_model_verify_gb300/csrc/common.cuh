// Shared device-side pieces of the verify-step library: constants, the
// workspace records, Philox4x32-10, warp reductions, the online-softmax
// merge, and thin inline-PTX wrappers for mbarrier, TMA and tcgen05.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "specdec_verify.h"

namespace specdec {

constexpr int kBlockV = 128;        // vocabulary rows per LM-head tile (MMA M)
constexpr int kBlockK = 64;         // bf16 per 128-byte swizzled smem row
constexpr int kMaxBT = 256;         // token rows per tile (MMA N) at most
constexpr int kChunkV = 4096;       // residual-sampler chunk (256 threads x 16)
constexpr int kSampleThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s per device-side wait

// Per (row, vocabulary tile) softmax partial of the target logits:
// m = max z over the tile, s = sum exp2((z - m) * c) with c = log2(e)/T,
// and the tile's argmax (value, lowest index) when requested.
struct PartialP {
  float m;
  float s;
  float amax_v;
  int amax_i;
};
// The same (m, s) pair for a draft row's logits.
struct PartialQ {
  float m;
  float s;
};
// What the sampler needs about the row each sequence samples from.
struct SelectedRow {
  float mp, lsp;      // max z and log2 of its sum, row j of the target
  float mq, lsq;      // the same for the draft row j (residual case)
  int residual;       // 1: w = max(0, p - q); 0: w = p (bonus)
  int j;              // the position sampled (n_accepted), or -1: nothing to draw
  int pad[2];
};

// Workspace header: device status word and per-sequence sampler counters
// follow it at fixed offsets computed on the host.
struct WsHeader {
  int status;
  int pad[63];
};

// ------------------------------------------------------------- status --

__device__ __forceinline__ void set_status(int* st, int code) {
  atomicCAS(st, 0, code);
}

// ------------------------------------------------------------- Philox --
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): returns output word 0
// for counter (c0, c1, c2, c3) and key (k0, k1).
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

// 24-bit integer of the verify step's stream for (seed, b, i, purpose).
__device__ __forceinline__ uint32_t uniform24(uint64_t seed, int b, int i, int purpose) {
  return philox_word0((uint32_t)b, (uint32_t)i, (uint32_t)purpose, 0u, (uint32_t)seed,
                      (uint32_t)(seed >> 32)) >> 8;
}
// r in (0, 1]: keep the draft iff r <= p/q.
__device__ __forceinline__ float accept_uniform(uint64_t seed, int b, int i) {
  return (float)(uniform24(seed, b, i, 0) + 1u) * 5.9604644775390625e-08f;
}
// u in [0, 1): inverse-CDF position of the replacement or bonus draw.
__device__ __forceinline__ float sample_uniform(uint64_t seed, int b, int i) {
  return (float)uniform24(seed, b, i, 1) * 5.9604644775390625e-08f;
}

// ------------------------------------------------------ warp reductions --

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
// (value, index) maximum with ties to the lower index; NaN never wins.
__device__ __forceinline__ bool argmax_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (argmax_better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Merge two (max, sum-of-exp2((z - max)*c)) pairs.
__device__ __forceinline__ void softmax_merge(float& m, float& s, float m2, float s2, float c) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) {
    m = mm;
    s = 0.f;
    return;
  }
  s = s * exp2f((m - mm) * c) + s2 * exp2f((m2 - mm) * c);
  m = mm;
}

__device__ __forceinline__ float load_logit(const __nv_bfloat16* p, size_t idx) {
  return __bfloat162float(p[idx]);
}
__device__ __forceinline__ float load_logit(const float* p, size_t idx) { return p[idx]; }

// ---------------------------------------------------------- PTX wrappers --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase. Gives up after kWaitLimitNs or when
// another role of the CTA has raised *abort; a timeout raises *abort and
// records SPECDEC_ERR_TIMEOUT in the status word. Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        set_status(status, SPECDEC_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 2-D tiled TMA load of box {x.., y..} into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int x,
                                            int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// tcgen05 (5th-generation tensor core, accumulators in tensor memory).
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// Each thread of the warp reads 16 consecutive fp32 columns of its lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
}

// Shared-memory matrix descriptor of a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)(16u >> 4) << 16;                 // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset: 8 rows
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}
// Instruction descriptor: bf16 x bf16 -> fp32, A and B K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------ LM-head tile epilogue --
// Shared by the tensor-core and the fp32 kernels: one thread per vocabulary
// row of a 128-row tile (4 warps, warp quarter q holds rows 32q..32q+31),
// each holding the logits of 16 consecutive token rows.

struct EpiParams {
  int M, V, gamma, P;      // P = vocabulary tiles = partial records per row
  float c;                 // log2(e) / T
  int sample;              // softmax partials for p and q
  int want_argmax;         // argmax partials
  float* zout;             // [M, V] logits, or NULL
  const void* dl;          // draft logits [B, gamma, V]
  PartialP* pp;            // [M, P]
  PartialQ* pq;            // [B*gamma, P]
};

struct RedSlot {
  float pm, ps, am;
  int ai;
  float qm, qs;
};

template <typename DL>
__device__ __forceinline__ void epilogue_chunk16(const float (&acc)[16], int m0, int v, int vt,
                                                 int q, int lane, int epi_tid, RedSlot* red,
                                                 const EpiParams& ep, int bar_id) {
  const bool vvalid = v < ep.V;
  const int g1 = ep.gamma + 1;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int m = m0 + n;
    if (m >= ep.M) break;
    const float z = acc[n];
    if (ep.zout != nullptr && vvalid) __stcs(ep.zout + (size_t)m * ep.V + v, z);
    RedSlot r;
    r.pm = -INFINITY;
    r.ps = 0.f;
    r.qm = -INFINITY;
    r.qs = 0.f;
    r.am = -INFINITY;
    r.ai = 0x7fffffff;
    if (ep.sample) {
      const float zm = vvalid ? z : -INFINITY;
      const float mx = warp_max(zm);
      const float e = vvalid ? exp2f((z - mx) * ep.c) : 0.f;
      r.pm = mx;
      r.ps = warp_sum(e);
      const int b = m / g1;
      const int i = m - b * g1;
      if (i < ep.gamma) {
        const DL* dl = static_cast<const DL*>(ep.dl);
        const float zq = vvalid ? load_logit(dl, ((size_t)b * ep.gamma + i) * ep.V + v) : -INFINITY;
        const float mq = warp_max(zq);
        const float eq = vvalid ? exp2f((zq - mq) * ep.c) : 0.f;
        r.qm = mq;
        r.qs = warp_sum(eq);
      }
    }
    if (ep.want_argmax) {
      float av = vvalid ? z : -INFINITY;
      int ai = vvalid ? v : 0x7fffffff;
      warp_argmax(av, ai);
      r.am = av;
      r.ai = ai;
    }
    if (lane == 0) red[q * 16 + n] = r;
  }
  named_bar_sync(bar_id, 128);
  if (epi_tid < 16) {
    const int m = m0 + epi_tid;
    if (m < ep.M) {
      RedSlot a = red[epi_tid];
#pragma unroll
      for (int qq = 1; qq < 4; ++qq) {
        const RedSlot o = red[qq * 16 + epi_tid];
        softmax_merge(a.pm, a.ps, o.pm, o.ps, ep.c);
        softmax_merge(a.qm, a.qs, o.qm, o.qs, ep.c);
        if (argmax_better(o.am, o.ai, a.am, a.ai)) {
          a.am = o.am;
          a.ai = o.ai;
        }
      }
      ep.pp[(size_t)m * ep.P + vt] = PartialP{a.pm, a.ps, a.am, a.ai};
      const int b = m / g1;
      const int i = m - b * g1;
      if (ep.sample && i < ep.gamma) ep.pq[((size_t)b * ep.gamma + i) * ep.P + vt] = PartialQ{a.qm, a.qs};
    }
  }
  named_bar_sync(bar_id, 128);
}

}  // namespace specdec
