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
constexpr int kMaxVocab = 1 << 22;  // V limit: the sampler stages 1024 chunk sums
constexpr int kQChunk = 8192;       // draft-logit columns per streamed q record
constexpr int kQWarpMaxRows = 16;   // draft rows up to which the LM-head q-warps reduce q
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
  int pad0;
  // Calls that have used this workspace (any initial value): the kernel
  // after the LM head adds one. Mixed into the LM head's fix-up tag, it keeps
  // tags distinct when a captured CUDA graph replays the same launch.
  unsigned long long calls;
  int pad[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header");

// Fix-up tag of one LM-head call: the host's per-launch tag mixed with the
// workspace's call count.
__device__ __forceinline__ unsigned long long call_tag(unsigned long long epoch,
                                                       const unsigned long long* calls) {
  return epoch ^ (*reinterpret_cast<const volatile unsigned long long*>(calls) *
                  0x9E3779B97F4A7C15ull);
}

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
// The draft draw's uniform (purpose 2), same map as the sampling uniform.
__device__ __forceinline__ float draft_uniform(uint64_t seed, int b, int i) {
  return (float)uniform24(seed, b, i, 2) * 5.9604644775390625e-08f;
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
// The same test with a suspend-time hint of zero: the thread polls instead of
// being suspended by the hardware between tests. The LM-head kernel's
// single-thread roles (TMA producer, MMA issuer) wait once per stage; there
// the default form's wake-up latency left the tensor core idle between
// stages (measured: 5-7 % fewer cycles per launch with the polling form).
__device__ __forceinline__ bool mbar_try_wait_poll(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 0;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase. Gives up after kWaitLimitNs or when
// another role of the CTA has raised *abort; a timeout raises *abort and
// records SPECDEC_ERR_TIMEOUT in the status word. Returns false on give-up.
// kPoll selects the polling test (mbar_try_wait_poll).
template <bool kPoll = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  auto test = [&]() { return kPoll ? mbar_try_wait_poll(bar, parity) : mbar_try_wait(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (test()) return true;
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
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
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

// CTA-pair (2-SM) tcgen05 forms. One warp in each CTA of the pair allocates
// collectively and both CTAs get the same tensor-memory address; an MMA
// issued by the pair's leader with M = 256 reads A as two 128-row halves,
// one in each CTA's shared memory at the same offset, and B as two halves
// of its N rows likewise, and writes each CTA's 128 rows of D into that
// CTA's tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc2_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// TMA loads of a CTA pair: the box lands in this CTA's shared memory and its
// bytes complete on `bar_cluster`, a barrier of either CTA of the pair (the
// leader's, so one barrier counts both halves of a stage).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap,
                                                 uint32_t bar_cluster, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
      ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap,
                                                 uint32_t bar_cluster, int x, int y, int z,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile"
      ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(z), "r"(bar_cluster), "l"(policy)
      : "memory");
}
// Arrive on `bar` in every CTA of `mask` once the pair MMAs issued so far are done.
__device__ __forceinline__ void tc2_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
      : "memory");
}
// The shared::cluster address of `addr` in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster_poll(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, 0;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for a barrier that CTAs of the cluster arrive on.
template <bool kPoll = false>
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, int* status) {
  auto test = [&]() {
    return kPoll ? mbar_try_wait_cluster_poll(bar, parity) : mbar_try_wait_cluster(bar, parity);
  };
  if (test()) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (test()) return true;
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
// Loads from another CTA's shared memory (address from mapa_shared).
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// 3-D tiled TMA load of box {x.., y.., z..} into shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x,
                                            int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
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
// Bulk tensor store (shared -> global) and its completion groups.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t smem, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
      "r"(smem), "r"(x), "r"(y)
      : "memory");
}
// The same with an L2 eviction-priority policy for the written lines.
__device__ __forceinline__ void tma_store_2d_hint(const void* tmap, uint32_t smem, int x, int y,
                                                  uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;"
      ::"l"(tmap), "r"(smem), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// Bulk prefetch of [addr, addr + bytes) into L2 (16-byte aligned, bytes a
// multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* addr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(addr), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

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

// 32 consecutive columns in one load.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
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

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (a no-op when this
// kernel was launched without the programmatic-serialisation attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next kernel in the stream start launching its CTAs now.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------- 16-column transposed reductions --
// Each lane holds one value for each of 16 columns (one vocabulary row of a
// tile). Five butterfly steps halve the columns a lane carries (16 -> 8 ->
// 4 -> 2 -> 1) while doubling the lanes folded in, so afterwards lanes 2c
// and 2c+1 both hold column c reduced over all 32 lanes. The 16 chains are
// independent, so the shuffles overlap instead of running one column at a
// time.

// Online-softmax pair merge with one exp2: (ma, sa) <- (ma, sa) + (mb, sb),
// s = sum of exp2((x - m) * c).
__device__ __forceinline__ void osm_merge(float& ma, float& sa, float mb, float sb, float c) {
  // Branch-free: scale the smaller side's sum by exp2(-|ma - mb| c).
  const float mm = fmaxf(ma, mb);
  const bool a_big = ma >= mb;
  const float e = exp2f(-fabsf(ma - mb) * c);
  const float s = fmaf(a_big ? sb : sa, e, a_big ? sa : sb);
  sa = mm == -INFINITY ? 0.f : s;   // both empty (the exponent is NaN then)
  ma = mm;
}

template <int N>
__device__ __forceinline__ void osm_halve(float (&m)[16], float (&s)[16], bool upper, int off,
                                          float c) {
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const float km = upper ? m[N + k] : m[k];
    const float ks = upper ? s[N + k] : s[k];
    const float sm = upper ? m[k] : m[N + k];
    const float ss = upper ? s[k] : s[N + k];
    const float rm = __shfl_xor_sync(0xffffffffu, sm, off);
    const float rs = __shfl_xor_sync(0xffffffffu, ss, off);
    m[k] = km;
    s[k] = ks;
    osm_merge(m[k], s[k], rm, rs, c);
  }
}

// Per-column (max, sum exp2((x - max) * c)) of x over the warp; -inf values
// are absent. Result for column (lane >> 1).
__device__ __forceinline__ void warp_softmax16(const float (&x)[16], float c, float& m_out,
                                               float& s_out) {
  const int lane = threadIdx.x & 31;
  float m[16], s[16];
  {
    const bool upper = (lane & 16) != 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float keep = upper ? x[8 + k] : x[k];
      const float send = upper ? x[k] : x[8 + k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      const float mm = fmaxf(keep, recv);
      m[k] = mm;
      s[k] = mm == -INFINITY ? 0.f : 1.f + exp2f(-fabsf(keep - recv) * c);
    }
  }
  osm_halve<4>(m, s, (lane & 8) != 0, 8, c);
  osm_halve<2>(m, s, (lane & 4) != 0, 4, c);
  osm_halve<1>(m, s, (lane & 2) != 0, 2, c);
  const float rm = __shfl_xor_sync(0xffffffffu, m[0], 1);
  const float rs = __shfl_xor_sync(0xffffffffu, s[0], 1);
  // The two lanes of a pair merge in the same order, so they agree exactly.
  float am = m[0], as = s[0];
  if (lane & 1) {
    am = rm;
    as = rs;
    osm_merge(am, as, m[0], s[0], c);
  } else {
    osm_merge(am, as, rm, rs, c);
  }
  m_out = am;
  s_out = as;
}

template <int N>
__device__ __forceinline__ void amax_halve(float (&v)[16], int (&i)[16], bool upper, int off) {
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const float kv = upper ? v[N + k] : v[k];
    const int ki = upper ? i[N + k] : i[k];
    const float sv = upper ? v[k] : v[N + k];
    const int si = upper ? i[k] : i[N + k];
    const float rv = __shfl_xor_sync(0xffffffffu, sv, off);
    const int ri = __shfl_xor_sync(0xffffffffu, si, off);
    v[k] = kv;
    i[k] = ki;
    if (argmax_better(rv, ri, v[k], i[k])) {
      v[k] = rv;
      i[k] = ri;
    }
  }
}

// Per-column (max value, lowest index) over the warp; every value of this
// lane carries the index `idx`. Result for column (lane >> 1).
__device__ __forceinline__ void warp_argmax16(const float (&x)[16], int idx, float& v_out,
                                              int& i_out) {
  const int lane = threadIdx.x & 31;
  float v[16];
  int i[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    v[k] = x[k];
    i[k] = idx;
  }
  amax_halve<8>(v, i, (lane & 16) != 0, 16);
  amax_halve<4>(v, i, (lane & 8) != 0, 8);
  amax_halve<2>(v, i, (lane & 4) != 0, 4);
  amax_halve<1>(v, i, (lane & 2) != 0, 2);
  const float rv = __shfl_xor_sync(0xffffffffu, v[0], 1);
  const int ri = __shfl_xor_sync(0xffffffffu, i[0], 1);
  if (argmax_better(rv, ri, v[0], i[0])) {
    v[0] = rv;
    i[0] = ri;
  }
  v_out = v[0];
  i_out = i[0];
}

// 32-column forms of the two reductions above, for one 32-column tensor
// memory load: five halving exchanges (xor 16, 8, 4, 2, 1) leave lane L
// holding column L, merged over all 32 rows exactly once (no duplicate
// pair). Twice the independent chains of the 16-column form at each level.
__device__ __forceinline__ void warp_softmax32(const float (&x)[32], float c, float& m_out,
                                               float& s_out) {
  const int lane = threadIdx.x & 31;
  float m[16], s[16];
  const bool upper = (lane & 16) != 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float keep = upper ? x[16 + k] : x[k];
    const float send = upper ? x[k] : x[16 + k];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    const float mm = fmaxf(keep, recv);
    m[k] = mm;
    s[k] = mm == -INFINITY ? 0.f : 1.f + exp2f(-fabsf(keep - recv) * c);
  }
  osm_halve<8>(m, s, (lane & 8) != 0, 8, c);
  osm_halve<4>(m, s, (lane & 4) != 0, 4, c);
  osm_halve<2>(m, s, (lane & 2) != 0, 2, c);
  osm_halve<1>(m, s, (lane & 1) != 0, 1, c);
  m_out = m[0];
  s_out = s[0];
}
__device__ __forceinline__ void warp_argmax32(const float (&x)[32], int idx, float& v_out,
                                              int& i_out) {
  const int lane = threadIdx.x & 31;
  float v[16];
  int i[16];
  const bool upper = (lane & 16) != 0;
  const int ridx = __shfl_xor_sync(0xffffffffu, idx, 16);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float keep = upper ? x[16 + k] : x[k];
    const float send = upper ? x[k] : x[16 + k];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    v[k] = keep;
    i[k] = idx;
    if (argmax_better(recv, ridx, v[k], i[k])) {
      v[k] = recv;
      i[k] = ridx;
    }
  }
  amax_halve<8>(v, i, (lane & 8) != 0, 8);
  amax_halve<4>(v, i, (lane & 4) != 0, 4);
  amax_halve<2>(v, i, (lane & 2) != 0, 2);
  amax_halve<1>(v, i, (lane & 1) != 0, 1);
  v_out = v[0];
  i_out = i[0];
}

// ------------------------------------------------ LM-head tile epilogue --
// Shared by the tensor-core and the fp32 kernels: one thread per vocabulary
// row of a 128-row tile (4 warps, warp quarter q holds rows 32q..32q+31),
// each holding the logits of 16 consecutive token rows.

struct RedSlot {
  float pm, ps, am;
  int ai;
  float qm, qs;
};

struct EpiParams {
  int M, V, gamma, P;      // P = partial records per row
  float c;                 // log2(e) / T
  int sample;              // softmax partials for p and q
  int want_argmax;         // argmax partials
  float* zout;             // [M, V] logits, or NULL
  const void* dl;          // draft logits [B, gamma, V]
  PartialP* pp;            // [M, P]
  PartialQ* pq;            // [B*gamma, P]
  RedSlot* run;            // shared memory [M]: fold tiles into one record per
                           // row and CTA (NULL: one record per row and tile)
  int q_in_epilogue;       // 1: the epilogue also reduces the draft logits
  int q_warps;             // 1: the LM-head kernel's q-warps reduce them per tile
  int q_stream;            // 1: its streamer warps reduce them per (row, kQChunk columns)
  int n_qrows;             // draft-logit rows the streamer reduces (rows of dl, in order)
  int Pq;                  // q records per draft row when streamed: ceil(V / kQChunk)
  int q_vec;               // streamed rows allow 16-byte loads (V % 8 == 0, aligned base)
  int* counters;           // sampler tickets the LM-head kernel clears (fused draw), or NULL
  int n_counters;
};

__device__ __forceinline__ void redslot_merge(RedSlot& a, const RedSlot& o, float c) {
  softmax_merge(a.pm, a.ps, o.pm, o.ps, c);
  softmax_merge(a.qm, a.qs, o.qm, o.qs, c);
  if (argmax_better(o.am, o.ai, a.am, a.ai)) {
    a.am = o.am;
    a.ai = o.ai;
  }
}

__device__ __forceinline__ void partialp_merge(PartialP& a, const PartialP& o, float c) {
  osm_merge(a.m, a.s, o.m, o.s, c);
  if (argmax_better(o.amax_v, o.amax_i, a.amax_v, a.amax_i)) {
    a.amax_v = o.amax_v;
    a.amax_i = o.amax_i;
  }
}

__device__ __forceinline__ RedSlot redslot_empty() {
  RedSlot r;
  r.pm = -INFINITY;
  r.ps = 0.f;
  r.am = -INFINITY;
  r.ai = 0x7fffffff;
  r.qm = -INFINITY;
  r.qs = 0.f;
  return r;
}

// Draft logits of this thread's vocabulary row v for the 16 token rows
// m0..m0+15 (-inf where the row is not a draft row or v >= V), loaded up
// front so the 16 loads are in flight together.
template <typename DL>
__device__ __forceinline__ void prefetch_draft16(float (&zq)[16], int m0, int v,
                                                 const EpiParams& ep) {
  const bool vvalid = v < ep.V;
  const int g1 = ep.gamma + 1;
  const DL* dl = static_cast<const DL*>(ep.dl);
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int m = m0 + n;
    const int b = m / g1;
    const int i = m - b * g1;
    zq[n] = (ep.sample && vvalid && m < ep.M && i < ep.gamma)
                ? load_logit(dl, ((size_t)b * ep.gamma + i) * ep.V + v)
                : -INFINITY;
  }
}

template <typename DL>
__device__ __forceinline__ void epilogue_chunk16(const float (&acc)[16], const float (&zqv)[16],
                                                 int m0, int v, int vt, int q, int lane,
                                                 int epi_tid, RedSlot* red, const EpiParams& ep,
                                                 int bar_id) {
  const bool vvalid = v < ep.V;
  const int g1 = ep.gamma + 1;
  if (ep.zout != nullptr && vvalid) {
#pragma unroll
    for (int n = 0; n < 16; ++n)
      if (m0 + n < ep.M) __stcs(ep.zout + (size_t)(m0 + n) * ep.V + v, acc[n]);
  }
  RedSlot r = redslot_empty();
  float zm[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) zm[n] = vvalid ? acc[n] : -INFINITY;
  if (ep.sample) {
    warp_softmax16(zm, ep.c, r.pm, r.ps);
    if (ep.q_in_epilogue) warp_softmax16(zqv, ep.c, r.qm, r.qs);
  }
  if (ep.want_argmax) warp_argmax16(zm, vvalid ? v : 0x7fffffff, r.am, r.ai);
  if ((lane & 1) == 0) red[q * 16 + (lane >> 1)] = r;
  named_bar_sync(bar_id, 128);
  if (epi_tid < 16) {
    const int m = m0 + epi_tid;
    if (m < ep.M) {
      RedSlot a = red[epi_tid];
#pragma unroll
      for (int qq = 1; qq < 4; ++qq) redslot_merge(a, red[qq * 16 + epi_tid], ep.c);
      if (ep.run != nullptr) {
        redslot_merge(ep.run[m], a, ep.c);   // this thread owns row m's slot
      } else {
        ep.pp[(size_t)m * ep.P + vt] = PartialP{a.pm, a.ps, a.am, a.ai};
        const int b = m / g1;
        const int i = m - b * g1;
        if (ep.sample && ep.q_in_epilogue && i < ep.gamma)
          ep.pq[((size_t)b * ep.gamma + i) * ep.P + vt] = PartialQ{a.qm, a.qs};
      }
    }
  }
  named_bar_sync(bar_id, 128);
}

}  // namespace specdec
