// LM-head scoring of all gamma+1 positions on the tcgen05 tensor cores.
//
// "推测解码" (world.lapla.si/zh/specdec), sections 一次一个词元 and 先让小模型猜:
// at small batch the step is bound by reading the weights, and the guessed
// positions ride on the same read. This kernel therefore streams W_lm
// through shared memory exactly once (for up to 256 token rows) and lets
// the otherwise idle tensor core score every token row against it.
//
// Layout: swap-AB. The MMA's M dimension is a 128-row tile of W_lm (the
// vocabulary), its N dimension the BT token rows, so z^T[v, m] lands in
// tensor memory with one vocabulary row per TMEM lane. Work units are
// (vocabulary tile, token tile) pairs, token tile fastest, dealt round-robin
// to one persistent CTA per SM; CTAs that run together share the W tile in
// L2 when there is more than one token tile.
//
// Warp roles (192 threads):
//   warp 0     one thread issues TMA loads of W and hidden k-slices into a
//              ring of shared-memory stages (full/empty mbarriers).
//   warp 1     allocates tensor memory; one thread issues tcgen05.mma into
//              one of two TMEM accumulators and commits to mbarriers.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, fp32 logits out,
//              per-tile softmax / argmax partials for p, and the matching
//              partials of the draft logits for q.
// Every wait is bounded (1 s); a timeout records SPECDEC_ERR_TIMEOUT, stops
// the other roles, waits for copies and MMAs already issued, frees tensor
// memory and returns.
#include <cuda.h>

#include "kernels.h"

namespace specdec {
namespace {

constexpr int kThreads = 192;
constexpr int kStageA = kBlockV * kBlockK * 2;   // 16 KB of W per stage
constexpr int kMaxStages = 12;
constexpr int kSmemLimit = 232448;               // 227 KB opt-in per CTA
constexpr int kMiscBytes = 4096;
constexpr unsigned long long kDrainLimitNs = 100000000ull;

struct TcParams {
  int M, V, d, gamma;
  int BT, n_tt, n_units, nk, stages;
  uint32_t stage_bytes, tmem_cols;
  int* status;
  EpiParams ep;
};

__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kDrainLimitNs) return false;
  }
  return true;
}

template <typename DL>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_h, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  const int S = p.stages;
  uint8_t* misc = smem + (size_t)S * p.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  // bars: full[S], empty[S], tfull[2], tempty[2], mma_done
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (2 * S + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_ok = reinterpret_cast<volatile int*>(tmem_slot + 2);
  RedSlot* red = reinterpret_cast<RedSlot*>(misc + 8 * (2 * S + 5) + 64);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 128);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer --
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      for (int unit = blockIdx.x; ok && unit < p.n_units; unit += gridDim.x) {
        const int vt = unit / p.n_tt;
        const int tt = unit - vt * p.n_tt;
        for (int kc = 0; kc < p.nk; ++kc) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), p.stage_bytes);
          const uint32_t a = sbase + (uint32_t)s * p.stage_bytes;
          tma_load_2d(a, &tmap_w, full_bar(s), kc * kBlockK, vt * kBlockV, pol_w);
          tma_load_2d(a + kStageA, &tmap_h, full_bar(s), kc * kBlockK, tt * p.BT, pol_h);
          issued_mask |= 1u << s;
          issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA exits.
        for (int t = 0; t < S; ++t)
          if (issued_mask & (1u << t)) mbar_wait_drain(full_bar(t), (issued_phase >> t) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuer --
      const uint32_t idesc = idesc_bf16_f32(kBlockV, p.BT);
      int s = 0;
      uint32_t ph = 0;
      int ul = 0;
      bool ok = true;
      for (int unit = blockIdx.x; ok && unit < p.n_units; unit += gridDim.x, ++ul) {
        const int acc = ul & 1;
        const uint32_t aph = (uint32_t)(ul >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.BT);
        for (int kc = 0; kc < p.nk; ++kc) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = sbase + (uint32_t)s * p.stage_bytes;
          const uint64_t adesc = smem_desc_sw128(a);
          const uint64_t bdesc = smem_desc_sw128(a + kStageA);
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k)
            tc_mma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kc | k) ? 1u : 0u);
          tc_commit(empty_bar(s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
      }
      // All MMAs this thread issued are complete once this phase ends.
      tc_commit(mma_done_bar);
      mbar_wait_drain(mma_done_bar, 0);
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int epi_tid = threadIdx.x - 64;
    int ul = 0;
    for (int unit = blockIdx.x; unit < p.n_units; unit += gridDim.x, ++ul) {
      const int acc = ul & 1;
      const uint32_t aph = (uint32_t)(ul >> 1) & 1u;
      if (epi_tid == 0) *epi_ok = mbar_wait(tfull_bar(acc), aph, abort_flag, p.status) ? 1 : 0;
      named_bar_sync(1, 128);
      const bool ok = *epi_ok != 0;
      named_bar_sync(2, 128);
      if (!ok) break;
      tc_fence_after();
      const int vt = unit / p.n_tt;
      const int tt = unit - vt * p.n_tt;
      const int v = vt * kBlockV + q * 32 + lane;
      const int m_base = tt * p.BT;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.BT);
      for (int c = 0; c < p.BT / 16; ++c) {
        const int m0 = m_base + c * 16;
        if (m0 >= p.M) break;
        float accv[16];
        tmem_ld16(tbase + (uint32_t)(c * 16), accv);
        epilogue_chunk16<DL>(accv, m0, v, vt, q, lane, epi_tid, red, p.ep, 1);
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

template <typename DL>
cudaError_t launch_typed(const TcLaunch& L, int num_sms, cudaStream_t stream) {
  const TcGeometry g = tc_geometry(L.M);
  TcParams p;
  p.M = L.M;
  p.V = L.V;
  p.d = L.d;
  p.gamma = L.gamma;
  p.BT = g.BT;
  p.n_tt = g.n_tt;
  const int n_vt = (L.V + kBlockV - 1) / kBlockV;
  p.n_units = n_vt * g.n_tt;
  p.nk = (L.d + kBlockK - 1) / kBlockK;
  p.stages = g.stages;
  p.stage_bytes = (uint32_t)g.stage_bytes;
  p.tmem_cols = (uint32_t)g.tmem_cols;
  p.status = L.status;
  p.ep = L.ep;
  auto kern = lmhead_tc_kernel<DL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       g.smem_bytes);
  if (e != cudaSuccess) return e;
  const int grid = p.n_units < num_sms ? p.n_units : num_sms;
  kern<<<grid, kThreads, g.smem_bytes, stream>>>(*L.tmap_w, *L.tmap_h, p);
  return cudaGetLastError();
}

}  // namespace

TcGeometry tc_geometry(int M) {
  TcGeometry g;
  g.n_tt = (M + kMaxBT - 1) / kMaxBT;
  if (g.n_tt < 1) g.n_tt = 1;
  const int per = (M + g.n_tt - 1) / g.n_tt;
  g.BT = ((per + 15) / 16) * 16;
  if (g.BT < 16) g.BT = 16;
  g.stage_bytes = kStageA + g.BT * kBlockK * 2;
  int stages = (kSmemLimit - 1024 - kMiscBytes) / g.stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  g.stages = stages;
  int cols = 32;
  while (cols < 2 * g.BT) cols <<= 1;
  g.tmem_cols = cols;
  g.smem_bytes = 1024 + g.stages * g.stage_bytes + kMiscBytes;
  return g;
}

cudaError_t launch_lmhead_tc(const TcLaunch& L, int num_sms, cudaStream_t stream) {
  // The tensor-core path exists for bf16 inputs; draft logits share the dtype.
  return launch_typed<__nv_bfloat16>(L, num_sms, stream);
}

}  // namespace specdec
