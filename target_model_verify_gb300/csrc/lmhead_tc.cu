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
// tensor memory with one vocabulary row per TMEM lane. Each k-step is one
// shared-memory stage of C adjacent 64-wide k-slices (C = 4 at small
// batch). With d % 64 == 0 the loads are 3-D boxes {64, rows, C}, so each W
// row gives C*128 contiguous bytes per request: fewer, longer DRAM bursts,
// which measured ~7.1 TB/s against ~6.8 TB/s for one 128-byte slice per row.
//
// CTA pairs: with large token tiles (BT >= 128) each SM would have to take in
// the whole token slice for every 128-row W slice (up to twice the W
// bytes), and that ingress, not DRAM, limited the kernel. There K = 2 CTAs
// form a cluster and run the 2-SM MMA (tcgen05.mma.cta_group::2, M = 256):
// each CTA loads its own W tile (128 vocabulary rows) and only its half of
// the token rows, and both CTAs' loads complete on the leader's (rank 0)
// barrier, so the leader issues the MMA as soon as both halves of a stage
// have landed and frees the stage in both CTAs with one multicast commit;
// each CTA's tensor memory receives its 128 rows x BT accumulator. The
// peer's epilogue releases an accumulator by arriving on the leader's
// barrier. K = 1 elsewhere.
//
// Row owner: a pair with token tiles of 256 rows swaps the operands back,
// tokens on the MMA's M side (A = 128 token rows per CTA, B = 128 W rows
// per CTA), so tensor-memory lane = token row. Each epilogue thread then
// owns one token row and keeps its softmax and argmax partials in
// registers (no shuffles), and the logits leave through bulk tensor stores
// of 32 x 32 fp32 tiles staged in shared memory.
//
// Scheduling, one persistent CTA per SM, in cluster units (K neighbouring
// vocabulary tiles x one token tile; CTA rank r of the cluster takes tile
// K*unit + r):
//   * one token tile (M <= 256): stream-K. The units x k-steps iterations
//     are cut into equal contiguous ranges, one per cluster, so every SM
//     streams the same number of W bytes. A tile cut between two clusters
//     leaves each CTA a partial accumulator; both write theirs to a fix-up
//     slot and take an atomic ticket, and the second to arrive adds the two
//     and runs the epilogue (nobody waits). Each CTA folds the softmax
//     partials of all its tiles into one record per token row. Tickets
//     hold a per-call tag: the host's launch epoch mixed with the
//     workspace's call count, which the kernel after this one advances, so
//     stale tickets never match, not even when a captured CUDA graph replays
//     the launch with identical parameters.
//   * several token tiles: units dealt round-robin with the token tile
//     fastest, so the clusters that share W tiles run together and read
//     them once from HBM and the rest from L2; one record per (row, tile).
//
// Warp roles (448 threads):
//   warp 0     one thread issues TMA loads of W and hidden k-slices into a
//              ring of shared-memory stages (full/empty mbarriers).
//   warp 1     allocates tensor memory; one thread issues tcgen05.mma into
//              one of two sets of TMEM accumulators (a narrow token tile
//              deals its k-slices across up to 16 accumulators per set, for
//              accuracy; see issue_stage) and commits to mbarriers.
//   warps 2-9  epilogue, two groups of four (one warp per TMEM lane quarter
//              in each) taking alternate 32-column chunks: tcgen05.ld of the
//              accumulator, fp32 logits out, softmax / argmax partials for p.
//   warps 10-13 q-warps: stream the draft logits of the same vocabulary tiles
//              (8 rows in flight per warp) and reduce their softmax
//              partials for q, off the epilogue's critical path. The CTA
//              holding a tile's first k-step scores that tile's draft rows.
//              With more than 16 draft rows, warps 10-12 instead stream
//              whole (draft row, 8192-column) items dealt across the grid,
//              one record each (warp 13 shares the MMA issuer's scheduler
//              and stays out).
// Every wait is bounded (1 s); a timeout records SPECDEC_ERR_TIMEOUT, stops
// the other roles, waits for copies and MMAs already issued, frees tensor
// memory and returns (a cluster partner's waits then run out as well, so
// the closing cluster barrier is always reached).
#include <cuda.h>

#include "kernels.h"

namespace specdec {
namespace {

constexpr int kThreads = 448;
constexpr int kEpiThreads = 256;   // warps 2-9
constexpr int kQWarp0 = 10;        // first q-warp
constexpr int kQRowsInFlight = 8;
constexpr int kQStreamWarps = 3;    // streamer q-warps: 10-12 (warp 13 shares the MMA issuer's scheduler)
constexpr int kStageA = kBlockV * kBlockK * 2;   // 16 KB of W per stage
constexpr int kMaxStagesC1 = 10;   // stage caps by slices per stage (measured)
constexpr int kMaxStagesC2 = 4;
constexpr int kMaxStagesC4 = 3;
constexpr int kSmemLimit = 232448;               // 227 KB opt-in per CTA
constexpr unsigned long long kDrainLimitNs = 100000000ull;
// Shared memory after the stages: mbarriers and flags (512 B), then per
// token column of the tile: the four epilogue warps' partials, the CTA's
// folded p record and its folded q record.
constexpr int kBarBytes = 512;
__host__ __device__ constexpr int misc_bytes(int BT) {
  return kBarBytes + BT * (4 * (int)sizeof(PartialP) + (int)sizeof(PartialP) + (int)sizeof(PartialQ));
}
constexpr int kMaxDevices = 64;
constexpr int kTmemCols = 512;     // tensor-memory columns per SM
constexpr int kMaxAcc = 16;        // accumulators per tile at most (issue_stage)
// Token tiles from this size run on CTA pairs. Single CTAs measured 1.5-2 %
// faster at 64-96 rows (their MMAs are short and a pair adds cluster
// waits) and the same at 128.
constexpr int kClusterMinBT = 128;
// Row-owner logit staging: one 32 x 32 fp32 tile (4 KB) per epilogue warp,
// written in the 128-byte swizzled layout the bulk tensor store reads.
constexpr int kZStageBytes = 4096;
constexpr int kZStaging = 8 * kZStageBytes;
__host__ __device__ constexpr int misc_span(int BT) { return (misc_bytes(BT) + 1023) & ~1023; }

struct TcParams {
  int M, V, d, gamma;
  int BT, n_tt, nk, stages;
  int n_vt;                      // vocabulary tiles
  int K;                         // CTAs per cluster (1, or 2 for the 2-SM MMA)
  int n_units;                   // cluster units: ceil(n_vt / K) * n_tt
  int kc;                        // 64-wide k slices per stage (C)
  int box3d;                     // 1: 3-D boxes {64, rows, C}; 0: 2-D boxes, C = 1
  int stream_k;                  // 1: contiguous iteration ranges (one token tile)
  long long total_iters;         // n_units * nk (k-steps)
  uint32_t stage_bytes, tmem_cols;
  int* status;
  float* fix;                    // [slots * 2][BT * 128] partial accumulators
  unsigned long long* fix_tickets;   // [slots]: epoch of the last part to arrive
  unsigned long long epoch;      // this launch's host tag (never repeats within a process)
  const unsigned long long* calls;   // the workspace's call count, mixed into the tag
  int withhold_loads;            // self-test: issue no loads, so the first wait runs out
  int z_tma;                     // row owner: logits leave through bulk tensor stores
  int n_acc;                     // accumulators per tile, each BT columns (see issue_stage)
  EpiParams ep;
};

// One stretch of work: k-steps [kb, ke) of cluster unit `unit`.
struct Piece {
  int unit, kb, ke;
};

// The sequence of pieces a cluster processes; all roles of all its CTAs
// walk it alike.
struct PieceIter {
  long long it, end;
  int unit;
  __device__ PieceIter(const TcParams& p) {
    const int cid = blockIdx.x / p.K;
    const int ncl = gridDim.x / p.K;
    if (p.stream_k) {
      it = p.total_iters * cid / ncl;
      end = p.total_iters * (cid + 1) / ncl;
    } else {
      unit = cid;
    }
  }
  __device__ bool next(const TcParams& p, Piece& pc) {
    if (p.stream_k) {
      if (it >= end) return false;
      const long long u = it / p.nk;
      pc.unit = (int)u;
      pc.kb = (int)(it - u * p.nk);
      const long long rem = end - it;
      pc.ke = (int)((long long)pc.kb + rem < (long long)p.nk ? pc.kb + rem : p.nk);
      it += pc.ke - pc.kb;
      return true;
    }
    if (unit >= p.n_units) return false;
    pc.unit = unit;
    pc.kb = 0;
    pc.ke = p.nk;
    unit += gridDim.x / p.K;
    return true;
  }
};

// q statistics streamed by spare warps: one (max, sum exp2) record per draft
// row and kQChunk columns, 16-byte loads (8 bf16) with 8 in flight per lane.
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

__device__ __forceinline__ PartialQ q_chunk_stats(const __nv_bfloat16* __restrict__ dl, int r,
                                                  int chunk, int V, float c, bool vec) {
  constexpr int kInFlight = 8;
  const int lane = threadIdx.x & 31;
  const int c0 = chunk * kQChunk;
  const int c1 = min(V, c0 + kQChunk);
  const __nv_bfloat16* row = dl + (size_t)r * V;
  float m = -INFINITY, s = 0.f;
  if (vec) {
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
  return PartialQ{m, s};
}

// One stage's MMAs: KC slices of four k16 steps. The descriptors advance by
// constant offsets from the stage's first A and B descriptors (a shared
// memory descriptor's low field is the byte address / 16), so the issue loop
// spends a few instructions per MMA: one thread issues every MMA of the CTA
// (or pair), and on shapes with narrow token tiles each MMA's tensor work is
// short enough that the issue rate, not the tensor core, would otherwise set
// the pace.
//
// Slice c of the stage goes to accumulator (sub0 + c) mod n_acc, each
// acc_cols columns from the last. The tensor core adds into its fp32
// accumulator with truncation, so the error of one accumulator grows with
// the number of additions and with the running sum's magnitude (a bias, not
// a random walk): dealing the slices across n_acc accumulators, which the
// epilogue adds in fp32 at the end, divides it by about n_acc. The first
// slice a piece gives each accumulator (fresh > c) starts it afresh.
//
// kMulti = false (one accumulator) compiles to the plain loop: the issuing
// thread's own instructions are on the critical path of the tensor-bound
// shapes, so nothing here may cost more than a few per MMA.
template <int KC, bool kPair, bool kRowOwn, bool kMulti>
__device__ __forceinline__ void issue_stage(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                            uint32_t b_slice16, uint32_t idesc, int sub0,
                                            int n_acc, uint32_t acc_cols, int fresh) {
  int sub = sub0;
#pragma unroll
  for (int c = 0; c < KC; ++c) {
    const uint32_t d = kMulti ? d_tmem + (uint32_t)sub * acc_cols : d_tmem;
#pragma unroll
    for (int k = 0; k < kBlockK / 16; ++k) {
      const uint64_t a = ad + (uint64_t)(c * (kStageA >> 4) + 2 * k);
      const uint64_t b = bd + (uint64_t)(c * b_slice16 + 2 * k);
      const uint32_t accum = (k == 0 && c < fresh) ? 0u : 1u;
      if constexpr (kRowOwn)   // A = token rows, B = W rows
        tc2_mma_bf16(d, b, a, idesc, accum);
      else if constexpr (kPair)
        tc2_mma_bf16(d, a, b, idesc, accum);
      else
        tc_mma_bf16(d, a, b, idesc, accum);
    }
    if (kMulti && ++sub == n_acc) sub = 0;
  }
}

// The tile's logits for 16 or 32 token columns at column `col`: the sum, in
// order, of the n_used accumulators (stride acc_cols) the piece wrote.
template <int N>
__device__ __forceinline__ void tmem_ld_acc(uint32_t tbase, int col, int n_used, uint32_t acc_cols,
                                            float (&z)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 16)
    tmem_ld16(tbase + (uint32_t)col, z);
  else
    tmem_ld32(tbase + (uint32_t)col, z);
  for (int j = 1; j < n_used; ++j) {
#pragma unroll
    for (int h = 0; h < N / 16; ++h) {   // 16 columns at a time: fewer live registers
      float t[16];
      tmem_ld16(tbase + (uint32_t)j * acc_cols + (uint32_t)(col + 16 * h), t);
#pragma unroll
      for (int n = 0; n < 16; ++n) z[16 * h + n] += t[n];
    }
  }
}

__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kDrainLimitNs) return false;
  }
  return true;
}

// kPair: the 2-SM (CTA pair) build; cta_group::1 and ::2 instructions cannot
// share a kernel. kRowOwn (pairs with 256-row token tiles): tokens on the
// MMA's M side, so tensor-memory lane = token row and each epilogue thread
// owns one token row.
template <typename DL, bool kPair, bool kRowOwn>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_h,
                     const __grid_constant__ CUtensorMap tmap_z, const TcParams p) {
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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (3 * S + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  PartialP* red = reinterpret_cast<PartialP*>(misc + kBarBytes);   // [4 warps][BT] column partials
  PartialP* run = red + 4 * p.BT;  // [BT] per-row records folded over the CTA's tiles
  PartialQ* qrun = reinterpret_cast<PartialQ*>(run + p.BT);  // [BT] draft rows, likewise

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)(blockIdx.x % p.K);      // rank within the cluster
  const int cid = (int)(blockIdx.x / p.K);
  constexpr bool pair = kPair;
  const int hid_rows = p.BT / p.K;               // token rows this CTA loads per slice

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), pair ? 2 : 1);   // one arrival per epilogue; a pair's leader counts both
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (p.stream_k)
    for (int r = threadIdx.x; r < p.BT; r += kThreads) {
      run[r] = PartialP{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
      qrun[r] = PartialQ{-INFINITY, 0.f};
    }
  if (warp == 1) {
    if constexpr (kPair)
      tmem_alloc_pair(smem_u32(tmem_slot), p.tmem_cols);
    else
      tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
  }
  // Launched with programmatic dependent launch: the set-up above overlaps
  // the previous kernel; global memory is touched only after this wait.
  grid_dependency_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) *(volatile int*)p.status = SPECDEC_OK;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.ep.n_counters; i += kThreads) p.ep.counters[i] = 0;
  // This call's fix-up tag; the call count only changes after this kernel.
  const unsigned long long tag = call_tag(p.epoch, p.calls);
  tc_fence_before();
  __syncthreads();
  if (pair) cluster_sync_all();   // the partner's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer --
      // A W tile read by one token tile leaves L2 first; with several token
      // tiles, the other tiles' CTAs read the same W tile at about the same
      // time, so it keeps the normal priority and outlives the logit stores.
      const uint64_t pol_w = p.n_tt > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      PieceIter itr(p);
      Piece pc;
      while (ok && !p.withhold_loads && itr.next(p, pc)) {
        const int vt = (pc.unit / p.n_tt) * p.K + rank;
        const int tt = pc.unit % p.n_tt;
        for (int kc = pc.kb; kc < pc.ke; ++kc) {
          const bool got = pair ? mbar_wait_cluster<true>(empty_bar(s), ph ^ 1u, abort_flag, p.status)
                                : mbar_wait<true>(empty_bar(s), ph ^ 1u, abort_flag, p.status);
          if (!got) {
            ok = false;
            break;
          }
          const uint32_t a = sbase + (uint32_t)s * p.stage_bytes;
          const uint32_t h = a + (uint32_t)(p.kc * kStageA);
          // Token rows [rank*BT/K, (rank+1)*BT/K) of the tile (all of them when K = 1).
          const int row = tt * p.BT + rank * hid_rows;
          if constexpr (kPair) {
            // Both halves of the stage complete on the leader's full barrier.
            const uint32_t lead_full = mapa_shared(full_bar(s), 0);
            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2u * p.stage_bytes);
            if (p.box3d) {
              tma_load_3d_pair(a, &tmap_w, lead_full, 0, vt * kBlockV, kc * p.kc, pol_w);
              tma_load_3d_pair(h, &tmap_h, lead_full, 0, row, kc * p.kc, pol_h);
            } else {
              tma_load_2d_pair(a, &tmap_w, lead_full, kc * kBlockK, vt * kBlockV, pol_w);
              tma_load_2d_pair(h, &tmap_h, lead_full, kc * kBlockK, row, pol_h);
            }
          } else {
            mbar_arrive_expect_tx(full_bar(s), p.stage_bytes);
            if (p.box3d) {
              tma_load_3d(a, &tmap_w, full_bar(s), 0, vt * kBlockV, kc * p.kc, pol_w);
              tma_load_3d(h, &tmap_h, full_bar(s), 0, row, kc * p.kc, pol_h);
            } else {
              tma_load_2d(a, &tmap_w, full_bar(s), kc * kBlockK, vt * kBlockV, pol_w);
              tma_load_2d(h, &tmap_h, full_bar(s), kc * kBlockK, row, pol_h);
            }
          }
          issued_mask |= 1u << s;
          issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && (!kPair || rank == 0)) {
        // Let every copy already issued land before the CTA exits (a pair's
        // copies all complete on the leader's barriers).
        for (int t = 0; t < S; ++t)
          if (issued_mask & (1u << t)) mbar_wait_drain(full_bar(t), (issued_phase >> t) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (kPair && rank == 1) {
        // The pair's MMAs are issued by the leader; nothing to do here.
      } else {
        // ---------------------------------------------------- MMA issuer --
        const uint32_t idesc = idesc_bf16_f32(pair ? 2 * kBlockV : kBlockV, p.BT);
        // Stage s, slice c: W rows [128 x 128 B] at sbase + s * stage_bytes + c * 16 KB,
        // then this CTA's token rows [BT/K x 128 B] per slice after the kc W slices.
        const uint64_t desc0 = smem_desc_sw128(sbase);
        const uint32_t stage16 = p.stage_bytes >> 4;
        const uint32_t hoff16 = (uint32_t)(p.kc * kStageA) >> 4;
        const uint32_t hsl16 = (uint32_t)(hid_rows * kBlockK * 2) >> 4;
        const int n_acc = p.n_acc, kcs = p.kc;
        const uint32_t acols = (uint32_t)p.BT;
        int s = 0;
        uint32_t ph = 0;
        int ul = 0;
        bool ok = true;
        PieceIter itr(p);
        Piece pc;
        while (ok && itr.next(p, pc)) {
          const int acc = ul & 1;
          const uint32_t aph = (uint32_t)(ul >> 1) & 1u;
          const bool empty_ok = pair ? mbar_wait_cluster<true>(tempty_bar(acc), aph ^ 1u, abort_flag, p.status)
                                     : mbar_wait<true>(tempty_bar(acc), aph ^ 1u, abort_flag, p.status);
          if (!empty_ok) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.BT * p.n_acc);
          int sub = 0;    // accumulator of the stage's first slice
          int srel = 0;   // slices of this piece issued so far
          for (int kc = pc.kb; kc < pc.ke; ++kc) {
            const bool got = pair ? mbar_wait_cluster<true>(full_bar(s), ph, abort_flag, p.status)
                                  : mbar_wait<true>(full_bar(s), ph, abort_flag, p.status);
            if (!got) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = desc0 + (uint64_t)((uint32_t)s * stage16);
            const uint64_t bd = ad + hoff16;
            const int fresh = n_acc - srel;   // slices c < fresh start their accumulator
            if (n_acc == 1) {
              if (kcs == 4)
                issue_stage<4, kPair, kRowOwn, false>(d_tmem, ad, bd, hsl16, idesc, 0, 1, acols, fresh);
              else if (kcs == 2)
                issue_stage<2, kPair, kRowOwn, false>(d_tmem, ad, bd, hsl16, idesc, 0, 1, acols, fresh);
              else
                issue_stage<1, kPair, kRowOwn, false>(d_tmem, ad, bd, hsl16, idesc, 0, 1, acols, fresh);
            } else {
              if (kcs == 4)
                issue_stage<4, kPair, kRowOwn, true>(d_tmem, ad, bd, hsl16, idesc, sub, n_acc, acols, fresh);
              else if (kcs == 2)
                issue_stage<2, kPair, kRowOwn, true>(d_tmem, ad, bd, hsl16, idesc, sub, n_acc, acols, fresh);
              else
                issue_stage<1, kPair, kRowOwn, true>(d_tmem, ad, bd, hsl16, idesc, sub, n_acc, acols, fresh);
              sub += kcs;   // kcs <= 4, so a few subtractions replace a division
              while (sub >= n_acc) sub -= n_acc;
            }
            srel += kcs;
            if constexpr (kPair)
              tc2_commit_mc(empty_bar(s), 3);   // the stage is free in both CTAs
            else
              tc_commit(empty_bar(s));
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          if constexpr (kPair)
            tc2_commit_mc(tfull_bar(acc), 3);
          else
            tc_commit(tfull_bar(acc));
          ++ul;
        }
        // All MMAs this thread issued are complete once this phase ends.
        if constexpr (kPair)
          tc2_commit_mc(mma_done_bar, 1);
        else
          tc_commit(mma_done_bar);
        mbar_wait_drain(mma_done_bar, 0);
      }
    }
  } else if (warp >= kQWarp0) {
    // ---------------------------------------------------------- q-warps --
    if (p.ep.q_stream && warp < kQWarp0 + kQStreamWarps) {
      // Many draft rows: stream them whole, (row, kQChunk-column chunk)
      // items dealt across the grid, while the tensor cores work. The warp
      // on the MMA issuer's scheduler (warp 13) stays out of it.
      const __nv_bfloat16* dl = static_cast<const __nv_bfloat16*>(p.ep.dl);
      const long long n_items = (long long)p.ep.n_qrows * p.ep.Pq;
      const int ns = gridDim.x * kQStreamWarps;
      for (long long it = (long long)blockIdx.x * kQStreamWarps + (warp - kQWarp0); it < n_items;
           it += ns) {
        const int r = (int)(it / p.ep.Pq);
        const int chunk = (int)(it - (long long)r * p.ep.Pq);
        const PartialQ q = q_chunk_stats(dl, r, chunk, p.V, p.ep.c, p.ep.q_vec != 0);
        if (lane == 0) p.ep.pq[(size_t)r * p.ep.Pq + chunk] = q;
      }
    } else if (p.ep.sample && p.ep.q_warps) {
      const int qw = warp - kQWarp0;
      const int g1 = p.gamma + 1;
      const __nv_bfloat16* dl = static_cast<const __nv_bfloat16*>(p.ep.dl);
      PieceIter itr(p);
      Piece pc;
      while (itr.next(p, pc)) {
        const int vt = (pc.unit / p.n_tt) * p.K + rank;
        if (pc.kb != 0 || vt >= p.n_vt) continue;
        const int tt = pc.unit % p.n_tt;
        const int m_lo = tt * p.BT;
        const int m_hi = min(p.M, m_lo + p.BT);
        // Draft rows of token rows [m_lo, m_hi): a contiguous range.
        const int dr_lo = (m_lo / g1) * p.gamma + min(m_lo % g1, p.gamma);
        const int dr_hi = (m_hi / g1) * p.gamma + min(m_hi % g1, p.gamma);
        const int v0 = vt * kBlockV;
        for (int r0 = dr_lo + qw; r0 < dr_hi; r0 += 4 * kQRowsInFlight) {
          float x[kQRowsInFlight][4];
#pragma unroll
          for (int g = 0; g < kQRowsInFlight; ++g) {
            const int r = r0 + 4 * g;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int v = v0 + lane + 32 * e;
              x[g][e] = (r < dr_hi && v < p.V) ? __bfloat162float(dl[(size_t)r * p.V + v])
                                                : -INFINITY;
            }
          }
#pragma unroll
          for (int g = 0; g < kQRowsInFlight; ++g) {
            const int r = r0 + 4 * g;
            float m = fmaxf(fmaxf(x[g][0], x[g][1]), fmaxf(x[g][2], x[g][3]));
            float sum = 0.f;
            if (m != -INFINITY) {
#pragma unroll
              for (int e = 0; e < 4; ++e) sum += exp2f((x[g][e] - m) * p.ep.c);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
              const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
              const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
              osm_merge(m, sum, m2, s2, p.ep.c);
            }
            if (lane == 0 && r < dr_hi) {
              if (p.stream_k) {
                osm_merge(qrun[r].m, qrun[r].s, m, sum, p.ep.c);   // warp r % 4 owns slot r
              } else {
                p.ep.pq[(size_t)r * p.ep.P + vt] = PartialQ{m, sum};
              }
            }
          }
        }
      }
      if (p.stream_k) {
        named_bar_sync(3, 128);
        const int n_draft = (p.M / g1) * p.gamma + min(p.M % g1, p.gamma);
        for (int r = threadIdx.x - 32 * kQWarp0; r < n_draft; r += 128)
          p.ep.pq[(size_t)r * p.ep.P + blockIdx.x] = qrun[r];
      }
    }
  } else if constexpr (kRowOwn) {
    // ------------------------------------------------ epilogue, row owner --
    // Tensor-memory lane = token row: thread (quarter q, lane) owns token
    // row r = 32q + lane of this CTA's 128 and reduces its softmax and
    // argmax partials in registers, 32 vocabulary columns per load; the two
    // warp groups take alternate chunks and merge once per record.
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const size_t slot_floats = (size_t)p.BT * kBlockV;
    const bool vsample = p.ep.sample != 0;
    const bool vargmax = p.ep.want_argmax != 0;
    const bool zvec = (p.V & 3) == 0 && ((uintptr_t)p.ep.zout & 15u) == 0;
    const bool ztma = p.z_tma != 0 && p.ep.zout != nullptr;
    const uint32_t zstg = sbase + (uint32_t)(S * p.stage_bytes + misc_span(p.BT)) +
                          (uint32_t)((warp - 2) * kZStageBytes);
    const int n32 = p.BT / 32;               // 32-column chunks of the 256-wide vocabulary tile
    PartialP st{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
    int m = rank * 128 + r;                  // token row (stream-K: the only token tile)
    int ul = 0;
    PieceIter itr(p);
    Piece pc;
    while (itr.next(p, pc)) {
      const int acc = ul & 1;
      const uint32_t aph = (uint32_t)(ul >> 1) & 1u;
      ++ul;
      const int vt2 = pc.unit / p.n_tt;      // vocabulary tile of 256 (both CTAs' W rows)
      const int tt = pc.unit % p.n_tt;
      m = tt * p.BT + rank * 128 + r;
      if (threadIdx.x == 64)
        *epi_flag = (mbar_wait_cluster<true>(tfull_bar(acc), aph, abort_flag, p.status)) ? 1 : 0;
      named_bar_sync(1, kEpiThreads);
      const bool ok = *epi_flag != 0;
      named_bar_sync(2, kEpiThreads);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.BT);
      bool finish = true;
      const float* other = nullptr;
      if (pc.kb > 0 || pc.ke < p.nk) {
        // Tile shared with the neighbouring cluster (see the swap-AB path).
        const int bnd = pc.kb > 0 ? cid : cid + 1;
        const int slot = bnd * p.K + rank;
        const int part = pc.kb > 0 ? 1 : 0;
        float* mine = p.fix + ((size_t)slot * 2 + part) * slot_floats;
        other = p.fix + ((size_t)slot * 2 + (1 - part)) * slot_floats;
        for (int c = grp; c < n32; c += 2) {
          float accv[32];
          tmem_ld32(tbase + (uint32_t)(c * 32), accv);
#pragma unroll
          for (int n = 0; n < 32; ++n) __stcg(mine + (size_t)(c * 32 + n) * kBlockV + r, accv[n]);
        }
        __threadfence();
        named_bar_sync(1, kEpiThreads);
        if (threadIdx.x == 64) {
          const unsigned long long prev = atomicExch(p.fix_tickets + slot, tag);
          __threadfence();
          *epi_flag = prev == tag ? 1 : 0;
        }
        named_bar_sync(1, kEpiThreads);
        finish = *epi_flag != 0;
        named_bar_sync(2, kEpiThreads);
        if (finish) __threadfence();
      }
      const bool mvalid = m < p.M;
      if (finish) {
        for (int c = grp; c < n32; c += 2) {
          float z[32];
          tmem_ld32(tbase + (uint32_t)(c * 32), z);
          if (other != nullptr) {
#pragma unroll
            for (int n = 0; n < 32; ++n) z[n] += __ldcg(other + (size_t)(c * 32 + n) * kBlockV + r);
          }
          const int v0 = vt2 * p.BT + c * 32;
          const bool full = v0 + 32 <= p.V;
          const int mw = m - lane;                 // the warp's first token row
          if (ztma) {
            // Through shared memory: this lane's row, 16-byte units swizzled
            // by row, then one bulk tensor store of the warp's 32 x 32 tile
            // (rows past M and columns past V are clipped by the copy).
            if (mw < p.M && v0 < p.V) {
              if (lane == 0) bulk_wait_read0();    // the previous tile has left the buffer
              __syncwarp();
              const uint32_t rowa = zstg + (uint32_t)(lane * 128);
#pragma unroll
              for (int k = 0; k < 8; ++k)
                st_shared_v4(rowa + (uint32_t)(((k ^ (lane & 7)) & 7) << 4), z[4 * k], z[4 * k + 1],
                             z[4 * k + 2], z[4 * k + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d_hint(&tmap_z, zstg, v0, mw, policy_evict_first());
                bulk_commit();
              }
            }
          } else if (p.ep.zout != nullptr && mvalid) {
            float* zr = p.ep.zout + (size_t)m * p.V + v0;
            if (full && zvec) {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                __stcs(reinterpret_cast<float4*>(zr) + k,
                       make_float4(z[4 * k], z[4 * k + 1], z[4 * k + 2], z[4 * k + 3]));
            } else {
#pragma unroll
              for (int n = 0; n < 32; ++n)
                if (v0 + n < p.V) __stcs(zr + n, z[n]);
            }
          }
          if (!full) {
#pragma unroll
            for (int n = 0; n < 32; ++n)
              if (v0 + n >= p.V) z[n] = -INFINITY;
          }
          if (vsample) {
            float mx = z[0];
#pragma unroll
            for (int n = 1; n < 32; ++n) mx = fmaxf(mx, z[n]);
            const float mm = fmaxf(st.m, mx);
            if (mm != -INFINITY) {
              float sum = st.m == -INFINITY ? 0.f : st.s * exp2f((st.m - mm) * p.ep.c);
#pragma unroll
              for (int n = 0; n < 32; ++n) sum += exp2f((z[n] - mm) * p.ep.c);
              st.m = mm;
              st.s = sum;
            }
          }
          if (vargmax) {
#pragma unroll
            for (int n = 0; n < 32; ++n)
              if (z[n] > st.amax_v) {   // ascending v: strict > keeps the lowest index
                st.amax_v = z[n];
                st.amax_i = v0 + n;
              }
          }
        }
      }
      // Every epilogue thread's tensor-memory loads are done; one thread per
      // CTA hands the accumulator back.
      tc_fence_before();
      named_bar_sync(1, kEpiThreads);
      if (threadIdx.x == 64) {
        if (rank == 1)
          mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
        else
          mbar_arrive(tempty_bar(acc));
      }
      if (!p.stream_k) {
        // One record per (token row, vocabulary tile): merge the two groups.
        if (grp == 1) red[r] = st;
        named_bar_sync(1, kEpiThreads);
        if (grp == 0 && mvalid) {
          PartialP a = st;
          partialp_merge(a, red[r], p.ep.c);
          p.ep.pp[(size_t)m * p.ep.P + vt2] = a;
        }
        named_bar_sync(1, kEpiThreads);
        st = PartialP{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
      }
    }
    if (ztma && lane == 0) bulk_wait0();   // every logit tile is written before the CTA ends
    if (p.stream_k) {
      // One record per token row and cluster for everything it finished.
      if (grp == 1) red[r] = st;
      named_bar_sync(1, kEpiThreads);
      if (grp == 0 && m < p.M) {
        PartialP a = st;
        partialp_merge(a, red[r], p.ep.c);
        p.ep.pp[(size_t)m * p.ep.P + cid] = a;
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int grp = (warp - 2) >> 2;        // chunk group: pairs 2*grp, 2*grp + 4, ...
    const int epi_tid = threadIdx.x - 64;
    const int row = q * 32 + lane;          // vocabulary row within the tile
    const size_t slot_floats = (size_t)p.BT * kBlockV;
    const bool vsample = p.ep.sample != 0;
    const bool vargmax = p.ep.want_argmax != 0;
    int ul = 0;
    PieceIter itr(p);
    Piece pc;
    while (itr.next(p, pc)) {
      const int acc = ul & 1;
      const uint32_t aph = (uint32_t)(ul >> 1) & 1u;
      ++ul;
      const int vt = (pc.unit / p.n_tt) * p.K + rank;
      const int tt = pc.unit % p.n_tt;
      const int v = vt * kBlockV + row;
      const int m_base = tt * p.BT;
      if (epi_tid == 0)
        *epi_flag = (pair ? mbar_wait_cluster<true>(tfull_bar(acc), aph, abort_flag, p.status)
                          : mbar_wait<true>(tfull_bar(acc), aph, abort_flag, p.status))
                        ? 1
                        : 0;
      named_bar_sync(1, kEpiThreads);
      const bool ok = *epi_flag != 0;
      named_bar_sync(2, kEpiThreads);
      if (!ok) break;
      tc_fence_after();
      const int n_chunks = (min(p.BT, p.M - m_base) + 15) / 16;
      const uint32_t tbase =
          tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.BT * p.n_acc);
      // accumulators this piece wrote (a short stream-K piece may not reach all)
      const int n_used = min(p.n_acc, (pc.ke - pc.kb) * p.kc);
      const uint32_t acols = (uint32_t)p.BT;

      // A tile past the vocabulary (odd tile count in a cluster) has nothing to report.
      bool finish = vt < p.n_vt;
      const float* other = nullptr;
      if (finish && (pc.kb > 0 || pc.ke < p.nk)) {
        // A tile shared with the neighbouring cluster: the piece holding
        // k-step 0 is part A of the boundary slot after its cluster, the
        // other part B. Slots are per boundary and cluster rank.
        const int bnd = pc.kb > 0 ? cid : cid + 1;
        const int slot = bnd * p.K + rank;
        const int part = pc.kb > 0 ? 1 : 0;
        float* mine = p.fix + ((size_t)slot * 2 + part) * slot_floats;
        other = p.fix + ((size_t)slot * 2 + (1 - part)) * slot_floats;
        for (int c = grp; c < n_chunks; c += 2) {
          float accv[16];
          tmem_ld_acc<16>(tbase, c * 16, n_used, acols, accv);
#pragma unroll
          for (int n = 0; n < 16; ++n) __stcg(mine + (size_t)(c * 16 + n) * kBlockV + row, accv[n]);
        }
        __threadfence();
        named_bar_sync(1, kEpiThreads);
        if (epi_tid == 0) {
          // The part that finds this call's tag already there arrives second.
          const unsigned long long prev = atomicExch(p.fix_tickets + slot, tag);
          __threadfence();
          *epi_flag = prev == tag ? 1 : 0;
        }
        named_bar_sync(1, kEpiThreads);
        finish = *epi_flag != 0;
        named_bar_sync(2, kEpiThreads);
        if (finish) __threadfence();
      }
      if (finish) {
        const bool vvalid = v < p.V;
        // Per 32-column chunk (one tensor-memory load): logits out, then each
        // warp's (max, sum exp2) and argmax per column into red[warp
        // quarter][column], lane L holding column L. The two warp groups take
        // alternate chunks; a 16-column tail goes to the group next in turn.
        const int n32 = n_chunks >> 1;
        for (int c = grp; c < n32; c += 2) {
          float z[32];
          tmem_ld_acc<32>(tbase, c * 32, n_used, acols, z);
          if (other != nullptr) {
#pragma unroll
            for (int n = 0; n < 32; ++n) z[n] += __ldcg(other + (size_t)(c * 32 + n) * kBlockV + row);
          }
          const int m0 = m_base + c * 32;
          if (p.ep.zout != nullptr && vvalid) {
#pragma unroll
            for (int n = 0; n < 32; ++n)
              if (m0 + n < p.M) __stcs(p.ep.zout + (size_t)(m0 + n) * p.V + v, z[n]);
          }
#pragma unroll
          for (int n = 0; n < 32; ++n) z[n] = vvalid ? z[n] : -INFINITY;
          PartialP r{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
          if (vsample) warp_softmax32(z, p.ep.c, r.m, r.s);
          if (vargmax) warp_argmax32(z, vvalid ? v : 0x7fffffff, r.amax_v, r.amax_i);
          red[q * p.BT + c * 32 + lane] = r;
        }
        if ((n_chunks & 1) && grp == (n32 & 1)) {
          const int cc = n_chunks - 1;
          float z[16];
          tmem_ld_acc<16>(tbase, cc * 16, n_used, acols, z);
          if (other != nullptr) {
#pragma unroll
            for (int n = 0; n < 16; ++n) z[n] += __ldcg(other + (size_t)(cc * 16 + n) * kBlockV + row);
          }
          const int m0 = m_base + cc * 16;
          if (p.ep.zout != nullptr && vvalid) {
#pragma unroll
            for (int n = 0; n < 16; ++n)
              if (m0 + n < p.M) __stcs(p.ep.zout + (size_t)(m0 + n) * p.V + v, z[n]);
          }
#pragma unroll
          for (int n = 0; n < 16; ++n) z[n] = vvalid ? z[n] : -INFINITY;
          PartialP r{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
          if (vsample) warp_softmax16(z, p.ep.c, r.m, r.s);
          if (vargmax) warp_argmax16(z, vvalid ? v : 0x7fffffff, r.amax_v, r.amax_i);
          if ((lane & 1) == 0) red[q * p.BT + cc * 16 + (lane >> 1)] = r;
        }
        named_bar_sync(1, kEpiThreads);
        // Columns across the four warp quarters, 256 columns at a time;
        // column col is always folded by thread col % 256.
        const int ncols = min(p.BT, p.M - m_base);
        for (int col = epi_tid; col < ncols; col += kEpiThreads) {
          PartialP a = red[col];
#pragma unroll
          for (int qq = 1; qq < 4; ++qq) partialp_merge(a, red[qq * p.BT + col], p.ep.c);
          const int m = m_base + col;
          if (p.stream_k)
            partialp_merge(run[m], a, p.ep.c);
          else
            p.ep.pp[(size_t)m * p.ep.P + vt] = a;
        }
        named_bar_sync(1, kEpiThreads);
      }
      // Every epilogue thread's tensor-memory loads are done; one thread per
      // CTA hands the accumulator back (a pair's to the leader, whose MMAs
      // reuse it).
      tc_fence_before();
      named_bar_sync(1, kEpiThreads);
      if (epi_tid == 0) {
        if (pair && rank == 1)
          mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
        else
          mbar_arrive(tempty_bar(acc));
      }
    }
    if (p.stream_k) {
      // One record per token row for everything this CTA finished.
      named_bar_sync(1, kEpiThreads);
      for (int m = epi_tid; m < p.M; m += kEpiThreads) p.ep.pp[(size_t)m * p.ep.P + blockIdx.x] = run[m];
    }
  }

  __syncthreads();
  // A pair deallocates collectively, once both CTAs are done with it and
  // with each other's barriers.
  if (pair) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, p.tmem_cols);
    else
      tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

int max_clusters_cached(int smem_bytes, int K) {
  static int cache[kMaxDevices][3] = {{0}};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev][0] == smem_bytes && cache[dev][1] == K) return cache[dev][2];
  auto kern = lmhead_tc_kernel<__nv_bfloat16, true, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(K * 512);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  cache[dev][0] = smem_bytes;
  cache[dev][1] = K;
  cache[dev][2] = n;
  return n;
}

}  // namespace

TcGeometry tc_geometry(int M, int V, int d, int num_sms, int max_clusters) {
  TcGeometry g;
  g.n_tt = (M + kMaxBT - 1) / kMaxBT;
  if (g.n_tt < 1) g.n_tt = 1;
  const int per = (M + g.n_tt - 1) / g.n_tt;
  g.BT = ((per + 15) / 16) * 16;
  if (g.BT < 16) g.BT = 16;
  // Slices per stage: 4 while three such stages fit, else 2 while four fit,
  // else 1 (the stream rates these caps were chosen from are in the kernel
  // header comment).
  g.n_vt = (V + kBlockV - 1) / kBlockV;
  g.K = (g.BT >= kClusterMinBT && g.n_vt >= 2) ? 2 : 1;
  // Token tiles of 256 on a CTA pair put the tokens on the MMA's M side
  // (row-owner epilogue, with its logit staging).
  g.rowown = (g.K == 2 && g.BT == 2 * kBlockV) ? 1 : 0;
  const int misc_total = g.rowown ? misc_span(g.BT) + kZStaging : misc_bytes(g.BT);
  const int budget = kSmemLimit - 1024 - misc_total;
  // A CTA holds 128 W rows and BT/K token rows of every slice.
  const int slice_bytes = kStageA + (g.BT / g.K) * kBlockK * 2;
  g.box3d = d % kBlockK == 0 ? 1 : 0;
  if (g.box3d && budget / (4 * slice_bytes) >= 3) {
    g.kc = 4;
  } else if (g.box3d && budget / (2 * slice_bytes) >= 4) {
    g.kc = 2;
  } else {
    g.kc = 1;
  }
  g.stage_bytes = g.kc * slice_bytes;
  const int cap = g.kc == 4 ? kMaxStagesC4 : g.kc == 2 ? kMaxStagesC2 : kMaxStagesC1;
  int stages = budget / g.stage_bytes;
  if (stages > cap) stages = cap;
  g.stages = stages;
  // Accumulators per tile (issue_stage): as many as two sets (the epilogue
  // drains one while the MMAs fill the other) leave room for in the 512
  // tensor-memory columns, up to 16; the row-owner layout fills them with one.
  g.n_acc = 1;
  if (!g.rowown)
    while (g.n_acc < kMaxAcc && 2 * g.BT * (g.n_acc + 1) <= kTmemCols) ++g.n_acc;
  int cols = 32;
  while (cols < 2 * g.BT * g.n_acc) cols <<= 1;
  g.tmem_cols = cols;
  g.smem_bytes = 1024 + g.stages * g.stage_bytes + misc_total;
  g.n_units = ((g.n_vt + g.K - 1) / g.K) * g.n_tt;
  g.nk = ((d + kBlockK - 1) / kBlockK + g.kc - 1) / g.kc;
  const int sms = num_sms < kMaxGrid ? num_sms : kMaxGrid;
  int clusters = sms / g.K;
  if (g.K > 1 && max_clusters > 0 && max_clusters < clusters) clusters = max_clusters;
  if (clusters > g.n_units) clusters = g.n_units;
  if (clusters < 1) clusters = 1;
  g.grid = clusters * g.K;
  g.stream_k = g.n_tt == 1 ? 1 : 0;
  // Row owner: one record per token row and cluster (stream-K) or per
  // 256-row vocabulary tile.
  if (g.rowown)
    g.records = g.stream_k ? g.grid / g.K : (g.n_vt + 1) / 2;
  else
    g.records = g.stream_k ? g.grid : g.n_vt;
  return g;
}

int tc_max_clusters(int M, int V, int d) {
  const TcGeometry g = tc_geometry(M, V, d, kMaxGrid, 0);
  if (g.K == 1) return 0;
  return max_clusters_cached(g.smem_bytes, g.K);
}

cudaError_t launch_lmhead_tc(const TcLaunch& L, int num_sms, cudaStream_t stream) {
  const TcGeometry g = tc_geometry(L.M, L.V, L.d, num_sms, L.max_clusters);
  TcParams p;
  p.M = L.M;
  p.V = L.V;
  p.d = L.d;
  p.gamma = L.gamma;
  p.BT = g.BT;
  p.n_tt = g.n_tt;
  p.nk = g.nk;
  p.stages = g.stages;
  p.n_vt = g.n_vt;
  p.K = g.K;
  p.n_units = g.n_units;
  p.kc = g.kc;
  p.box3d = g.box3d;
  p.stream_k = g.stream_k;
  p.total_iters = (long long)g.n_units * g.nk;
  p.stage_bytes = (uint32_t)g.stage_bytes;
  p.tmem_cols = (uint32_t)g.tmem_cols;
  p.status = L.status;
  p.fix = L.fix;
  p.fix_tickets = L.fix_tickets;
  p.epoch = L.epoch;
  p.calls = L.calls;
  p.withhold_loads = L.withhold_loads;
  p.z_tma = (g.rowown && L.tmap_z != nullptr) ? 1 : 0;
  p.n_acc = g.n_acc;
  p.ep = L.ep;
  p.ep.P = g.records;
  p.ep.run = nullptr;
  p.ep.q_in_epilogue = 0;   // q-warps (ep.q_warps) or the standalone stream reduce q
  // The tensor-core path exists for bf16 inputs; draft logits share the dtype.
  auto kern = g.rowown ? lmhead_tc_kernel<__nv_bfloat16, true, true>
               : g.K > 1 ? lmhead_tc_kernel<__nv_bfloat16, true, false>
                         : lmhead_tc_kernel<__nv_bfloat16, false, false>;
  // The shared-memory opt-in is set once per device, build and size.
  static int smem_set[kMaxDevices][3] = {{0}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int which = g.rowown ? 2 : g.K > 1 ? 1 : 0;
  if (dev < 0 || dev >= kMaxDevices || smem_set[dev][which] != g.smem_bytes) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) smem_set[dev][which] = g.smem_bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = g.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = g.K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, *L.tmap_w, *L.tmap_h,
                            L.tmap_z != nullptr ? *L.tmap_z : *L.tmap_w, p);
}

}  // namespace specdec
