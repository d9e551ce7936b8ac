// C ABI of the verify step: argument checks, workspace plan, tensor maps
// and the stream-ordered launch sequence
//   LM-head scoring (+ softmax/argmax partials)  ->  acceptance scan
//   ->  residual / bonus draw (sampling mode only).
#include <cstddef>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <mutex>

#include "kernels.h"

using namespace specdec;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Plan {
  int M, P, nchunks;
  size_t off_tickets, off_sel, off_counters, off_pp, off_pq, off_z, off_chunks, off_fix, total;

};

// Checks the shape; returns SPECDEC_OK or an error code.
int check_shape(int B, int gamma, int d, int V, int dtype, int mode) {
  if (dtype != SPECDEC_BF16 && dtype != SPECDEC_FP32) return SPECDEC_ERR_INVALID_ARG;
  if (mode != SPECDEC_SAMPLE && mode != SPECDEC_GREEDY) return SPECDEC_ERR_INVALID_ARG;
  if (B < 0 || gamma < 1 || gamma > SPECDEC_MAX_GAMMA || d < 1 || V < 1 || V > kMaxVocab)
    return SPECDEC_ERR_UNSUPPORTED;
  if (dtype == SPECDEC_BF16 && d % 8 != 0) return SPECDEC_ERR_UNSUPPORTED;
  const long long M = (long long)B * (gamma + 1);
  if (M * (long long)V >= (1ll << 31)) return SPECDEC_ERR_UNSUPPORTED;
  if ((M + 15) / 16 > 65535) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}

Plan make_plan(int B, int gamma, int d, int V, int dtype, int mode) {
  Plan p;
  p.M = B * (gamma + 1);
  p.P = (V + kBlockV - 1) / kBlockV + 2;   // record capacity per row (>= any grid used)
  p.nchunks = (V + kChunkV - 1) / kChunkV;
  const bool sample = mode == SPECDEC_SAMPLE;
  size_t off = align_up(sizeof(WsHeader));
  p.off_tickets = off;
  off = align_up(off + sizeof(unsigned long long) * kFixSlots);
  p.off_sel = off;
  off = align_up(off + sizeof(SelectedRow) * (size_t)B);
  p.off_counters = off;
  off = align_up(off + sizeof(int) * (size_t)B);
  p.off_pp = off;
  off = align_up(off + sizeof(PartialP) * (size_t)p.M * p.P);
  p.off_pq = off;
  if (sample) off = align_up(off + sizeof(PartialQ) * (size_t)B * gamma * p.P);
  p.off_z = off;
  if (sample) off = align_up(off + sizeof(float) * (size_t)p.M * V);
  p.off_chunks = off;
  if (sample) off = align_up(off + sizeof(float) * (size_t)B * p.nchunks);
  p.off_fix = off;
  if (dtype == SPECDEC_BF16) off = align_up(off + sizeof(float) * tc_fix_floats(p.M, V, d));
  p.total = off;
  return p;
}

int num_sms_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 0 || dev >= 64) return -1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = n;
  }
  return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] as a 2-D tensor map with a
// {64, box_rows} box and the 128-byte swizzle; out-of-range rows read 0.
bool encode_bf16_rows(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBlockK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same matrix as a 3-D tensor {64, rows, cols/64} whose slices of 64
// columns are the outer dimension, with a {64, box_rows, box_slices} box:
// one load brings box_slices adjacent 128-byte pieces of every row, stored
// slice-major as box_slices standard [box_rows x 128 B] swizzled tiles.
// Needs cols % 64 == 0.
// fp32 logits [rows, cols] as 32 x 32 tiles in the 128-byte swizzled layout
// (the row-owner epilogue's bulk stores). Needs cols % 4 == 0 and a 16-byte
// aligned base.
bool encode_f32_tiles(CUtensorMap* map, void* base, int rows, int cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_rows3d(CUtensorMap* map, const void* base, int rows, int cols, int box_rows,
                        int box_slices) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kBlockK, (cuuint64_t)rows,
                              (cuuint64_t)(cols / kBlockK)};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)kBlockK * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)box_rows, (cuuint32_t)box_slices};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One layer's K or V cache [B, Lmax, Hkv, 128] (bf16) as a 4-D tensor
// {128, Hkv, Lmax, B} with a {64, 1, 64, 1} box (64 keys x 64 dims) and the
// 128-byte swizzle; keys past Lmax read 0.
bool encode_kv_cache(CUtensorMap* map, const void* base, int B, int Lmax, int Hkv) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {128, (cuuint64_t)Hkv, (cuuint64_t)Lmax, (cuuint64_t)B};
  const cuuint64_t strides[3] = {256, (cuuint64_t)Hkv * 256, (cuuint64_t)Lmax * Hkv * 256};
  const cuuint32_t box[4] = {64, 1, 64, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The call count in the header that starts every workspace (its status
// word is the header's first field).
unsigned long long* header_calls(int* status) {
  return reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(status) +
                                               offsetof(WsHeader, calls));
}

struct Extras {
  float* logits_out = nullptr;
  float* lse_p = nullptr;
  float* lse_q = nullptr;
  float* p_x = nullptr;
  float* q_x = nullptr;
  int32_t* argmax_out = nullptr;
  cudaEvent_t ev0 = nullptr;
  cudaEvent_t ev1 = nullptr;
};

// The bf16 LM-head stage shared by the chain and tree steps: tensor maps,
// geometry and the launch. *records = partial records per row it writes.
int lmhead_stage_bf16(const void* hidden, const void* W, int M, int d, int V, const EpiParams& ep,
                      int* status, char* ws, size_t off_tickets, size_t off_fix,
                      unsigned long long epoch, int nsm, cudaStream_t stream, int* records) {
  const int max_clusters = tc_max_clusters(M, V, d);
  const TcGeometry g = tc_geometry(M, V, d, nsm, max_clusters);
  // A CTA of a pair loads its BT/K token rows of all kc slices of a stage.
  const int h_rows = g.BT / g.K;
  const int h_slices = g.kc;
  CUtensorMap tw, th;
  const bool ok = g.box3d ? (encode_bf16_rows3d(&tw, W, V, d, kBlockV, g.kc) &&
                             encode_bf16_rows3d(&th, hidden, M, d, h_rows, h_slices))
                          : (encode_bf16_rows(&tw, W, V, d, kBlockV) &&
                             encode_bf16_rows(&th, hidden, M, d, h_rows));
  if (!ok) return SPECDEC_ERR_CUDA;
  float* z = ep.zout;
  CUtensorMap tz;
  const bool ztma = g.rowown && z != nullptr && V % 4 == 0 && ((uintptr_t)z & 15u) == 0 &&
                    encode_f32_tiles(&tz, z, M, V);
  TcLaunch L;
  L.tmap_w = &tw;
  L.tmap_h = &th;
  L.tmap_z = ztma ? &tz : nullptr;
  L.M = M;
  L.V = V;
  L.d = d;
  L.gamma = ep.gamma;
  L.status = status;
  L.fix = reinterpret_cast<float*>(ws + off_fix);
  L.fix_tickets = reinterpret_cast<unsigned long long*>(ws + off_tickets);
  L.epoch = epoch;
  L.calls = header_calls(status);
  L.max_clusters = max_clusters;
  L.withhold_loads = 0;
  L.ep = ep;
  *records = g.records;
  return launch_lmhead_tc(L, nsm, stream) == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

int verify_impl(const void* hidden, const void* W, const int32_t* draft_tokens,
                const void* draft_logits, int B, int gamma, int d, int V, int dtype, float T,
                uint64_t seed, int mode, int32_t* out_tokens, int32_t* n_accepted, void* workspace,
                size_t workspace_bytes, void* stream_ptr, const Extras& ex) {
  int rc = check_shape(B, gamma, d, V, dtype, mode);
  if (rc != SPECDEC_OK) return rc;
  if (B == 0) return SPECDEC_OK;   // empty batch: nothing is read or written
  const bool sample = mode == SPECDEC_SAMPLE;
  if (!hidden || !W || !draft_tokens || !out_tokens || !n_accepted) return SPECDEC_ERR_INVALID_ARG;
  if (sample && (!draft_logits || !(T > 0.f) || !std::isfinite(T))) return SPECDEC_ERR_INVALID_ARG;
  if (dtype == SPECDEC_BF16 &&
      (((uintptr_t)hidden & 15u) != 0 || ((uintptr_t)W & 15u) != 0))
    return SPECDEC_ERR_INVALID_ARG;
  const Plan pl = make_plan(B, gamma, d, V, dtype, mode);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || workspace_bytes < pl.total)
    return SPECDEC_ERR_WORKSPACE;
  const int nsm = num_sms_current();
  if (nsm <= 0) return SPECDEC_ERR_CUDA;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  SelectedRow* sel = reinterpret_cast<SelectedRow*>(ws + pl.off_sel);
  int* counters = reinterpret_cast<int*>(ws + pl.off_counters);
  PartialP* pp = reinterpret_cast<PartialP*>(ws + pl.off_pp);
  PartialQ* pq = reinterpret_cast<PartialQ*>(ws + pl.off_pq);
  float* z = ex.logits_out ? ex.logits_out : (sample ? reinterpret_cast<float*>(ws + pl.off_z) : nullptr);
  float* chunk_sums = reinterpret_cast<float*>(ws + pl.off_chunks);
  const float c = sample ? kLog2e / T : kLog2e;

  // Nothing is cleared up front: the LM-head kernel resets the status word
  // after its dependency wait, and fix-up tickets are tagged with this call's
  // epoch, so every kernel of the step can launch as a programmatic dependent.
  const unsigned long long epoch = next_call_epoch();
  int P = (V + kBlockV - 1) / kBlockV;   // records per row written by the fp32 kernel

  EpiParams ep;
  ep.M = pl.M;
  ep.V = V;
  ep.gamma = gamma;
  ep.P = P;
  ep.c = c;
  ep.sample = sample ? 1 : 0;
  ep.want_argmax = (!sample || ex.argmax_out) ? 1 : 0;
  ep.zout = z;
  ep.dl = draft_logits;
  ep.pp = pp;
  ep.pq = pq;
  ep.run = nullptr;
  ep.q_in_epilogue = 1;
  // Many draft rows: the LM-head kernel's streamer warps reduce whole rows
  // (records of kQChunk columns) instead of the per-tile q-warps.
  const bool q_stream = sample && dtype == SPECDEC_BF16 && B * gamma > kQWarpMaxRows;
  ep.q_warps = q_stream ? 0 : 1;
  ep.q_stream = q_stream ? 1 : 0;
  ep.n_qrows = B * gamma;
  const int Pq = q_stream ? (V + kQChunk - 1) / kQChunk : 0;
  ep.Pq = Pq;
  ep.q_vec = (V % 8 == 0 && ((uintptr_t)draft_logits & 15u) == 0) ? 1 : 0;
  // Small batches draw in the same kernel as the acceptance test; its
  // tickets are cleared by the LM-head kernel.
  const bool fused = sample && fused_accept_sample(B, pl.nchunks);
  ep.counters = fused ? counters : nullptr;
  ep.n_counters = fused ? B : 0;

  if (ex.ev0 && cudaEventRecord(ex.ev0, stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (dtype == SPECDEC_BF16) {
    rc = lmhead_stage_bf16(hidden, W, pl.M, d, V, ep, status, ws, pl.off_tickets, pl.off_fix, epoch,
                           nsm, stream, &P);
    if (rc != SPECDEC_OK) return rc;
  } else if (launch_lmhead_f32(static_cast<const float*>(hidden), static_cast<const float*>(W), d,
                               ep, status, stream) != cudaSuccess) {
    return SPECDEC_ERR_CUDA;
  }
  if (ex.ev1 && cudaEventRecord(ex.ev1, stream) != cudaSuccess) return SPECDEC_ERR_CUDA;

  AcceptLaunch A;
  A.B = B;
  A.gamma = gamma;
  A.V = V;
  A.P = P;
  A.Pq = q_stream ? Pq : P;
  A.mode = mode;
  A.dl_bf16 = dtype == SPECDEC_BF16;
  A.c = c;
  A.seed = seed;
  A.pp = pp;
  A.pq = pq;
  A.z = z;
  A.dl = draft_logits;
  A.draft_tokens = draft_tokens;
  A.out_tokens = out_tokens;
  A.n_accepted = n_accepted;
  A.sel = sel;
  A.counters = counters;
  A.status = status;
  A.calls = header_calls(status);
  A.lse_p = ex.lse_p;
  A.lse_q = ex.lse_q;
  A.p_x = ex.p_x;
  A.q_x = ex.q_x;
  A.argmax_out = ex.argmax_out;
  A.tok_offset = 0;
  if (!fused && launch_accept(A, stream) != cudaSuccess) return SPECDEC_ERR_CUDA;

  if (sample) {
    SampleLaunch S;
    S.B = B;
    S.gamma = gamma;
    S.V = V;
    S.nchunks = pl.nchunks;
    S.dl_bf16 = dtype == SPECDEC_BF16;
    S.c = c;
    S.seed = seed;
    S.z = z;
    S.dl = draft_logits;
    S.sel = sel;
    S.chunk_sums = chunk_sums;
    S.counters = counters;
    S.out_tokens = out_tokens;
    const cudaError_t e = fused ? launch_accept_sample(A, S, stream) : launch_sample(S, stream);
    if (e != cudaSuccess) return SPECDEC_ERR_CUDA;
  }
  return SPECDEC_OK;
}

size_t host_staging_bytes(int B, int gamma, int d, int V, int dtype, int mode) {
  const size_t e = dtype == SPECDEC_BF16 ? 2 : 4;
  const size_t M = (size_t)B * (gamma + 1);
  size_t n = align_up(M * d * e);                                   // hidden
  n += align_up((size_t)B * gamma * 4);                             // draft tokens
  if (mode == SPECDEC_SAMPLE) n += align_up((size_t)B * gamma * V * e);   // draft logits
  n += align_up(M * 4) + align_up((size_t)B * 4);                   // outputs
  return n;
}

// ---------------------------------------------------------------- tree --

struct TreePlan {
  int M, P, Pq;
  size_t off_tickets, off_pp, off_pq, off_z, off_fix, total;
};

int check_tree_shape(int B, int N, int d, int V, int dtype, int mode) {
  if (dtype != SPECDEC_BF16 && dtype != SPECDEC_FP32) return SPECDEC_ERR_INVALID_ARG;
  if (mode != SPECDEC_SAMPLE && mode != SPECDEC_GREEDY) return SPECDEC_ERR_INVALID_ARG;
  if (dtype != SPECDEC_BF16) return SPECDEC_ERR_UNSUPPORTED;
  if (B < 0 || N < 1 || N > SPECDEC_MAX_TREE_NODES || d < 1 || d % 8 != 0 || V < 1 ||
      V > kMaxVocab)
    return SPECDEC_ERR_UNSUPPORTED;
  const long long M = (long long)B * N;
  if (M * (long long)V >= (1ll << 31)) return SPECDEC_ERR_UNSUPPORTED;
  if ((M + 15) / 16 > 65535) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}

TreePlan make_tree_plan(int B, int N, int d, int V, int mode) {
  TreePlan p;
  p.M = B * N;
  p.P = (V + kBlockV - 1) / kBlockV + 2;
  p.Pq = (V + kQChunk - 1) / kQChunk;
  const bool sample = mode == SPECDEC_SAMPLE;
  size_t off = align_up(sizeof(WsHeader));
  p.off_tickets = off;
  off = align_up(off + sizeof(unsigned long long) * kFixSlots);
  p.off_pp = off;
  off = align_up(off + sizeof(PartialP) * (size_t)p.M * p.P);
  p.off_pq = off;
  if (sample) off = align_up(off + sizeof(PartialQ) * (size_t)p.M * p.Pq);
  p.off_z = off;
  if (sample) off = align_up(off + sizeof(float) * (size_t)p.M * V);
  p.off_fix = off;
  off = align_up(off + sizeof(float) * tc_fix_floats(p.M, V, d));
  p.total = off;
  return p;
}

// ----------------------------------------------------------- attention --

struct AttnPlan {
  int n_splits, split_len;
  size_t off_m, off_l, off_o, total;
};

int check_attn_shape(int B, int n_new, int Hq, int Hkv, int D, int Lmax) {
  if (B < 0 || n_new < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || D != 128 || Lmax < n_new)
    return SPECDEC_ERR_UNSUPPORTED;
  if ((long long)n_new * (Hq / Hkv) > 64) return SPECDEC_ERR_UNSUPPORTED;
  if ((long long)B * Lmax * Hkv * D >= (1ll << 40)) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}

// Splits of the key range. The split kernel keeps two CTAs resident per SM
// (one when the query rows need four row tiles), so a 152-SM part holds
// `slots` CTAs at once. Once the (sequence, KV head) pairs alone fill that,
// no split. Otherwise the splits stay within one wave (a small last wave
// would run with too few CTAs to keep HBM busy) and aim at 1.5 CTAs per SM,
// at least 256 keys each (fixed targets, so the workspace size does not
// depend on the device).
AttnPlan make_attn_plan(int B, int n_new, int Hq, int Hkv, int Lmax) {
  AttnPlan p;
  const long long pairs = (long long)B * Hkv;
  const int n_mt = (n_new * (Hq / Hkv) + 15) / 16;
  const long long slots = 152ll * (n_mt <= 3 ? 2 : 1);
  const long long target = 228;
  long long want = 1;
  if (pairs > 0 && pairs < slots) {
    want = (target + pairs - 1) / pairs;
    if (want > slots / pairs) want = slots / pairs;
    const long long most = (Lmax + 255) / 256;
    if (want > most) want = most;
    if (want < 1) want = 1;
  }
  int split = (int)((Lmax + want - 1) / want);
  split = (split + 63) / 64 * 64;
  p.split_len = split;
  p.n_splits = (Lmax + split - 1) / split;
  size_t off = align_up(sizeof(WsHeader));
  const size_t rows = (size_t)B * Hkv * p.n_splits * 64;
  p.off_m = off;
  p.off_l = off;
  p.off_o = off;
  if (p.n_splits > 1) {
    p.off_l = align_up(off + sizeof(float) * rows);
    p.off_o = align_up(p.off_l + sizeof(float) * rows);
    off = align_up(p.off_o + sizeof(float) * rows * 128);
  }
  p.total = off;
  return p;
}

// -------------------------------------------------------- cluster head --

struct ClusterPlan {
  int max_members, sort_n;
  size_t off_y, off_offs, off_z, off_ids, total;
};

int check_cluster_shape(int M, int d, int V, int n_c, int top_k, int max_cluster) {
  if (M < 0 || M > 64 || d < 8 || d % 8 != 0 || d > SPECDEC_CLUSTER_MAX_D || V < 1 || n_c < 1 ||
      top_k < 1 || top_k > SPECDEC_CLUSTER_MAX_TOP_K || top_k > n_c || max_cluster < 1 ||
      (long long)top_k * max_cluster > SPECDEC_CLUSTER_MAX_MEMBERS)
    return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}

ClusterPlan make_cluster_plan(int M, int n_c, int top_k, int max_cluster) {
  ClusterPlan p;
  p.max_members = top_k * max_cluster;
  p.sort_n = 1;
  while (p.sort_n < p.max_members) p.sort_n <<= 1;
  size_t off = align_up(sizeof(WsHeader));
  p.off_y = off;
  off = align_up(off + sizeof(float) * (size_t)M * n_c);
  p.off_offs = off;
  off = align_up(off + sizeof(int) * (size_t)M * (top_k + 1));
  p.off_z = off;
  off = align_up(off + sizeof(float) * (size_t)M * p.max_members);
  p.off_ids = off;
  off = align_up(off + sizeof(int) * (size_t)M * p.max_members);
  p.total = off;
  return p;
}

}  // namespace

namespace specdec {
unsigned long long next_call_epoch() {
  // Starts from the clock so that tags left in reused memory by another
  // process are unlikely to match; then strictly increasing.
  static std::atomic<unsigned long long> counter{
      (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() |
      (1ull << 63)};
  return counter.fetch_add(1, std::memory_order_relaxed);
}
}  // namespace specdec

extern "C" {

size_t specdec_verify_workspace_size(int B, int gamma, int d, int V, int dtype, int mode) {
  if (check_shape(B, gamma, d, V, dtype, mode) != SPECDEC_OK) return 0;
  return make_plan(B, gamma, d, V, dtype, mode).total;
}

int specdec_verify(const void* hidden, const void* W_lm, const int32_t* draft_tokens,
                   const void* draft_logits, int B, int gamma, int d, int V, int dtype,
                   float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                   int32_t* n_accepted, void* workspace, size_t workspace_bytes, void* stream) {
  return verify_impl(hidden, W_lm, draft_tokens, draft_logits, B, gamma, d, V, dtype, temperature,
                     seed, mode, out_tokens, n_accepted, workspace, workspace_bytes, stream,
                     Extras());
}

int specdec_verify_debug(const void* hidden, const void* W_lm, const int32_t* draft_tokens,
                         const void* draft_logits, int B, int gamma, int d, int V, int dtype,
                         float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                         int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                         void* stream, float* logits_out, float* lse_p, float* lse_q, float* p_x,
                         float* q_x, int32_t* argmax_out) {
  Extras ex;
  ex.logits_out = logits_out;
  ex.lse_p = lse_p;
  ex.lse_q = lse_q;
  ex.p_x = p_x;
  ex.q_x = q_x;
  ex.argmax_out = argmax_out;
  return verify_impl(hidden, W_lm, draft_tokens, draft_logits, B, gamma, d, V, dtype, temperature,
                     seed, mode, out_tokens, n_accepted, workspace, workspace_bytes, stream, ex);
}

int specdec_verify_timed(const void* hidden, const void* W_lm, const int32_t* draft_tokens,
                         const void* draft_logits, int B, int gamma, int d, int V, int dtype,
                         float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                         int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                         void* stream, void* lmhead_start_event, void* lmhead_end_event) {
  Extras ex;
  ex.ev0 = static_cast<cudaEvent_t>(lmhead_start_event);
  ex.ev1 = static_cast<cudaEvent_t>(lmhead_end_event);
  return verify_impl(hidden, W_lm, draft_tokens, draft_logits, B, gamma, d, V, dtype, temperature,
                     seed, mode, out_tokens, n_accepted, workspace, workspace_bytes, stream, ex);
}

size_t specdec_verify_host_workspace_size(int B, int gamma, int d, int V, int dtype, int mode) {
  const size_t base = specdec_verify_workspace_size(B, gamma, d, V, dtype, mode);
  if (base == 0) return 0;
  return base + host_staging_bytes(B, gamma, d, V, dtype, mode);
}

// Device address of a pinned host buffer that is mapped into the GPU's
// address space, or nullptr (pageable memory, or not mapped).
void* mapped_device_ptr(const void* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();   // not a pointer the runtime knows: the copy path handles it
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
  return a.devicePointer;
}

// One staging segment, in the widest units both ends are aligned to.
void host_seg(HostSeg& g, const void* src, void* dst, size_t bytes) {
  const uintptr_t a = (uintptr_t)src | (uintptr_t)dst;
  g.src = src;
  g.dst = dst;
  g.bytes = (long long)bytes;
  g.unit = a % 16 == 0 ? 16 : a % 4 == 0 ? 4 : 1;
}

int specdec_verify_host(const void* hidden_host, const void* W_lm, const int32_t* draft_tokens_host,
                        const void* draft_logits_host, int B, int gamma, int d, int V, int dtype,
                        float temperature, uint64_t seed, int mode, int32_t* out_tokens_host,
                        int32_t* n_accepted_host, void* workspace, size_t workspace_bytes,
                        void* stream_ptr) {
  int rc = check_shape(B, gamma, d, V, dtype, mode);
  if (rc != SPECDEC_OK) return rc;
  if (B == 0) return SPECDEC_OK;
  const bool sample = mode == SPECDEC_SAMPLE;
  if (!hidden_host || !W_lm || !draft_tokens_host || !out_tokens_host || !n_accepted_host)
    return SPECDEC_ERR_INVALID_ARG;
  if (sample && !draft_logits_host) return SPECDEC_ERR_INVALID_ARG;
  const size_t base = specdec_verify_workspace_size(B, gamma, d, V, dtype, mode);
  const size_t need = base + host_staging_bytes(B, gamma, d, V, dtype, mode);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || workspace_bytes < need)
    return SPECDEC_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const size_t e = dtype == SPECDEC_BF16 ? 2 : 4;
  const size_t M = (size_t)B * (gamma + 1);
  char* p = static_cast<char*>(workspace) + base;
  void* d_hidden = p;
  p += align_up(M * d * e);
  int32_t* d_tokens = reinterpret_cast<int32_t*>(p);
  p += align_up((size_t)B * gamma * 4);
  void* d_logits = nullptr;
  if (sample) {
    d_logits = p;
    p += align_up((size_t)B * gamma * V * e);
  }
  int32_t* d_out = reinterpret_cast<int32_t*>(p);
  p += align_up(M * 4);
  int32_t* d_nacc = reinterpret_cast<int32_t*>(p);

  // Mapped pinned host buffers: the GPU gathers the inputs and writes the
  // results itself (one kernel each way). Otherwise copy-engine transfers.
  void* m_hidden = mapped_device_ptr(hidden_host);
  void* m_tokens = mapped_device_ptr(draft_tokens_host);
  void* m_logits = sample ? mapped_device_ptr(draft_logits_host) : nullptr;
  void* m_out = mapped_device_ptr(out_tokens_host);
  void* m_nacc = mapped_device_ptr(n_accepted_host);
  StageInLaunch S;
  S.nseg = sample ? 3 : 2;
  const bool mapped = m_hidden && m_tokens && (!sample || m_logits) && m_out && m_nacc &&
                     ((uintptr_t)m_out | (uintptr_t)m_nacc) % 4 == 0;
  if (mapped) {
    host_seg(S.seg[0], m_hidden, d_hidden, M * d * e);
    host_seg(S.seg[1], m_tokens, d_tokens, (size_t)B * gamma * 4);
    if (sample) host_seg(S.seg[2], m_logits, d_logits, (size_t)B * gamma * V * e);
    if (launch_stage_in(S, num_sms_current(), stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  } else {
    if (cudaMemcpyAsync(d_hidden, hidden_host, M * d * e, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess ||
        cudaMemcpyAsync(d_tokens, draft_tokens_host, (size_t)B * gamma * 4,
                        cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return SPECDEC_ERR_CUDA;
    if (sample && cudaMemcpyAsync(d_logits, draft_logits_host, (size_t)B * gamma * V * e,
                                  cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return SPECDEC_ERR_CUDA;
  }
  // Mapped outputs: the accept and sample kernels write the results straight
  // into the caller's host buffers (they only ever store to them).
  if (mapped) {
    d_out = static_cast<int32_t*>(m_out);
    d_nacc = static_cast<int32_t*>(m_nacc);
  }
  rc = verify_impl(d_hidden, W_lm, d_tokens, d_logits, B, gamma, d, V, dtype, temperature, seed,
                   mode, d_out, d_nacc, workspace, base, stream_ptr, Extras());
  if (rc != SPECDEC_OK) return rc;
  if (!mapped &&
      (cudaMemcpyAsync(out_tokens_host, d_out, M * 4, cudaMemcpyDeviceToHost, stream) !=
           cudaSuccess ||
       cudaMemcpyAsync(n_accepted_host, d_nacc, (size_t)B * 4, cudaMemcpyDeviceToHost, stream) !=
           cudaSuccess))
    return SPECDEC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  return SPECDEC_OK;
}

int specdec_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream_ptr,
                                  int32_t* status) {
  // A small sampling-free shape: M = 5 rows, V = 256, d = 64.
  const int B = 1, gamma = 4, d = 64, V = 256;
  if (!workspace || !status || ((uintptr_t)workspace % kAlign) != 0) return SPECDEC_ERR_INVALID_ARG;
  const Plan pl = make_plan(B, gamma, d, V, SPECDEC_BF16, SPECDEC_GREEDY);
  if (workspace_bytes < pl.total) return SPECDEC_ERR_WORKSPACE;
  const int nsm = num_sms_current();
  if (nsm <= 0) return SPECDEC_ERR_CUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  const TcGeometry g = tc_geometry(pl.M, V, d, nsm, 0);
  // The tensor maps point at the workspace; no load is ever issued through them.
  CUtensorMap tw, th;
  if (!encode_bf16_rows3d(&tw, ws, V, d, kBlockV, g.kc) ||
      !encode_bf16_rows3d(&th, ws, pl.M, d, g.BT, g.kc))
    return SPECDEC_ERR_CUDA;
  EpiParams ep;
  ep.M = pl.M;
  ep.V = V;
  ep.gamma = gamma;
  ep.P = pl.P;
  ep.c = kLog2e;
  ep.sample = 0;
  ep.want_argmax = 0;
  ep.zout = nullptr;
  ep.dl = nullptr;
  ep.pp = reinterpret_cast<PartialP*>(ws + pl.off_pp);
  ep.pq = reinterpret_cast<PartialQ*>(ws + pl.off_pq);
  ep.run = nullptr;
  ep.q_in_epilogue = 0;
  ep.q_warps = 0;
  ep.q_stream = 0;
  ep.n_qrows = 0;
  ep.Pq = 0;
  ep.q_vec = 0;
  ep.counters = nullptr;
  ep.n_counters = 0;
  TcLaunch L;
  L.tmap_w = &tw;
  L.tmap_h = &th;
  L.tmap_z = nullptr;
  L.M = pl.M;
  L.V = V;
  L.d = d;
  L.gamma = gamma;
  L.status = reinterpret_cast<int*>(ws);
  L.fix = reinterpret_cast<float*>(ws + pl.off_fix);
  L.fix_tickets = reinterpret_cast<unsigned long long*>(ws + pl.off_tickets);
  L.epoch = next_call_epoch();
  L.calls = header_calls(L.status);
  L.max_clusters = 0;
  L.withhold_loads = 1;
  L.ep = ep;
  if (launch_lmhead_tc(L, nsm, stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (cudaMemcpy(status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  return SPECDEC_OK;
}

size_t specdec_verify_tree_workspace_size(int B, int n_nodes, int d, int V, int dtype, int mode) {
  if (check_tree_shape(B, n_nodes, d, V, dtype, mode) != SPECDEC_OK) return 0;
  return make_tree_plan(B, n_nodes, d, V, mode).total;
}

int specdec_verify_tree_timed(const void* hidden, const void* W_lm, const int32_t* parent,
                              const int32_t* node_tokens, const void* draft_logits, int B,
                              int n_nodes, int d, int V, int dtype, float temperature,
                              uint64_t seed, int mode, int32_t* out_tokens, int32_t* out_nodes,
                              int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                              void* stream_ptr, void* lmhead_start_event,
                              void* lmhead_end_event) {
  int rc = check_tree_shape(B, n_nodes, d, V, dtype, mode);
  if (rc != SPECDEC_OK) return rc;
  const int N = n_nodes;
  if (!parent) return SPECDEC_ERR_INVALID_ARG;
  // The topology: parent[0] = -1, parent[n] an earlier node; children are
  // linked in increasing index.
  TreeLaunch T;
  if (parent[0] != -1) return SPECDEC_ERR_INVALID_ARG;
  for (int n = 0; n < SPECDEC_MAX_TREE_NODES; ++n)
    T.first_child[n] = T.next_sibling[n] = T.parent[n] = -1;
  for (int n = N - 1; n >= 1; --n) {
    const int pa = parent[n];
    if (pa < 0 || pa >= n) return SPECDEC_ERR_INVALID_ARG;
    T.parent[n] = (int16_t)pa;
    T.next_sibling[n] = T.first_child[pa];
    T.first_child[pa] = (int16_t)n;
  }
  if (B == 0) return SPECDEC_OK;
  const bool sample = mode == SPECDEC_SAMPLE;
  if (!hidden || !W_lm || !node_tokens || !out_tokens || !out_nodes || !n_accepted)
    return SPECDEC_ERR_INVALID_ARG;
  if (sample && (!draft_logits || !(temperature > 0.f) || !std::isfinite(temperature)))
    return SPECDEC_ERR_INVALID_ARG;
  if (((uintptr_t)hidden & 15u) != 0 || ((uintptr_t)W_lm & 15u) != 0)
    return SPECDEC_ERR_INVALID_ARG;
  const TreePlan pl = make_tree_plan(B, N, d, V, mode);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || workspace_bytes < pl.total)
    return SPECDEC_ERR_WORKSPACE;
  const int nsm = num_sms_current();
  if (nsm <= 0) return SPECDEC_ERR_CUDA;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  PartialP* pp = reinterpret_cast<PartialP*>(ws + pl.off_pp);
  PartialQ* pq = reinterpret_cast<PartialQ*>(ws + pl.off_pq);
  float* z = sample ? reinterpret_cast<float*>(ws + pl.off_z) : nullptr;
  const float c = sample ? kLog2e / temperature : kLog2e;

  EpiParams ep;
  ep.M = pl.M;
  ep.V = V;
  ep.gamma = 1;               // unused: no per-tile q-warps for trees
  ep.P = 0;
  ep.c = c;
  ep.sample = sample ? 1 : 0;
  ep.want_argmax = sample ? 0 : 1;
  ep.zout = z;
  ep.dl = draft_logits;
  ep.pp = pp;
  ep.pq = pq;
  ep.run = nullptr;
  ep.q_in_epilogue = 0;
  ep.q_warps = 0;
  // Every node's draft row is reduced by the LM-head kernel's streamer warps.
  ep.q_stream = sample ? 1 : 0;
  ep.n_qrows = pl.M;
  ep.Pq = pl.Pq;
  ep.q_vec = (V % 8 == 0 && ((uintptr_t)draft_logits & 15u) == 0) ? 1 : 0;
  ep.counters = nullptr;
  ep.n_counters = 0;
  int P = 0;
  cudaEvent_t ev0 = static_cast<cudaEvent_t>(lmhead_start_event);
  cudaEvent_t ev1 = static_cast<cudaEvent_t>(lmhead_end_event);
  if (ev0 && cudaEventRecord(ev0, stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  rc = lmhead_stage_bf16(hidden, W_lm, pl.M, d, V, ep, status, ws, pl.off_tickets, pl.off_fix,
                         next_call_epoch(), nsm, stream, &P);
  if (rc != SPECDEC_OK) return rc;
  if (ev1 && cudaEventRecord(ev1, stream) != cudaSuccess) return SPECDEC_ERR_CUDA;

  T.B = B;
  T.N = N;
  T.V = V;
  T.P = P;
  T.Pq = pl.Pq;
  T.mode = mode;
  T.vec = (V % 4 == 0 && ((uintptr_t)draft_logits & 7u) == 0) ? 1 : 0;
  T.c = c;
  T.seed = seed;
  T.pp = pp;
  T.pq = pq;
  T.z = z;
  T.dl = static_cast<const __nv_bfloat16*>(draft_logits);
  T.tok = node_tokens;
  T.out_tokens = out_tokens;
  T.out_nodes = out_nodes;
  T.n_accepted = n_accepted;
  T.status = status;
  T.calls = header_calls(status);
  return launch_tree_walk(T, stream) == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

int specdec_verify_tree(const void* hidden, const void* W_lm, const int32_t* parent,
                        const int32_t* node_tokens, const void* draft_logits, int B, int n_nodes,
                        int d, int V, int dtype, float temperature, uint64_t seed, int mode,
                        int32_t* out_tokens, int32_t* out_nodes, int32_t* n_accepted,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return specdec_verify_tree_timed(hidden, W_lm, parent, node_tokens, draft_logits, B, n_nodes, d,
                                   V, dtype, temperature, seed, mode, out_tokens, out_nodes,
                                   n_accepted, workspace, workspace_bytes, stream, nullptr,
                                   nullptr);
}

size_t specdec_verify_attention_workspace_size(int B, int n_new, int Hq, int Hkv, int D,
                                               int Lmax) {
  if (check_attn_shape(B, n_new, Hq, Hkv, D, Lmax) != SPECDEC_OK) return 0;
  return make_attn_plan(B, n_new, Hq, Hkv, Lmax).total;
}

int specdec_verify_attention(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* seq_lens, int B, int n_new, int Hq, int Hkv, int D,
                             int Lmax, float scale, float* out, void* workspace,
                             size_t workspace_bytes, void* stream_ptr) {
  int rc = check_attn_shape(B, n_new, Hq, Hkv, D, Lmax);
  if (rc != SPECDEC_OK) return rc;
  if (B == 0) return SPECDEC_OK;
  if (!q || !k_cache || !v_cache || !seq_lens || !out) return SPECDEC_ERR_INVALID_ARG;
  if ((((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)out) & 15u) != 0)
    return SPECDEC_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return SPECDEC_ERR_INVALID_ARG;
  const AttnPlan pl = make_attn_plan(B, n_new, Hq, Hkv, Lmax);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || workspace_bytes < pl.total)
    return SPECDEC_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  AttnLaunch A;
  A.B = B;
  A.n_new = n_new;
  A.Hq = Hq;
  A.Hkv = Hkv;
  A.Lmax = Lmax;
  A.n_splits = pl.n_splits;
  A.split_len = pl.split_len;
  A.n_stages = attn_n_stages(B, n_new, Hq, Hkv);
  A.scale_log2 = (scale > 0.f ? scale : 1.f / std::sqrt((float)D)) * kLog2e;
  A.q = static_cast<const __nv_bfloat16*>(q);
  A.k = static_cast<const __nv_bfloat16*>(k_cache);
  A.v = static_cast<const __nv_bfloat16*>(v_cache);
  A.seq_lens = seq_lens;
  A.out = out;
  A.part_m = reinterpret_cast<float*>(ws + pl.off_m);
  A.part_l = reinterpret_cast<float*>(ws + pl.off_l);
  A.part_o = reinterpret_cast<float*>(ws + pl.off_o);
  A.status = reinterpret_cast<int*>(ws);
  CUtensorMap tk, tv;
  if (!encode_kv_cache(&tk, k_cache, B, Lmax, Hkv) || !encode_kv_cache(&tv, v_cache, B, Lmax, Hkv))
    return SPECDEC_ERR_CUDA;
  return launch_attention(A, tk, tv, stream) == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

size_t specdec_cluster_head_workspace_size(int M, int n_c, int top_k, int max_cluster) {
  if (check_cluster_shape(M, 8, 1, n_c, top_k, max_cluster) != SPECDEC_OK) return 0;
  return make_cluster_plan(M, n_c, top_k, max_cluster).total;
}

int specdec_cluster_head(const void* hidden, const void* cluster_emb, const void* W_sorted,
                         const int32_t* starts, const int32_t* token_of_row, int M, int d, int V,
                         int n_c, int top_k, int max_cluster, float temperature, uint64_t seed,
                         int position, int mode, int32_t* out_tokens, int32_t* out_clusters,
                         float* logits_out, void* workspace, size_t workspace_bytes,
                         void* stream_ptr) {
  if (mode != SPECDEC_SAMPLE && mode != SPECDEC_GREEDY) return SPECDEC_ERR_INVALID_ARG;
  int rc = check_cluster_shape(M, d, V, n_c, top_k, max_cluster);
  if (rc != SPECDEC_OK) return rc;
  if (M == 0) return SPECDEC_OK;
  if (!hidden || !cluster_emb || !W_sorted || !starts || !token_of_row || !out_tokens ||
      !out_clusters)
    return SPECDEC_ERR_INVALID_ARG;
  if ((((uintptr_t)hidden | (uintptr_t)cluster_emb | (uintptr_t)W_sorted) & 15u) != 0)
    return SPECDEC_ERR_INVALID_ARG;
  const bool sample = mode == SPECDEC_SAMPLE;
  if (sample && (!(temperature > 0.f) || !std::isfinite(temperature))) return SPECDEC_ERR_INVALID_ARG;
  const ClusterPlan pl = make_cluster_plan(M, n_c, top_k, max_cluster);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || workspace_bytes < pl.total)
    return SPECDEC_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  ClusterLaunch L;
  L.M = M;
  L.d = d;
  L.V = V;
  L.n_c = n_c;
  L.top_k = top_k;
  L.max_cluster = max_cluster;
  L.max_members = pl.max_members;
  L.sort_n = pl.sort_n;
  L.sample = sample ? 1 : 0;
  L.position = position;
  L.c = sample ? kLog2e / temperature : kLog2e;
  L.seed = seed;
  L.h = static_cast<const __nv_bfloat16*>(hidden);
  L.E = static_cast<const __nv_bfloat16*>(cluster_emb);
  L.W = static_cast<const __nv_bfloat16*>(W_sorted);
  L.starts = starts;
  L.token_of_row = token_of_row;
  L.y = reinterpret_cast<float*>(ws + pl.off_y);
  L.offs = reinterpret_cast<int*>(ws + pl.off_offs);
  L.z = reinterpret_cast<float*>(ws + pl.off_z);
  L.ids = reinterpret_cast<int*>(ws + pl.off_ids);
  L.clusters = out_clusters;
  L.tokens = out_tokens;
  L.logits_out = logits_out;
  L.status = reinterpret_cast<int*>(ws);
  return launch_cluster_head(L, stream) == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

int specdec_read_status(const void* workspace, void* stream, int32_t* status) {
  if (!workspace || !status) return SPECDEC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (cudaMemcpy(status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  return SPECDEC_OK;
}

int specdec_philox_uniforms(uint64_t seed, int B, int n_pos, int purpose, float* out,
                            void* stream) {
  if (!out || B < 0 || n_pos < 0 || (purpose != 0 && purpose != 1)) return SPECDEC_ERR_INVALID_ARG;
  if ((long long)B * n_pos >= (1ll << 31)) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0 || n_pos == 0) return SPECDEC_OK;
  return launch_philox_uniforms(seed, B, n_pos, purpose, out, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SPECDEC_OK
             : SPECDEC_ERR_CUDA;
}

// ------------------------------------------------ vocabulary-parallel --

size_t specdec_shard_record_bytes(int B, int gamma) {
  if (B < 0 || gamma < 1 || gamma > SPECDEC_MAX_GAMMA) return 0;
  return shard_record_bytes(B, gamma);
}

size_t specdec_shard_workspace_size(int B, int gamma, int d, int V_shard, int mode) {
  if (check_shape(B, gamma, d, V_shard, SPECDEC_BF16, mode) != SPECDEC_OK) return 0;
  const Plan pl = make_plan(B, gamma, d, V_shard, SPECDEC_BF16, mode);
  return pl.total + align_up(sizeof(float) * (size_t)B * pl.nchunks);
}

namespace {
// Arguments every call of the vocabulary-parallel step shares.
int shard_check(int B, int gamma, int d, int V_shard, int v_begin, int V, float T, int mode,
                const void* workspace, size_t workspace_bytes, Plan* pl) {
  int rc = check_shape(B, gamma, d, V_shard, SPECDEC_BF16, mode);
  if (rc != SPECDEC_OK) return rc;
  if (V < 1 || V > kMaxVocab || v_begin < 0 || (long long)v_begin + V_shard > V)
    return SPECDEC_ERR_UNSUPPORTED;
  if (mode == SPECDEC_SAMPLE && (!(T > 0.f) || !std::isfinite(T))) return SPECDEC_ERR_INVALID_ARG;
  *pl = make_plan(B, gamma, d, V_shard, SPECDEC_BF16, mode);
  const size_t need = pl->total + align_up(sizeof(float) * (size_t)B * pl->nchunks);
  if (!workspace || ((uintptr_t)workspace % kAlign) != 0 || workspace_bytes < need)
    return SPECDEC_ERR_WORKSPACE;
  return SPECDEC_OK;
}

SampleLaunch shard_sample_launch(const Plan& pl, char* ws, const void* dl_shard, int B, int gamma,
                                 int V_shard, float T, uint64_t seed, int32_t* out_tokens) {
  SampleLaunch S;
  S.B = B;
  S.gamma = gamma;
  S.V = V_shard;
  S.nchunks = pl.nchunks;
  S.dl_bf16 = 1;
  S.vec = 0;
  S.prefetch = 0;
  S.c = kLog2e / T;
  S.seed = seed;
  S.z = reinterpret_cast<float*>(ws + pl.off_z);
  S.dl = dl_shard;
  S.sel = reinterpret_cast<SelectedRow*>(ws + pl.off_sel);
  S.chunk_sums = reinterpret_cast<float*>(ws + pl.off_chunks);
  S.counters = reinterpret_cast<int*>(ws + pl.off_counters);
  S.out_tokens = out_tokens;
  return S;
}
}  // namespace

int specdec_shard_score(const void* hidden, const void* W_shard, const int32_t* draft_tokens,
                        const void* draft_logits_shard, int B, int gamma, int d, int V_shard,
                        int v_begin, int V, float temperature, int mode, void* records,
                        void* workspace, size_t workspace_bytes, void* stream_ptr) {
  Plan pl;
  int rc = shard_check(B, gamma, d, V_shard, v_begin, V, temperature, mode, workspace,
                       workspace_bytes, &pl);
  if (rc != SPECDEC_OK) return rc;
  if (B == 0) return SPECDEC_OK;
  const bool sample = mode == SPECDEC_SAMPLE;
  if (!hidden || !W_shard || !draft_tokens || !records || (sample && !draft_logits_shard))
    return SPECDEC_ERR_INVALID_ARG;
  if ((((uintptr_t)hidden | (uintptr_t)W_shard) & 15u) != 0 || ((uintptr_t)records & 15u) != 0)
    return SPECDEC_ERR_INVALID_ARG;
  const int nsm = num_sms_current();
  if (nsm <= 0) return SPECDEC_ERR_CUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  PartialP* pp = reinterpret_cast<PartialP*>(ws + pl.off_pp);
  PartialQ* pq = reinterpret_cast<PartialQ*>(ws + pl.off_pq);
  float* z = sample ? reinterpret_cast<float*>(ws + pl.off_z) : nullptr;
  const float c = sample ? kLog2e / temperature : kLog2e;
  EpiParams ep;
  ep.M = pl.M;
  ep.V = V_shard;
  ep.gamma = gamma;
  ep.P = 0;
  ep.c = c;
  ep.sample = sample ? 1 : 0;
  ep.want_argmax = sample ? 0 : 1;
  ep.zout = z;
  ep.dl = draft_logits_shard;
  ep.pp = pp;
  ep.pq = pq;
  ep.run = nullptr;
  ep.q_in_epilogue = 1;
  const bool q_stream = sample && B * gamma > kQWarpMaxRows;
  ep.q_warps = q_stream ? 0 : 1;
  ep.q_stream = q_stream ? 1 : 0;
  ep.n_qrows = B * gamma;
  const int Pq = q_stream ? (V_shard + kQChunk - 1) / kQChunk : 0;
  ep.Pq = Pq;
  ep.q_vec = (V_shard % 8 == 0 && ((uintptr_t)draft_logits_shard & 15u) == 0) ? 1 : 0;
  // the chunk tickets of the fused accept-and-sums kernel
  ep.counters = sample ? reinterpret_cast<int*>(ws + pl.off_counters) : nullptr;
  ep.n_counters = sample ? B : 0;
  int P = 0;
  rc = lmhead_stage_bf16(hidden, W_shard, pl.M, d, V_shard, ep, status, ws, pl.off_tickets,
                         pl.off_fix, next_call_epoch(), nsm, stream, &P);
  if (rc != SPECDEC_OK) return rc;
  AcceptLaunch A;
  A.B = B;
  A.gamma = gamma;
  A.V = V_shard;
  A.P = P;
  A.Pq = q_stream ? Pq : P;
  A.mode = mode;
  A.dl_bf16 = 1;
  A.c = c;
  A.seed = 0;
  A.pp = pp;
  A.pq = pq;
  A.z = z;
  A.dl = draft_logits_shard;
  A.draft_tokens = draft_tokens;
  A.out_tokens = nullptr;
  A.n_accepted = nullptr;
  A.sel = nullptr;
  A.counters = nullptr;
  A.status = status;
  A.calls = header_calls(status);
  A.lse_p = A.lse_q = A.p_x = A.q_x = nullptr;
  A.argmax_out = nullptr;
  A.tok_offset = v_begin;
  return launch_shard_fold(A, records, stream) == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

int specdec_shard_accept(const void* all_records, int n_shards, const int32_t* draft_tokens,
                         const void* draft_logits_shard, int B, int gamma, int d, int V_shard,
                         int v_begin, int V, float temperature, uint64_t seed, int mode,
                         int32_t* out_tokens, int32_t* n_accepted, float* shard_sums,
                         void* workspace, size_t workspace_bytes, void* stream_ptr) {
  Plan pl;
  int rc = shard_check(B, gamma, d, V_shard, v_begin, V, temperature, mode, workspace,
                       workspace_bytes, &pl);
  if (rc != SPECDEC_OK) return rc;
  if (B == 0) return SPECDEC_OK;
  const bool sample = mode == SPECDEC_SAMPLE;
  if (!all_records || n_shards < 1 || n_shards > SPECDEC_MAX_SHARDS || !draft_tokens ||
      !out_tokens || !n_accepted || (sample && (!draft_logits_shard || !shard_sums)))
    return SPECDEC_ERR_INVALID_ARG;
  if (((uintptr_t)all_records & 15u) != 0 || ((uintptr_t)shard_sums & 7u) != 0)
    return SPECDEC_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  const float c = sample ? kLog2e / temperature : kLog2e;
  AcceptLaunch A;
  A.B = B;
  A.gamma = gamma;
  A.V = V;
  A.P = 0;
  A.Pq = 0;
  A.mode = mode;
  A.dl_bf16 = 1;
  A.c = c;
  A.seed = seed;
  A.pp = nullptr;
  A.pq = nullptr;
  A.z = nullptr;
  A.dl = nullptr;
  A.draft_tokens = draft_tokens;
  A.out_tokens = out_tokens;
  A.n_accepted = n_accepted;
  A.sel = reinterpret_cast<SelectedRow*>(ws + pl.off_sel);
  A.counters = reinterpret_cast<int*>(ws + pl.off_counters);
  A.status = status;
  A.calls = header_calls(status);
  A.lse_p = A.lse_q = A.p_x = A.q_x = nullptr;
  A.argmax_out = nullptr;
  A.tok_offset = 0;
  const size_t rb = shard_record_bytes(B, gamma);
  float* cs_p = reinterpret_cast<float*>(ws + pl.total);
  if (sample && shard_fused_accept_sums(B, pl.nchunks)) {
    const SampleLaunch S = shard_sample_launch(pl, ws, draft_logits_shard, B, gamma, V_shard,
                                               temperature, seed, out_tokens);
    return launch_shard_accept_sums(A, S, all_records, rb, n_shards, cs_p,
                                    reinterpret_cast<float2*>(shard_sums), stream) == cudaSuccess
               ? SPECDEC_OK
               : SPECDEC_ERR_CUDA;
  }
  if (launch_shard_accept(A, all_records, rb, n_shards, stream) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  if (!sample) return SPECDEC_OK;
  const SampleLaunch S = shard_sample_launch(pl, ws, draft_logits_shard, B, gamma, V_shard,
                                             temperature, seed, out_tokens);
  return launch_shard_sums(S, cs_p, reinterpret_cast<float2*>(shard_sums), stream) == cudaSuccess
             ? SPECDEC_OK
             : SPECDEC_ERR_CUDA;
}

int specdec_shard_draw(const float* all_shard_sums, int n_shards, int shard,
                       const void* draft_logits_shard, int B, int gamma, int d, int V_shard,
                       int v_begin, int V, float temperature, uint64_t seed, int mode,
                       int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                       void* stream_ptr) {
  Plan pl;
  int rc = shard_check(B, gamma, d, V_shard, v_begin, V, temperature, mode, workspace,
                       workspace_bytes, &pl);
  if (rc != SPECDEC_OK) return rc;
  if (B == 0 || mode == SPECDEC_GREEDY) return SPECDEC_OK;
  if (!all_shard_sums || n_shards < 1 || n_shards > SPECDEC_MAX_SHARDS || shard < 0 ||
      shard >= n_shards || !draft_logits_shard || !out_tokens ||
      ((uintptr_t)all_shard_sums & 7u) != 0)
    return SPECDEC_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  const SampleLaunch S = shard_sample_launch(pl, ws, draft_logits_shard, B, gamma, V_shard,
                                             temperature, seed, out_tokens);
  const float* cs_p = reinterpret_cast<const float*>(ws + pl.total);
  return launch_shard_draw(S, cs_p, reinterpret_cast<const float2*>(all_shard_sums), n_shards,
                           shard, v_begin, stream) == cudaSuccess
             ? SPECDEC_OK
             : SPECDEC_ERR_CUDA;
}

const char* specdec_status_string(int status) {
  switch (status) {
    case SPECDEC_OK: return "ok";
    case SPECDEC_ERR_INVALID_ARG: return "invalid argument";
    case SPECDEC_ERR_UNSUPPORTED: return "unsupported shape";
    case SPECDEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPECDEC_ERR_CUDA: return "CUDA error";
    case SPECDEC_ERR_TIMEOUT: return "device-side wait timed out";
    case SPECDEC_ERR_TOKEN_RANGE: return "draft token outside [0, V)";
    default: return "unknown status";
  }
}

}  // extern "C"
