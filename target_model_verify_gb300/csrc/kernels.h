// Host-side launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace specdec {

// LM-head scoring on the tensor cores (bf16 inputs): logits z = hidden.W^T
// for every token row, with the per-tile softmax / argmax partials and the
// draft-logit partials fused into the epilogue.
struct TcLaunch {
  const CUtensorMap* tmap_w;     // W_lm [V, d], box {64, 128}, 128B swizzle
  const CUtensorMap* tmap_h;     // hidden [M, d], box {64, BT}, 128B swizzle
  const CUtensorMap* tmap_z;     // logits [M, V] fp32, box {32, 32}, 128B swizzle; or null
  int M, V, d, gamma;
  int* status;
  float* fix;                    // stream-K fix-up slots (tc_fix_floats floats)
  unsigned long long* fix_tickets;   // kFixSlots tags, any initial contents
  unsigned long long epoch;      // per-call tag (next_call_epoch)
  const unsigned long long* calls;   // the workspace header's call count
  int max_clusters;              // co-resident clusters of the launch shape (0: unknown)
  int withhold_loads;            // self-test of the bounded waits (normally 0)
  EpiParams ep;
};
cudaError_t launch_lmhead_tc(const TcLaunch& L, int num_sms, cudaStream_t stream);

// The same scoring for fp32 inputs on the CUDA cores.
cudaError_t launch_lmhead_f32(const float* hidden, const float* W, int d, const EpiParams& ep,
                              int* status, cudaStream_t stream);

// A tag that no earlier call in this process used.
unsigned long long next_call_epoch();

// Combine the partials, apply the acceptance rule, write the kept prefix.
struct AcceptLaunch {
  int B, gamma, V, P, Pq, mode, dl_bf16;   // P, Pq: records per p row and per q row
  float c;                       // log2(e) / T
  uint64_t seed;
  const PartialP* pp;
  const PartialQ* pq;
  const float* z;
  const void* dl;
  const int32_t* draft_tokens;
  int32_t* out_tokens;
  int32_t* n_accepted;
  SelectedRow* sel;
  int* counters;
  int* status;
  unsigned long long* calls;     // the workspace header's call count (one added per call)
  float* lse_p;
  float* lse_q;
  float* p_x;
  float* q_x;
  int32_t* argmax_out;
  int tok_offset;                // vocabulary-parallel shard: first token ID it holds (else 0)
};
cudaError_t launch_accept(const AcceptLaunch& L, cudaStream_t stream);

// Residual / bonus draw for every sequence (sampling mode).
struct SampleLaunch {
  int B, gamma, V, nchunks, dl_bf16;
  int vec;          // set by the launcher: 16-byte logit and draft-logit loads are aligned
  int prefetch;     // set by the launcher: small batch, rows prefetched into L2 early
  float c;
  uint64_t seed;
  const float* z;
  const void* dl;
  const SelectedRow* sel;
  float* chunk_sums;
  int* counters;
  int32_t* out_tokens;
};
// Up to kSampleOneKernelItems (sequence, chunk) pairs one kernel sums the
// chunks and draws (the last CTA of each sequence to finish draws); beyond,
// a kernel of chunk sums and a kernel of one drawing CTA per sequence.
constexpr long long kSampleOneKernelItems = 608;
cudaError_t launch_sample(const SampleLaunch& L, cudaStream_t stream);
// Small batches in sampling mode: acceptance and draw in one kernel (every
// drawing CTA folds its sequence's records itself). The sampler tickets
// must be zero when it starts: the LM-head kernel clears them
// (EpiParams::counters). kFusedAcceptItems bounds B * nchunks.
constexpr long long kFusedAcceptItems = 128;
bool fused_accept_sample(int B, int nchunks);
cudaError_t launch_accept_sample(const AcceptLaunch& A, const SampleLaunch& L,
                                 cudaStream_t stream);

// Vocabulary-parallel step (one slice of the vocabulary per GPU). A slice's
// records: target rows [M] (max z, sum exp2, argmax value and global token
// ID), draft rows [B*gamma] (max, sum exp2), guessed tokens [B*gamma] (the
// two logits when this slice holds the token); segments 256-byte aligned.
struct ShardRec {
  float m, s, amax_v;
  int amax_i;
};
struct ShardQRec {
  float m, s;
};
struct ShardXRec {
  float zx, zqx;
  int owned, pad;
};
size_t shard_record_bytes(int B, int gamma);
// Fold the slice's LM-head records into one record per row (A.V = the
// slice's vocabulary, A.tok_offset = its first token ID).
cudaError_t launch_shard_fold(const AcceptLaunch& A, void* records, cudaStream_t stream);
// Fold the gathered records of all slices and decide (A.V = the whole vocabulary).
cudaError_t launch_shard_accept(const AcceptLaunch& A, const void* all_records,
                                size_t record_bytes, int n_shards, cudaStream_t stream);
// The slice's (residual, p) weight sums of each sequence's drawn row.
// Few sequences (B * chunks <= kFusedAcceptItems): accept and the slice sums
// in one kernel; its chunk tickets use counters the LM head zeroed.
bool shard_fused_accept_sums(int B, int nchunks);
cudaError_t launch_shard_accept_sums(const AcceptLaunch& A, const SampleLaunch& L,
                                     const void* all_records, size_t record_bytes, int n_shards,
                                     float* cs_p, float2* shard_sums, cudaStream_t stream);
cudaError_t launch_shard_sums(const SampleLaunch& L, float* cs_p, float2* shard_sums,
                              cudaStream_t stream);
// The draw: the slice holding t = u * S writes its token, the others -1.
cudaError_t launch_shard_draw(const SampleLaunch& L, const float* cs_p, const float2* all_sums,
                              int n_shards, int shard, int tok_offset, cudaStream_t stream);

// Tree verification walk: one cluster of kTreeCluster CTAs per sequence
// (sampling; the CTAs split the vocabulary), kTreeClusterWide when every
// sequence's cluster of that size can be resident at once, or one CTA
// (greedy).
constexpr int kTreeCluster = 8;
constexpr int kTreeClusterWide = 16;
struct TreeLaunch {
  int B, N, V, P, Pq, mode, vec;
  float c;
  uint64_t seed;
  const PartialP* pp;            // [B*N, P] target records
  const PartialQ* pq;            // [B*N, Pq] draft records (sampling)
  const float* z;                // [B*N, V] fp32 logits (sampling)
  const __nv_bfloat16* dl;       // [B*N, V] draft logits (sampling)
  const int32_t* tok;            // [B, N] node tokens (column 0 unused)
  int16_t first_child[SPECDEC_MAX_TREE_NODES];    // -1: none; children in increasing index
  int16_t next_sibling[SPECDEC_MAX_TREE_NODES];
  int16_t parent[SPECDEC_MAX_TREE_NODES];         // parent[0] = -1
  int32_t* out_tokens;           // [B, N]
  int32_t* out_nodes;            // [B, N]
  int32_t* n_accepted;           // [B]
  int* status;
  unsigned long long* calls;     // the workspace header's call count (one added per call)
};
cudaError_t launch_tree_walk(const TreeLaunch& L, cudaStream_t stream);

// Host entry point staging through mapped pinned host memory: segments of
// `bytes` copied from host to the workspace in `unit`-byte pieces (16, 4 or
// 1; both ends aligned to it), the remainder byte by byte.
struct HostSeg {
  const void* src;
  void* dst;
  long long bytes;
  int unit;
};
struct StageInLaunch {
  HostSeg seg[3];
  int nseg;
};
cudaError_t launch_stage_in(const StageInLaunch& S, int num_sms, cudaStream_t stream);

// Verify-step attention (one layer): split-KV partials and their merge.
struct AttnLaunch {
  int B, n_new, Hq, Hkv, Lmax, n_splits, split_len;
  int n_stages;                      // K/V blocks in flight per CTA (attn_n_stages)
  float scale_log2;                  // softmax scale times log2(e)
  const __nv_bfloat16* q;            // [B, n_new, Hq, 128]
  const __nv_bfloat16* k;            // [B, Lmax, Hkv, 128]
  const __nv_bfloat16* v;
  const int32_t* seq_lens;           // [B]
  float* out;                        // [B, n_new, Hq, 128]
  float* part_m;                     // [B, Hkv, n_splits, 64] (n_splits > 1)
  float* part_l;
  float* part_o;                     // [B, Hkv, n_splits, 64, 128]
  int* status;
};
// tmap_k, tmap_v: the caches as 4-D bf16 tensors {128, Hkv, Lmax, B} with a
// {64, 1, 64, 1} box and the 128-byte swizzle.
cudaError_t launch_attention(const AttnLaunch& A, const CUtensorMap& tmap_k,
                             const CUtensorMap& tmap_v, cudaStream_t stream);
int attn_n_stages(int B, int n_new, int Hq, int Hkv);
int attn_smem_bytes(int n_mt, int n_stages);

// The drafter's clustered LM head.
struct ClusterLaunch {
  int M, d, V, n_c, top_k, max_cluster, max_members, sort_n, sample, position;
  float c;                           // log2(e) / T
  uint64_t seed;
  const __nv_bfloat16* h;            // [M, d]
  const __nv_bfloat16* E;            // [n_c, d]
  const __nv_bfloat16* W;            // [V, d] rows grouped by cluster
  const int32_t* starts;             // [n_c + 1]
  const int32_t* token_of_row;       // [V]
  float* y;                          // [M, n_c] cluster logits
  int* offs;                         // [M, top_k + 1] kept members' prefix
  float* z;                          // [M, max_members] kept members' logits
  int* ids;                          // [M, max_members] their token IDs
  int32_t* clusters;                 // [M, top_k]
  int32_t* tokens;                   // [M]
  float* logits_out;                 // [M, V] or null
  int* status;
};
cudaError_t launch_cluster_head(const ClusterLaunch& L, cudaStream_t stream);

cudaError_t launch_philox_uniforms(uint64_t seed, int B, int n_pos, int purpose, float* out,
                                   cudaStream_t stream);

// Tile geometry and schedule of the tensor-core path, shared by the
// workspace planner and the launcher.
constexpr int kMaxGrid = 256;    // persistent CTAs at most (one per SM)
constexpr int kFixSlots = kMaxGrid + 2;   // stream-K boundaries x cluster ranks
struct TcGeometry {
  int BT;                        // token rows per tile: multiple of 16, <= 256
  int n_tt;                      // token tiles
  int kc;                        // 64-wide k slices per shared-memory stage
  int box3d;                     // 3-D boxes {64, rows, kc} (d % 64 == 0)
  int stages, stage_bytes, tmem_cols, smem_bytes;
  int n_vt;                      // vocabulary tiles of 128
  int K;                         // CTAs per cluster sharing hidden slices
  int n_units, nk, grid;
  int stream_k;                  // one token tile: contiguous k-iteration ranges
  int records;                   // partial records per row (grid or vocabulary tiles)
  int rowown;                    // 1: tokens on the MMA's M side (pairs, 256-row token tiles)
  int n_acc;                     // accumulators a tile's k-slices are dealt across (swap-AB)
};
TcGeometry tc_geometry(int M, int V, int d, int num_sms, int max_clusters);
// Co-resident clusters of the kernel for this shape on the current device
// (0 when the shape runs without clusters).
int tc_max_clusters(int M, int V, int d);
// Floats of stream-K fix-up storage for a shape (0 without stream-K).
inline size_t tc_fix_floats(int M, int V, int d) {
  const TcGeometry g = tc_geometry(M, V, d, kMaxGrid, 0);
  return g.stream_k ? (size_t)kFixSlots * 2 * g.BT * kBlockV : 0;
}

}  // namespace specdec
