/*
 * specdec_verify.h -- C ABI of the speculative-decoding verify step on one
 * NVIDIA GB300 (sm_103a).
 *
 * What one call computes ("推测解码", world.lapla.si/zh/specdec):
 *   - section 先让小模型猜: the large model reads its LM-head weights once and
 *     scores the gamma guessed positions plus one more. Row (b, i) of
 *     `hidden` is the target state whose next-token distribution p_{b,i}
 *     scores draft x_{b,i} (i < gamma); row (b, gamma) is the extra
 *     position. Logits z = hidden . W_lm^T, p = softmax(z / T).
 *   - section 通过的规则: draft x is kept iff r <= p(x)/q(x) with a uniform r
 *     (tested as r*q(x) <= p(x)); q = softmax(draft_logits / T).
 *   - section 留下对的，换掉错的: the first rejected draft j is replaced by a
 *     token drawn from max(0, p_j - q_j) renormalised, and every later draft
 *     is dropped; if all gamma drafts pass, a bonus token is drawn from
 *     p_gamma. One call writes 1 .. gamma+1 tokens per sequence.
 *   - greedy mode (maxstudionews.com article 1664, the verify paragraph):
 *     keep drafts while each equals argmax z, and write the argmax at the
 *     first mismatch (or at position gamma when all match).
 *
 * Random draws: Philox4x32-10 (Salmon et al., SC'11) with key = (seed low
 * 32 bits, seed high 32 bits) and counter = (b, i, purpose, 0); k = word0
 * >> 8; the acceptance uniform is r = (k+1)/2^24 (purpose 0) and the
 * sampling uniform u = k/2^24 (purpose 1), drawn at the position where the
 * replacement or bonus is written. The draw is the smallest token v with
 * C_v > u*S, C the prefix sum of the weights in token-ID order and S its
 * total; if S is 0 the draw falls back to p_j.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise, owned
 *     by the caller, row-major and contiguous. The library allocates nothing
 *     and keeps no state between calls (apart from a per-device cache of the
 *     SM count and kernel attributes).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising, except where
 *     stated.
 *   - Return value: SPECDEC_OK (0) or a negative SPECDEC_ERR_* code.
 *     Argument errors are detected on the host before anything is enqueued.
 *     Errors found on the device (draft token out of [0, V), a kernel wait
 *     that timed out) are written to a status word in the workspace; the
 *     call then writes n_accepted = -1 and out_tokens = -1 for the affected
 *     sequences (a token out of range: its sequence; a timeout: every
 *     sequence). specdec_read_status() returns that word.
 *   - Shapes: B >= 0 (B == 0 returns SPECDEC_OK and touches no pointer),
 *     1 <= gamma <= SPECDEC_MAX_GAMMA,
 *     d >= 1 with d % 8 == 0 for bf16 (rows must be 16-byte aligned),
 *     1 <= V <= 2^22, M = B*(gamma+1), and M*V < 2^31. Pointers to bf16 data must
 *     be 16-byte aligned.
 */
#ifndef SPECDEC_VERIFY_H_
#define SPECDEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPECDEC_MAX_GAMMA 32
#define SPECDEC_MAX_TREE_NODES 128

/* mode */
#define SPECDEC_SAMPLE 0
#define SPECDEC_GREEDY 1

/* dtype of hidden, W_lm and draft_logits */
#define SPECDEC_BF16 0
#define SPECDEC_FP32 1

/* status codes */
#define SPECDEC_OK 0
#define SPECDEC_ERR_INVALID_ARG (-1)   /* null pointer, bad enum, T <= 0 in sampling mode */
#define SPECDEC_ERR_UNSUPPORTED (-2)   /* shape outside the limits above */
#define SPECDEC_ERR_WORKSPACE (-3)     /* workspace NULL, misaligned or too small */
#define SPECDEC_ERR_CUDA (-4)          /* a CUDA runtime/driver call failed */
#define SPECDEC_ERR_TIMEOUT (-5)       /* a device-side wait ran out (status word) */
#define SPECDEC_ERR_TOKEN_RANGE (-6)   /* a draft token outside [0, V) (status word) */

/*
 * Bytes of device workspace specdec_verify() needs for this shape. The
 * workspace must be 256-byte aligned; its contents need no initialisation
 * and are overwritten by every call. Calls that share a workspace must be
 * ordered (same stream, or synchronised). Returns 0 for invalid shapes.
 * Takes the mode besides the shape: greedy mode keeps no fp32 logits, no
 * draft-logit records and no sampler chunk sums (it never reads the draft
 * logits), so its workspace is a small fraction of the sampling one (at
 * B = 256 on the Llama-3-8B-shaped head, 0.2 GB instead of 1.1 GB).
 */
size_t specdec_verify_workspace_size(int B, int gamma, int d, int V, int dtype, int mode);

/*
 * The verify step.
 *   hidden       [B, gamma+1, d]  dtype   target hidden states (see above)
 *   W_lm         [V, d]           dtype   LM-head weights, row v = token v
 *   draft_tokens [B, gamma]       int32   the small model's guesses x
 *   draft_logits [B, gamma, V]    dtype   the small model's logits for q;
 *                                         may be NULL in greedy mode
 *   temperature  T > 0 (sampling mode; ignored in greedy mode)
 *   seed         Philox key (see above)
 *   mode         SPECDEC_SAMPLE or SPECDEC_GREEDY
 *   out_tokens   [B, gamma+1]     int32   written: kept drafts, then the
 *                                         replacement or bonus token, then -1
 *   n_accepted   [B]              int32   j = number of kept drafts, 0..gamma
 *   workspace    device scratch of specdec_verify_workspace_size() bytes
 */
int specdec_verify(const void* hidden, const void* W_lm, const int32_t* draft_tokens,
                   const void* draft_logits, int B, int gamma, int d, int V, int dtype,
                   float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                   int32_t* n_accepted, void* workspace, size_t workspace_bytes, void* stream);

/*
 * specdec_verify() that also exposes its intermediates, for parity checks.
 * Every extra pointer is an optional device buffer (NULL = not wanted):
 *   logits_out [M, V] fp32  the target logits z
 *   lse_p      [M]    fp32  log sum_v exp(z_v / T)           (sampling mode)
 *   lse_q      [B*gamma]    log sum_v exp(draft_logit_v / T) (sampling mode)
 *   p_x, q_x   [B*gamma]    p_i(x_i) and q_i(x_i)            (sampling mode)
 *   argmax_out [M]   int32  argmax_v z (lowest v among equal maxima)
 * Same results as specdec_verify() for the same inputs and seed. There is
 * no first-reject output: n_accepted already is that position (the first
 * rejected draft sits at index n_accepted, or none when it equals gamma).
 * The per-row argmax takes its place, since greedy parity needs the argmax
 * of every scored row, not only of the rows the walk reached.
 */
int specdec_verify_debug(const void* hidden, const void* W_lm, const int32_t* draft_tokens,
                         const void* draft_logits, int B, int gamma, int d, int V, int dtype,
                         float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                         int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                         void* stream, float* logits_out, float* lse_p, float* lse_q,
                         float* p_x, float* q_x, int32_t* argmax_out);

/*
 * specdec_verify() with two caller-created CUDA events (cudaEvent_t)
 * recorded on `stream` immediately before and after the LM-head kernel, so
 * a caller can time that kernel inside a real step. Either may be NULL.
 */
int specdec_verify_timed(const void* hidden, const void* W_lm, const int32_t* draft_tokens,
                         const void* draft_logits, int B, int gamma, int d, int V, int dtype,
                         float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                         int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                         void* stream, void* lmhead_start_event, void* lmhead_end_event);

/*
 * End-to-end form: hidden, draft_tokens, draft_logits, out_tokens and
 * n_accepted are HOST pointers; W_lm and the workspace stay on the device.
 * The call moves the inputs in, runs the step and moves the outputs back on
 * `stream`, then synchronises that stream before returning. When all five
 * host buffers are pinned and mapped into the GPU's address space (the
 * runtime reports a device address for each; the two outputs 4-byte
 * aligned), one kernel
 * reads the inputs from host memory into the workspace and the step's
 * kernels store the results straight into the output buffers (on
 * Grace-Blackwell over NVLink-C2C); otherwise the copy engines move them
 * (pageable memory is allowed there). Host buffers must
 * hold the sizes the shape implies. Workspace:
 * specdec_verify_host_workspace_size().
 */
size_t specdec_verify_host_workspace_size(int B, int gamma, int d, int V, int dtype, int mode);
int specdec_verify_host(const void* hidden_host, const void* W_lm, const int32_t* draft_tokens_host,
                        const void* draft_logits_host, int B, int gamma, int d, int V, int dtype,
                        float temperature, uint64_t seed, int mode, int32_t* out_tokens_host,
                        int32_t* n_accepted_host, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * specdec_verify() for callers that cannot allocate device memory. The
 * source pages have no counterpart to this entry point: it exists because
 * some callers cannot hand the library a workspace -- code running inside a
 * host program that owns all device memory and gives its plug-ins no
 * allocator, or a decode loop whose memory was planned up front, where a
 * cudaMalloc would synchronise the device or fail against a caching
 * allocator's reservation.
 *
 * Same arguments and results as specdec_verify(), minus the workspace: the
 * scratch is a static device array of SPECDEC_NOALLOC_SCRATCH_BYTES
 * (16 MiB) that every GPU which loads the library holds until the process
 * exits. Shapes whose specdec_verify_workspace_size() exceeds that are
 * rejected with SPECDEC_ERR_WORKSPACE before anything is enqueued (one
 * sequence fits at every head shape here, e.g. 6.6 MiB for the
 * Llama-3-8B-shaped head, 13.4 MiB for the Gemma-E2B head at gamma = 8).
 * The call allocates nothing. Its first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture. All calls share the one
 * array and each clears what must start at zero, but calls whose work
 * overlaps on the GPU (different streams, or different host threads
 * without ordering) race on it and must be serialised by the caller.
 * specdec_read_status() does not apply: the status word lives in the array,
 * so the exact device-side error code cannot be read. A step that failed
 * on the device (a draft token outside [0, V), or a wait that ran out)
 * shows in its outputs instead: n_accepted[b] = -1 and out_tokens[b, :] =
 * -1 for every affected sequence (for a timeout, every sequence). The
 * array's address is looked up again whenever the current context changes
 * (after cudaDeviceReset, or with another context current on the device),
 * so a reset does not leave the call writing through a stale address; that
 * look-up, too, is best made before any stream capture.
 */
#define SPECDEC_NOALLOC_SCRATCH_BYTES (16u << 20)
int specdec_verify_noalloc(const void* hidden, const void* W_lm, const int32_t* draft_tokens,
                           const void* draft_logits, int B, int gamma, int d, int V, int dtype,
                           float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                           int32_t* n_accepted, void* stream);

/*
 * Tree verification ("推测解码", section 不要第二个模型: guesses arranged as
 * a tree are checked in one pass, with the acceptance rule applied at every
 * fork). One tree topology for the whole batch, given by `parent`, a HOST
 * array of n_nodes int32: parent[0] = -1 (the root, the position after the
 * committed text) and 0 <= parent[n] < n for n >= 1, so 1 <= n_nodes <=
 * SPECDEC_MAX_TREE_NODES. Node n >= 1 holds one guessed token.
 *   hidden       [B, N, d]   dtype   target state after the path root -> n;
 *                                    p_n = softmax(z_n / T) scores n's children
 *   W_lm         [V, d]      dtype   LM-head weights
 *   node_tokens  [B, N]      int32   guessed token of every node (column 0
 *                                    ignored); in [0, V) else the status word
 *                                    gets SPECDEC_ERR_TOKEN_RANGE
 *   draft_logits [B, N, V]   dtype   q_n, the distribution n's children were
 *                                    drawn from (rows of leaves are read but
 *                                    unused); may be NULL in greedy mode
 *   out_tokens   [B, N]      int32   kept path tokens, then the drawn (or argmax)
 *                                    token, then -1
 *   out_nodes    [B, N]      int32   kept node indices in path order, then -1
 *   n_accepted   [B]         int32   number of kept nodes
 * Sampling rule at node u: children in increasing index; child c is kept iff
 * r_c * q_u(x_c) <= f(x_c), with f = p_u for the first child and f =
 * max(0, f - q_u) / S after each rejection (S its sum over the vocabulary);
 * a kept child becomes the node; otherwise one token is drawn from the last
 * residual max(0, f - q_u) (or from p_u when u has no children) by the
 * inversion above. Random draws: child c uses the acceptance uniform of
 * position c - 1, the draw at depth j the sampling uniform of position j,
 * so a chain-shaped tree (parent[n] = n - 1) gives the same tokens as
 * specdec_verify(). Greedy: move to the first child whose token is the
 * target argmax; else write the argmax. Only dtype SPECDEC_BF16; limits as
 * specdec_verify() with M = B*N rows. Asynchronous on `stream`.
 */
size_t specdec_verify_tree_workspace_size(int B, int n_nodes, int d, int V, int dtype, int mode);
int specdec_verify_tree(const void* hidden, const void* W_lm, const int32_t* parent,
                        const int32_t* node_tokens, const void* draft_logits, int B, int n_nodes,
                        int d, int V, int dtype, float temperature, uint64_t seed, int mode,
                        int32_t* out_tokens, int32_t* out_nodes, int32_t* n_accepted,
                        void* workspace, size_t workspace_bytes, void* stream);
/* specdec_verify_tree() with events around its LM-head kernel (see
 * specdec_verify_timed). */
int specdec_verify_tree_timed(const void* hidden, const void* W_lm, const int32_t* parent,
                              const int32_t* node_tokens, const void* draft_logits, int B,
                              int n_nodes, int d, int V, int dtype, float temperature,
                              uint64_t seed, int mode, int32_t* out_tokens, int32_t* out_nodes,
                              int32_t* n_accepted, void* workspace, size_t workspace_bytes,
                              void* stream, void* lmhead_start_event, void* lmhead_end_event);

/*
 * Verify-step attention for one layer ("推测解码", section 几段话一起写:
 * every sequence reads its own KV cache each step). The n_new = gamma + 1
 * new positions of every sequence attend to their causal window of the
 * sequence's cache:
 *   q        [B, n_new, Hq, D]   bf16   queries of the new positions
 *   k_cache  [B, Lmax, Hkv, D]   bf16   keys; rows < seq_lens[b] are valid and
 *   v_cache  [B, Lmax, Hkv, D]   bf16   the last n_new of them are the new positions
 *   seq_lens [B]                 int32  (device) valid rows, n_new <= L <= Lmax;
 *                                       otherwise the status word gets
 *                                       SPECDEC_ERR_INVALID_ARG and that
 *                                       sequence's output is 0
 *   out      [B, n_new, Hq, D]   fp32   o = sum_j softmax_j(scale q.k_j) v_j over
 *                                       rows j <= seq_len - n_new + i
 * Query head h reads KV head h / (Hq / Hkv). scale <= 0 selects 1/sqrt(D).
 * Limits: D = 128, Hq % Hkv == 0, n_new * Hq / Hkv <= 64, B >= 0 (0 is a
 * no-op), Lmax >= n_new; q, caches and out 16-byte aligned. The status word
 * sits at the start of the workspace (specdec_read_status). Asynchronous.
 */
size_t specdec_verify_attention_workspace_size(int B, int n_new, int Hq, int Hkv, int D, int Lmax);
int specdec_verify_attention(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* seq_lens, int B, int n_new, int Hq, int Hkv, int D,
                             int Lmax, float scale, float* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * The drafter's clustered LM head ("多詞元預測視覺化指南", section 高效嵌入器):
 * cluster logits y = h E^T, the top_k clusters of every row (largest y, ties
 * to the lower index), token logits z = h . W_r for the kept clusters'
 * member rows only, and the draft token: greedy, the argmax of z (lowest
 * token ID on ties); sampling, the smallest token ID whose prefix sum (in
 * token-ID order) of exp((z - max z) / T) passes u * S, with u from Philox
 * counter (row m, position, purpose 2).
 *   hidden        [M, d]       bf16   drafter hidden states, M <= 64
 *   cluster_emb   [n_c, d]     bf16   one embedding per cluster
 *   W_sorted      [V, d]       bf16   token embeddings grouped by cluster
 *   starts        [n_c + 1]    int32  (device) cluster c owns rows starts[c] ..
 *                                     starts[c+1] - 1 of W_sorted
 *   token_of_row  [V]          int32  (device) token ID of every W_sorted row
 *   max_cluster   host bound on any cluster's size; a kept cluster above it
 *                 sets SPECDEC_ERR_INVALID_ARG in the status word
 *   out_tokens    [M] int32, out_clusters [M, top_k] int32 (best first)
 *   logits_out    [M, V] fp32 or NULL: the kept tokens' logits are written
 *                 there (other entries are left as the caller set them)
 * Limits: 1 <= top_k <= SPECDEC_CLUSTER_MAX_TOP_K, d % 8 == 0,
 * d <= SPECDEC_CLUSTER_MAX_D, top_k * max_cluster <=
 * SPECDEC_CLUSTER_MAX_MEMBERS, top_k <= n_c; bf16 pointers 16-byte aligned.
 * Asynchronous; status word at the start of the workspace.
 */
#define SPECDEC_CLUSTER_MAX_TOP_K 8
#define SPECDEC_CLUSTER_MAX_D 4096
#define SPECDEC_CLUSTER_MAX_MEMBERS 4096
size_t specdec_cluster_head_workspace_size(int M, int n_c, int top_k, int max_cluster);
int specdec_cluster_head(const void* hidden, const void* cluster_emb, const void* W_sorted,
                         const int32_t* starts, const int32_t* token_of_row, int M, int d, int V,
                         int n_c, int top_k, int max_cluster, float temperature, uint64_t seed,
                         int position, int mode, int32_t* out_tokens, int32_t* out_clusters,
                         float* logits_out, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Vocabulary-parallel verify step, for a tensor-parallel target model whose
 * LM head is split by vocabulary rows across G GPUs ("推测解码", section
 * 几段话一起写: the weight read is the step's cost, so each GPU reads only
 * its slice). GPU g holds rows [v_begin, v_begin + V_shard) of W_lm and the
 * same columns of every draft row; hidden and draft_tokens are replicated.
 * The slices must cover [0, V) without overlap. A step is three calls on
 * every GPU, with the caller's collectives between them (the library holds
 * no communicator):
 *
 *   specdec_shard_score   LM head on the slice; writes this GPU's records
 *                         (specdec_shard_record_bytes bytes, 16-byte aligned
 *                         device buffer): per target row (max z, sum exp2,
 *                         argmax value and global token ID), per draft row
 *                         (max, sum exp2), per guessed token its two logits
 *                         when the slice holds it.
 *   -- all-gather the G records, in rank order, into one device buffer --
 *   specdec_shard_accept  folds the G records of every row in one fixed
 *                         order (so every GPU decides alike), writes out_tokens'
 *                         kept prefix and n_accepted (greedy mode: the whole
 *                         result; nothing follows), and in sampling mode the
 *                         slice's weight sums of the drawn row:
 *                         shard_sums[2b] = sum of max(0, p - q) (of p for the
 *                         bonus row), shard_sums[2b+1] = sum of p.
 *   -- all-gather the G shard_sums [B, 2] fp32, in rank order --
 *   specdec_shard_draw    every GPU forms the same prefix over slices and
 *                         t = u * S (S the residual total, or the p total if
 *                         no residual mass is left); the GPU whose slice
 *                         holds t writes the drawn token's global ID at
 *                         out_tokens[b, n_accepted[b]], the others -1.
 *   -- all-reduce out_tokens with max --
 *
 * Same rule, uniforms and token order as specdec_verify(); the draw's
 * position t is split across slices, so a token can differ from the
 * single-GPU step's only where u sits within rounding of a CDF boundary.
 * Every call takes the same shape arguments and the same workspace
 * (specdec_shard_workspace_size bytes, 256-byte aligned; it carries the
 * slice's logits and sums from one call to the next, and the score call
 * resets the counters the accept call uses, so each accept follows the
 * score of its own step on that workspace). dtype bf16 only;
 * 1 <= n_shards <= SPECDEC_MAX_SHARDS. Errors as specdec_verify(); a guessed
 * token that no slice holds sets SPECDEC_ERR_TOKEN_RANGE in the status word
 * and that sequence's outputs to -1. Asynchronous on `stream`.
 */
#define SPECDEC_MAX_SHARDS 64
size_t specdec_shard_record_bytes(int B, int gamma);
size_t specdec_shard_workspace_size(int B, int gamma, int d, int V_shard, int mode);
int specdec_shard_score(const void* hidden, const void* W_shard, const int32_t* draft_tokens,
                        const void* draft_logits_shard, int B, int gamma, int d, int V_shard,
                        int v_begin, int V, float temperature, int mode, void* records,
                        void* workspace, size_t workspace_bytes, void* stream);
int specdec_shard_accept(const void* all_records, int n_shards, const int32_t* draft_tokens,
                         const void* draft_logits_shard, int B, int gamma, int d, int V_shard,
                         int v_begin, int V, float temperature, uint64_t seed, int mode,
                         int32_t* out_tokens, int32_t* n_accepted, float* shard_sums,
                         void* workspace, size_t workspace_bytes, void* stream);
int specdec_shard_draw(const float* all_shard_sums, int n_shards, int shard,
                       const void* draft_logits_shard, int B, int gamma, int d, int V_shard,
                       int v_begin, int V, float temperature, uint64_t seed, int mode,
                       int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * Reads the device status word of a workspace after synchronising `stream`:
 * SPECDEC_OK, SPECDEC_ERR_TIMEOUT, SPECDEC_ERR_TOKEN_RANGE (verify and tree
 * steps) or SPECDEC_ERR_INVALID_ARG (attention lengths, clustered-head
 * tables) of the last call that used it. *status receives the value; the
 * return code reports the read itself.
 */
int specdec_read_status(const void* workspace, void* stream, int32_t* status);

/*
 * Self-test of the device-side failure detection: runs the LM-head kernel on
 * a small internal shape with its loads withheld, so the first wait of the
 * MMA stage finds a barrier that nothing will ever arm. The wait gives up
 * after its bound (about 1 s), the kernel frees what it holds and returns,
 * and *status receives the status word it left: SPECDEC_ERR_TIMEOUT when the
 * detection works. Nothing faults, traps or hangs, and the CUDA context stays
 * usable. Synchronises `stream`. workspace: at least
 * specdec_verify_workspace_size(1, 4, 64, 256, SPECDEC_BF16, SPECDEC_GREEDY)
 * bytes, 256-byte aligned; its contents are overwritten.
 */
int specdec_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream,
                                  int32_t* status);

/*
 * The library's own uniforms, for checking them against another
 * implementation: out[b*n_pos + i] = r (purpose 0) or u (purpose 1) for
 * sequence b < B and position i < n_pos. `out` is a device fp32 buffer.
 */
int specdec_philox_uniforms(uint64_t seed, int B, int n_pos, int purpose, float* out,
                            void* stream);

/* A static, human-readable name for a status code. */
const char* specdec_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_VERIFY_H_ */
