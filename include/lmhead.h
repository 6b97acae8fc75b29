/*
 * lmhead.h - C ABI of liblmhead.so, a GB300 (sm_103a) two-stage draft LM head.
 *
 * The operation is the "EAGLE Efficient LM Head" of the EAGLE-4 design notes
 * (qingkeai.online/blog/EAGLE): stage 1 scores the whole vocabulary with a
 * rank-r factor of the full head, A (n x r) and B (r x d), built offline by
 * the Freq-aware SVD of that page's section "A training-free version:
 * Freq-aware SVD", and keeps candidates by Top-k (globally, or per vocabulary
 * tile as in the section "A Local Top-k based variant"); stage 2 gathers the
 * candidates' rows of the full head W (n x d), recomputes their exact logits
 * from the same hidden states h (M x d) and softmaxes them into the draft
 * distribution q that a speculative-decoding drafter samples from.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Element types: bf16 tensors are passed as raw 16-bit patterns
 *    (lmhead_bf16); scores, logits and q are fp32; ids are int32 vocabulary
 *    ids. All matrices are dense row-major with no padding.
 *  - Memory: every pointer is a DEVICE pointer owned by the caller, aligned
 *    to 16 bytes; d and r must be multiples of 8. The library allocates no
 *    device memory; scratch comes from the caller's `workspace`
 *    (size from lmhead_workspace_size). `workspace` may be reused across
 *    calls but not by two calls in flight at once.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream). All
 *    calls enqueue asynchronous work on it and return without synchronising,
 *    except lmhead_last_device_error.
 *  - Errors: arguments are validated on the host before anything is
 *    launched; a negative lmhead_status is returned and nothing is enqueued.
 *    A failed launch returns LMHEAD_ERR_CUDA. Kernels that read caller ids
 *    bounds-check them; a bad id sets a device error word (read with
 *    lmhead_last_device_error) and its outputs are NaN; nothing faults.
 *    NaN/Inf inputs are not checked (outputs undefined).
 *  - Ties: equal scores are ordered by the smaller vocabulary id.
 */
#ifndef LMHEAD_H
#define LMHEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lmhead_bf16; /* bf16 bit pattern */
typedef void* lmhead_stream; /* a cudaStream_t */

typedef enum {
  LMHEAD_OK = 0,
  LMHEAD_ERR_NULL = -1,         /* a required pointer is NULL */
  LMHEAD_ERR_SHAPE = -2,        /* a size is out of range or inconsistent */
  LMHEAD_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned */
  LMHEAD_ERR_WORKSPACE = -4,    /* workspace missing or too small */
  LMHEAD_ERR_UNSUPPORTED = -5,  /* valid but not supported by this build */
  LMHEAD_ERR_CUDA = -6,         /* a CUDA runtime call or launch failed */
  LMHEAD_ERR_DEVICE_CHECK = -7, /* a kernel's own check failed (bad id, ...) */
  LMHEAD_ERR_TIMEOUT = -8       /* a kernel's bounded wait ran out */
} lmhead_status;

typedef enum {
  LMHEAD_GLOBAL = 0, /* ids = Top-C of the full-vocabulary scores */
  LMHEAD_LOCAL = 1   /* ids = concat over vocabulary tiles of each tile's top-k_tile */
} lmhead_mode;

/* Library version (major*10000 + minor*100 + patch). */
int lmhead_version(void);

/* Human-readable name of a status code; never NULL. */
const char* lmhead_status_string(int status);

/*
 * Candidates per hidden vector for a mode (EAGLE-4 notes, "A Local Top-k
 * based variant": the candidate count is about tiles x k_tile).
 *   GLOBAL: C (C_or_tile), requires 1 <= C <= n.
 *   LOCAL : T = C_or_tile rows per tile, tiles = ceil(n/T); each full tile
 *           keeps k_tile and a short last tile keeps min(k_tile, rows).
 * Returns the count, or a negative lmhead_status for invalid sizes.
 */
int64_t lmhead_candidate_count(int mode, int64_t n, int C_or_tile, int k_tile);

/*
 * Bytes of device workspace that lmhead_lowrank_score_topk and
 * lmhead_two_stage need for these sizes. Depends only on its arguments.
 * Returns 0 for invalid sizes.
 */
size_t lmhead_workspace_size(int mode, int64_t n, int d, int r, int M,
                             int C_or_tile, int k_tile);

/*
 * Stage-1 projection u = B.h (EAGLE-4 notes, "A Local Top-k based variant",
 * first line of both flows).
 *   B  r x d bf16, h  M x d bf16  ->  u  M x r bf16.
 * Accumulates in fp32 and rounds each u element to bf16 (nearest-even).
 */
int lmhead_project_u(const lmhead_bf16* B, const lmhead_bf16* h, int d, int r, int M,
                     lmhead_bf16* u, lmhead_stream stream);

/*
 * Stage 1: candidate selection with the low-rank head (EAGLE-4 notes,
 * "A training-free version: Freq-aware SVD": Top-k of A(Bh); and
 * "A Local Top-k based variant").
 *   A          n x r bf16, rows in POSITION order (pre-shuffled: position p
 *              holds vocabulary row token_ids[p]).
 *   B          r x d bf16.
 *   h          M x d bf16 hidden states; each row is selected independently.
 *   token_ids  n int32, position -> vocabulary id; NULL means identity.
 *              Must be a permutation of 0..n-1 (ids are range-checked).
 *   mode       LMHEAD_GLOBAL: C_or_tile = C, k_tile ignored (0).
 *              LMHEAD_LOCAL : C_or_tile = T >= 1, 1 <= k_tile <= T.
 *   out_ids    M x K int32 (K = lmhead_candidate_count). GLOBAL rows are in
 *              descending score order; LOCAL rows are in tile order, each
 *              tile's ids in descending score order.
 *   out_scores M x K fp32 low-rank scores of out_ids, or NULL.
 *   workspace  >= lmhead_workspace_size(...) bytes, 256-byte aligned.
 * LOCAL mode with k_tile <= 32 runs the fused score + tile top-k kernel
 * (no score writeback); GLOBAL mode and larger k_tile write the fp32 scores
 * to the workspace and run a radix select.
 */
int lmhead_lowrank_score_topk(int mode, const lmhead_bf16* A, const lmhead_bf16* B,
                              const lmhead_bf16* h, const int32_t* token_ids,
                              int64_t n, int d, int r, int M, int C_or_tile, int k_tile,
                              int32_t* out_ids, float* out_scores,
                              void* workspace, size_t workspace_bytes,
                              lmhead_stream stream);

/*
 * Stage 2: exact logits of the candidates (EAGLE-4 notes, "EAGLE Efficient
 * LM Head": index the full head's rows of the candidates and recompute the
 * logits with the original hidden states; logits = W[ids] @ h).
 *   W  n x d bf16 (vocabulary order), h  M x d bf16, ids  M x K int32.
 *   out_logits M x K fp32: out_logits[m,j] = sum_i W[ids[m,j], i] * h[m,i],
 *   fp32 accumulation. An id outside [0, n) gives NaN and sets the device
 *   error word.
 */
int lmhead_gather_logits(const lmhead_bf16* W, const lmhead_bf16* h, const int32_t* ids,
                         int64_t n, int d, int M, int K, float* out_logits,
                         lmhead_stream stream);

/*
 * Draft distribution over each row's candidates: q[m,j] = exp((L[m,j] -
 * max_j L[m,:]) / temperature) / sum. The drafter samples its next token
 * from this distribution (EAGLE -> EAGLE-2 -> EAGLE-3 -> DFlash overview,
 * course.zhidx.com, section 1.3; the accept/reject rule of "Speculative
 * decoding and EAGLE", ai-engineering.com.cn, consumes it). Tokens that are
 * not candidates have probability 0. temperature > 0. out_q may alias logits.
 */
int lmhead_candidate_softmax(const float* logits, int M, int K, float temperature,
                             float* out_q, lmhead_stream stream);

/*
 * The whole two-stage head in one call: projection, selection (mode as in
 * lmhead_lowrank_score_topk), gather of W[ids], exact logits and softmax.
 * Outputs: out_ids, out_logits, out_q, each M x K (K from
 * lmhead_candidate_count). No host synchronisation.
 */
int lmhead_two_stage(int mode, const lmhead_bf16* W, const lmhead_bf16* A,
                     const lmhead_bf16* B, const lmhead_bf16* h, const int32_t* token_ids,
                     int64_t n, int d, int r, int M, int C_or_tile, int k_tile,
                     float temperature, int32_t* out_ids, float* out_logits, float* out_q,
                     void* workspace, size_t workspace_bytes, lmhead_stream stream);

/*
 * lmhead_two_stage with timing marks for profiling: records events[0] on
 * `stream` before the first kernel and events[i] after the i-th stage, for
 * i < n_events (events are cudaEvent_t created by the caller). The stages are
 * the projection, the scoring, the selection (global mode and local k_tile
 * > 32 only; for long rows it is several kernels), the gather and the
 * softmax; lmhead_two_stage_launches gives their number.
 * Same arguments, outputs and errors as lmhead_two_stage otherwise.
 */
int lmhead_two_stage_profiled(int mode, const lmhead_bf16* W, const lmhead_bf16* A,
                              const lmhead_bf16* B, const lmhead_bf16* h,
                              const int32_t* token_ids, int64_t n, int d, int r, int M,
                              int C_or_tile, int k_tile, float temperature, int32_t* out_ids,
                              float* out_logits, float* out_q, void* workspace,
                              size_t workspace_bytes, void* const* events, int n_events,
                              lmhead_stream stream);
int lmhead_two_stage_launches(int mode, int k_tile);

/*
 * Comparison head: the dense full-vocabulary head whose cost the method
 * avoids (EAGLE-4 notes, "EAGLE Efficient LM Head": the LM head can be about
 * half of a one-layer drafter's forward).
 *   out_logits M x n fp32 = h W^T; out_q M x n softmax over the whole
 *   vocabulary, or NULL for logits only.
 */
int lmhead_dense_head(const lmhead_bf16* W, const lmhead_bf16* h, int64_t n, int d, int M,
                      float temperature, float* out_logits, float* out_q,
                      lmhead_stream stream);

/*
 * Comparison head: the frequency-pruned vocabulary (FR-Spec style, 32000
 * most frequent tokens in the EAGLE-4 notes, "EAGLE Efficient LM Head").
 *   W_pruned  n_keep x d bf16: the kept rows of W, copied contiguously by the
 *             caller in the order of its kept-id list.
 *   out_logits, out_q  M x n_keep fp32 over the kept tokens (out_q may be NULL).
 */
int lmhead_pruned_head(const lmhead_bf16* W_pruned, const lmhead_bf16* h, int n_keep,
                       int d, int M, float temperature, float* out_logits, float* out_q,
                       lmhead_stream stream);

/*
 * Local-mode two-stage head that allocates nothing and takes no workspace.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory or hand over a workspace, such as a
 * serving engine that gives all free HBM to its KV-cache pool at start-up and
 * forbids allocation in its decode loop, or C/C++ code embedding the library
 * with no device allocator of its own. Arguments, outputs and results are
 * those of lmhead_two_stage with mode = LMHEAD_LOCAL, C_or_tile = T.
 *   Speed: it scores as lmhead_two_stage does (the warp-per-row GEMV kernel
 *   for up to four hidden vectors at r = 256 or 512, the tensor-core kernel for
 *   tiles of a multiple of 128 rows), except that tiles of other sizes score
 *   on the CUDA-core tile kernel (the tensor-core form for them needs scratch
 *   that grows with M and n), and the gather never overlaps the scoring
 *   kernel, so at 9 to 256 hidden vectors it is somewhat slower than
 *   lmhead_two_stage.
 *   Scratch: a fixed static device array of 513 KiB (u for M <= 256 and
 *   r <= 1024, plus the scoring kernel's tile counters) held by every GPU
 *   that loads the library until the process exits. M > 256, r > 1024 or k_tile > 32
 *   returns LMHEAD_ERR_UNSUPPORTED and enqueues nothing.
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   contents (the call zeroes what must start at zero). Calls whose work
 *   overlaps on the GPU (other streams, other host threads) race on the
 *   array and corrupt each other's outputs: serialise them.
 *   Never calls cudaMalloc, cudaFree or any allocating library routine.
 */
int lmhead_two_stage_local_noalloc(const lmhead_bf16* W, const lmhead_bf16* A,
                                   const lmhead_bf16* B, const lmhead_bf16* h,
                                   const int32_t* token_ids, int64_t n, int d, int r, int M,
                                   int T, int k_tile, float temperature, int32_t* out_ids,
                                   float* out_logits, float* out_q, lmhead_stream stream);

/*
 * Cluster-level two-stage head: the third route of the EAGLE-4 notes,
 * "EAGLE Efficient LM Head" (split the tokens into groups, 128 per group in
 * the notes' example; select a few groups; compute the logits of every token
 * inside them and sample from those). The notes leave the group make-up and
 * the selector open; this library reads them as:
 *   - a group is `group` consecutive rows of the head as stored, group g =
 *     rows [g*group, (g+1)*group), so every selected group is one contiguous
 *     block of W; `group` must divide n;
 *   - a group's score is the largest low-rank score A(Bh) among its rows
 *     (the token-level route's own first stage, u rounded to bf16), and each
 *     row of h keeps the G best groups, best first, ties by the smaller
 *     group index.
 * Per row m of h (M x d):
 *   out_groups        M x G int32 selected group indices, best first.
 *   out_group_scores  M x G fp32 their scores, or NULL.
 *   out_ids           M x (G*group) int32: the rows of each selected group in
 *                     selection order, ascending within a group.
 *   out_logits, out_q M x (G*group) fp32: exact W[ids].h and their softmax
 *                     (temperature > 0).
 * Sizes: 1 <= G <= n/group, G <= 4096, M*G*group <= 2^31-1, d and r as for
 * lmhead_two_stage. Scratch from `workspace`, at least
 * lmhead_cluster_workspace_size bytes, 256-byte aligned. W, A, B, h must be
 * 16-byte aligned (LMHEAD_ERR_ALIGN otherwise); bad sizes give
 * LMHEAD_ERR_SHAPE (a group size that does not divide n included) and
 * nothing is enqueued. Six kernels, no host synchronisation.
 */
int64_t lmhead_cluster_candidate_count(int64_t n, int group, int G);
size_t lmhead_cluster_workspace_size(int64_t n, int d, int r, int M, int group, int G);
int lmhead_cluster_two_stage(const lmhead_bf16* W, const lmhead_bf16* A, const lmhead_bf16* B,
                             const lmhead_bf16* h, int64_t n, int d, int r, int M, int group,
                             int G, float temperature, int32_t* out_groups,
                             float* out_group_scores, int32_t* out_ids, float* out_logits,
                             float* out_q, void* workspace, size_t workspace_bytes,
                             lmhead_stream stream);

/*
 * Draft-token selection on q ("EAGLE -> EAGLE-2 -> EAGLE-3 -> DFlash", the
 * EAGLE-2 dynamic draft tree, Expansion Phase: a node is expanded into its
 * most likely draft tokens, and a token's value is the product of the draft
 * confidences along its path). Per row m of q (one tree node):
 *   q, ids        M x K fp32 / int32: the node's draft distribution over its
 *                 candidates (lmhead_two_stage's out_q and out_ids).
 *   k_sel         1 <= k_sel <= min(K, 16).
 *   parent_value  M fp32, the node's own value, or NULL (value 1).
 *   uniforms      M x K fp32 in (0, 1), or NULL for no draw.
 *   out_top_ids, out_top_q, out_top_value  M x k_sel: the k_sel largest q
 *                 (ties: smaller vocabulary id), descending, and
 *                 parent_value * q (fp32). out_top_value may be NULL.
 *   out_sample_id, out_sample_q  M (may be NULL): one token drawn from q by
 *                 Gumbel-max, argmax_j log q_j - log(-log uniforms_j) (ties:
 *                 smaller id), and its q. Ignored when uniforms is NULL.
 * Returns LMHEAD_ERR_SHAPE for bad sizes; everything else as above.
 */
int lmhead_draft_select(const float* q, const int32_t* ids, int M, int K, int k_sel,
                        const float* parent_value, const float* uniforms, int32_t* out_top_ids,
                        float* out_top_q, float* out_top_value, int32_t* out_sample_id,
                        float* out_sample_q, lmhead_stream stream);

/*
 * Chain verification of drafted tokens ("Speculative decoding and EAGLE",
 * the exactness rule): for t = 0..Kd-1, accept x_t if r_t < p_t(x_t) /
 * q_t(x_t) (fp32); otherwise draw the replacement from (p_t - q_t)+
 * normalised and stop; when every draft is accepted, draw a bonus token from
 * p_Kd. q_t is the head's distribution over row t's candidates, zero
 * elsewhere (the pointwise residual, as the page's exactness claim requires).
 * Draws: the smallest vocabulary id v whose running sum of weights exceeds
 * u * (total weight), in vocabulary order.
 *   p         B x (Kd + 1) x n fp32: target distributions (rows sum to 1).
 *   x         B x Kd int32: drafted tokens; each must be a candidate of its row.
 *   cand_ids, cand_q  B x Kd x K: the drafter's candidates and q (1 <= K <= 4096).
 *   r         B x Kd fp32 accept uniforms; u  B x (Kd + 1) fp32 draw uniforms.
 *   out_tokens  B x (Kd + 1) int32: the accepted drafts, then the replacement
 *             or bonus token, then -1; out_count  B int32: drafts accepted
 *             (0..Kd), or -1 when a drafted token is not a candidate (also
 *             recorded as LMHEAD_ERR_DEVICE_CHECK, see lmhead_last_device_error).
 * One 8-CTA thread-block cluster per chain (the vocabulary split over its CTAs); Kd may be
 * 0 (bonus draw only).
 */
int lmhead_verify_chain(const float* p, int64_t n, int B, int Kd, const int32_t* x,
                        const int32_t* cand_ids, const float* cand_q, int K, const float* r,
                        const float* u, int32_t* out_tokens, int32_t* out_count,
                        lmhead_stream stream);

/*
 * Vocabulary-sharded local head, one shard of G (one GPU each). The EAGLE-4
 * notes' local Top-k ("A Local Top-k based variant") picks every tile's
 * candidates from that tile alone, so when the shuffled positions are split
 * into contiguous ranges of whole tiles the shards select independently and
 * the union of their candidates is the unsharded head's. Each shard gathers
 * its own candidates' rows; only the softmax spans the shards: every shard
 * reduces its candidates to (max, sum of exponentials) per row, the caller
 * exchanges those M x 2 floats (an all-gather), and lmhead_shard_softmax
 * finishes each shard's q. Offline, per shard holding positions [p0, p1):
 *   A_shard          n_shard x r bf16: rows p0.. of the shuffled A.
 *   token_ids_shard  n_shard int32: the vocabulary ids of those positions.
 *   W_shard          n_shard x d bf16: W_shard[i] = W[token_ids_shard[i]].
 *   row_of_id        n_vocab int32: the local row of each vocabulary id held
 *                    by this shard, -1 for the others.
 * B r x d and h M x d are replicated. T, k_tile, temperature as for
 * lmhead_two_stage in local mode; every shard but the last should hold a
 * multiple of T positions (otherwise its last tile is short, as at the end
 * of the head).
 *   out_ids     M x K_s int32 vocabulary ids (K_s = lmhead_candidate_count(
 *               LMHEAD_LOCAL, n_shard, T, k_tile)), tile order.
 *   out_logits  M x K_s fp32 exact W[id].h.
 *   out_stats   M x 2 fp32: (max_j logits/T, sum_j exp(logits/T - max)).
 * Workspace: lmhead_shard_workspace_size bytes, 256-byte aligned. Errors as
 * for lmhead_two_stage; token_ids_shard and row_of_id are required, and an
 * id whose row_of_id is -1 is a bad id (NaN logit, LMHEAD_ERR_DEVICE_CHECK).
 */
size_t lmhead_shard_workspace_size(int64_t n_shard, int d, int r, int M, int T, int k_tile);
int lmhead_shard_two_stage(const lmhead_bf16* W_shard, const lmhead_bf16* A_shard,
                           const lmhead_bf16* B, const lmhead_bf16* h,
                           const int32_t* token_ids_shard, const int32_t* row_of_id,
                           int64_t n_vocab, int64_t n_shard, int d, int r, int M, int T,
                           int k_tile, float temperature, int32_t* out_ids, float* out_logits,
                           float* out_stats, void* workspace, size_t workspace_bytes,
                           lmhead_stream stream);

/*
 * The draft distribution of one shard's candidates from every shard's stats:
 *   all_stats  G x M x 2 fp32 (the shards' out_stats, in any shard order).
 *   logits     M x K fp32 this shard's out_logits; out_q M x K fp32 (may
 *              alias logits): exp(logits/T - Mx) / Z with Mx the largest of
 *              the shards' maxima and Z = sum_g sum_g exp(max_g - Mx), so that
 *              the shards' q together are the softmax over all candidates.
 */
int lmhead_shard_softmax(const float* all_stats, int G, const float* logits, int M, int K,
                         float temperature, float* out_q, lmhead_stream stream);

/*
 * Test hook for the timeout path (the pages have no counterpart). Every wait
 * between the warp roles of the tensor-core kernels (the fused score + tile
 * top-k, the global path's score writeback, the dense and pruned heads) is
 * bounded by a budget of SM clock cycles, about a second by default; on
 * expiry the kernel records LMHEAD_ERR_TIMEOUT in the device error word,
 * waits for its own copies and MMAs in flight, frees its tensor memory and
 * returns, leaving that call's outputs undefined and the context usable.
 *   cycles > 0   sets the budget for kernels launched from now on;
 *   cycles == 0  makes each such wait test its barrier once and give up
 *                unless it is already complete (a call then almost surely
 *                times out: this is how the tests exercise the path);
 *   cycles < 0   restores the default.
 * Process-wide, read at launch (a captured CUDA graph keeps the budget of its
 * capture). Returns the previous budget. Not meant for production use.
 */
int64_t lmhead_debug_set_wait_cycles(int64_t cycles);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word. Returns LMHEAD_OK, LMHEAD_ERR_DEVICE_CHECK, LMHEAD_ERR_TIMEOUT, or
 * LMHEAD_ERR_CUDA if the synchronisation itself failed.
 */
int lmhead_last_device_error(lmhead_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* LMHEAD_H */
