// Internal launch functions of liblmhead (host side). Each returns a
// cudaError_t from the launch; arguments have been validated by api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lmhead {

typedef uint16_t bf16_t;

// Largest k_tile handled by the fused score + tile top-k kernels.
constexpr int kFusedMaxKTile = 32;
// Largest selection budget of the radix select (global C or k_tile).
constexpr int kSelectMaxK = 4096;

// K1: u = bf16(B h), fp32 accumulation. Tensor cores (cluster split over d)
// up to d = kProjTcMaxD, CUDA cores beyond. Also zeroes `zero_ints` ints at
// `zero_ptr` (tickets of the fused kernels that follow), if non-null.
constexpr int kProjTcMaxD = 5120;
cudaError_t launch_project_u(const bf16_t* B, const bf16_t* h, int d, int r, int M, bf16_t* u,
                             int* zero_ptr, int zero_ints, cudaStream_t s);

// K4 (CUDA cores): fused tile scores + per-tile top-k_tile, no score writeback.
// For M <= kLocalGemvMaxM and tiles of 32..256 rows dividing 256 (k_tile <= 8,
// r = 256 or 512) it runs the warp-per-row GEMV kernel (measured faster than
// the tensor-core kernel up to four hidden vectors; at five to eight the
// GEMV's registers leave too few warps per SM).
constexpr int kLocalGemvMaxM = 4;  // compiled up to; gemv_max_m() is the limit in use
int gemv_max_m();
bool local_topk_gemv_supported(int M, int r, int T, int k_tile);
// The GEMV score writeback (below): one or two hidden vectors.
bool scores_gemv_supported(int M, int r);
// The same GEMV kernel writing every score to S (M x n fp32 by position)
// instead of selecting: the global path's writeback for one or two hidden
// vectors at r = 256 or 512. hist0 != nullptr: it also adds the counts of the
// scores' top kSelectHistBits order bits of hidden vector m into
// hist0 + m * hist0_stride (kSelectHistBins ints; the multi-CTA selection's
// first histogram).
cudaError_t launch_scores_gemv(const bf16_t* A, const bf16_t* u, int64_t n, int r, int M, float* S,
                               cudaStream_t s, int* hist0 = nullptr, int hist0_stride = 0);
// ready: the gather's ready counters (GEMV kernel only; may be nullptr).
cudaError_t launch_local_topk_fma(const bf16_t* A, const bf16_t* u, const int32_t* token_ids,
                                  int64_t n, int r, int M, int T, int k_tile, int32_t* out_ids,
                                  float* out_scores, cudaStream_t s, int* ready = nullptr);

// K4 (tensor cores): tcgen05 MMA with TMA-staged A chunks, persistent CTAs.
constexpr int kLocalTcMaxR = 512;
constexpr int kLocalTcMaxCtas = 256;
bool local_topk_tc_supported(int r, int T, int k_tile);
// workspace bytes for the split-tile partial lists; tile tickets are counted separately
size_t local_topk_tc_scratch_bytes(int64_t n, int M, int T);
int local_topk_tc_tickets(int64_t n, int M, int T);
// ready: the gather's ready counters (tiles of a multiple of 128 rows only;
// may be nullptr).
cudaError_t launch_local_topk_tc(const bf16_t* A, const bf16_t* u, const int32_t* token_ids,
                                 int64_t n, int r, int M, int T, int k_tile, int32_t* out_ids,
                                 float* out_scores, void* partials, int* tile_tickets, int* err,
                                 cudaStream_t s, int* ready = nullptr);

// K3: per row m, per segment of `seg_len` positions, exact top-k of S by
// (score desc, vocabulary id asc). k <= kSelectMaxK.
cudaError_t launch_segment_topk(const float* S, const int32_t* token_ids, int64_t n, int M,
                                int64_t seg_len, int k, int32_t* out_ids, float* out_scores,
                                int* err, cudaStream_t s);

// Overlap of the gather with the fused scoring kernel (local mode): the
// scoring kernel counts, per block of kReadyTiles consecutive tiles, the
// hidden rows whose ids of the block's tiles it has written (ready[b] reaches
// tiles_in_block * M when block b is complete); the gather waits on those
// counters instead of on the scoring kernel's completion. The counters, and
// after them one stop word that the scoring kernel sets if it aborts, live in
// the workspace's ticket area, zeroed by the projection kernel every call.
constexpr int kReadyTiles = 16;
__host__ __device__ inline int ready_blocks(int64_t tiles) {
  return (int)((tiles + kReadyTiles - 1) / kReadyTiles);
}
inline int ready_words(int64_t tiles) { return ready_blocks(tiles) + 1; }  // counters + stop

// K3 for long rows and few of them (global Top-k, several CTAs per row):
// `zero` holds row_select_multi_ints(M) ints that are zero on entry (the
// projection kernel zeroes them), `scratch` row_select_multi_bytes(M, k)
// bytes (no initial value). Same result and order as launch_segment_topk with
// one segment per row. The first histogram of row m (kSelectHistBins counts of
// the scores' top kSelectHistBits order bits, float_key(score) >> 20) is at
// zero + row_select_multi_hist0(m); hist0_filled: the score writeback has
// counted it already.
constexpr int kSelectHistBits = 12;
constexpr int kSelectHistBins = 1 << kSelectHistBits;
bool row_select_multi(int64_t n, int M, int k);
int row_select_multi_ints(int M);
int row_select_multi_hist0(int m);
size_t row_select_multi_bytes(int M, int k);
cudaError_t launch_row_select_multi(const float* S, const int32_t* token_ids, int64_t n, int M,
                                    int k, int32_t* out_ids, float* out_scores, int* zero,
                                    void* scratch, bool hist0_filled, cudaStream_t s);

// K5 (+K6 fused when q != nullptr): L[m,j] = W[ids[m,j]] . h[m]; q = softmax.
// `tickets` (M ints, zero on entry, left zero on exit) enable the fusion.
// span > 0: warps take the candidates in blocks of `span` columns (all rows
// of a block together) instead of row by row; see the kernel.
// ready != nullptr: wait on the scoring kernel's ready counters (tiles of
// k_tile columns, `tiles` in all) instead of on its completion.
// row_of_id != nullptr: W holds n_rows rows, the row of vocabulary id i being
// row_of_id[i] (a vocabulary shard; ids outside it are bad ids).
cudaError_t launch_gather_logits(const bf16_t* W, const bf16_t* h, const int32_t* ids, int64_t n,
                                 int d, int M, int K, float* logits, float* q, float inv_temp,
                                 int* tickets, int* err, cudaStream_t s, int span = 0,
                                 const int* ready = nullptr, int k_tile = 0, int64_t tiles = 0,
                                 const int32_t* row_of_id = nullptr, int64_t n_rows = 0);

// Vocabulary shards: per row of L (M x K), stats[m] = (max_j L/T, sum_j
// exp(L/T - max)); and q of one shard's candidates from all G shards' stats
// (G x M x 2, any order): q = exp(L/T - Mx) / Z, Mx = max of the maxima,
// Z = sum_g sum_g exp(max_g - Mx).
cudaError_t launch_row_stats(const float* L, int M, int K, float inv_temp, float* stats,
                             cudaStream_t s);
cudaError_t launch_shard_softmax(const float* all_stats, int G, const float* L, int M, int K,
                                 float inv_temp, float* q, cudaStream_t s);

// K6 standalone: row softmax of an M x K matrix (any K).
cudaError_t launch_row_softmax(const float* L, int M, int64_t K, float inv_temp, float* q,
                               cudaStream_t s);

// Tensor-core row products (rows_tc.cu): out[m * ldo + j] = X[j] . Y[m] for
// every row j of X (n x kdim) and hidden vector m of Y (M x kdim); any M
// (blocks of kRowsTcMaxN). Used for the dense and pruned heads and the
// global path's score writeback.
constexpr int kRowsTcMaxN = 256;
cudaError_t launch_rows_dense_tc(const bf16_t* X, int64_t n, int kdim, const bf16_t* Y, int M,
                                 float* out, int64_t ldo, int* err, cudaStream_t s);

// Cluster-level route: ids[m, j*group + t] = groups[m, j]*group + t (M x G*group).
cudaError_t launch_expand_groups(const int32_t* groups, int M, int G, int group, int64_t ngroups,
                                 int32_t* ids, int* err, cudaStream_t s);

// K8: per row, the k_sel (<= kDraftMaxK) largest q (ties: smaller id) with
// value parent * q, and optionally a Gumbel-max draw from q (uniforms M x K).
constexpr int kDraftMaxK = 16;
cudaError_t launch_draft_select(const float* q, const int32_t* ids, int M, int K, int k_sel,
                                const float* parent_value, const float* uniforms, int32_t* top_ids,
                                float* top_q, float* top_value, int32_t* sample_id,
                                float* sample_q, cudaStream_t s);
// K9: chain verification of B chains of Kd drafted tokens against dense
// target rows p (B x (Kd + 1) x n), candidate lists B x Kd x K.
cudaError_t launch_verify_chain(const float* p, int64_t n, int B, int Kd, const int32_t* x,
                                const int32_t* cand_ids, const float* cand_q, int K, const float* r,
                                const float* u, int32_t* out_tokens, int32_t* out_count, int* err,
                                cudaStream_t s);

int* device_error_word();  // this device's error word (nullptr on failure)
// Budget (SM cycles) of the tensor-core kernels' role waits; tc::kWaitCycles
// unless lmhead_debug_set_wait_cycles changed it.
long long role_wait_cycles();

// TMA map of a rows x cols bf16 row-major matrix: box_rows x box_cols
// (box_cols * 2 == 128 bytes), 128-byte swizzle, zero fill out of bounds.
bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows, uint32_t box_cols);
int sm_count();  // SMs of the current device (cached)

}  // namespace lmhead
