// The C ABI of liblmhead (include/lmhead.h): host-side validation, workspace
// carve-up and the launch sequence of each entry point. No entry point
// allocates device memory or synchronises (except lmhead_last_device_error).
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "lmhead.h"
#include "tc_util.cuh"

namespace lmhead {

__device__ int g_device_error;

// Role-wait budget of the tensor-core kernels (-1: the default).
static std::atomic<long long> g_role_wait{-1};

long long role_wait_cycles() {
  const long long v = g_role_wait.load(std::memory_order_relaxed);
  return v < 0 ? tc::kWaitCycles : v;
}

int* device_error_word() {
  static int* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(p);
  }
  return cache[dev];
}

namespace {

constexpr int kMaxR = 2048;
constexpr int kMaxD = 65536;
constexpr int kMaxM = 65535 * 8;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t u = 0, tickets = 0, scores = 0, partials = 0, select = 0, total = 0;
  // ints at `tickets` zeroed by K1: row tickets, the scoring kernel's tile
  // tickets, the gather's ready counters (n_ready, 0 when not used), then the
  // multi-CTA global selection's row states and histograms (at ms_at)
  int n_tickets = 0, ready_at = 0, n_ready = 0, ms_at = 0;
  bool ms = false;  // global Top-C through several CTAs per row
};

// The fused scoring kernel of local mode: up to four hidden vectors take the
// warp-per-row GEMV kernel, more the tensor cores, where each applies.
bool use_tc(int mode, int r, int T, int k_tile, int M) {
  return mode == LMHEAD_LOCAL && local_topk_tc_supported(r, T, k_tile) &&
         !local_topk_gemv_supported(M, r, T, k_tile);
}

bool needs_score_buffer(int mode, int k_tile) {
  return mode == LMHEAD_GLOBAL || k_tile > kFusedMaxKTile;
}

// The gather waits on per-block ready counters of the fused scoring kernel
// (instead of its completion) where that kernel publishes them: the dynamic
// tensor-core kernel (tiles of a multiple of 128 rows) and the GEMV kernel.
// Measured on the 128256-row head: 2-4 us faster per call at 16-64 hidden
// vectors, no gain at one, 1.4 us slower at eight, so it is used above eight.
// LMHEAD_OVERLAP=0 turns it off, =2 uses it at every M (measurements only).
constexpr int kOverlapMinM = 9;

// Up to this many hidden vectors the softmax can run inside the gather: the
// warp that finishes a row's last candidate (per-row ticket, no waiting)
// normalises the row, saving a launch. Measured on the 128256-row head it is
// slower (one hidden vector 25.4 -> 35.7 us, eight 47.7 -> 59.9 us: every
// gather warp waits on its ticket's round trip and one warp normalises the
// row), so it is off; LMHEAD_FUSED_SOFTMAX_M sets the limit (measurements).
int fused_softmax_max_m() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LMHEAD_FUSED_SOFTMAX_M");
    v = e ? atoi(e) : 0;
  }
  return v;
}
int overlap_setting() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LMHEAD_OVERLAP");
    v = e ? atoi(e) : 1;
  }
  return v;
}

bool gather_overlaps(int mode, int r, int T, int k_tile, int M) {
  const int ov = overlap_setting();
  if (ov == 0 || (ov == 1 && M < kOverlapMinM)) return false;
  if (mode != LMHEAD_LOCAL || needs_score_buffer(mode, k_tile)) return false;
  if (use_tc(mode, r, T, k_tile, M)) return T % 128 == 0;
  return local_topk_gemv_supported(M, r, T, k_tile);
}

// Columns per block of the warp gather's candidate order in local mode (a
// block of tiles); LMHEAD_GATHER_SPAN overrides it (0 = row by row).
int gather_span(int k_tile) {
  static int v = -2;
  if (v == -2) {
    const char* e = getenv("LMHEAD_GATHER_SPAN");
    v = e ? atoi(e) : -1;
  }
  return v >= 0 ? v : 16 * k_tile;
}

Layout layout_for(int mode, int64_t n, int d, int r, int M, int C_or_tile, int k_tile) {
  Layout L;
  size_t off = 0;
  L.u = off;
  off = round_up(off + (size_t)M * r * sizeof(bf16_t), 256);
  L.tickets = off;
  const bool tc = use_tc(mode, r, C_or_tile, k_tile, M);
  L.ready_at = M + (tc ? local_topk_tc_tickets(n, M, C_or_tile) : 0);
  L.n_ready = gather_overlaps(mode, r, C_or_tile, k_tile, M)
                  ? ready_words((n + C_or_tile - 1) / C_or_tile) : 0;
  L.ms = mode == LMHEAD_GLOBAL && row_select_multi(n, M, C_or_tile);
  L.ms_at = (int)round_up((size_t)(L.ready_at + L.n_ready), 4);  // 16-byte aligned
  L.n_tickets = L.ms ? L.ms_at + row_select_multi_ints(M) : L.ready_at + L.n_ready;
  off = round_up(off + (size_t)L.n_tickets * sizeof(int), 256);
  if (L.ms) {
    L.select = off;
    off = round_up(off + row_select_multi_bytes(M, C_or_tile), 256);
  }
  if (tc) {
    L.partials = off;
    off = round_up(off + local_topk_tc_scratch_bytes(n, M, C_or_tile), 256);
  }
  if (needs_score_buffer(mode, k_tile)) {
    L.scores = off;
    off = round_up(off + (size_t)M * (size_t)n * sizeof(float), 256);
  }
  L.total = off;
  return L;
}

int64_t candidate_count(int mode, int64_t n, int C_or_tile, int k_tile) {
  if (n < 1 || n > INT32_MAX) return LMHEAD_ERR_SHAPE;
  if (mode == LMHEAD_GLOBAL) {
    if (C_or_tile < 1 || C_or_tile > n) return LMHEAD_ERR_SHAPE;
    return C_or_tile;
  }
  if (mode == LMHEAD_LOCAL) {
    if (C_or_tile < 1 || k_tile < 1 || k_tile > C_or_tile) return LMHEAD_ERR_SHAPE;
    const int64_t T = C_or_tile;
    const int64_t full = n / T, tail = n - full * T;
    return full * k_tile + (tail ? (tail < k_tile ? tail : k_tile) : 0);
  }
  return LMHEAD_ERR_SHAPE;
}

int check_select(int mode, int64_t n, int d, int r, int M, int C_or_tile, int k_tile) {
  if (d < 8 || d % 8 || d > kMaxD || r < 8 || r % 8 || r > kMaxR) return LMHEAD_ERR_SHAPE;
  if (M < 1 || M > kMaxM) return LMHEAD_ERR_SHAPE;
  const int64_t K = candidate_count(mode, n, C_or_tile, k_tile);
  if (K < 0) return (int)K;
  if (mode == LMHEAD_GLOBAL && C_or_tile > kSelectMaxK) return LMHEAD_ERR_UNSUPPORTED;
  if (mode == LMHEAD_LOCAL && k_tile > kSelectMaxK) return LMHEAD_ERR_UNSUPPORTED;
  if ((int64_t)M * K > INT32_MAX) return LMHEAD_ERR_SHAPE;
  return LMHEAD_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LMHEAD_OK : LMHEAD_ERR_CUDA; }

// Optional timing marks between launches (lmhead_two_stage_profiled).
struct Marks {
  void* const* events = nullptr;
  int n = 0;
  int next = 0;
  cudaError_t mark(cudaStream_t s) {
    if (next < n && events && events[next]) {
      // inside a stream capture the record must be external to stay observable
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      cudaError_t e = cudaStreamIsCapturing(s, &cs);
      if (e != cudaSuccess) return e;
      e = cs == cudaStreamCaptureStatusActive
              ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[next]), s,
                                         cudaEventRecordExternal)
              : cudaEventRecord(static_cast<cudaEvent_t>(events[next]), s);
      ++next;
      return e;
    }
    ++next;
    return cudaSuccess;
  }
};

// Stage 1 on validated arguments; u lives in the workspace.
// ready: the gather's counters when it overlaps the scoring kernel, else nullptr.
int run_select(int mode, const bf16_t* A, const bf16_t* B, const bf16_t* h,
               const int32_t* token_ids, int64_t n, int d, int r, int M, int C_or_tile,
               int k_tile, int32_t* out_ids, float* out_scores, char* ws, const Layout& L,
               bool zero_tickets, Marks& mk, cudaStream_t s, int* ready = nullptr) {
  bf16_t* u = reinterpret_cast<bf16_t*>(ws + L.u);
  int* tickets = reinterpret_cast<int*>(ws + L.tickets);
  if (mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
  const bool tc = use_tc(mode, r, C_or_tile, k_tile, M);
  const bool zero = zero_tickets || tc || ready || L.ms;
  cudaError_t e = launch_project_u(B, h, d, r, M, u, zero ? tickets : nullptr,
                                   zero ? L.n_tickets : 0, s);
  if (e != cudaSuccess || mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
  if (tc) {
    e = launch_local_topk_tc(A, u, token_ids, n, r, M, C_or_tile, k_tile, out_ids, out_scores,
                             ws + L.partials, tickets + M, device_error_word(), s, ready);
    if (e != cudaSuccess || mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
    return LMHEAD_OK;
  }
  if (!needs_score_buffer(mode, k_tile)) {
    e = launch_local_topk_fma(A, u, token_ids, n, r, M, C_or_tile, k_tile, out_ids, out_scores, s,
                              ready);
    if (e != cudaSuccess || mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
    return LMHEAD_OK;
  }
  // score writeback: the GEMV kernel for one or two hidden vectors, else the
  // tensor-core row products
  // (the GEMV form also counts the multi-CTA selection's first histogram)
  float* S = reinterpret_cast<float*>(ws + L.scores);
  const bool gemv = scores_gemv_supported(M, r);
  int* ms_zero = L.ms ? tickets + L.ms_at : nullptr;
  e = gemv ? launch_scores_gemv(A, u, n, r, M, S, s,
                                ms_zero ? ms_zero + row_select_multi_hist0(0) : nullptr,
                                row_select_multi_hist0(1) - row_select_multi_hist0(0))
           : launch_rows_dense_tc(A, n, r, u, M, S, n, device_error_word(), s);
  if (e != cudaSuccess || mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
  const int64_t seg = mode == LMHEAD_GLOBAL ? n : C_or_tile;
  const int k = mode == LMHEAD_GLOBAL ? C_or_tile : k_tile;
  if (L.ms)
    e = launch_row_select_multi(S, token_ids, n, M, k, out_ids, out_scores, ms_zero,
                                ws + L.select, gemv, s);
  else
    e = launch_segment_topk(S, token_ids, n, M, seg, k, out_ids, out_scores, device_error_word(),
                            s);
  if (e != cudaSuccess || mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
  return LMHEAD_OK;
}

// Cluster-level route: the local selection with one candidate per group
// (tile = group, k_tile = 1) leaves every group's best score in the
// workspace; the segment top-k picks the G best groups from those.
struct ClusterLayout {
  Layout sel;
  size_t best_ids = 0, gscores = 0, total = 0;
};

int64_t cluster_count(int64_t n, int group, int G) {
  if (n < 1 || n > INT32_MAX || group < 1 || n % group) return LMHEAD_ERR_SHAPE;
  if (G < 1 || G > n / group) return LMHEAD_ERR_SHAPE;
  return (int64_t)G * group;
}

int check_cluster(int64_t n, int d, int r, int M, int group, int G) {
  const int64_t K = cluster_count(n, group, G);
  if (K < 0) return (int)K;
  const int st = check_select(LMHEAD_LOCAL, n, d, r, M, group, 1);
  if (st != LMHEAD_OK) return st;
  if (G > kSelectMaxK) return LMHEAD_ERR_UNSUPPORTED;
  if ((int64_t)M * K > INT32_MAX || (int64_t)M * (n / group) > INT32_MAX) return LMHEAD_ERR_SHAPE;
  return LMHEAD_OK;
}

ClusterLayout cluster_layout(int64_t n, int d, int r, int M, int group) {
  ClusterLayout C;
  C.sel = layout_for(LMHEAD_LOCAL, n, d, r, M, group, 1);
  const size_t cells = (size_t)M * (size_t)(n / group);
  C.best_ids = round_up(C.sel.total, 256);
  C.gscores = round_up(C.best_ids + cells * sizeof(int32_t), 256);
  C.total = round_up(C.gscores + cells * sizeof(float), 256);
  return C;
}

// Stages of a call (each one timing mark): projection, scoring, selection
// when the mode needs one (the multi-CTA global selection launches seven
// kernels inside its stage), gather, softmax.
int launches_for(int mode, int k_tile) { return needs_score_buffer(mode, k_tile) ? 5 : 4; }

bool valid_temperature(float t) { return t > 0.f && isfinite(t); }

}  // namespace
}  // namespace lmhead

using namespace lmhead;

extern "C" {

int lmhead_version(void) { return 100; }

const char* lmhead_status_string(int status) {
  switch (status) {
    case LMHEAD_OK: return "ok";
    case LMHEAD_ERR_NULL: return "null pointer argument";
    case LMHEAD_ERR_SHAPE: return "invalid size argument";
    case LMHEAD_ERR_ALIGN: return "pointer not 16-byte aligned";
    case LMHEAD_ERR_WORKSPACE: return "workspace missing or too small";
    case LMHEAD_ERR_UNSUPPORTED: return "unsupported configuration";
    case LMHEAD_ERR_CUDA: return "CUDA error";
    case LMHEAD_ERR_DEVICE_CHECK: return "device-side check failed (e.g. id out of range)";
    case LMHEAD_ERR_TIMEOUT: return "device-side bounded wait timed out";
    default: return "unknown status";
  }
}

int64_t lmhead_candidate_count(int mode, int64_t n, int C_or_tile, int k_tile) {
  return candidate_count(mode, n, C_or_tile, k_tile);
}

size_t lmhead_workspace_size(int mode, int64_t n, int d, int r, int M, int C_or_tile,
                             int k_tile) {
  if (check_select(mode, n, d, r, M, C_or_tile, k_tile) != LMHEAD_OK) return 0;
  return layout_for(mode, n, d, r, M, C_or_tile, k_tile).total;
}

int lmhead_project_u(const lmhead_bf16* B, const lmhead_bf16* h, int d, int r, int M,
                     lmhead_bf16* u, lmhead_stream stream) {
  if (!B || !h || !u) return LMHEAD_ERR_NULL;
  if (d < 8 || d % 8 || d > kMaxD || r < 1 || r > 65535 * 8 || M < 1 || M > kMaxM)
    return LMHEAD_ERR_SHAPE;
  if (!aligned16(B) || !aligned16(h)) return LMHEAD_ERR_ALIGN;
  return cuda_status(launch_project_u(B, h, d, r, M, u, nullptr, 0, (cudaStream_t)stream));
}

int lmhead_lowrank_score_topk(int mode, const lmhead_bf16* A, const lmhead_bf16* B,
                              const lmhead_bf16* h, const int32_t* token_ids, int64_t n, int d,
                              int r, int M, int C_or_tile, int k_tile, int32_t* out_ids,
                              float* out_scores, void* workspace, size_t workspace_bytes,
                              lmhead_stream stream) {
  if (!A || !B || !h || !out_ids) return LMHEAD_ERR_NULL;
  if (mode == LMHEAD_GLOBAL) k_tile = 0;
  int st = check_select(mode, n, d, r, M, C_or_tile, k_tile);
  if (st != LMHEAD_OK) return st;
  if (!aligned16(A) || !aligned16(B) || !aligned16(h) || (token_ids && !aligned16(token_ids)) ||
      !aligned16(out_ids) || (out_scores && !aligned16(out_scores)))
    return LMHEAD_ERR_ALIGN;
  const Layout L = layout_for(mode, n, d, r, M, C_or_tile, k_tile);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return LMHEAD_ERR_WORKSPACE;
  Marks none;
  return run_select(mode, A, B, h, token_ids, n, d, r, M, C_or_tile, k_tile, out_ids, out_scores,
                    static_cast<char*>(workspace), L, false, none, (cudaStream_t)stream);
}

int lmhead_gather_logits(const lmhead_bf16* W, const lmhead_bf16* h, const int32_t* ids,
                         int64_t n, int d, int M, int K, float* out_logits,
                         lmhead_stream stream) {
  if (!W || !h || !ids || !out_logits) return LMHEAD_ERR_NULL;
  if (n < 1 || n > INT32_MAX || d < 8 || d % 8 || d > kMaxD || M < 1 || K < 1 ||
      (int64_t)M * K > INT32_MAX)
    return LMHEAD_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(h)) return LMHEAD_ERR_ALIGN;
  return cuda_status(launch_gather_logits(W, h, ids, n, d, M, K, out_logits, nullptr, 1.f,
                                          nullptr, device_error_word(), (cudaStream_t)stream));
}

int lmhead_candidate_softmax(const float* logits, int M, int K, float temperature, float* out_q,
                             lmhead_stream stream) {
  if (!logits || !out_q) return LMHEAD_ERR_NULL;
  if (M < 1 || K < 1 || M > 2147483647 / K) return LMHEAD_ERR_SHAPE;
  if (!valid_temperature(temperature)) return LMHEAD_ERR_SHAPE;
  return cuda_status(launch_row_softmax(logits, M, K, 1.f / temperature, out_q,
                                        (cudaStream_t)stream));
}

static int two_stage_impl(int mode, const lmhead_bf16* W, const lmhead_bf16* A,
                          const lmhead_bf16* B, const lmhead_bf16* h, const int32_t* token_ids,
                          int64_t n, int d, int r, int M, int C_or_tile, int k_tile,
                          float temperature, int32_t* out_ids, float* out_logits, float* out_q,
                          void* workspace, size_t workspace_bytes, Marks& mk,
                          lmhead_stream stream) {
  if (!W || !A || !B || !h || !out_ids || !out_logits || !out_q) return LMHEAD_ERR_NULL;
  if (mode == LMHEAD_GLOBAL) k_tile = 0;
  int st = check_select(mode, n, d, r, M, C_or_tile, k_tile);
  if (st != LMHEAD_OK) return st;
  if (!valid_temperature(temperature)) return LMHEAD_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(A) || !aligned16(B) || !aligned16(h) ||
      (token_ids && !aligned16(token_ids)) || !aligned16(out_ids))
    return LMHEAD_ERR_ALIGN;
  const Layout L = layout_for(mode, n, d, r, M, C_or_tile, k_tile);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return LMHEAD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;
  int* ready = L.n_ready ? reinterpret_cast<int*>(ws + L.tickets) + L.ready_at : nullptr;
  st = run_select(mode, A, B, h, token_ids, n, d, r, M, C_or_tile, k_tile, out_ids, nullptr, ws,
                  L, true, mk, s, ready);
  if (st != LMHEAD_OK) return st;
  const int K = (int)candidate_count(mode, n, C_or_tile, k_tile);
  // stage 2: exact logits of the candidates (block by block as the scoring
  // kernel finishes them, when it publishes ready counters), then their
  // softmax: inside the gather for a few hidden vectors (per-row tickets,
  // zeroed by K1), else one CTA per row
  const bool fuse = M <= fused_softmax_max_m();
  cudaError_t e = launch_gather_logits(W, h, out_ids, n, d, M, K, out_logits,
                                       fuse ? out_q : nullptr, 1.f / temperature,
                                       fuse ? reinterpret_cast<int*>(ws + L.tickets) : nullptr,
                                       device_error_word(), s,
                                       mode == LMHEAD_LOCAL ? gather_span(k_tile) : 0, ready,
                                       k_tile, (n + C_or_tile - 1) / C_or_tile);
  if (e != cudaSuccess || mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
  if (!fuse) e = launch_row_softmax(out_logits, M, K, 1.f / temperature, out_q, s);
  if (e != cudaSuccess || mk.mark(s) != cudaSuccess) return LMHEAD_ERR_CUDA;
  return LMHEAD_OK;
}

int lmhead_two_stage(int mode, const lmhead_bf16* W, const lmhead_bf16* A, const lmhead_bf16* B,
                     const lmhead_bf16* h, const int32_t* token_ids, int64_t n, int d, int r,
                     int M, int C_or_tile, int k_tile, float temperature, int32_t* out_ids,
                     float* out_logits, float* out_q, void* workspace, size_t workspace_bytes,
                     lmhead_stream stream) {
  Marks none;
  return two_stage_impl(mode, W, A, B, h, token_ids, n, d, r, M, C_or_tile, k_tile, temperature,
                        out_ids, out_logits, out_q, workspace, workspace_bytes, none, stream);
}

int lmhead_two_stage_profiled(int mode, const lmhead_bf16* W, const lmhead_bf16* A,
                              const lmhead_bf16* B, const lmhead_bf16* h,
                              const int32_t* token_ids, int64_t n, int d, int r, int M,
                              int C_or_tile, int k_tile, float temperature, int32_t* out_ids,
                              float* out_logits, float* out_q, void* workspace,
                              size_t workspace_bytes, void* const* events, int n_events,
                              lmhead_stream stream) {
  if (n_events < 0 || (n_events > 0 && !events)) return LMHEAD_ERR_NULL;
  Marks mk;
  mk.events = events;
  mk.n = n_events;
  return two_stage_impl(mode, W, A, B, h, token_ids, n, d, r, M, C_or_tile, k_tile, temperature,
                        out_ids, out_logits, out_q, workspace, workspace_bytes, mk, stream);
}

int lmhead_two_stage_launches(int mode, int k_tile) {
  if (mode == LMHEAD_GLOBAL) k_tile = 0;
  return launches_for(mode, k_tile);
}

int lmhead_dense_head(const lmhead_bf16* W, const lmhead_bf16* h, int64_t n, int d, int M,
                      float temperature, float* out_logits, float* out_q, lmhead_stream stream) {
  if (!W || !h || !out_logits) return LMHEAD_ERR_NULL;
  if (n < 1 || n > INT32_MAX || d < 8 || d % 8 || d > kMaxD || M < 1 || M > 65535)
    return LMHEAD_ERR_SHAPE;
  if (out_q && !valid_temperature(temperature)) return LMHEAD_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(h)) return LMHEAD_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_rows_dense_tc(W, n, d, h, M, out_logits, n, device_error_word(), s);
  if (e != cudaSuccess || !out_q) return cuda_status(e);
  return cuda_status(launch_row_softmax(out_logits, M, n, 1.f / temperature, out_q, s));
}

int lmhead_pruned_head(const lmhead_bf16* W_pruned, const lmhead_bf16* h, int n_keep, int d,
                       int M, float temperature, float* out_logits, float* out_q,
                       lmhead_stream stream) {
  return lmhead_dense_head(W_pruned, h, n_keep, d, M, temperature, out_logits, out_q, stream);
}

int lmhead_draft_select(const float* q, const int32_t* ids, int M, int K, int k_sel,
                        const float* parent_value, const float* uniforms, int32_t* out_top_ids,
                        float* out_top_q, float* out_top_value, int32_t* out_sample_id,
                        float* out_sample_q, lmhead_stream stream) {
  if (!q || !ids || !out_top_ids || !out_top_q) return LMHEAD_ERR_NULL;
  if (M < 1 || M > 2147483647 || K < 1 || K > kSelectMaxK || k_sel < 1 || k_sel > K ||
      k_sel > kDraftMaxK)
    return LMHEAD_ERR_SHAPE;
  return cuda_status(launch_draft_select(q, ids, M, K, k_sel, parent_value, uniforms, out_top_ids,
                                         out_top_q, out_top_value, uniforms ? out_sample_id : nullptr,
                                         uniforms ? out_sample_q : nullptr, (cudaStream_t)stream));
}

int lmhead_verify_chain(const float* p, int64_t n, int B, int Kd, const int32_t* x,
                        const int32_t* cand_ids, const float* cand_q, int K, const float* r,
                        const float* u, int32_t* out_tokens, int32_t* out_count,
                        lmhead_stream stream) {
  if (!p || !u || !out_tokens || !out_count) return LMHEAD_ERR_NULL;
  if (Kd > 0 && (!x || !cand_ids || !cand_q || !r)) return LMHEAD_ERR_NULL;
  if (n < 1 || n > INT32_MAX || B < 1 || B > 65535 || Kd < 0 || Kd > 1024 || K < 1 ||
      K > kSelectMaxK)
    return LMHEAD_ERR_SHAPE;
  return cuda_status(launch_verify_chain(p, n, B, Kd, x, cand_ids, cand_q, K, r, u, out_tokens,
                                         out_count, device_error_word(), (cudaStream_t)stream));
}

int64_t lmhead_cluster_candidate_count(int64_t n, int group, int G) {
  return cluster_count(n, group, G);
}

size_t lmhead_cluster_workspace_size(int64_t n, int d, int r, int M, int group, int G) {
  if (check_cluster(n, d, r, M, group, G) != LMHEAD_OK) return 0;
  return cluster_layout(n, d, r, M, group).total;
}

int lmhead_cluster_two_stage(const lmhead_bf16* W, const lmhead_bf16* A, const lmhead_bf16* B,
                             const lmhead_bf16* h, int64_t n, int d, int r, int M, int group,
                             int G, float temperature, int32_t* out_groups,
                             float* out_group_scores, int32_t* out_ids, float* out_logits,
                             float* out_q, void* workspace, size_t workspace_bytes,
                             lmhead_stream stream) {
  if (!W || !A || !B || !h || !out_groups || !out_ids || !out_logits || !out_q)
    return LMHEAD_ERR_NULL;
  int st = check_cluster(n, d, r, M, group, G);
  if (st != LMHEAD_OK) return st;
  if (!valid_temperature(temperature)) return LMHEAD_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(A) || !aligned16(B) || !aligned16(h)) return LMHEAD_ERR_ALIGN;
  const ClusterLayout C = cluster_layout(n, d, r, M, group);
  if (!workspace || workspace_bytes < C.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return LMHEAD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* best_ids = reinterpret_cast<int32_t*>(ws + C.best_ids);
  float* gscores = reinterpret_cast<float*>(ws + C.gscores);
  Marks none;
  // stage 1: every group's best low-rank score, then the G best groups
  st = run_select(LMHEAD_LOCAL, A, B, h, nullptr, n, d, r, M, group, 1, best_ids, gscores, ws,
                  C.sel, true, none, s);
  if (st != LMHEAD_OK) return st;
  const int64_t ngroups = n / group;
  const int K = G * group;
  cudaError_t e = launch_segment_topk(gscores, nullptr, ngroups, M, ngroups, G, out_groups,
                                      out_group_scores, device_error_word(), s);
  if (e == cudaSuccess)
    e = launch_expand_groups(out_groups, M, G, group, ngroups, out_ids, device_error_word(), s);
  // stage 2: exact logits of every row of the selected groups, then softmax
  if (e == cudaSuccess)
    e = launch_gather_logits(W, h, out_ids, n, d, M, K, out_logits, nullptr, 1.f, nullptr,
                             device_error_word(), s, 0);
  if (e == cudaSuccess) e = launch_row_softmax(out_logits, M, K, 1.f / temperature, out_q, s);
  return cuda_status(e);
}

size_t lmhead_shard_workspace_size(int64_t n_shard, int d, int r, int M, int T, int k_tile) {
  return lmhead_workspace_size(LMHEAD_LOCAL, n_shard, d, r, M, T, k_tile);
}

int lmhead_shard_two_stage(const lmhead_bf16* W_shard, const lmhead_bf16* A_shard,
                           const lmhead_bf16* B, const lmhead_bf16* h,
                           const int32_t* token_ids_shard, const int32_t* row_of_id,
                           int64_t n_vocab, int64_t n_shard, int d, int r, int M, int T,
                           int k_tile, float temperature, int32_t* out_ids, float* out_logits,
                           float* out_stats, void* workspace, size_t workspace_bytes,
                           lmhead_stream stream) {
  if (!W_shard || !A_shard || !B || !h || !token_ids_shard || !row_of_id || !out_ids ||
      !out_logits || !out_stats)
    return LMHEAD_ERR_NULL;
  if (n_vocab < 1 || n_vocab > INT32_MAX || n_shard > n_vocab) return LMHEAD_ERR_SHAPE;
  int st = check_select(LMHEAD_LOCAL, n_shard, d, r, M, T, k_tile);
  if (st != LMHEAD_OK) return st;
  if (!valid_temperature(temperature)) return LMHEAD_ERR_SHAPE;
  if (!aligned16(W_shard) || !aligned16(A_shard) || !aligned16(B) || !aligned16(h) ||
      !aligned16(token_ids_shard) || !aligned16(out_ids))
    return LMHEAD_ERR_ALIGN;
  const Layout L = layout_for(LMHEAD_LOCAL, n_shard, d, r, M, T, k_tile);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return LMHEAD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;
  int* ready = L.n_ready ? reinterpret_cast<int*>(ws + L.tickets) + L.ready_at : nullptr;
  Marks none;
  // stage 1 over the shard's positions; ids come out in vocabulary space
  st = run_select(LMHEAD_LOCAL, A_shard, B, h, token_ids_shard, n_shard, d, r, M, T, k_tile,
                  out_ids, nullptr, ws, L, true, none, s, ready);
  if (st != LMHEAD_OK) return st;
  const int K = (int)candidate_count(LMHEAD_LOCAL, n_shard, T, k_tile);
  // stage 2 on the shard's own rows of W (row_of_id: vocabulary id -> local row)
  cudaError_t e = launch_gather_logits(W_shard, h, out_ids, n_vocab, d, M, K, out_logits, nullptr,
                                       1.f, nullptr, device_error_word(), s, gather_span(k_tile),
                                       ready, k_tile, (n_shard + T - 1) / T, row_of_id, n_shard);
  if (e == cudaSuccess) e = launch_row_stats(out_logits, M, K, 1.f / temperature, out_stats, s);
  return cuda_status(e);
}

int lmhead_shard_softmax(const float* all_stats, int G, const float* logits, int M, int K,
                         float temperature, float* out_q, lmhead_stream stream) {
  if (!all_stats || !logits || !out_q) return LMHEAD_ERR_NULL;
  if (G < 1 || G > 65536 || M < 1 || K < 1 || M > 2147483647 / K) return LMHEAD_ERR_SHAPE;
  if (!valid_temperature(temperature)) return LMHEAD_ERR_SHAPE;
  return cuda_status(launch_shard_softmax(all_stats, G, logits, M, K, 1.f / temperature, out_q,
                                          (cudaStream_t)stream));
}

int64_t lmhead_debug_set_wait_cycles(int64_t cycles) {
  const long long prev = role_wait_cycles();
  g_role_wait.store(cycles < 0 ? -1 : (long long)cycles, std::memory_order_relaxed);
  return prev;
}

int lmhead_last_device_error(lmhead_stream stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LMHEAD_ERR_CUDA;
  int* p = device_error_word();
  if (!p) return LMHEAD_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LMHEAD_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return LMHEAD_ERR_CUDA;
  }
  if (v == kDevErrBadId) return LMHEAD_ERR_DEVICE_CHECK;
  if (v == kDevErrTimeout) return LMHEAD_ERR_TIMEOUT;
  return v == 0 ? LMHEAD_OK : LMHEAD_ERR_DEVICE_CHECK;
}

}  // extern "C"
