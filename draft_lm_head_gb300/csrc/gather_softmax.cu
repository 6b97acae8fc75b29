// Stage 2 (EAGLE-4 notes, "EAGLE Efficient LM Head"): gather the full head's
// rows of the candidates and recompute their exact logits with the original
// hidden states, logits = W[ids] @ h; then the draft distribution q =
// softmax(logits / temperature) over each row's candidates.
//
// K5: one warp per candidate (m, j). The W row (d bf16, 0.5-10 KB) is read
// once with 16-byte non-allocating loads; h[m] comes through L1 (all of a
// row's candidates share it). fp32 accumulation, butterfly reduction.
// K6 fused: the warp that finishes a row's last candidate (a per-row atomic
// ticket, no waiting) computes that row's softmax and resets the ticket.
// K6 standalone: one CTA per row, any row length.
#include <math.h>
#include <stdlib.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace lmhead {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kGatherMinCtas = 6;  // CTAs per SM the register budget is sized for
constexpr int kSmallGatherPerSm = 2 * kWarpsPerCta;  // candidates per SM of a "small" gather

// Online max/sum over a row, lane-strided, then combined across the warp.
__device__ __forceinline__ void warp_row_softmax(const float* L, float* q, int K,
                                                 float inv_temp) {
  const int lane = threadIdx.x & 31;
  float mx = -INFINITY, sum = 0.f;
  for (int j = lane; j < K; j += 32) {
    const float z = __ldcg(L + j) * inv_temp;
    if (z > mx) {
      sum = sum * __expf(mx - z) + 1.f;
      mx = z;
    } else {
      sum += __expf(z - mx);
    }
  }
  const float gmx = warp_max(mx);
  sum = (mx == -INFINITY) ? 0.f : sum * __expf(mx - gmx);
  const float inv = 1.f / warp_sum(sum);
  for (int j = lane; j < K; j += 32) q[j] = __expf(__ldcg(L + j) * inv_temp - gmx) * inv;
}

// warp c -> candidate (m, j), returned as the flat index m * K + j.
// Row-major, or by blocks of `span` columns: every row's candidates of one
// block are taken together, so a W row that several rows picked is requested
// several times within a short window (the repeats hit L2), while consecutive
// warps still share h[m].
// (M * K < 2^31 is checked on the host, so 32-bit arithmetic suffices.)
__device__ __forceinline__ uint32_t candidate_of(uint32_t c, uint32_t M, uint32_t K, uint32_t span,
                                                 int* m_out) {
  if (span > 0 && span < K) {
    const uint32_t full = K / span, cut = full * M * span;
    uint32_t j0, w, r;
    if (c < cut) {
      const uint32_t b = c / (M * span);
      r = c - b * M * span;
      j0 = b * span;
      w = span;
    } else {
      r = c - cut;
      j0 = full * span;
      w = K - j0;
    }
    const uint32_t m = r / w;
    *m_out = (int)m;
    return m * K + j0 + (r - m * w);
  }
  *m_out = (int)(c / K);
  return c;
}

// WPC warps per CTA, UNR 16-byte loads of W in flight per lane, at least
// MINB CTAs per SM. When SH and all warps of the CTA share one hidden vector,
// h[m] is staged in shared memory once (before waiting for the ids: h is an
// input), so only the W row streams through L1 per candidate. Measured on the
// n=128256, d=4096, M=64 workload: 8 warps, 4 loads, 6 CTAs per SM (48 warps)
// with staging is the fastest of the shapes tried (4-16 warps, 2-16 loads).
// FUSED: the softmax-in-gather path (q, tickets) is compiled in; ROWMAP: ids
// are mapped to W rows through row_of_id (a vocabulary shard); OVL: the
// warps wait on the scoring kernel's ready counters. Without them (the usual
// case) the kernel needs fewer registers.
template <int WPC, int UNR, int MINB, bool SH, bool FUSED, bool ROWMAP, bool OVL>
__global__ void __launch_bounds__(WPC * 32, MINB)
gather_logits_kernel(const bf16_t* __restrict__ W, const bf16_t* __restrict__ h,
                     const int32_t* __restrict__ ids, int64_t n, int d, int M, int K,
                     int span, float* __restrict__ logits, float* __restrict__ q,
                     float inv_temp, int* __restrict__ tickets, int* __restrict__ err,
                     const int* __restrict__ ready, int k_tile, int tiles,
                     const int32_t* __restrict__ row_of_id, int64_t n_rows) {
  extern __shared__ uint4 h_s[];
  const int lane = threadIdx.x & 31;
  const uint32_t MK = (uint32_t)M * (uint32_t)K;
  const uint32_t c = blockIdx.x * WPC + (threadIdx.x >> 5);
  const int nvec = d >> 3;
  pdl_trigger();
  bool staged = false;
  if (SH) {
    const uint32_t cb = blockIdx.x * WPC;
    const uint32_t ce = cb + WPC - 1 < MK ? cb + WPC - 1 : MK - 1;
    int mb, me;
    candidate_of(cb, M, K, span, &mb);
    candidate_of(ce, M, K, span, &me);
    staged = mb == me;  // the same for every thread of the CTA
    if (staged) {
      const uint4* hrow = reinterpret_cast<const uint4*>(h + (size_t)mb * d);
      for (int v = threadIdx.x; v < nvec; v += WPC * 32) h_s[v] = __ldg(hrow + v);
      cta_sync();
    }
  }
  // ids come from the previous kernel: wait for all of it, or (ready) only
  // for the block of tiles that holds this warp's candidate
  if (!OVL) pdl_wait();
  if (c >= MK) return;
  int m;
  const uint32_t flat = candidate_of(c, M, K, span, &m);
  if (OVL) {
    if (lane == 0) {
      const int b = (int)((flat - (uint32_t)m * (uint32_t)K) / (uint32_t)k_tile) / kReadyTiles;
      wait_count(ready + b, min(kReadyTiles, tiles - b * kReadyTiles) * M,
                 ready + ready_blocks(tiles), err);
    }
    __syncwarp();
  }
  // overlapping the scoring kernel, ids may be written while this CTA runs:
  // read them from L2; otherwise through L1, where a CTA's warps share a line
  const int32_t id = OVL ? __ldcg(ids + flat) : __ldg(ids + flat);
  // the W row of the id: the id itself, or (a vocabulary shard) its local row
  int64_t row = id;
  bool bad = id < 0 || (int64_t)id >= n;
  if (ROWMAP && !bad) {
    row = __ldg(row_of_id + id);
    bad = row < 0 || row >= n_rows;
  }
  float s;
  if (bad) {
    if (lane == 0) record_error(err, kDevErrBadId);
    s = __int_as_float(0x7FC00000);  // NaN
  } else {
    const uint4* wrow = reinterpret_cast<const uint4*>(W + (size_t)row * d);
    const uint4* hrow = reinterpret_cast<const uint4*>(h + (size_t)m * d);
    float acc = 0.f;
    if (staged) {
#pragma unroll UNR
      for (int v = lane; v < nvec; v += 32) acc += dot8(ldg_nc_v4(wrow + v), h_s[v]);
    } else {
#pragma unroll UNR
      for (int v = lane; v < nvec; v += 32) acc += dot8(ldg_nc_v4(wrow + v), __ldg(hrow + v));
    }
    s = warp_sum(acc);
  }
  if (lane == 0) logits[flat] = s;
  if constexpr (!FUSED) return;
  if (q == nullptr) return;
  int ticket = 0;
  if (lane == 0) {
    __threadfence();
    ticket = atomicAdd(tickets + m, 1);
  }
  ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
  if (ticket != K - 1) return;
  __threadfence();
  warp_row_softmax(logits + (size_t)m * K, q + (size_t)m * K, K, inv_temp);
  if (lane == 0) tickets[m] = 0;
}

// Long rows (the dense and pruned heads' full-vocabulary softmax): one
// cluster of kSmCluster CTAs per row, each CTA holding kSmThreads * EPT elements
// of the row in registers. The CTAs exchange their (max, sum) through
// distributed shared memory, so the row is read once and q written once.
constexpr int kSmCluster = 8;
constexpr int kSmThreads = 512;

template <int EPT>
__global__ void __cluster_dims__(kSmCluster, 1, 1) __launch_bounds__(kSmThreads)
row_softmax_cluster_kernel(const float* __restrict__ L, int64_t K, float inv_temp,
                           float* __restrict__ q) {
  constexpr int kWarps = kSmThreads / 32;
  __shared__ float red[kWarps];
  __shared__ float part[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = tc::cluster_ctarank();
  const int64_t per = (K + kSmCluster - 1) / kSmCluster;
  const int64_t beg = (int64_t)rank * per;
  const int64_t end = beg + per < K ? beg + per : K;
  const float* row = L + (size_t)blockIdx.y * K;
  float* qrow = q + (size_t)blockIdx.y * K;
  pdl_wait();  // the logits come from the previous kernel
  float z[EPT];
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int64_t j = beg + tid + kSmThreads * e;
    z[e] = j < end ? row[j] * inv_temp : -INFINITY;
    mx = fmaxf(mx, z[e]);
  }
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  cta_sync();
  float bm = red[0];
  for (int w = 1; w < kWarps; ++w) bm = fmaxf(bm, red[w]);
  cta_sync();  // red is reused below
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < EPT; ++e) sum += bm == -INFINITY ? 0.f : __expf(z[e] - bm);
  sum = warp_sum(sum);
  if (lane == 0) red[warp] = sum;
  cta_sync();
  if (tid == 0) {
    float bs = 0.f;
    for (int w = 0; w < kWarps; ++w) bs += red[w];
    part[0] = bm;
    part[1] = bs;
  }
  tc::cluster_sync();  // every CTA's (max, sum) is published
  float gm = -INFINITY, ms[kSmCluster], ss[kSmCluster];
  const uint32_t pa = tc::smem_addr(part);
#pragma unroll
  for (int c = 0; c < kSmCluster; ++c) {
    const uint32_t a = tc::map_to_rank(pa, (uint32_t)c);
    ms[c] = tc::ld_cluster_f32(a);
    ss[c] = tc::ld_cluster_f32(a + 4);
    gm = fmaxf(gm, ms[c]);
  }
  float gs = 0.f;
#pragma unroll
  for (int c = 0; c < kSmCluster; ++c) gs += ms[c] == -INFINITY ? 0.f : ss[c] * __expf(ms[c] - gm);
  const float inv = 1.f / gs;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int64_t j = beg + tid + kSmThreads * e;
    if (j < end) qrow[j] = __expf(z[e] - gm) * inv;
  }
  tc::cluster_sync();  // no CTA leaves while another may still read its (max, sum)
}

// One CTA per row.
__global__ void __launch_bounds__(256)
row_softmax_kernel(const float* __restrict__ L, int64_t K, float inv_temp, float* __restrict__ q) {
  __shared__ float red_m[8], red_s[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();  // the logits come from the previous kernel
  const float* row = L + (size_t)blockIdx.x * K;
  float* qrow = q + (size_t)blockIdx.x * K;
  float mx = -INFINITY, sum = 0.f;
  for (int64_t j = tid; j < K; j += blockDim.x) {
    const float z = row[j] * inv_temp;
    if (z > mx) {
      sum = sum * __expf(mx - z) + 1.f;
      mx = z;
    } else {
      sum += __expf(z - mx);
    }
  }
  float wm = warp_max(mx);
  float ws = (mx == -INFINITY) ? 0.f : sum * __expf(mx - wm);
  ws = warp_sum(ws);
  if (lane == 0) { red_m[warp] = wm; red_s[warp] = ws; }
  cta_sync();
  float gm = red_m[0];
  for (int w = 1; w < 8; ++w) gm = fmaxf(gm, red_m[w]);
  float gs = 0.f;
  for (int w = 0; w < 8; ++w) gs += (red_m[w] == -INFINITY) ? 0.f : red_s[w] * __expf(red_m[w] - gm);
  const float inv = 1.f / gs;
  cta_sync();  // q may alias L: every read of the row is done
  for (int64_t j = tid; j < K; j += blockDim.x) qrow[j] = __expf(row[j] * inv_temp - gm) * inv;
}

// Rows of up to 256 * EPT logits: every element is read once into registers,
// the row max and sum are block reductions, and q is written from registers.
template <int EPT>
__global__ void __launch_bounds__(256)
row_softmax_reg_kernel(const float* __restrict__ L, int K, float inv_temp, float* __restrict__ q) {
  __shared__ float red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();  // the logits come from the previous kernel
  const size_t row0 = (size_t)blockIdx.x * K;
  float* qrow = q + row0;
  float z[EPT];
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int j = tid + 256 * e;
    z[e] = j < K ? L[row0 + j] * inv_temp : -INFINITY;
    mx = fmaxf(mx, z[e]);
  }
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  cta_sync();
  float gm = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) gm = fmaxf(gm, red[w]);
  cta_sync();  // red is reused below
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    z[e] = __expf(z[e] - gm);  // exp(-inf) = 0 for padding
    sum += z[e];
  }
  sum = warp_sum(sum);
  if (lane == 0) red[warp] = sum;
  cta_sync();
  float gs = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) gs += red[w];
  const float inv = 1.f / gs;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int j = tid + 256 * e;
    if (j < K) qrow[j] = z[e] * inv;
  }
}

}  // namespace

int overlap_ctas() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LMHEAD_GATHER_OVL_CTAS");
    v = e ? atoi(e) : kGatherMinCtas;
  }
  return v;
}

template <int WPC, int UNR, int MINB, bool SH, bool FUSED, bool ROWMAP, bool OVL>
cudaError_t launch_gather_v(const bf16_t* W, const bf16_t* h, const int32_t* ids, int64_t n, int d,
                            int M, int K, float* logits, float* q, float inv_temp, int* tickets,
                            int* err, cudaStream_t s, int span, const int* ready, int k_tile,
                            int64_t tiles, const int32_t* row_of_id, int64_t n_rows) {
  const int64_t total = (int64_t)M * K;
  const unsigned grid = (unsigned)((total + WPC - 1) / WPC);
  const size_t smem = SH ? (size_t)d * 2 : 0;
  static int smem_set[64] = {0};
  if (SH) {
    cudaError_t e =
        ensure_dynamic_smem(gather_logits_kernel<WPC, UNR, MINB, SH, FUSED, ROWMAP, OVL>, smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(true, gather_logits_kernel<WPC, UNR, MINB, SH, FUSED, ROWMAP, OVL>, dim3(grid),
                       dim3(WPC * 32), smem, s, W, h, ids, n, d, M, K, span, logits, q,
                       inv_temp, tickets, err, ready, k_tile, (int)tiles, row_of_id, n_rows);
}

cudaError_t launch_gather_logits(const bf16_t* W, const bf16_t* h, const int32_t* ids, int64_t n,
                                 int d, int M, int K, float* logits, float* q, float inv_temp,
                                 int* tickets, int* err, cudaStream_t s, int span,
                                 const int* ready, int k_tile, int64_t tiles,
                                 const int32_t* row_of_id, int64_t n_rows) {
  if (ready && (k_tile < 1 || tiles < 1)) return cudaErrorInvalidValue;
#define GATHER_U(UNR, MINB, FUSED, ROWMAP, OVL)                                           \
  return launch_gather_v<kWarpsPerCta, UNR, MINB, true, FUSED, ROWMAP, OVL>(               \
      W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s, span, ready, k_tile, tiles, \
      row_of_id, n_rows)
#define GATHER(MINB, FUSED, ROWMAP, OVL) GATHER_U(4, MINB, FUSED, ROWMAP, OVL)
  if (q) GATHER(6, true, false, false);  // softmax fused (the no-allocation entry point)
  if (row_of_id) {                       // a vocabulary shard
    if (ready) GATHER(6, false, true, true);
    GATHER(6, false, true, false);
  }
  if (!ready && (int64_t)M * K <= (int64_t)kSmallGatherPerSm * sm_count()) {
    // a thousand or two candidates (one or two hidden vectors): the warps are
    // too few to hide DRAM latency, so each lane keeps 16 loads in flight (a
    // whole 8 KB row per warp request round) instead of 4; at 122 registers
    // two CTAs fit per SM, so only gathers that fit one such wave take it
    // (measured: one hidden vector 25.4 -> 23.1 us a call, eight 47.2 -> 49.8)
    GATHER_U(16, 2, false, false, false);
  }
  if (ready) {
    // overlapping the scoring kernel, the gather's CTAs share SMs with it and
    // registers bound how many fit; LMHEAD_GATHER_OVL_CTAS=8 compiles the
    // kernel for eight CTAs per SM (32 registers, some spilled; measurements)
    if (overlap_ctas() == 8) GATHER(8, false, false, true);
    GATHER(kGatherMinCtas, false, false, true);
  }
  GATHER(6, false, false, false);
#undef GATHER
#undef GATHER_U
}

cudaError_t launch_row_softmax(const float* L, int M, int64_t K, float inv_temp, float* q,
                               cudaStream_t s) {
  if (K <= 256 * 4)
    return launch_kernel(true, row_softmax_reg_kernel<4>, dim3(M), dim3(256), 0, s, L, (int)K,
                         inv_temp, q);
  if (K <= 256 * 16)
    return launch_kernel(true, row_softmax_reg_kernel<16>, dim3(M), dim3(256), 0, s, L, (int)K,
                         inv_temp, q);
  const int64_t per = (K + kSmCluster - 1) / kSmCluster;
  if (per <= kSmThreads * 32)
    return launch_kernel(true, row_softmax_cluster_kernel<32>, dim3(kSmCluster, M), dim3(kSmThreads),
                         0, s, L, K, inv_temp, q);
  if (per <= kSmThreads * 56)
    return launch_kernel(true, row_softmax_cluster_kernel<56>, dim3(kSmCluster, M), dim3(kSmThreads),
                         0, s, L, K, inv_temp, q);
  return launch_kernel(true, row_softmax_kernel, dim3(M), dim3(256), 0, s, L, K, inv_temp, q);
}

}  // namespace lmhead
