// Stage-1 scoring on CUDA cores (EAGLE-4 notes, "A Local Top-k based
// variant"): scores = A u over the vocabulary rows of a tile, kept on chip,
// reduced to the tile's top k_tile and written out through token_ids (no
// score writeback). It serves the tile shapes the tensor-core kernel does not
// (tiles under 32 rows, k_tile not in {1, 2, 4, 8}, r > 512).
//
// This is the small-batch engine: A is read once with 16-byte loads, one warp
// per row with the rank dimension split across lanes; u (M x r) sits in
// shared memory as fp32. A CTA covers a block of up to kMB hidden vectors.
#include <math.h>
#include <stdlib.h>

#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

constexpr int kMB = 8;         // hidden vectors per CTA (one selection warp each)
constexpr int kChunk = 256;    // vocabulary rows scored per pass
constexpr int kThreads = 256;  // 8 warps

// Stage u[m0 .. m0+mb) into shared memory as fp32 (rows beyond mb are zero).
__device__ void stage_u(const bf16_t* __restrict__ u, int r, int m0, int mb, float* us) {
  for (int i = threadIdx.x; i < kMB * r; i += blockDim.x) {
    const int mm = i / r, k = i - mm * r;
    float v = 0.f;
    if (mm < mb) {
      const uint32_t b = u[(size_t)(m0 + mm) * r + k];
      v = __uint_as_float(b << 16);
    }
    us[i] = v;
  }
}

// Score rows [p0, p0+rows) of A against the staged u; result for row j of
// this chunk and hidden vector mm goes to out(mm, j).
template <typename Out>
__device__ __forceinline__ void score_chunk(const bf16_t* __restrict__ A, int r, int64_t p0,
                                            int rows, int mb, const float* us, Out out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < rows; j += kThreads / 32) {
    const bf16_t* arow = A + (size_t)(p0 + j) * r;
    float part[kMB];
#pragma unroll
    for (int mm = 0; mm < kMB; ++mm) part[mm] = 0.f;
    for (int k = lane * 8; k < r; k += 256) {
      float a[8];
      unpack8(ldg_nc_v4(arow + k), a);
#pragma unroll
      for (int mm = 0; mm < kMB; ++mm) {
        if (mm < mb) {
          const float4 u0 = *reinterpret_cast<const float4*>(us + mm * r + k);
          const float4 u1 = *reinterpret_cast<const float4*>(us + mm * r + k + 4);
          float s = part[mm];
          s = fmaf(a[0], u0.x, s); s = fmaf(a[1], u0.y, s);
          s = fmaf(a[2], u0.z, s); s = fmaf(a[3], u0.w, s);
          s = fmaf(a[4], u1.x, s); s = fmaf(a[5], u1.y, s);
          s = fmaf(a[6], u1.z, s); s = fmaf(a[7], u1.w, s);
          part[mm] = s;
        }
      }
    }
#pragma unroll
    for (int mm = 0; mm < kMB; ++mm) {
      if (mm < mb) {
        const float s = warp_sum(part[mm]);
        if (lane == 0) out(mm, j, s);
      }
    }
  }
}

// ---------------------------------------------------------------- K4 (fma)
// grid: (tiles, ceil(M / kMB)). Dynamic smem: us[kMB*r] fp32.
__global__ void __launch_bounds__(kThreads)
local_topk_fma_kernel(const bf16_t* __restrict__ A, const bf16_t* __restrict__ u,
                      const int32_t* __restrict__ token_ids, int64_t n, int r, int M, int T,
                      int k_tile, int K, int32_t* __restrict__ out_ids,
                      float* __restrict__ out_scores) {
  extern __shared__ float us[];
  __shared__ float sc[kMB][kChunk];
  __shared__ int32_t sid[kChunk];
  __shared__ float ls[kMB][kFusedMaxKTile];
  __shared__ int32_t li[kMB][kFusedMaxKTile];
  __shared__ float ns[kMB][kFusedMaxKTile];
  __shared__ int32_t ni[kMB][kFusedMaxKTile];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tile = blockIdx.x;
  const int m0 = blockIdx.y * kMB;
  const int mb = min(kMB, M - m0);
  const int64_t t0 = tile * (int64_t)T;
  const int64_t t1 = min(n, t0 + (int64_t)T);
  stage_u(u, r, m0, mb, us);
  int lcount = 0;  // entries in this warp's list (uniform in the warp)

  for (int64_t p0 = t0; p0 < t1; p0 += kChunk) {
    const int rows = (int)min((int64_t)kChunk, t1 - p0);
    cta_sync();  // us staged / previous chunk's selection done
    for (int j = threadIdx.x; j < rows; j += blockDim.x)
      sid[j] = token_ids ? token_ids[p0 + j] : (int32_t)(p0 + j);
    score_chunk(A, r, p0, rows, mb, us,
                [&](int mm, int j, float s) { sc[mm][j] = s; });
    cta_sync();
    if (warp < mb) {
      // new list = top-k_tile of (current list U this chunk)
      const int want = min(k_tile, lcount + rows);
      for (int round = 0; round < want; ++round) {
        float bs = -INFINITY;
        int32_t bi = 0x7FFFFFFF;
        int bslot = -1;
        for (int j = lane; j < rows; j += 32) {
          const float s = sc[warp][j];
          if (s != -INFINITY && (bslot < 0 || beats(s, sid[j], bs, bi))) {
            bs = s; bi = sid[j]; bslot = j;
          }
        }
        for (int j = lane; j < lcount; j += 32) {
          const float s = ls[warp][j];
          if (s != -INFINITY && (bslot < 0 || beats(s, li[warp][j], bs, bi))) {
            bs = s; bi = li[warp][j]; bslot = kChunk + j;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float os = __shfl_xor_sync(0xFFFFFFFFu, bs, o);
          const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
          const int oslot = __shfl_xor_sync(0xFFFFFFFFu, bslot, o);
          if (oslot >= 0 && (bslot < 0 || beats(os, oi, bs, bi))) {
            bs = os; bi = oi; bslot = oslot;
          }
        }
        if (lane == 0) {
          ns[warp][round] = bs;
          ni[warp][round] = bi;
          if (bslot >= 0 && bslot < kChunk) sc[warp][bslot] = -INFINITY;
          else if (bslot >= kChunk) ls[warp][bslot - kChunk] = -INFINITY;
        }
        __syncwarp();
      }
      for (int j = lane; j < want; j += 32) {
        ls[warp][j] = ns[warp][j];
        li[warp][j] = ni[warp][j];
      }
      lcount = want;
      __syncwarp();
    }
  }
  if (warp < mb) {
    const size_t base = (size_t)(m0 + warp) * K + (size_t)tile * k_tile;
    for (int j = lane; j < lcount; j += 32) {
      out_ids[base + j] = li[warp][j];
      if (out_scores) out_scores[base + j] = ls[warp][j];
    }
  }
}

// ---------------------------------------------------------------- K4 (gemv)
// Up to four hidden vectors with tiles of 32-256 rows that divide 256: the
// contraction is a GEMV (one to four FLOP per byte of A), so CUDA cores keep
// pace with HBM and the tensor-core kernel's machinery (TMA ring, MMA issue,
// TMEM) only adds latency. A warp scores eight rows at a time at r = 256 (four
// at r = 512), each lane reading one (two) 16-byte pieces of every row
// (coalesced 512-byte requests), the first rows requested before waiting for u
// (u comes from the projection kernel, A does not); the lane's share of u
// sits in registers and a warp reduction gives each row's score. The CTA's
// 256 rows hold 256 / T whole tiles; each tile's top k_tile per hidden vector
// comes from one warp: every lane keeps a
// sorted register list of its strided share of the tile's scores, then
// k_tile rounds of a warp arg-best over the list heads (score descending,
// then the smaller vocabulary id).
constexpr int kGemvThreads = 256;

__device__ __forceinline__ bool gemv_beats(float sa, int32_t ia, float sb, int32_t ib) {
  return sa > sb || (sa == sb && ia < ib);
}

// DB: the next batch of rows is requested before the current one is used
// (more registers, so fewer CTAs per SM).
// WB: write the scores to S (M x n by position: the global path's score
// writeback) instead of selecting.
// P: 16-byte pieces of a row per lane (r = 256 P): a batch is 8 / P rows, so
// a lane keeps eight loads in flight at either rank.
template <int MB, int KT, bool DB, bool WB = false, int P = 1>
__global__ void __launch_bounds__(kGemvThreads,
                                  DB ? (MB == 1 ? 3 : 2) : (MB == 1 ? 4 : (MB == 2 ? 3 : 2)))
local_topk_gemv_kernel(const bf16_t* __restrict__ A, const bf16_t* __restrict__ u,
                       const int32_t* __restrict__ token_ids, int64_t n, int r, int M, int T,
                       int k_tile, int K, int32_t* __restrict__ out_ids,
                       float* __restrict__ out_scores, int* __restrict__ ready,
                       float* __restrict__ S, int* __restrict__ hist0, int hist0_stride) {
  __shared__ float sc[MB][kGemvThreads];
  __shared__ int32_t svid[kGemvThreads];
  // writeback: score-digit counts, two 16-bit bins a word (a CTA counts at
  // most 256 scores per hidden vector)
  __shared__ uint32_t hh[WB ? MB * kSelectHistBins / 2 : 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row0 = (int64_t)blockIdx.x * kGemvThreads;
  const int m0 = blockIdx.y * MB;
  const int mb = min(MB, M - m0);
  if constexpr (WB) {
    if (hist0)
      for (int i = tid; i < MB * kSelectHistBins / 2; i += kGemvThreads) hh[i] = 0u;
  }
  constexpr int kRows = 8 / P;  // rows per batch and warp (8 loads in flight per lane)
  {
    const int64_t pos = row0 + tid;
    svid[tid] = pos < n ? (token_ids ? __ldg(token_ids + pos) : (int32_t)pos) : 0x7FFFFFFF;
  }
  // warp w scores rows w, w + 8, ... of the CTA's 256; lane L reads pieces
  // L, L + 32, ... of a row (coalesced 512-byte requests)
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 a[kRows * P];
  auto load_batch = [&](int bt) {
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int64_t pos = row0 + (int64_t)(bt * kRows + i) * 8 + warp;
      const uint4* arow = reinterpret_cast<const uint4*>(A + (size_t)(pos < n ? pos : 0) * r);
#pragma unroll
      for (int q = 0; q < P; ++q) a[i * P + q] = pos < n ? ldg_nc_v4(arow + lane + 32 * q) : zero;
    }
  };
  load_batch(0);  // A before waiting for u
  pdl_wait();     // u is written by the previous kernel
  // the gather may launch once every thread has triggered, which is after
  // the projection kernel (that zeroes the ready counters) completed
  pdl_trigger();
  float uf[MB][8 * P];
#pragma unroll
  for (int mm = 0; mm < MB; ++mm) {
#pragma unroll
    for (int q = 0; q < P; ++q) {
      uint4 uv = zero;
      if (mm < mb)
        uv = *reinterpret_cast<const uint4*>(u + (size_t)(m0 + mm) * r + (lane + 32 * q) * 8);
      unpack8(uv, uf[mm] + 8 * q);
    }
  }
  constexpr int kBatches = kGemvThreads / 8 / kRows;  // batches of kRows rows per warp
  for (int bt = 0; bt < kBatches; ++bt) {
    if (!DB && bt > 0) load_batch(bt);
    uint4 cur[kRows * P];  // this batch; with DB the next one is requested before it is used
#pragma unroll
    for (int i = 0; i < kRows * P; ++i) cur[i] = a[i];
    if (DB && bt + 1 < kBatches) load_batch(bt + 1);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      float part[MB];
#pragma unroll
      for (int mm = 0; mm < MB; ++mm) part[mm] = 0.f;
#pragma unroll
      for (int q = 0; q < P; ++q) {
        float f[8];
        unpack8(cur[i * P + q], f);
#pragma unroll
        for (int mm = 0; mm < MB; ++mm) {
#pragma unroll
          for (int e = 0; e < 8; ++e) part[mm] = fmaf(f[e], uf[mm][8 * q + e], part[mm]);
        }
      }
      const int rl = (bt * kRows + i) * 8 + warp;  // row within the CTA
      const bool live = row0 + rl < n;
#pragma unroll
      for (int mm = 0; mm < MB; ++mm) {
        const float sres = warp_sum(part[mm]);
        if (lane == 0) sc[mm][rl] = live ? sres : -INFINITY;
      }
    }
  }
  cta_sync();
  if constexpr (WB) {  // the global path: every score to HBM, rows in position order
    for (int i = tid; i < mb * kGemvThreads; i += kGemvThreads) {
      const int mm = i / kGemvThreads, rl = i - mm * kGemvThreads;
      if (row0 + rl < n) {
        const float x = sc[mm][rl];
        S[(size_t)(m0 + mm) * n + row0 + rl] = x;
        if (hist0) {
          const uint32_t b = mm * kSelectHistBins + (float_key(x) >> (32 - kSelectHistBits));
          atomicAdd(&hh[b >> 1], 1u << ((b & 1u) * 16));
        }
      }
    }
    if (hist0) {  // this CTA's counts into the rows' first selection histograms
      cta_sync();
      for (int w = tid; w < mb * kSelectHistBins / 2; w += kGemvThreads) {
        const uint32_t c2 = hh[w];
        if (!c2) continue;
        const int mm = (2 * w) / kSelectHistBins, b = 2 * w - mm * kSelectHistBins;
        int* hrow = hist0 + (size_t)(m0 + mm) * hist0_stride;
        if (c2 & 0xFFFFu) atomicAdd(hrow + b, (int)(c2 & 0xFFFFu));
        if (c2 >> 16) atomicAdd(hrow + b + 1, (int)(c2 >> 16));
      }
    }
    return;
  }
  // one warp per (tile, hidden vector)
  const int tpc = kGemvThreads / T;
  const int jobs = tpc * mb;
  for (int job = warp; job < jobs; job += kGemvThreads / 32) {
    const int tl = job / mb, mm = job - tl * mb;
    const int64_t tile = (int64_t)blockIdx.x * tpc + tl;
    const int64_t t0 = tile * T;
    if (t0 >= n) continue;
    const int rows = (int)min((int64_t)T, n - t0);
    float ls[KT];
    int32_t lv[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) { ls[i] = -INFINITY; lv[i] = 0x7FFFFFFF; }
    for (int j = lane; j < rows; j += 32) {
      const float x = sc[mm][tl * T + j];
      const int32_t id = svid[tl * T + j];
      bool c[KT];
#pragma unroll
      for (int i = 0; i < KT; ++i) c[i] = gemv_beats(x, id, ls[i], lv[i]);
#pragma unroll
      for (int i = KT - 1; i > 0; --i) {
        ls[i] = c[i] ? (c[i - 1] ? ls[i - 1] : x) : ls[i];
        lv[i] = c[i] ? (c[i - 1] ? lv[i - 1] : id) : lv[i];
      }
      ls[0] = c[0] ? x : ls[0];
      lv[0] = c[0] ? id : lv[0];
    }
    const int count = min(k_tile, rows);
    const size_t base = (size_t)(m0 + mm) * K + (size_t)tile * k_tile;
    for (int k = 0; k < count; ++k) {
      float key = ls[0];
      int32_t id = lv[0];
      int who = lane;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ok = __shfl_xor_sync(0xFFFFFFFFu, key, off);
        const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, id, off);
        const int ow = __shfl_xor_sync(0xFFFFFFFFu, who, off);
        if (gemv_beats(ok, oi, key, id)) { key = ok; id = oi; who = ow; }
      }
      if (lane == who) {  // pop the head
#pragma unroll
        for (int i = 0; i + 1 < KT; ++i) { ls[i] = ls[i + 1]; lv[i] = lv[i + 1]; }
        ls[KT - 1] = -INFINITY;
        lv[KT - 1] = 0x7FFFFFFF;
      }
      if (lane == 0) {
        out_ids[base + k] = id;
        if (out_scores) out_scores[base + k] = key;
      }
    }
  }
  if (ready) {  // this CTA's tiles (one ready block: 256 / T divides 16) are written
    __threadfence();
    cta_sync();
    if (tid == 0) {
      const int64_t tile0 = (int64_t)blockIdx.x * tpc;
      const int64_t tiles_here = min((int64_t)tpc, (n + T - 1) / T - tile0);
      signal_count(ready + tile0 / kReadyTiles, (int)tiles_here * mb);
    }
  }
}

template <int MB, bool DB>
cudaError_t launch_gemv_mb(const bf16_t* A, const bf16_t* u, const int32_t* token_ids, int64_t n,
                           int r, int M, int T, int k_tile, int K, int32_t* out_ids,
                           float* out_scores, cudaStream_t s, int* ready) {
  dim3 grid((unsigned)((n + kGemvThreads - 1) / kGemvThreads), (unsigned)((M + MB - 1) / MB));
#define GV(KT, P)                                                                                \
  return launch_kernel(true, local_topk_gemv_kernel<MB, KT, DB, false, P>, grid, dim3(kGemvThreads), \
                       0, s, A, u, token_ids, n, r, M, T, k_tile, K, out_ids, out_scores, ready,   \
                       (float*)nullptr, (int*)nullptr, 0);
#define GVR(KT) do { if (r == 512) GV(KT, 2); GV(KT, 1); } while (0)
  if (k_tile <= 1) GVR(1);
  if (k_tile <= 2) GVR(2);
  if (k_tile <= 4) GVR(4);
  GVR(8);
#undef GVR
#undef GV
}

// LMHEAD_K4_GEMV = 0 keeps small batches off the GEMV kernel (measurements only).
bool gemv_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LMHEAD_K4_GEMV");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

}  // namespace

cudaError_t launch_scores_gemv(const bf16_t* A, const bf16_t* u, int64_t n, int r, int M, float* S,
                               cudaStream_t s, int* hist0, int hist0_stride) {
  if (!scores_gemv_supported(M, r)) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((n + kGemvThreads - 1) / kGemvThreads), 1);
#define WBK(MB, DB, P)                                                                          \
  return launch_kernel(true, local_topk_gemv_kernel<MB, 1, DB, true, P>, grid, dim3(kGemvThreads), \
                       0, s, A, u, (const int32_t*)nullptr, n, r, M, kGemvThreads, 1, 0,           \
                       (int32_t*)nullptr, (float*)nullptr, (int*)nullptr, S, hist0, hist0_stride)
  if (M <= 1) {
    if (r == 512) WBK(1, false, 2);
    WBK(1, false, 1);
  }
  if (r == 512) WBK(2, true, 2);
  WBK(2, true, 1);
#undef WBK
}

// LMHEAD_GEMV_MAX_M = m (0..4) moves the hand-over to the tensor cores
// (measurements only).
int gemv_max_m() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LMHEAD_GEMV_MAX_M");
    v = e ? atoi(e) : kLocalGemvMaxM;
    if (v < 0) v = 0;
    if (v > 8) v = 8;  // five to eight: two grid rows of four (A streamed twice)
  }
  return v;
}

// measured: at three and four hidden vectors the tensor-core row products and a
// histogram pass beat a four-vector GEMV writeback (global calls 53.3 vs 58.3
// us at three, 59.3 vs 63.5 at four)
bool scores_gemv_supported(int M, int r) {
  return gemv_enabled() && M <= 2 && (r == 256 || r == 512);
}

bool local_topk_gemv_supported(int M, int r, int T, int k_tile) {
  return gemv_enabled() && M <= gemv_max_m() && (r == 256 || r == 512) && T >= 32 &&
         T <= kGemvThreads && kGemvThreads % T == 0 && k_tile <= 8;
}

cudaError_t launch_local_topk_fma(const bf16_t* A, const bf16_t* u, const int32_t* token_ids,
                                  int64_t n, int r, int M, int T, int k_tile, int32_t* out_ids,
                                  float* out_scores, cudaStream_t s, int* ready) {
  const int64_t tiles = (n + T - 1) / T;
  const int64_t full = n / T, tail = n - full * T;
  const int K = (int)(full * k_tile + (tail ? (tail < k_tile ? tail : k_tile) : 0));
  if (local_topk_gemv_supported(M, r, T, k_tile)) {
    // measured: one hidden vector, four CTAs per SM (all 501 CTAs of the
    // 128256-row head resident at once); two, the next rows requested early
    if (M <= 1)
      return launch_gemv_mb<1, false>(A, u, token_ids, n, r, M, T, k_tile, K, out_ids, out_scores,
                                      s, ready);
    if (M <= 2)
      return launch_gemv_mb<2, true>(A, u, token_ids, n, r, M, T, k_tile, K, out_ids, out_scores,
                                     s, ready);
    // three or four: 128 registers, two CTAs per SM (measured: the call
    // 45.0 -> 40.9 us at three, 46.7 -> 42.9 at four, the wide head at four
    // 87.9 -> 70.7 us)
    return launch_gemv_mb<4, false>(A, u, token_ids, n, r, M, T, k_tile, K, out_ids, out_scores,
                                    s, ready);
  }
  // the kernel also has ~13 KB of static shared memory, so the opt-in is
  // needed below 48 KB of dynamic memory too: always raise the limit (cached)
  const size_t smem = (size_t)kMB * r * sizeof(float);
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(local_topk_fma_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)tiles, (M + kMB - 1) / kMB);
  return launch_kernel(false, local_topk_fma_kernel, grid, dim3(kThreads), smem, s, A, u, token_ids,
                       n, r, M, T, k_tile, K, out_ids, out_scores);
}

}  // namespace lmhead
