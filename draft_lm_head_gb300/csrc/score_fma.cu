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

}  // namespace

cudaError_t launch_local_topk_fma(const bf16_t* A, const bf16_t* u, const int32_t* token_ids,
                                  int64_t n, int r, int M, int T, int k_tile, int32_t* out_ids,
                                  float* out_scores, cudaStream_t s) {
  const int64_t tiles = (n + T - 1) / T;
  const int64_t full = n / T, tail = n - full * T;
  const int K = (int)(full * k_tile + (tail ? (tail < k_tile ? tail : k_tile) : 0));
  const size_t smem = (size_t)kMB * r * sizeof(float);
  if (smem > 48 * 1024) {
    static int smem_set[64] = {0};
    cudaError_t e = ensure_dynamic_smem(local_topk_fma_kernel, smem, smem_set);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)tiles, (M + kMB - 1) / kMB);
  return launch_kernel(false, local_topk_fma_kernel, grid, dim3(kThreads), smem, s, A, u, token_ids,
                       n, r, M, T, k_tile, K, out_ids, out_scores);
}

}  // namespace lmhead
