// K1: the skinny projection u = B h of stage 1 (EAGLE-4 notes, "A Local
// Top-k based variant": both flows start with u = B @ h).
//
// B is r x d (2-5 MB at the workloads' sizes), h is M x d, u is M x r bf16.
// One warp owns one row of B and streams it once with 16-byte loads; a CTA
// holds 8 rows and a block of up to kMB hidden vectors, whose d-chunks are
// staged in shared memory and shared by the 8 warps. fp32 accumulation, one
// bf16 rounding (nearest-even) at the end.
#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

constexpr int kRowsPerCta = 8;
constexpr int kMB = 16;
constexpr int kDChunk = 1024;  // bf16 elements of h per staged chunk

__global__ void __launch_bounds__(256) project_u_kernel(const bf16_t* __restrict__ B,
                                                        const bf16_t* __restrict__ h, int d, int r,
                                                        int M, bf16_t* __restrict__ u,
                                                        int* zero_ptr, int zero_ints) {
  __shared__ uint4 hs[kMB * kDChunk / 8];
  if (zero_ptr) {
    const int nb = gridDim.x * gridDim.y, bid = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = bid * blockDim.x + threadIdx.x; i < zero_ints; i += nb * blockDim.x) zero_ptr[i] = 0;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = blockIdx.x * kRowsPerCta + warp;
  const int m0 = blockIdx.y * kMB;
  const int mb = min(kMB, M - m0);
  float acc[kMB];
#pragma unroll
  for (int i = 0; i < kMB; ++i) acc[i] = 0.f;

  const uint4* brow = reinterpret_cast<const uint4*>(B + (size_t)min(k, r - 1) * d);
  for (int c0 = 0; c0 < d; c0 += kDChunk) {
    const int nvec = min(kDChunk, d - c0) / 8;
    __syncthreads();
    for (int i = threadIdx.x; i < mb * nvec; i += blockDim.x) {
      const int mm = i / nvec, v = i - mm * nvec;
      hs[mm * (kDChunk / 8) + v] =
          *reinterpret_cast<const uint4*>(h + (size_t)(m0 + mm) * d + c0 + v * 8);
    }
    __syncthreads();
    if (k < r) {
#pragma unroll 2
      for (int v = lane; v < nvec; v += 32) {
        float bf[8];
        unpack8(ldg_nc_v4(brow + c0 / 8 + v), bf);
#pragma unroll
        for (int mm = 0; mm < kMB; ++mm) {
          if (mm < mb) {
            float hf[8];
            unpack8(hs[mm * (kDChunk / 8) + v], hf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[mm] = fmaf(bf[e], hf[e], acc[mm]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int mm = 0; mm < kMB; ++mm) {
    if (mm < mb) {
      const float s = warp_sum(acc[mm]);
      if (lane == 0 && k < r) {
        const __nv_bfloat16 b = __float2bfloat16_rn(s);
        u[(size_t)(m0 + mm) * r + k] = *reinterpret_cast<const bf16_t*>(&b);
      }
    }
  }
}

}  // namespace

cudaError_t launch_project_u(const bf16_t* B, const bf16_t* h, int d, int r, int M, bf16_t* u,
                             int* zero_ptr, int zero_ints, cudaStream_t s) {
  dim3 grid((r + kRowsPerCta - 1) / kRowsPerCta, (M + kMB - 1) / kMB);
  project_u_kernel<<<grid, 256, 0, s>>>(B, h, d, r, M, u, zero_ptr, zero_ints);
  return cudaGetLastError();
}

}  // namespace lmhead
