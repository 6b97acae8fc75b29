// K7: the dense full-vocabulary head, logits = h W^T over all n rows (the
// cost the two-stage method avoids; EAGLE-4 notes, "EAGLE Efficient LM
// Head"). Also serves the frequency-pruned head, which is the same product
// over a caller-built contiguous copy of the kept rows.
//
// CUDA-core engine: one warp per vocabulary row, 16-byte loads of W, hidden
// vectors in blocks of 8 through L1.
#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kMB = 8;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
dense_logits_kernel(const bf16_t* __restrict__ W, const bf16_t* __restrict__ h, int64_t n, int d,
                    int M, float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int64_t j = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (j >= n) return;
  const uint4* wrow = reinterpret_cast<const uint4*>(W + (size_t)j * d);
  const int nvec = d >> 3;
  for (int m0 = 0; m0 < M; m0 += kMB) {
    const int mb = min(kMB, M - m0);
    float acc[kMB];
#pragma unroll
    for (int mm = 0; mm < kMB; ++mm) acc[mm] = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 w = m0 == 0 ? ldg_nc_v4(wrow + v) : __ldg(wrow + v);
#pragma unroll
      for (int mm = 0; mm < kMB; ++mm)
        if (mm < mb) acc[mm] += dot8(w, __ldg(reinterpret_cast<const uint4*>(h + (size_t)(m0 + mm) * d) + v));
    }
#pragma unroll
    for (int mm = 0; mm < kMB; ++mm) {
      if (mm < mb) {
        const float s = warp_sum(acc[mm]);
        if (lane == 0) logits[(size_t)(m0 + mm) * n + j] = s;
      }
    }
  }
}

}  // namespace

cudaError_t launch_dense_logits(const bf16_t* W, const bf16_t* h, int64_t n, int d, int M,
                                float* logits, cudaStream_t s) {
  const unsigned grid = (unsigned)((n + kWarpsPerCta - 1) / kWarpsPerCta);
  dense_logits_kernel<<<grid, kWarpsPerCta * 32, 0, s>>>(W, h, n, d, M, logits);
  return cudaGetLastError();
}

}  // namespace lmhead
