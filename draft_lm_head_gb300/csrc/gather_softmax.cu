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

#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

constexpr int kWarpsPerCta = 8;

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

__global__ void __launch_bounds__(kWarpsPerCta * 32)
gather_logits_kernel(const bf16_t* __restrict__ W, const bf16_t* __restrict__ h,
                     const int32_t* __restrict__ ids, int64_t n, int d, int M, int K,
                     float* __restrict__ logits, float* __restrict__ q, float inv_temp,
                     int* __restrict__ tickets, int* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int64_t c = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (c >= (int64_t)M * K) return;
  const int m = (int)(c / K);
  const int32_t id = __ldg(ids + c);
  float s;
  if (id < 0 || (int64_t)id >= n) {
    if (lane == 0) record_error(err, kDevErrBadId);
    s = __int_as_float(0x7FC00000);  // NaN
  } else {
    const uint4* wrow = reinterpret_cast<const uint4*>(W + (size_t)id * d);
    const uint4* hrow = reinterpret_cast<const uint4*>(h + (size_t)m * d);
    const int nvec = d >> 3;
    float acc = 0.f;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) acc += dot8(ldg_nc_v4(wrow + v), __ldg(hrow + v));
    s = warp_sum(acc);
  }
  if (lane == 0) logits[c] = s;
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

// One CTA per row.
__global__ void __launch_bounds__(256)
row_softmax_kernel(const float* __restrict__ L, int64_t K, float inv_temp, float* __restrict__ q) {
  __shared__ float red_m[8], red_s[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
  __syncthreads();
  float gm = red_m[0];
  for (int w = 1; w < 8; ++w) gm = fmaxf(gm, red_m[w]);
  float gs = 0.f;
  for (int w = 0; w < 8; ++w) gs += (red_m[w] == -INFINITY) ? 0.f : red_s[w] * __expf(red_m[w] - gm);
  const float inv = 1.f / gs;
  __syncthreads();  // q may alias L: every read of the row is done
  for (int64_t j = tid; j < K; j += blockDim.x) qrow[j] = __expf(row[j] * inv_temp - gm) * inv;
}

}  // namespace

cudaError_t launch_gather_logits(const bf16_t* W, const bf16_t* h, const int32_t* ids, int64_t n,
                                 int d, int M, int K, float* logits, float* q, float inv_temp,
                                 int* tickets, int* err, cudaStream_t s) {
  const int64_t total = (int64_t)M * K;
  const unsigned grid = (unsigned)((total + kWarpsPerCta - 1) / kWarpsPerCta);
  gather_logits_kernel<<<grid, kWarpsPerCta * 32, 0, s>>>(W, h, ids, n, d, M, K, logits, q,
                                                          inv_temp, tickets, err);
  return cudaGetLastError();
}

cudaError_t launch_row_softmax(const float* L, int M, int64_t K, float inv_temp, float* q,
                               cudaStream_t s) {
  row_softmax_kernel<<<M, 256, 0, s>>>(L, K, inv_temp, q);
  return cudaGetLastError();
}

}  // namespace lmhead
