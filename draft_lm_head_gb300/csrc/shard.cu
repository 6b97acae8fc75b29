// The softmax of a vocabulary-sharded head. With the vocabulary positions
// split into contiguous, tile-aligned ranges, one per shard, the local Top-k
// of the EAGLE-4 notes ("A Local Top-k based variant": every tile picks its
// own k_tile candidates) needs no exchange between shards, and each shard
// gathers and scores its own candidates. Only the softmax over a row's
// candidates spans the shards. It is split in two: every shard reduces its
// candidates' logits to (max, sum of exponentials), the shards exchange
// those 8 bytes per row (an all-gather, done by the caller), and every shard
// then normalises its own candidates with the combined pair:
//   Mx = max_g max_g,  Z = sum_g sum_g * exp(max_g - Mx),  q = exp(L/T - Mx) / Z.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

constexpr int kStatThreads = 256;

// Combine per-thread (max, sum) pairs across the CTA; result in every thread.
__device__ __forceinline__ float2 block_max_sum(float mx, float sum, float2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float wm = warp_max(mx);
  float ws = (mx == -INFINITY) ? 0.f : sum * __expf(mx - wm);
  ws = warp_sum(ws);
  if (lane == 0) red[warp] = make_float2(wm, ws);
  cta_sync();
  float gm = red[0].x;
  for (int w = 1; w < kStatThreads / 32; ++w) gm = fmaxf(gm, red[w].x);
  float gs = 0.f;
  for (int w = 0; w < kStatThreads / 32; ++w)
    gs += (red[w].x == -INFINITY) ? 0.f : red[w].y * __expf(red[w].x - gm);
  return make_float2(gm, gs);
}

// One CTA per row: stats[m] = (max_j L[m,j]/T, sum_j exp(L[m,j]/T - max)).
__global__ void __launch_bounds__(kStatThreads)
row_stats_kernel(const float* __restrict__ L, int K, float inv_temp, float* __restrict__ stats) {
  __shared__ float2 red[kStatThreads / 32];
  pdl_wait();  // the logits come from the previous kernel
  const float* row = L + (size_t)blockIdx.x * K;
  float mx = -INFINITY, sum = 0.f;
  for (int j = threadIdx.x; j < K; j += kStatThreads) {
    const float z = row[j] * inv_temp;
    if (z > mx) {
      sum = sum * __expf(mx - z) + 1.f;
      mx = z;
    } else {
      sum += __expf(z - mx);
    }
  }
  const float2 r = block_max_sum(mx, sum, red);
  if (threadIdx.x == 0) {
    stats[2 * (size_t)blockIdx.x] = r.x;
    stats[2 * (size_t)blockIdx.x + 1] = r.y;
  }
}

// One CTA per row: q of this shard's candidates from every shard's stats.
__global__ void __launch_bounds__(kStatThreads)
shard_softmax_kernel(const float* __restrict__ all_stats, int G, int M,
                     const float* __restrict__ L, int K, float inv_temp, float* __restrict__ q) {
  pdl_wait();
  const int m = blockIdx.x;
  float gm = -INFINITY;
  for (int g = 0; g < G; ++g) gm = fmaxf(gm, all_stats[2 * ((size_t)g * M + m)]);
  float gs = 0.f;
  for (int g = 0; g < G; ++g) {
    const float mg = all_stats[2 * ((size_t)g * M + m)];
    if (mg != -INFINITY) gs += all_stats[2 * ((size_t)g * M + m) + 1] * __expf(mg - gm);
  }
  const float inv = 1.f / gs;
  const float* row = L + (size_t)m * K;
  float* qrow = q + (size_t)m * K;
  for (int j = threadIdx.x; j < K; j += kStatThreads) qrow[j] = __expf(row[j] * inv_temp - gm) * inv;
}

}  // namespace

cudaError_t launch_row_stats(const float* L, int M, int K, float inv_temp, float* stats,
                             cudaStream_t s) {
  return launch_kernel(true, row_stats_kernel, dim3(M), dim3(kStatThreads), 0, s, L, K, inv_temp,
                       stats);
}

cudaError_t launch_shard_softmax(const float* all_stats, int G, const float* L, int M, int K,
                                 float inv_temp, float* q, cudaStream_t s) {
  return launch_kernel(true, shard_softmax_kernel, dim3(M), dim3(kStatThreads), 0, s, all_stats, G,
                       M, L, K, inv_temp, q);
}

}  // namespace lmhead
