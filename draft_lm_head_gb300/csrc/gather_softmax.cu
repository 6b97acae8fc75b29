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
  pdl_trigger();
  pdl_wait();  // ids come from the previous kernel
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

// v3 (persistent, TMA bulk): CTA b owns a contiguous range of the M*K
// candidates (row-major). One producer thread streams each candidate's W row
// (d bf16, contiguous) into a ring of shared-memory slots with
// cp.async.bulk; kConsumers warps take the slots in turn and dot the row with
// h[m], which each consumer keeps in registers (reloaded when m changes).
// The fused softmax is decided per row by a ticket that each CTA advances by
// the number of that row's candidates it finished; the CTA that completes a
// row normalises it.
constexpr int kConsumers = 8;
// Engine choice for A/B measurements: LMHEAD_GATHER=staged selects this
// kernel, anything else the one-warp-per-candidate kernel.
int gather_engine() {
  static int e = -1;
  if (e < 0) {
    const char* v = getenv("LMHEAD_GATHER");
    e = (v && v[0] == 's') ? 3 : 1;
  }
  return e;
}
constexpr int kMaxSlots = 32;
constexpr int kV3Threads = 32 * (kConsumers + 1);

template <int VPL>
__global__ void __launch_bounds__(kV3Threads, 1)
gather_logits_v3_kernel(const bf16_t* __restrict__ W, const bf16_t* __restrict__ h,
                        const int32_t* __restrict__ ids, int64_t n, int d, int M, int K,
                        int slots, float* __restrict__ logits, float* __restrict__ q,
                        float inv_temp, int* __restrict__ tickets, int* __restrict__ err) {
  extern __shared__ uint4 ring[];  // slots x (d/8) 16-byte vectors
  __shared__ uint64_t full[kMaxSlots], empty[kMaxSlots];
  __shared__ int slot_id[kMaxSlots];
  __shared__ volatile int abort_flag;
  __shared__ int finish_row[64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t total = (int64_t)M * K;
  const int64_t c0 = total * blockIdx.x / gridDim.x;
  const int64_t c1 = total * (blockIdx.x + 1) / gridDim.x;
  const int cnt = (int)(c1 - c0);
  const int nvec = d >> 3;
  const uint32_t row_bytes = (uint32_t)d * 2u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < slots; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // ids come from the previous kernel

  if (warp == 0) {
    // ids are fetched 32 at a time by the whole warp (next batch prefetched)
    // and broadcast with shuffles; lane 0 runs the slot protocol
    int issued = 0;
    int32_t cur = lane < cnt ? __ldg(ids + c0 + lane) : 0;
    for (int base = 0; base < cnt; base += 32) {
      const int nb = min(32, cnt - base);
      const int nxt_i = base + 32 + lane;
      const int32_t nxt = nxt_i < cnt ? __ldg(ids + c0 + nxt_i) : 0;
      for (int t = 0; t < nb; ++t) {
        const int32_t id = __shfl_sync(0xFFFFFFFFu, cur, t);
        if (lane == 0) {
          const int i = base + t;
          const int s = i % slots;
          if (tc::mbar_wait(&empty[s], ((i / slots) & 1) ^ 1, &abort_flag)) {
            slot_id[s] = id;
            if (id < 0 || (int64_t)id >= n) {
              tc::mbar_arrive(&full[s]);  // nothing to copy: the consumer writes NaN
            } else {
              tc::mbar_arrive_expect_tx(&full[s], row_bytes);
              tc::bulk_load(ring + (size_t)s * nvec, W + (size_t)id * d, row_bytes, &full[s]);
            }
            issued = i + 1;
          } else {
            abort_flag = 1;
            record_error(err, kDevErrTimeout);
          }
        }
        if (__shfl_sync(0xFFFFFFFFu, abort_flag, 0)) break;  // uniform decision
      }
      cur = nxt;
      if (__shfl_sync(0xFFFFFFFFu, abort_flag, 0)) break;
    }
    if (lane == 0 && abort_flag) {
      // drain (bounded) the copies issued last on every slot before exiting
      for (int j = max(0, issued - slots); j < issued; ++j) {
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(&full[j % slots], (j / slots) & 1) &&
               clock64() - t0 < tc::kWaitCycles) {
        }
      }
    }
  } else {
    const int cw = warp - 1;
    int cur_m = -1;
    uint4 hv[VPL];
    for (int i = cw; i < cnt; i += kConsumers) {
      const int64_t c = c0 + i;
      const int m = (int)(c / K);
      if (m != cur_m) {
        const uint4* hrow = reinterpret_cast<const uint4*>(h + (size_t)m * d);
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
          const int v = lane + 32 * k;
          hv[k] = v < nvec ? __ldg(hrow + v) : make_uint4(0, 0, 0, 0);
        }
        cur_m = m;
      }
      const int s = i % slots;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait(&full[s], (i / slots) & 1, &abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) { abort_flag = 1; record_error(err, kDevErrTimeout); }
        break;
      }
      const int32_t id = slot_id[s];
      float val;
      if (id < 0 || (int64_t)id >= n) {
        if (lane == 0) record_error(err, kDevErrBadId);
        val = __int_as_float(0x7FC00000);
      } else {
        const uint4* row = ring + (size_t)s * nvec;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
          const int v = lane + 32 * k;
          if (v < nvec) acc += dot8(row[v], hv[k]);
        }
        val = warp_sum(acc);
      }
      __syncwarp();
      if (lane == 0) {
        logits[c] = val;
        tc::mbar_arrive(&empty[s]);
      }
    }
  }
  __syncthreads();
  if (q == nullptr) return;
  // rows this CTA touched: advance their tickets by the candidates done here;
  // the CTA that completes a row normalises it (rows in batches of 64)
  const int m_first = (int)(c0 / K), m_last = (int)((c1 - 1) / K);
  for (int mb = m_first; mb <= m_last; mb += 64) {
    const int me = min(m_last, mb + 63);
    if (threadIdx.x == 0) {
      __threadfence();
      for (int m = mb; m <= me; ++m) {
        const int64_t lo = max(c0, (int64_t)m * K), hi = min(c1, (int64_t)(m + 1) * K);
        const int done = (int)(hi - lo);
        const int old = atomicAdd(tickets + m, done);
        finish_row[m - mb] = (old + done == K) ? 1 : 0;
      }
    }
    __syncthreads();
    for (int m = mb + warp; m <= me; m += kConsumers + 1) {
      if (!finish_row[m - mb]) continue;
      __threadfence();
      warp_row_softmax(logits + (size_t)m * K, q + (size_t)m * K, K, inv_temp);
      if (lane == 0) tickets[m] = 0;
    }
    __syncthreads();
  }
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
  __syncthreads();
  float gm = red_m[0];
  for (int w = 1; w < 8; ++w) gm = fmaxf(gm, red_m[w]);
  float gs = 0.f;
  for (int w = 0; w < 8; ++w) gs += (red_m[w] == -INFINITY) ? 0.f : red_s[w] * __expf(red_m[w] - gm);
  const float inv = 1.f / gs;
  __syncthreads();  // q may alias L: every read of the row is done
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
  const float* row = L + (size_t)blockIdx.x * K;
  float* qrow = q + (size_t)blockIdx.x * K;
  float z[EPT];
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int j = tid + 256 * e;
    z[e] = j < K ? row[j] * inv_temp : -INFINITY;
    mx = fmaxf(mx, z[e]);
  }
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float gm = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) gm = fmaxf(gm, red[w]);
  __syncthreads();  // red is reused below
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    z[e] = __expf(z[e] - gm);  // exp(-inf) = 0 for padding
    sum += z[e];
  }
  sum = warp_sum(sum);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
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

template <int VPL>
cudaError_t launch_v3(const bf16_t* W, const bf16_t* h, const int32_t* ids, int64_t n, int d,
                      int M, int K, float* logits, float* q, float inv_temp, int* tickets,
                      int* err, cudaStream_t s) {
  const size_t row_bytes = (size_t)d * 2;
  int slots = (int)((200 * 1024) / row_bytes);
  if (slots > kMaxSlots) slots = kMaxSlots;
  const size_t smem = (size_t)slots * row_bytes;
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(gather_logits_v3_kernel<VPL>, smem, smem_set);
  if (e != cudaSuccess) return e;
  const int64_t total = (int64_t)M * K;
  const int grid = (int)(total < (int64_t)sm_count() ? total : (int64_t)sm_count());
  gather_logits_v3_kernel<VPL><<<grid, kV3Threads, smem, s>>>(W, h, ids, n, d, M, K, slots,
                                                              logits, q, inv_temp, tickets, err);
  return cudaGetLastError();
}

cudaError_t launch_gather_logits(const bf16_t* W, const bf16_t* h, const int32_t* ids, int64_t n,
                                 int d, int M, int K, float* logits, float* q, float inv_temp,
                                 int* tickets, int* err, cudaStream_t s) {
  const int vpl = (d + 255) / 256;  // 16-byte vectors per lane
  if (gather_engine() == 3 && vpl <= 20) {
  if (vpl <= 1) return launch_v3<1>(W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s);
  if (vpl <= 2) return launch_v3<2>(W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s);
  if (vpl <= 4) return launch_v3<4>(W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s);
  if (vpl <= 8) return launch_v3<8>(W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s);
  if (vpl <= 12) return launch_v3<12>(W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s);
  if (vpl <= 16) return launch_v3<16>(W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s);
  if (vpl <= 20) return launch_v3<20>(W, h, ids, n, d, M, K, logits, q, inv_temp, tickets, err, s);
  }
  const int64_t total = (int64_t)M * K;
  const unsigned grid = (unsigned)((total + kWarpsPerCta - 1) / kWarpsPerCta);
  return launch_kernel(true, gather_logits_kernel, dim3(grid), dim3(kWarpsPerCta * 32), 0, s, W, h,
                       ids, n, d, M, K, logits, q, inv_temp, tickets, err);
}

cudaError_t launch_row_softmax(const float* L, int M, int64_t K, float inv_temp, float* q,
                               cudaStream_t s) {
  if (K <= 256 * 4)
    return launch_kernel(true, row_softmax_reg_kernel<4>, dim3(M), dim3(256), 0, s, L, (int)K,
                         inv_temp, q);
  if (K <= 256 * 16)
    return launch_kernel(true, row_softmax_reg_kernel<16>, dim3(M), dim3(256), 0, s, L, (int)K,
                         inv_temp, q);
  return launch_kernel(true, row_softmax_kernel, dim3(M), dim3(256), 0, s, L, K, inv_temp, q);
}

}  // namespace lmhead
