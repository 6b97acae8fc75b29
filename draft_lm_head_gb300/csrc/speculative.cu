// The steps after the draft distribution q.
//
// K8 draft selection ("EAGLE -> EAGLE-2 -> EAGLE-3 -> DFlash", EAGLE-2
// dynamic draft tree, Expansion Phase): per row (one node of the draft tree)
// the k_sel most likely draft tokens by q (ties: smaller vocabulary id) with
// their path values parent_value * q, and optionally one token drawn from q
// by the Gumbel-max construction on caller-supplied uniforms. One CTA per row.
//
// K9 chain verification ("Speculative decoding and EAGLE", exactness rule):
// for each drafted token x_t, accept if r_t < p_t(x_t) / q_t(x_t); otherwise
// draw the replacement from (p_t - q_t)+ normalised (q_t is the head's
// candidate-supported distribution, zero outside the row's candidates) and
// stop; when every draft is accepted, draw a bonus token from p_Kd. Draws
// use the inverse CDF in vocabulary order with one caller-supplied uniform.
// One CTA per chain: the candidates of the rejected position go into a
// shared-memory hash table, each thread sums the residual over a contiguous
// slice of the vocabulary, a block scan places the draw.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

constexpr int kSelThreads = 256;

// a beats b: larger q, then smaller id
__device__ __forceinline__ bool q_beats(float qa, int32_t ia, float qb, int32_t ib) {
  return qa > qb || (qa == qb && ia < ib);
}

// Block-wide arg-best over (key, id) pairs: larger key wins, then smaller id.
// Every thread returns the winner. sh: 2 * kSelThreads / 32 words.
__device__ __forceinline__ void block_best(float& key, int32_t& id, int& who, float* shk, int* shi,
                                           int* shw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ok = __shfl_xor_sync(0xFFFFFFFFu, key, off);
    const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, id, off);
    const int ow = __shfl_xor_sync(0xFFFFFFFFu, who, off);
    if (q_beats(ok, oi, key, id)) { key = ok; id = oi; who = ow; }
  }
  if (lane == 0) { shk[warp] = key; shi[warp] = id; shw[warp] = who; }
  cta_sync();
  key = shk[0]; id = shi[0]; who = shw[0];
  for (int w = 1; w < nw; ++w)
    if (q_beats(shk[w], shi[w], key, id)) { key = shk[w]; id = shi[w]; who = shw[w]; }
  cta_sync();  // the scratch is reused by the next call
}

template <int KT>
__global__ void __launch_bounds__(kSelThreads)
draft_select_kernel(const float* __restrict__ q, const int32_t* __restrict__ ids, int K, int k_sel,
                    const float* __restrict__ parent_value, const float* __restrict__ uniforms,
                    int32_t* __restrict__ top_ids, float* __restrict__ top_q,
                    float* __restrict__ top_value, int32_t* __restrict__ sample_id,
                    float* __restrict__ sample_q) {
  __shared__ float lq[kSelThreads][KT];
  __shared__ int32_t li[kSelThreads][KT];
  __shared__ float shk[kSelThreads / 32];
  __shared__ int shi[kSelThreads / 32], shw[kSelThreads / 32];
  const int tid = threadIdx.x;
  const size_t row = (size_t)blockIdx.x * K;
  pdl_wait();  // q comes from the previous kernel
  // this thread's sorted top-KT of its strided share, kept in shared memory
  for (int i = 0; i < KT; ++i) { lq[tid][i] = -INFINITY; li[tid][i] = 0x7FFFFFFF; }
  float gk = -INFINITY;  // Gumbel-max: best perturbed log q of this thread
  int32_t gi = 0x7FFFFFFF;
  int gj = -1;
  for (int j = tid; j < K; j += kSelThreads) {
    const float qj = q[row + j];
    const int32_t id = ids[row + j];
    if (q_beats(qj, id, lq[tid][KT - 1], li[tid][KT - 1])) {
      int pos = KT - 1;
      while (pos > 0 && q_beats(qj, id, lq[tid][pos - 1], li[tid][pos - 1])) {
        lq[tid][pos] = lq[tid][pos - 1];
        li[tid][pos] = li[tid][pos - 1];
        --pos;
      }
      lq[tid][pos] = qj;
      li[tid][pos] = id;
    }
    if (uniforms) {
      const float s = qj > 0.f ? logf(qj) - logf(-logf(uniforms[row + j])) : -INFINITY;
      if (gj < 0 || q_beats(s, id, gk, gi)) { gk = s; gi = id; gj = j; }
    }
  }
  // k_sel rounds: the best head over all threads' lists is the next output
  int head = 0;
  const float pv = parent_value ? parent_value[blockIdx.x] : 1.f;
  for (int k = 0; k < k_sel; ++k) {
    float key = head < KT ? lq[tid][head] : -INFINITY;
    int32_t id = head < KT ? li[tid][head] : 0x7FFFFFFF;
    int who = tid;
    block_best(key, id, who, shk, shi, shw);
    if (tid == who) ++head;
    if (tid == 0) {
      const size_t o = (size_t)blockIdx.x * k_sel + k;
      top_ids[o] = id;
      top_q[o] = key;
      if (top_value) top_value[o] = pv * key;
    }
  }
  if (uniforms) {
    int who = gj;  // carries the index of the winner's element
    block_best(gk, gi, who, shk, shi, shw);
    if (tid == 0) {
      if (sample_id) sample_id[blockIdx.x] = gi;
      if (sample_q) sample_q[blockIdx.x] = who >= 0 ? q[row + who] : 0.f;
    }
  }
}

// ---------------------------------------------------------------- K9
constexpr int kVerThreads = 1024;
constexpr int kHashSlots = 8192;  // >= 2 x kSelectMaxK

__device__ __forceinline__ uint32_t hash_slot(int32_t id) {
  return ((uint32_t)id * 2654435761u) >> (32 - 13);
}

// Inverse-CDF draw over w_v = max(0, p_v - q(v)) (q from the hash table, or
// none when use_q is false): the smallest v whose running sum exceeds u * W.
// Each thread sums a contiguous slice of the vocabulary; one thread turns the
// slice sums into prefix sums sequentially, so the slices' intervals
// [start_i, start_{i+1}) partition [0, W) exactly. The thread whose interval
// holds u * W walks its slice; if rounding keeps the walk from crossing, or
// u * W rounds up to W, the last positive weight of the slice (of the whole
// vocabulary) is taken. W == 0 falls back to p itself. Returns the token on
// every thread.
__device__ int residual_draw(const float* __restrict__ prow, int64_t n, bool use_q,
                             const int32_t* tkey, const float* tval, float u, float* start,
                             int* s_tok) {
  const int64_t per = (n + kVerThreads - 1) / kVerThreads;
  const int64_t v0 = (int64_t)threadIdx.x * per;
  const int64_t v1 = v0 + per < n ? v0 + per : n;
  auto weight = [&](int64_t v, bool sub) -> float {
    float w = prow[v];
    if (sub) {
      uint32_t h = hash_slot((int32_t)v);
      for (int probe = 0; probe < kHashSlots; ++probe) {
        const int32_t k = tkey[h];
        if (k == (int32_t)v) { w -= tval[h]; break; }
        if (k < 0) break;
        h = (h + 1) & (kHashSlots - 1);
      }
    }
    return w > 0.f ? w : 0.f;
  };
  for (int pass = 0; pass < 2; ++pass) {
    const bool sub = use_q && pass == 0;
    float local = 0.f;
    for (int64_t v = v0; v < v1; ++v) local += weight(v, sub);
    start[threadIdx.x + 1] = local;
    cta_sync();
    if (threadIdx.x == 0) {
      float acc = 0.f;
      start[0] = 0.f;
      for (int i = 1; i <= kVerThreads; ++i) {
        acc += start[i];
        start[i] = acc;
      }
      *s_tok = -1;
    }
    cta_sync();
    const float total = start[kVerThreads];
    if (!(total > 0.f)) {  // (p - q)+ vanishes: draw from p
      cta_sync();
      continue;
    }
    const float target = u * total;
    const float lo = start[threadIdx.x], hi = start[threadIdx.x + 1];
    if (lo <= target && target < hi) {
      float acc = lo;
      int64_t pick = -1, last_pos = -1;
      for (int64_t v = v0; v < v1; ++v) {
        const float w = weight(v, sub);
        if (w > 0.f) last_pos = v;
        acc += w;
        if (acc > target) { pick = v; break; }
      }
      *s_tok = (int)(pick >= 0 ? pick : last_pos);
    }
    cta_sync();
    if (*s_tok < 0 && hi > lo) {  // target at or past W: the last positive weight
      int64_t last_pos = -1;
      for (int64_t v = v1 - 1; v >= v0; --v)
        if (weight(v, sub) > 0.f) { last_pos = v; break; }
      if (last_pos >= 0) atomicMax(s_tok, (int)last_pos);
    }
    cta_sync();
    const int tok = *s_tok;
    cta_sync();
    return tok;
  }
  return (int)(n - 1);
}

__global__ void __launch_bounds__(kVerThreads)
verify_chain_kernel(const float* __restrict__ p, int64_t n, int Kd, const int32_t* __restrict__ x,
                    const int32_t* __restrict__ cand_ids, const float* __restrict__ cand_q, int K,
                    const float* __restrict__ r, const float* __restrict__ u,
                    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_count,
                    int* __restrict__ err) {
  extern __shared__ int32_t vsm[];
  int32_t* tkey = vsm;                                          // [kHashSlots]
  float* tval = reinterpret_cast<float*>(vsm + kHashSlots);     // [kHashSlots]
  __shared__ float start[kVerThreads + 1];
  __shared__ int s_hit, s_tok;
  const int b = blockIdx.x;
  const float* pb = p + (size_t)b * (Kd + 1) * n;
  int32_t* ob = out_tokens + (size_t)b * (Kd + 1);
  pdl_wait();  // the candidate lists may come from the previous kernel
  for (int i = threadIdx.x; i <= Kd; i += kVerThreads) ob[i] = -1;
  for (int t = 0; t < Kd; ++t) {
    const int32_t xt = x[(size_t)b * Kd + t];
    const int32_t* ci = cand_ids + ((size_t)b * Kd + t) * K;
    const float* cq = cand_q + ((size_t)b * Kd + t) * K;
    if (threadIdx.x == 0) s_hit = K;
    cta_sync();
    for (int j = threadIdx.x; j < K; j += kVerThreads)
      if (ci[j] == xt) atomicMin(&s_hit, j);
    cta_sync();
    const int hit = s_hit;
    if (hit >= K || xt < 0 || (int64_t)xt >= n) {  // not a candidate of its row
      if (threadIdx.x == 0) {
        record_error(err, kDevErrBadId);
        out_count[b] = -1;
      }
      return;
    }
    const float px = pb[(size_t)t * n + xt];
    const float qx = cq[hit];
    if (r[(size_t)b * Kd + t] < px / qx) {
      if (threadIdx.x == 0) ob[t] = xt;
      continue;
    }
    // rejected: the residual (p_t - q_t)+ over the vocabulary
    for (int i = threadIdx.x; i < kHashSlots; i += kVerThreads) tkey[i] = -1;
    cta_sync();
    for (int j = threadIdx.x; j < K; j += kVerThreads) {
      const int32_t id = ci[j];
      if (id < 0 || (int64_t)id >= n) continue;
      uint32_t h = hash_slot(id);
      for (int probe = 0; probe < kHashSlots; ++probe) {
        const int old = atomicCAS(&tkey[h], -1, id);
        if (old == -1 || old == id) {
          if (old == -1) tval[h] = cq[j];
          break;
        }
        h = (h + 1) & (kHashSlots - 1);
      }
    }
    cta_sync();
    const int tok = residual_draw(pb + (size_t)t * n, n, true, tkey, tval,
                                  u[(size_t)b * (Kd + 1) + t], start, &s_tok);
    if (threadIdx.x == 0) {
      ob[t] = tok;
      out_count[b] = t;
    }
    return;
  }
  const int tok = residual_draw(pb + (size_t)Kd * n, n, false, tkey, tval,
                                u[(size_t)b * (Kd + 1) + Kd], start, &s_tok);
  if (threadIdx.x == 0) {
    ob[Kd] = tok;
    out_count[b] = Kd;
  }
}

}  // namespace

cudaError_t launch_draft_select(const float* q, const int32_t* ids, int M, int K, int k_sel,
                                const float* parent_value, const float* uniforms, int32_t* top_ids,
                                float* top_q, float* top_value, int32_t* sample_id,
                                float* sample_q, cudaStream_t s) {
#define DS(KT)                                                                                  \
  return launch_kernel(true, draft_select_kernel<KT>, dim3(M), dim3(kSelThreads), 0, s, q, ids, K, \
                       k_sel, parent_value, uniforms, top_ids, top_q, top_value, sample_id,     \
                       sample_q)
  if (k_sel <= 1) DS(1);
  if (k_sel <= 2) DS(2);
  if (k_sel <= 4) DS(4);
  if (k_sel <= 8) DS(8);
  DS(16);
#undef DS
}

cudaError_t launch_verify_chain(const float* p, int64_t n, int B, int Kd, const int32_t* x,
                                const int32_t* cand_ids, const float* cand_q, int K, const float* r,
                                const float* u, int32_t* out_tokens, int32_t* out_count, int* err,
                                cudaStream_t s) {
  const size_t smem = (size_t)kHashSlots * (sizeof(int32_t) + sizeof(float));
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(verify_chain_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_kernel(true, verify_chain_kernel, dim3(B), dim3(kVerThreads), smem, s, p, n, Kd, x,
                       cand_ids, cand_q, K, r, u, out_tokens, out_count, err);
}

}  // namespace lmhead
