// The steps after the draft distribution q.
//
// K8 draft selection ("EAGLE -> EAGLE-2 -> EAGLE-3 -> DFlash", EAGLE-2
// dynamic draft tree, Expansion Phase): per row (one node of the draft tree)
// the k_sel most likely draft tokens by q (ties: smaller vocabulary id) with
// their path values parent_value * q, and optionally one token drawn from q
// by the Gumbel-max construction on caller-supplied uniforms. One warp per row.
//
// K9 chain verification ("Speculative decoding and EAGLE", exactness rule):
// for each drafted token x_t, accept if r_t < p_t(x_t) / q_t(x_t); otherwise
// draw the replacement from (p_t - q_t)+ normalised (q_t is the head's
// candidate-supported distribution, zero outside the row's candidates) and
// stop; when every draft is accepted, draw a bonus token from p_Kd. Draws
// use the inverse CDF in vocabulary order with one caller-supplied uniform.
// One 8-CTA cluster per chain: every CTA takes the accept decisions, puts
// the candidates of the rejected position into a shared-memory hash table and
// sums the residual over its eighth of the vocabulary (warps over contiguous
// runs, coalesced loads); the CTA totals meet in distributed shared memory and
// the CTA holding the draw places it with a scan of its run sums.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace lmhead {
namespace {

constexpr int kSelThreads = 64;  // two rows (warps) per CTA

// a beats b: larger q, then smaller id
__device__ __forceinline__ bool q_beats(float qa, int32_t ia, float qb, int32_t ib) {
  return qa > qb || (qa == qb && ia < ib);
}

// Warp-wide arg-best over (key, id) pairs: larger key wins, then smaller id;
// `who` travels with the winner. Every lane returns the winner.
__device__ __forceinline__ void warp_best(float& key, int32_t& id, int& who) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ok = __shfl_xor_sync(0xFFFFFFFFu, key, off);
    const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, id, off);
    const int ow = __shfl_xor_sync(0xFFFFFFFFu, who, off);
    if (q_beats(ok, oi, key, id)) { key = ok; id = oi; who = ow; }
  }
}

// One warp per row: every lane keeps the sorted top KT of its strided share
// of the row in registers (branch-free insertion: the comparisons against a
// sorted list are monotone, so each slot takes its own value, its upper
// neighbour's or the new one); k_sel rounds of a warp arg-best over the list
// heads then pick the outputs in order, the winning lane popping its head.
template <int KT>
__global__ void __launch_bounds__(kSelThreads)
draft_select_kernel(const float* __restrict__ q, const int32_t* __restrict__ ids, int M, int K,
                    int k_sel, const float* __restrict__ parent_value,
                    const float* __restrict__ uniforms, int32_t* __restrict__ top_ids,
                    float* __restrict__ top_q, float* __restrict__ top_value,
                    int32_t* __restrict__ sample_id, float* __restrict__ sample_q) {
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * (kSelThreads / 32) + (threadIdx.x >> 5);
  pdl_wait();  // q comes from the previous kernel
  if (m >= M) return;
  const size_t row = (size_t)m * K;
  float lq[KT];
  int32_t li[KT];
#pragma unroll
  for (int i = 0; i < KT; ++i) { lq[i] = -INFINITY; li[i] = 0x7FFFFFFF; }
  float gk = -INFINITY;  // Gumbel-max: best perturbed log q of this lane
  int32_t gi = 0x7FFFFFFF;
  int gj = -1;
  constexpr int kBatch = 8;  // elements per lane loaded together (one latency per batch)
  for (int j0 = 0; j0 < K; j0 += 32 * kBatch) {
    float qb[kBatch], ub[kBatch];
    int32_t ib[kBatch];
#pragma unroll
    for (int bb = 0; bb < kBatch; ++bb) {
      const int j = j0 + bb * 32 + lane;
      const bool in = j < K;
      qb[bb] = in ? __ldg(q + row + j) : -INFINITY;
      ib[bb] = in ? __ldg(ids + row + j) : 0x7FFFFFFF;
      ub[bb] = (in && uniforms) ? __ldg(uniforms + row + j) : 0.5f;
    }
#pragma unroll
    for (int bb = 0; bb < kBatch; ++bb) {
      const int j = j0 + bb * 32 + lane;
      if (j >= K) break;
      const float qj = qb[bb];
      const int32_t id = ib[bb];
      bool c[KT];
#pragma unroll
      for (int i = 0; i < KT; ++i) c[i] = q_beats(qj, id, lq[i], li[i]);
#pragma unroll
      for (int i = KT - 1; i > 0; --i) {
        lq[i] = c[i] ? (c[i - 1] ? lq[i - 1] : qj) : lq[i];
        li[i] = c[i] ? (c[i - 1] ? li[i - 1] : id) : li[i];
      }
      lq[0] = c[0] ? qj : lq[0];
      li[0] = c[0] ? id : li[0];
      if (uniforms) {
        const float sj = qj > 0.f ? logf(qj) - logf(-logf(ub[bb])) : -INFINITY;
        if (gj < 0 || q_beats(sj, id, gk, gi)) { gk = sj; gi = id; gj = j; }
      }
    }
  }
  const float pv = parent_value ? parent_value[m] : 1.f;
  for (int k = 0; k < k_sel; ++k) {
    float key = lq[0];
    int32_t id = li[0];
    int who = lane;
    warp_best(key, id, who);
    if (lane == who) {  // pop the head
#pragma unroll
      for (int i = 0; i + 1 < KT; ++i) { lq[i] = lq[i + 1]; li[i] = li[i + 1]; }
      lq[KT - 1] = -INFINITY;
      li[KT - 1] = 0x7FFFFFFF;
    }
    if (lane == 0) {
      const size_t o = (size_t)m * k_sel + k;
      top_ids[o] = id;
      top_q[o] = key;
      if (top_value) top_value[o] = pv * key;
    }
  }
  if (uniforms) {
    int who = gj;  // carries the index of the winner's element
    warp_best(gk, gi, who);
    if (lane == 0) {
      if (sample_id) sample_id[m] = gi;
      if (sample_q) sample_q[m] = who >= 0 ? q[row + who] : 0.f;
    }
  }
}

// ---------------------------------------------------------------- K9
constexpr int kVerThreads = 1024;
constexpr int kVerCluster = 8;     // CTAs per chain (the vocabulary is split over them)
constexpr int kMaxDrafts = 1024;   // drafts per chain (the entry point's bound)
constexpr int kMaxCpw = 64;        // chunk sums kept per warp for the walk
constexpr int kHashSlots = 8192;  // >= 2 x kSelectMaxK

__device__ __forceinline__ uint32_t hash_slot(int32_t id) {
  return ((uint32_t)id * 2654435761u) >> (32 - 13);
}

// Inverse-CDF draw over w_v = max(0, p_v - q(v)) (q from the hash table, or
// none when use_q is false): the smallest v whose running sum exceeds u * W.
// The vocabulary is split over the kVerCluster CTAs of the chain's cluster
// (CTA `rank` owns a contiguous run of 32-entry chunks) and, inside a CTA,
// over its warps. Every warp sums its run (coalesced loads, lane partials,
// one warp reduction); CTA totals are summed in warp order and exchanged
// through distributed shared memory, so every CTA sees the same CTA totals
// and the same W, and the target u * W falls into exactly one CTA's interval
// (CTA offsets chain the totals in rank order). Inside that CTA the warp
// whose interval holds the target walks its run again in blocks of 32 chunks
// (one chunk sum per lane, a scan over them) and, in the crossing chunk,
// takes the first entry whose running sum passes the target. Where rounding
// keeps a walk from crossing, or u * W rounds up to W, the last positive
// weight of the run (of the vocabulary) is taken. W == 0 falls back to p
// itself. Returns the token in the CTA that drew it and -1 in the others.
__device__ int residual_draw(const float* __restrict__ prow, int64_t n, bool use_q,
                             const int32_t* tkey, const float* tval, float u, float* wtot,
                             int* s_tok, float* cta_tot, float* csum, int rank) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kVerThreads / 32;
  const int64_t nch = (n + 31) / 32;
  const int64_t cpc = (nch + kVerCluster - 1) / kVerCluster;  // chunks per CTA
  const int64_t s0 = rank * cpc < nch ? rank * cpc : nch;
  const int64_t s1 = s0 + cpc < nch ? s0 + cpc : nch;
  const int64_t cpw = (s1 - s0 + kWarps - 1) / kWarps;
  const int64_t c0 = s0 + warp * cpw < s1 ? s0 + warp * cpw : s1;
  const int64_t c1 = c0 + cpw < s1 ? c0 + cpw : s1;
  auto weight = [&](int64_t v, bool sub) -> float {
    if (v >= n) return 0.f;
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
  // runs of at most kMaxCpw chunks keep their chunk sums in shared memory, so
  // the walk reads the vocabulary again only in the crossing chunk
  const bool keep = cpw <= kMaxCpw;
  float* cs_w = csum + warp * kMaxCpw;
  for (int pass = 0; pass < 2; ++pass) {
    const bool sub = use_q && pass == 0;
    float run = 0.f;  // chunk sums added in chunk order (identical in every lane)
#pragma unroll 8
    for (int64_t c = c0; c < c1; ++c) {
      const float cs = warp_sum(weight(c * 32 + lane, sub));  // coalesced: one chunk per load
      if (keep && lane == 0) cs_w[c - c0] = cs;
      run += cs;
    }
    if (lane == 0) wtot[warp] = run;
    if (threadIdx.x == 0) *s_tok = -1;
    cta_sync();
    float woff = 0.f, ctot = 0.f;  // this warp's offset inside the CTA, the CTA total
    for (int w = 0; w < kWarps; ++w) {
      if (w == warp) woff = ctot;
      ctot += wtot[w];
    }
    if (threadIdx.x == 0) *cta_tot = ctot;
    tc::cluster_sync();  // every CTA total is published
    float coff = 0.f, total = 0.f;
    int last_pos_rank = -1;
    const uint32_t tot_addr = tc::smem_addr(cta_tot);
    for (int rr = 0; rr < kVerCluster; ++rr) {
      const float tr = tc::ld_cluster_f32(tc::map_to_rank(tot_addr, (uint32_t)rr));
      if (rr == rank) coff = total;
      if (tr > 0.f) last_pos_rank = rr;
      total += tr;
    }
    tc::cluster_sync();  // the totals have been read before any CTA moves on or exits
    if (!(total > 0.f)) continue;  // (p - q)+ vanishes: draw from p (same in every CTA)
    const float target = u * total;
    const float chi = rank + 1 < kVerCluster ? coff + ctot : total;
    const bool past_end = !(target < total);  // u * W rounded up to W
    const bool mine = (coff <= target && target < chi) || (past_end && rank == last_pos_rank);
    if (!mine) return -1;
    const float off = coff + woff;
    const float hi = warp + 1 < kWarps ? off + wtot[warp] : chi;
    if (!past_end && off <= target && target < hi) {
      float acc = off;
      int64_t pick = -1, last_pos = -1;
      for (int64_t b = c0; b < c1 && pick < 0; b += 32) {
        const int64_t c = b + lane;
        float cs = 0.f;
        if (c < c1) {
          if (keep) {
            cs = cs_w[c - c0];
          } else {
#pragma unroll 8
            for (int i = 0; i < 32; ++i) cs += weight(c * 32 + i, sub);
          }
        }
        float sc = cs;  // inclusive scan of the chunk sums
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(0xFFFFFFFFu, sc, o);
          if (lane >= o) sc += t;
        }
        const uint32_t pos = __ballot_sync(0xFFFFFFFFu, cs > 0.f);
        if (pos) last_pos = b + 31 - __clz(pos);  // last chunk with weight (refined below)
        const uint32_t cross = __ballot_sync(0xFFFFFFFFu, c < c1 && cs > 0.f && acc + sc > target);
        if (cross) {
          const int k = __ffs(cross) - 1;
          const float before = acc + __shfl_sync(0xFFFFFFFFu, sc - cs, k);
          const int64_t cc = b + k;
          const float wl = weight(cc * 32 + lane, sub);
          float se = wl;  // inclusive scan over the chunk's entries
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xFFFFFFFFu, se, o);
            if (lane >= o) se += t;
          }
          const uint32_t hit = __ballot_sync(0xFFFFFFFFu, wl > 0.f && before + se > target);
          const uint32_t wpos = __ballot_sync(0xFFFFFFFFu, wl > 0.f);
          pick = hit ? cc * 32 + __ffs(hit) - 1 : cc * 32 + 31 - __clz(wpos);
        }
        acc += __shfl_sync(0xFFFFFFFFu, sc, 31);
      }
      if (pick < 0 && last_pos >= 0) {  // rounding kept the walk short: last positive entry
        const uint32_t wpos = __ballot_sync(0xFFFFFFFFu, weight(last_pos * 32 + lane, sub) > 0.f);
        pick = last_pos * 32 + 31 - __clz(wpos);
      }
      if (lane == 0) *s_tok = (int)pick;
    }
    cta_sync();
    if (*s_tok < 0 && wtot[warp] > 0.f) {  // target at or past this CTA's end: last positive weight
      int64_t last_pos = -1;
      for (int64_t c = c1 - 1; c >= c0 && last_pos < 0; --c) {
        const uint32_t pos = __ballot_sync(0xFFFFFFFFu, weight(c * 32 + lane, sub) > 0.f);
        if (pos) last_pos = c * 32 + 31 - __clz(pos);
      }
      if (lane == 0 && last_pos >= 0) atomicMax(s_tok, (int)last_pos);
    }
    cta_sync();
    const int tok = *s_tok;
    cta_sync();
    return tok;
  }
  // p itself sums to zero (invalid input): the last entry, drawn by the last CTA
  return rank == kVerCluster - 1 ? (int)(n - 1) : -1;
}

__global__ void __cluster_dims__(kVerCluster, 1, 1) __launch_bounds__(kVerThreads, 1)
verify_chain_kernel(const float* __restrict__ p, int64_t n, int Kd, const int32_t* __restrict__ x,
                    const int32_t* __restrict__ cand_ids, const float* __restrict__ cand_q, int K,
                    const float* __restrict__ r, const float* __restrict__ u,
                    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_count,
                    int* __restrict__ err) {
  extern __shared__ int32_t vsm[];
  int32_t* tkey = vsm;                                          // [kHashSlots]
  float* tval = reinterpret_cast<float*>(vsm + kHashSlots);     // [kHashSlots]
  __shared__ float wtot[kVerThreads / 32];
  __shared__ float cta_tot;
  __shared__ float csum[(kVerThreads / 32) * kMaxCpw];
  __shared__ int s_tok;
  __shared__ int s_hit[kMaxDrafts];              // each draft's position in its candidates
  __shared__ unsigned char s_state[kMaxDrafts];  // 0 not a candidate, 1 accepted, 2 rejected
  const int b = blockIdx.y;
  const int rank = (int)tc::cluster_ctarank();
  const float* pb = p + (size_t)b * (Kd + 1) * n;
  int32_t* ob = out_tokens + (size_t)b * (Kd + 1);
  pdl_wait();  // the candidate lists may come from the previous kernel
  // CTA 0 writes the accepted drafts and the count; the CTA that draws the
  // last token writes it (after the cluster barriers inside the draw, so
  // after CTA 0's initialisation below)
  if (rank == 0)
    for (int i = threadIdx.x; i <= Kd; i += kVerThreads) ob[i] = -1;
  // every draft's accept test at once (each CTA of the cluster computes the
  // same decisions): its position among its row's candidates, then
  // r_t < p_t(x_t) / q_t(x_t) in fp32
  for (int t = threadIdx.x; t < Kd; t += kVerThreads) s_hit[t] = K;
  cta_sync();
  const int64_t pairs = (int64_t)Kd * K;
  for (int64_t e = threadIdx.x; e < pairs; e += kVerThreads) {
    const int t = (int)(e / K);
    const int j = (int)(e - (int64_t)t * K);
    if (cand_ids[(size_t)b * Kd * K + e] == x[(size_t)b * Kd + t]) atomicMin(&s_hit[t], j);
  }
  cta_sync();
  for (int t = threadIdx.x; t < Kd; t += kVerThreads) {
    const int32_t xt = x[(size_t)b * Kd + t];
    const int hit = s_hit[t];
    int st = 0;  // not a candidate of its row
    if (hit < K && xt >= 0 && (int64_t)xt < n) {
      const float px = pb[(size_t)t * n + xt];
      const float qx = cand_q[((size_t)b * Kd + t) * K + hit];
      st = r[(size_t)b * Kd + t] < px / qx ? 1 : 2;  // accepted : rejected
    }
    s_state[t] = (unsigned char)st;
  }
  cta_sync();
  int stop = Kd;  // the first draft not accepted, in order
  bool bad = false;
  for (int t = 0; t < Kd; ++t) {
    const int st = s_state[t];
    if (st == 1) continue;
    bad = st == 0;
    stop = t;
    break;
  }
  if (bad) {
    if (rank == 0 && threadIdx.x == 0) {
      record_error(err, kDevErrBadId);
      out_count[b] = -1;
    }
    return;
  }
  if (rank == 0)
    for (int t = threadIdx.x; t < stop; t += kVerThreads) ob[t] = x[(size_t)b * Kd + t];
  if (stop < Kd) {
    // rejected: the residual (p_t - q_t)+ over the vocabulary
    const int t = stop;
    const int32_t* ci = cand_ids + ((size_t)b * Kd + t) * K;
    const float* cq = cand_q + ((size_t)b * Kd + t) * K;
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
                                  u[(size_t)b * (Kd + 1) + t], wtot, &s_tok, &cta_tot, csum, rank);
    if (threadIdx.x == 0) {
      if (tok >= 0) ob[t] = tok;
      if (rank == 0) out_count[b] = t;
    }
    return;
  }
  const int tok = residual_draw(pb + (size_t)Kd * n, n, false, tkey, tval,
                                u[(size_t)b * (Kd + 1) + Kd], wtot, &s_tok, &cta_tot, csum, rank);
  if (threadIdx.x == 0) {
    if (tok >= 0) ob[Kd] = tok;
    if (rank == 0) out_count[b] = Kd;
  }
}

}  // namespace

cudaError_t launch_draft_select(const float* q, const int32_t* ids, int M, int K, int k_sel,
                                const float* parent_value, const float* uniforms, int32_t* top_ids,
                                float* top_q, float* top_value, int32_t* sample_id,
                                float* sample_q, cudaStream_t s) {
  const unsigned grid = (unsigned)((M + kSelThreads / 32 - 1) / (kSelThreads / 32));
#define DS(KT)                                                                                  \
  return launch_kernel(true, draft_select_kernel<KT>, dim3(grid), dim3(kSelThreads), 0, s, q, ids, \
                       M, K, k_sel, parent_value, uniforms, top_ids, top_q, top_value,          \
                       sample_id, sample_q)
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
  return launch_kernel(true, verify_chain_kernel, dim3(kVerCluster, B), dim3(kVerThreads), smem, s,
                       p, n, Kd, x, cand_ids, cand_q, K, r, u, out_tokens, out_count, err);
}

}  // namespace lmhead
