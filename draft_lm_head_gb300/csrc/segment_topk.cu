// K3: exact Top-k over segments of a score matrix (EAGLE-4 notes, "A Local
// Top-k based variant": the original flow's ids = topk(scores, C) reads the
// full-vocabulary scores back from HBM).
//
// A segment is `seg_len` consecutive positions of one row of S (M x n fp32);
// the global Top-C is one segment of length n, the local variant with a large
// k_tile is one segment per tile. Order: score descending, then the smaller
// vocabulary id (token_ids[p], identity when null). Every element maps to a
// unique 64-bit key (order-preserving score bits, then the complemented id),
// so the k-th largest key is a unique threshold.
//
// Long segments: multi-pass radix select on 12-bit digits of the key (each
// pass one read of the segment, histogram in shared memory) until the
// boundary digit holds few enough keys for shared memory, then one collection
// pass and a bitonic sort of the survivors. Short segments (<= 8192 keys):
// loaded whole and bitonic-sorted.
#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

constexpr int kThreads = 1024;
constexpr int kCap = kSelectMaxK;  // keys of the selected / candidate regions
constexpr int kBins = 4096;        // 12-bit digits
constexpr int kDigit = 12;

__device__ __forceinline__ uint64_t key_at(const float* __restrict__ row,
                                           const int32_t* __restrict__ token_ids, int64_t p) {
  const int32_t id = token_ids ? __ldg(token_ids + p) : (int32_t)p;
  return select_key(__ldcg(row + p), id);
}

// Sort keys[0..P) descending, P a power of two, all threads participate
// (blockDim.x a multiple of 32). Pair i of a stage touches elements of the
// 64-element chunk i / 32 when the stride is at most 32, and warp w handles
// pairs w*32 + 32*blockDim.x/32*k + lane, i.e. only its own chunks: such
// stages need only a warp barrier after them unless the next stage reaches
// across chunks (stride 64 and up), which needs the CTA barrier.
__device__ void bitonic_desc(uint64_t* keys, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        const int pos = 2 * i - (i & (stride - 1));
        const int par = pos + stride;
        const uint64_t a = keys[pos], b = keys[par];
        const bool desc_block = (pos & size) == 0;
        if (desc_block ? (a < b) : (a > b)) {
          keys[pos] = b;
          keys[par] = a;
        }
      }
      const int next = stride > 1 ? stride >> 1 : size;  // the next stage's stride
      if (stride >= 64 || next >= 64) {
        cta_sync();
      } else {
        __syncwarp();
      }
    }
  }
  cta_sync();
}

__device__ __forceinline__ int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// grid: (segments, M). Dynamic smem: 2*kCap keys + kBins counters + scan.
__global__ void __launch_bounds__(kThreads)
segment_topk_kernel(const float* __restrict__ S, const int32_t* __restrict__ token_ids,
                    int64_t n, int64_t seg_len, int k, int K, int32_t* __restrict__ out_ids,
                    float* __restrict__ out_scores) {
  extern __shared__ uint64_t keys[];  // [0,kCap) selected, [kCap,2kCap) candidates
  uint32_t* hist = reinterpret_cast<uint32_t*>(keys + 2 * kCap);
  uint32_t* part = hist + kBins;  // kThreads partial sums
  __shared__ uint64_t s_lo, s_hi;
  __shared__ int s_gt, s_bin_count, s_sel, s_cand;

  const int tid = threadIdx.x;
  const int m = blockIdx.y;
  const int64_t seg = blockIdx.x;
  const int64_t p0 = seg * seg_len;
  const int64_t p1 = min(n, p0 + seg_len);
  const int len = (int)(p1 - p0);
  const int kk = min(k, len);
  const float* row = S + (size_t)m * n;
  const size_t obase = (size_t)m * K + (size_t)seg * k;

  if (len <= 2 * kCap) {
    const int P = pow2_at_least(len);
    for (int i = tid; i < P; i += blockDim.x) keys[i] = i < len ? key_at(row, token_ids, p0 + i) : 0ull;
    cta_sync();
    bitonic_desc(keys, P);
    for (int j = tid; j < kk; j += blockDim.x) {
      out_ids[obase + j] = key_id(keys[j]);
      if (out_scores) out_scores[obase + j] = key_score(keys[j]);
    }
    return;
  }

  uint64_t lo = 0ull, hi = ~0ull;
  int gt = 0;  // keys above hi (all selected)
  for (int shift = 64 - kDigit;; shift = shift >= kDigit ? shift - kDigit : 0) {
    for (int i = tid; i < kBins; i += blockDim.x) hist[i] = 0;
    cta_sync();
    for (int64_t p = p0 + tid; p < p1; p += blockDim.x) {
      const uint64_t key = key_at(row, token_ids, p);
      if (key >= lo && key <= hi) atomicAdd(&hist[(key >> shift) & (kBins - 1)], 1u);
    }
    cta_sync();
    // suffix sums over threads' groups of 4 bins (bins descending = keys descending)
    const int g = kThreads - 1 - tid;  // thread tid owns bins [4g, 4g+4)
    uint32_t local = hist[4 * g] + hist[4 * g + 1] + hist[4 * g + 2] + hist[4 * g + 3];
    part[tid] = local;
    cta_sync();
    for (int off = 1; off < kThreads; off <<= 1) {
      const uint32_t v = tid >= off ? part[tid - off] : 0u;
      cta_sync();
      part[tid] += v;
      cta_sync();
    }
    // part[tid] = keys in bins >= 4g (inclusive); above = keys in bins >= 4g+4
    uint32_t above = part[tid] - local;
    const uint32_t need = (uint32_t)(kk - gt);
    if (above < need && above + local >= need) {
      for (int b = 4 * g + 3; b >= 4 * g; --b) {
        if (above + hist[b] >= need) {
          s_gt = gt + (int)above;
          s_bin_count = (int)hist[b];
          const uint64_t prefix = (lo & ~((((uint64_t)kBins - 1) << shift) | ((1ull << shift) - 1ull)));
          const uint64_t nlo = prefix | ((uint64_t)b << shift);
          s_lo = nlo;
          s_hi = nlo | ((1ull << shift) - 1ull);
          break;
        }
        above += hist[b];
      }
    }
    cta_sync();
    lo = s_lo;
    hi = s_hi;
    gt = s_gt;
    const int bin_count = s_bin_count;
    cta_sync();
    if (bin_count <= kCap || shift == 0) break;
  }

  if (tid == 0) { s_sel = 0; s_cand = 0; }
  cta_sync();
  for (int64_t p = p0 + tid; p < p1; p += blockDim.x) {
    const uint64_t key = key_at(row, token_ids, p);
    if (key > hi) {
      keys[atomicAdd(&s_sel, 1)] = key;
    } else if (key >= lo) {
      const int c = atomicAdd(&s_cand, 1);
      if (c < kCap) keys[kCap + c] = key;
    }
  }
  cta_sync();
  const int ncand = min(s_cand, kCap);
  const int P = pow2_at_least(ncand);
  for (int i = ncand + tid; i < P; i += blockDim.x) keys[kCap + i] = 0ull;
  cta_sync();
  bitonic_desc(keys + kCap, P);
  const int take = kk - gt;
  for (int i = tid; i < take; i += blockDim.x) keys[gt + i] = keys[kCap + i];
  const int Ps = pow2_at_least(kk);
  for (int i = kk + tid; i < Ps; i += blockDim.x) keys[i] = 0ull;
  cta_sync();
  bitonic_desc(keys, Ps);
  for (int j = tid; j < kk; j += blockDim.x) {
    out_ids[obase + j] = key_id(keys[j]);
    if (out_scores) out_scores[obase + j] = key_score(keys[j]);
  }
}

// ---------------------------------------------------------------- long rows, few rows
// Global Top-k of rows too long for one CTA to sweep quickly (one CTA per row
// does every radix pass over the whole row: ~100 us at n = 128256). Here G
// CTAs share a row. Pass kernels (kMsPasses launches, 12-bit digits from the
// top of the key): each CTA histograms the keys of its segment that lie in
// the row's current range [lo, hi] and adds the histogram into the row's
// global one; the last CTA of the row to finish (atomic ticket, no waiting)
// finds the boundary digit, narrows [lo, hi], counts the keys above it and
// marks the row done once the range holds at most kMsDone keys (fp32 scores
// need two passes in practice: the first 12-bit digit is a sign, the
// exponent and three mantissa bits). Collection kernel: every CTA appends its keys above
// the range and inside it to two per-row lists; the last CTA sorts the
// survivors (at most k + kCap keys) and writes the row's Top-k, score
// descending, ties by the smaller vocabulary id (the keys are unique). A row
// the passes left unfinished (more than kCap keys sharing 24 key bits) is
// finished by the collection kernel's last CTA alone, with the remaining
// passes over the whole row.
constexpr int kMsThreads = 1024;
constexpr int kMsPasses = 2;      // launched passes; later digits in the fallback
constexpr int kMsStateInts = 16;  // per-row state, then the row's kBins histogram
// A row is done once its boundary range holds at most this many keys: the
// collection's last CTA then sorts about C + kMsDone keys, not C + kCap (the
// first digit of fp32 scores often leaves a few thousand keys in range).
constexpr int kMsDone = 512;

struct MsState {
  unsigned long long lo, hi;  // current key range (meaningful once pass > 0)
  int gt;                     // keys above hi
  int done;                   // the range holds <= kCap keys
  int ticket;                 // CTAs of the row finished with the current kernel
  int pass;                   // passes completed
  int n_sel, n_cand;          // collection counters
};
static_assert(sizeof(MsState) <= kMsStateInts * sizeof(int), "state slot");

struct MsBoundary {
  unsigned long long lo, hi;
  int above, count;
};

__device__ __forceinline__ int64_t ms_seg(int64_t n, int G) { return (n + G - 1) / G; }
__device__ __forceinline__ int ms_shift(int pass) { return max(0, 64 - kDigit * (pass + 1)); }

// Every thread of the CTA (kMsThreads): with hist[] the kBins counts of the
// keys in [lo, hi] by the digit at `shift`, find the bin holding the need-th
// largest such key; thread that finds it writes *out (the narrowed range, the
// keys above the bin, the bin's count).
__device__ void ms_boundary(const uint32_t* hist, uint32_t* part, uint32_t need, int shift,
                            uint64_t lo, MsBoundary* out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = kMsThreads - 1 - tid;  // thread tid owns bins [4g, 4g+4), descending order
  const uint32_t local = hist[4 * g] + hist[4 * g + 1] + hist[4 * g + 2] + hist[4 * g + 3];
  // inclusive prefix over threads (thread 0 holds the top bins): a warp scan,
  // then a scan of the 32 warp totals by warp 0 (part[] holds them)
  uint32_t v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) part[warp] = v;
  cta_sync();
  if (warp == 0) {
    const uint32_t tot = part[lane];
    uint32_t w = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += t;
    }
    part[lane] = w - tot;  // keys in the bins of the warps before
  }
  cta_sync();
  uint32_t above = v + part[warp] - local;  // keys in bins above this thread's
  if (above < need && above + local >= need) {
    for (int b = 4 * g + 3; b >= 4 * g; --b) {
      if (above + hist[b] >= need) {
        const uint64_t prefix = lo & ~((((uint64_t)kBins - 1) << shift) | ((1ull << shift) - 1ull));
        const uint64_t nlo = prefix | ((uint64_t)b << shift);
        out->lo = nlo;
        out->hi = nlo | ((1ull << shift) - 1ull);
        out->above = (int)above;
        out->count = (int)hist[b];
        break;
      }
      above += hist[b];
    }
  }
  cta_sync();
}

// grid (G, M). `zero`: M x (kMsStateInts + kBins) ints, zero before the
// first pass of a call.
__global__ void __launch_bounds__(kMsThreads)
ms_pass_kernel(const float* __restrict__ S, const int32_t* __restrict__ token_ids, int64_t n,
               int k, int* __restrict__ zero) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t part[kMsThreads];
  __shared__ MsBoundary bnd;
  __shared__ int s_last;
  const int tid = threadIdx.x, G = gridDim.x, m = blockIdx.y;
  int* zr = zero + (size_t)m * (kMsStateInts + kBins);
  MsState* st = reinterpret_cast<MsState*>(zr);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(zr + kMsStateInts);
  pdl_wait();  // scores, and the state the previous pass left
  pdl_trigger();
  if (*reinterpret_cast<volatile int*>(&st->done)) return;
  const int pass = st->pass;
  const uint64_t lo = pass ? st->lo : 0ull, hi = pass ? st->hi : ~0ull;
  const int gt = st->gt;
  const int shift = ms_shift(pass);
  const int64_t per = ms_seg(n, G);
  const int64_t p0 = (int64_t)blockIdx.x * per, p1 = min(n, p0 + per);
  const float* row = S + (size_t)m * n;
  for (int i = tid; i < kBins; i += kMsThreads) hist[i] = 0;
  cta_sync();
  for (int64_t p = p0 + tid; p < p1; p += kMsThreads) {
    const uint64_t key = key_at(row, token_ids, p);
    if (key >= lo && key <= hi) atomicAdd(&hist[(key >> shift) & (kBins - 1)], 1u);
  }
  cta_sync();
  for (int i = tid; i < kBins; i += kMsThreads)
    if (hist[i]) atomicAdd(&ghist[i], hist[i]);
  __threadfence();
  cta_sync();
  if (tid == 0) s_last = atomicAdd(&st->ticket, 1) == G - 1;
  cta_sync();
  if (!s_last) return;
  // the last CTA of the row: the row's histogram is complete
  __threadfence();
  for (int i = tid; i < kBins; i += kMsThreads) {
    hist[i] = __ldcg(ghist + i);
    ghist[i] = 0;  // ready for the next pass
  }
  cta_sync();
  ms_boundary(hist, part, (uint32_t)(min((int64_t)k, n) - gt), shift, lo, &bnd);
  if (tid == 0) {
    st->lo = bnd.lo;
    st->hi = bnd.hi;
    st->gt = gt + bnd.above;
    st->done = (bnd.count <= kMsDone || shift == 0) ? 1 : 0;
    st->pass = pass + 1;
    st->ticket = 0;
  }
}

// grid (G, M); dynamic shared memory: the last CTA's sort buffer (2 kCap
// keys), then a histogram and scan space for the fallback passes.
__global__ void __launch_bounds__(kMsThreads)
ms_collect_kernel(const float* __restrict__ S, const int32_t* __restrict__ token_ids, int64_t n,
                  int k, int* __restrict__ zero, uint64_t* __restrict__ sel,
                  uint64_t* __restrict__ cand, int32_t* __restrict__ out_ids,
                  float* __restrict__ out_scores) {
  extern __shared__ uint64_t keys[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(keys + 2 * kCap);
  uint32_t* part = hist + kBins;
  __shared__ MsBoundary bnd;
  __shared__ int s_last, s_sel, s_cand, s_base_sel, s_base_cand;
  const int tid = threadIdx.x, G = gridDim.x, m = blockIdx.y;
  MsState* st = reinterpret_cast<MsState*>(zero + (size_t)m * (kMsStateInts + kBins));
  pdl_wait();
  pdl_trigger();
  const bool done = st->done != 0;
  uint64_t lo = st->lo, hi = st->hi;
  const int kk = (int)min((int64_t)k, n);
  uint64_t* rsel = sel + (size_t)m * k;
  uint64_t* rcand = cand + (size_t)m * kCap;
  const float* row = S + (size_t)m * n;
  if (done) {
    // this CTA's keys above the range and inside it go to shared memory first
    // (at most kk and kCap: the row's lists are no longer), then to the row's
    // lists through one global reservation per list
    if (tid == 0) { s_sel = 0; s_cand = 0; }
    cta_sync();
    const int64_t per = ms_seg(n, G);
    const int64_t p0 = (int64_t)blockIdx.x * per, p1 = min(n, p0 + per);
    for (int64_t p = p0 + tid; p < p1; p += kMsThreads) {
      const uint64_t key = key_at(row, token_ids, p);
      if (key > hi) {
        const int i = atomicAdd(&s_sel, 1);
        if (i < kCap) keys[i] = key;
      } else if (key >= lo) {
        const int i = atomicAdd(&s_cand, 1);
        if (i < kCap) keys[kCap + i] = key;
      }
    }
    cta_sync();
    const int ls = min(s_sel, kCap), lc = min(s_cand, kCap);
    if (tid == 0) {
      s_base_sel = ls ? atomicAdd(&st->n_sel, ls) : 0;
      s_base_cand = lc ? atomicAdd(&st->n_cand, lc) : 0;
    }
    cta_sync();
    for (int i = tid; i < ls; i += kMsThreads)
      if (s_base_sel + i < kk) rsel[s_base_sel + i] = keys[i];
    for (int i = tid; i < lc; i += kMsThreads)
      if (s_base_cand + i < kCap) rcand[s_base_cand + i] = keys[kCap + i];
    __threadfence();
  }
  cta_sync();
  if (tid == 0) s_last = atomicAdd(&st->ticket, 1) == G - 1;
  cta_sync();
  if (!s_last) return;
  __threadfence();
  int ns, nc;
  if (done) {
    ns = min(__ldcg(&st->n_sel), kk);
    nc = min(__ldcg(&st->n_cand), kCap);
    const int P = pow2_at_least(ns + nc);
    for (int i = tid; i < P; i += kMsThreads)
      keys[i] = i < ns ? __ldcg(rsel + i) : (i < ns + nc ? __ldcg(rcand + i - ns) : 0ull);
  } else {
    // fallback: the remaining passes over the whole row by this CTA alone
    int gt = st->gt;
    for (int pass = st->pass;; ++pass) {
      const int shift = ms_shift(pass);
      for (int i = tid; i < kBins; i += kMsThreads) hist[i] = 0;
      cta_sync();
      for (int64_t p = tid; p < n; p += kMsThreads) {
        const uint64_t key = key_at(row, token_ids, p);
        if (key >= lo && key <= hi) atomicAdd(&hist[(key >> shift) & (kBins - 1)], 1u);
      }
      cta_sync();
      ms_boundary(hist, part, (uint32_t)(kk - gt), shift, lo, &bnd);
      lo = bnd.lo;
      hi = bnd.hi;
      gt += bnd.above;
      const int count = bnd.count;
      cta_sync();
      if (count <= kCap || shift == 0) break;
    }
    if (tid == 0) { s_sel = 0; s_cand = 0; }
    cta_sync();
    for (int64_t p = tid; p < n; p += kMsThreads) {
      const uint64_t key = key_at(row, token_ids, p);
      if (key > hi) {
        const int i = atomicAdd(&s_sel, 1);
        if (i < kk) keys[i] = key;
      } else if (key >= lo) {
        const int i = atomicAdd(&s_cand, 1);
        if (i < kCap) keys[kCap + i] = key;
      }
    }
    cta_sync();
    ns = min(s_sel, kk);
    nc = min(s_cand, kCap);
    // move the candidates next to the selected keys (read all, then write)
    uint64_t mv[kCap / kMsThreads];
#pragma unroll
    for (int r = 0; r < kCap / kMsThreads; ++r) {
      const int i = tid + r * kMsThreads;
      mv[r] = i < nc ? keys[kCap + i] : 0ull;
    }
    cta_sync();
#pragma unroll
    for (int r = 0; r < kCap / kMsThreads; ++r) {
      const int i = tid + r * kMsThreads;
      if (i < nc) keys[ns + i] = mv[r];
    }
    const int P = pow2_at_least(ns + nc);
    for (int i = ns + nc + tid; i < P; i += kMsThreads) keys[i] = 0ull;
  }
  cta_sync();
  const int P = pow2_at_least(ns + nc);
  bitonic_desc(keys, P);
  const int take = min(kk, ns + nc);
  for (int j = tid; j < take; j += kMsThreads) {
    out_ids[(size_t)m * k + j] = key_id(keys[j]);
    if (out_scores) out_scores[(size_t)m * k + j] = key_score(keys[j]);
  }
}

int ms_ctas(int64_t n, int M, int sms) {
  const int64_t want = (4 * (int64_t)sms + M - 1) / M;
  const int64_t cap = (n + 2047) / 2048;  // at least ~2 keys per thread
  return (int)max((int64_t)1, min(want, cap));
}

}  // namespace

bool row_select_multi(int64_t n, int M, int k) {
  return n > 2 * kCap && k <= kCap && M <= 2 * 152;
}

int row_select_multi_ints(int M) { return M * (kMsStateInts + kBins); }

size_t row_select_multi_bytes(int M, int k) {
  return (size_t)M * ((size_t)k + kCap) * sizeof(uint64_t);
}

cudaError_t launch_row_select_multi(const float* S, const int32_t* token_ids, int64_t n, int M,
                                    int k, int32_t* out_ids, float* out_scores, int* zero,
                                    void* scratch, cudaStream_t s) {
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const dim3 grid((unsigned)ms_ctas(n, M, sms), (unsigned)M);
  for (int pass = 0; pass < kMsPasses; ++pass) {
    cudaError_t e = launch_kernel(true, ms_pass_kernel, grid, dim3(kMsThreads), 0, s, S, token_ids,
                                  n, k, zero);
    if (e != cudaSuccess) return e;
  }
  uint64_t* sel = static_cast<uint64_t*>(scratch);
  uint64_t* cand = sel + (size_t)M * k;
  // k + kCap <= 2 kCap keys, then the fallback's histogram and scan space
  const size_t smem = (size_t)2 * kCap * sizeof(uint64_t) + (kBins + kMsThreads) * sizeof(uint32_t);
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(ms_collect_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_kernel(true, ms_collect_kernel, grid, dim3(kMsThreads), smem, s, S, token_ids, n, k,
                       zero, sel, cand, out_ids, out_scores);
}

cudaError_t launch_segment_topk(const float* S, const int32_t* token_ids, int64_t n, int M,
                                int64_t seg_len, int k, int32_t* out_ids, float* out_scores,
                                int* err, cudaStream_t s) {
  (void)err;
  const int64_t segs = (n + seg_len - 1) / seg_len;
  const int64_t full = n / seg_len, tail = n - full * seg_len;
  const int K = (int)(full * k + (tail ? (tail < k ? tail : k) : 0));
  const size_t smem = 2 * kCap * sizeof(uint64_t) + (kBins + kThreads) * sizeof(uint32_t);
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(segment_topk_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)segs, M);
  return launch_kernel(false, segment_topk_kernel, grid, dim3(kThreads), smem, s, S, token_ids, n,
                       seg_len, k, K, out_ids, out_scores);
}

}  // namespace lmhead
