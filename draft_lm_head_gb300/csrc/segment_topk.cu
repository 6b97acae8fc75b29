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
// loaded whole and bitonic-sorted. Long rows and few of them (the global
// Top-C at up to 304 rows) use several CTAs per row instead (below).
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
// CTAs share a row, and no CTA waits on another. Histogram p (p = 0 .. kMsPasses-1)
// counts the row's keys inside the range left by histograms 0 .. p-1 by
// their 12-bit digit p from the top of the key; each CTA adds its segment's
// counts into the row's global histogram. The kernel after it (the next pass,
// or the collection) derives the narrowed range itself in every CTA, from
// the finished histogram: the bin holding the k-th largest key, the keys above
// it, and whether the bin holds at most kMsDone keys (then no further
// histogram is needed). The first histogram may come from the score
// writeback (it needs only the score's top 12 bits); fp32 scores need two in
// practice (the first digit is a sign, the exponent and three mantissa bits).
// Collection kernel: every CTA appends its keys above the range and inside it
// to two per-row lists. Rank kernel: every kept key's place in the row's
// Top-k (score descending, ties by the smaller vocabulary id; the keys are
// unique) is the number of larger keys in its own list, plus the length of
// the list above for a key inside the range; the keys are spread over many
// CTAs, so no single SM sorts a row. A row whose range still holds more than
// kCap keys after the last histogram is finished by the collection kernel's
// first CTA of the row alone, with the remaining passes over the whole row.
constexpr int kMsThreads = 1024;
constexpr int kMsPasses = 2;      // histograms; later digits in the fallback
constexpr int kMsStateInts = 32;  // per-row ranges and counters, then the histograms
constexpr int kMsRowInts = kMsStateInts + kMsPasses * kBins;
// A range of at most this many keys needs no further histogram: the rank
// kernel then places about k + kMsDone keys.
constexpr int kMsDone = 512;
static_assert(kBins == 1 << kSelectHistBits && kDigit == kSelectHistBits, "digit width");
// The histograms' digits lie in the score's order bits (the key's top 32), so
// the passes read only scores, and a range they leave decides every key by
// its score bits alone (its low 32 bits are all free): the collection reads
// a vocabulary id only for the keys it keeps.
static_assert(64 - kDigit * kMsPasses >= 32, "histogram digits inside the score bits");

struct MsRange {
  unsigned long long lo, hi;  // keys in [lo, hi] are still undecided
  int gt;                     // keys above hi (all selected)
  int count;                  // keys in [lo, hi]
  int done;                   // no further histogram
  int pad;
};

struct MsRow {
  MsRange range[kMsPasses];  // range[p]: what histogram p counts (p >= 1; 0 is the whole row)
  int n_sel, n_cand;         // collection list lengths
};
static_assert(sizeof(MsRow) <= kMsStateInts * sizeof(int), "row state");

struct MsBoundary {
  unsigned long long lo, hi;
  int above, count;
};

__device__ __forceinline__ int64_t ms_seg(int64_t n, int G) { return (n + G - 1) / G; }
__device__ __forceinline__ int ms_shift(int pass) { return max(0, 64 - kDigit * (pass + 1)); }

// A CTA's scan of the scores of positions [p0, p1) of one row (row = S + off,
// off = m * n floats from a 16-byte aligned S): 16-byte loads of four scores
// over the aligned middle, one score each for the at most three positions
// before and after it. start() requests the thread's first four scores (so
// they travel while the caller does other work); run() calls f(score, position)
// for every score of the thread, in no particular order.
struct MsScan {
  int64_t p0, p1, pa, nb;
  float4 pre;

  __device__ __forceinline__ void start(const float* row, int64_t off, int64_t p0_, int64_t p1_) {
    p0 = p0_;
    p1 = p1_;
    pa = min(p1, p0 + ((4 - ((off + p0) & 3)) & 3));
    nb = (p1 - pa) >> 2;
    pre = (int64_t)threadIdx.x < nb ? __ldcg(reinterpret_cast<const float4*>(row + pa) + threadIdx.x)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  template <typename F>
  __device__ __forceinline__ void run(const float* row, F&& f) const {
    const int tid = threadIdx.x;
    const int64_t pe = pa + nb * 4;
    if (tid < pa - p0) f(__ldcg(row + p0 + tid), p0 + tid);
    if (tid < p1 - pe) f(__ldcg(row + pe + tid), pe + tid);
    const float4* v = reinterpret_cast<const float4*>(row + pa);
    auto four = [&](const float4& a, int64_t i) {
      const int64_t q = pa + 4 * i;
      f(a.x, q);
      f(a.y, q + 1);
      f(a.z, q + 2);
      f(a.w, q + 3);
    };
    if (tid < nb) four(pre, tid);
    int64_t i = tid + kMsThreads;
    for (; i + kMsThreads < nb; i += 2 * kMsThreads) {  // two vectors in flight
      const float4 a = __ldcg(v + i), b = __ldcg(v + i + kMsThreads);
      four(a, i);
      four(b, i + kMsThreads);
    }
    if (i < nb) four(__ldcg(v + i), i);
  }
};

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

__device__ __forceinline__ MsRange ms_load_range(const MsRange* r) {
  MsRange x;
  x.lo = __ldcg(&r->lo);
  x.hi = __ldcg(&r->hi);
  x.gt = __ldcg(&r->gt);
  x.count = __ldcg(&r->count);
  x.done = __ldcg(&r->done);
  x.pad = 0;
  return x;
}

// Every thread of the CTA, after the kernel that finished histogram p - 1
// (p >= 1): the range left by histograms 0 .. p - 1. hist, part: shared
// scratch (kBins and kMsThreads words).
__device__ MsRange ms_range(const MsRow* row, const uint32_t* H, int p, int64_t n, int kk,
                            uint32_t* hist, uint32_t* part, MsBoundary* bnd) {
  MsRange prev;
  if (p == 1) {
    prev.lo = 0ull;
    prev.hi = ~0ull;
    prev.gt = 0;
    prev.count = (int)n;
    prev.done = 0;
    prev.pad = 0;
  } else {
    prev = ms_load_range(&row->range[p - 1]);
  }
  if (prev.done) return prev;
  const uint32_t* h = H + (size_t)(p - 1) * kBins;
  for (int i = threadIdx.x; i < kBins; i += kMsThreads) hist[i] = __ldcg(h + i);
  cta_sync();
  const int shift = ms_shift(p - 1);
  ms_boundary(hist, part, (uint32_t)(kk - prev.gt), shift, prev.lo, bnd);
  MsRange cur;
  cur.lo = bnd->lo;
  cur.hi = bnd->hi;
  cur.gt = prev.gt + bnd->above;
  cur.count = bnd->count;
  cur.done = (bnd->count <= kMsDone || shift == 0) ? 1 : 0;
  cur.pad = 0;
  return cur;
}

// grid (G, M), pass p < kMsPasses. `zero`: M x kMsRowInts ints, zero before
// the first histogram of a call. Histogram p of the keys in the range left by
// histograms 0 .. p - 1 (all of them for p = 0).
__global__ void __launch_bounds__(kMsThreads, 2)
ms_pass_kernel(const float* __restrict__ S, const int32_t* __restrict__ token_ids, int64_t n,
               int k, int* __restrict__ zero, int p) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t part[kMsThreads];
  __shared__ MsBoundary bnd;
  const int tid = threadIdx.x, G = gridDim.x, m = blockIdx.y;
  int* zr = zero + (size_t)m * kMsRowInts;
  MsRow* row_state = reinterpret_cast<MsRow*>(zr);
  uint32_t* H = reinterpret_cast<uint32_t*>(zr + kMsStateInts);
  const int kk = (int)min((int64_t)k, n);
  const int64_t per = ms_seg(n, G);
  const int64_t p0 = (int64_t)blockIdx.x * per, p1 = min(n, p0 + per);
  const float* row = S + (size_t)m * n;
  pdl_wait();  // scores, and the histogram the previous pass left
  pdl_trigger();
  MsScan scan;
  scan.start(row, (int64_t)m * n, p0, p1);  // in flight while the range is derived
  uint32_t lo = 0u, hi = 0xFFFFFFFFu;  // the range's score bits
  if (p > 0) {
    const MsRange cur = ms_range(row_state, H, p, n, kk, hist, part, &bnd);
    if (blockIdx.x == 0 && tid == 0) row_state->range[p] = cur;
    if (cur.done) return;
    lo = (uint32_t)(cur.lo >> 32);
    hi = (uint32_t)(cur.hi >> 32);
  }
  const int shift = ms_shift(p) - 32;
  for (int i = tid; i < kBins; i += kMsThreads) hist[i] = 0;
  cta_sync();
  scan.run(row, [&](float x, int64_t) {
    const uint32_t key = float_key(x);
    if (key >= lo && key <= hi) atomicAdd(&hist[(key >> shift) & (kBins - 1)], 1u);
  });
  cta_sync();
  uint32_t* Hp = H + (size_t)p * kBins;
  for (int i = tid; i < kBins; i += kMsThreads)
    if (hist[i]) atomicAdd(&Hp[i], hist[i]);
}

// grid (G, M); dynamic shared memory: 2 kCap keys of list space, then kBins
// + kMsThreads words of histogram and scan space. Appends the row's keys above
// the final range to its `sel` list and those inside it to its `cand` list;
// ms_rank_kernel orders them.
__global__ void __launch_bounds__(kMsThreads, 2)
ms_collect_kernel(const float* __restrict__ S, const int32_t* __restrict__ token_ids, int64_t n,
                  int k, int* __restrict__ zero, uint64_t* __restrict__ sel,
                  uint64_t* __restrict__ cand) {
  extern __shared__ uint64_t keys[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(keys + 2 * kCap);
  uint32_t* part = hist + kBins;
  __shared__ MsBoundary bnd;
  __shared__ int s_sel, s_cand, s_base_sel, s_base_cand;
  const int tid = threadIdx.x, G = gridDim.x, m = blockIdx.y;
  int* zr = zero + (size_t)m * kMsRowInts;
  MsRow* st = reinterpret_cast<MsRow*>(zr);
  const uint32_t* H = reinterpret_cast<const uint32_t*>(zr + kMsStateInts);
  const int kk = (int)min((int64_t)k, n);
  uint64_t* rsel = sel + (size_t)m * k;
  uint64_t* rcand = cand + (size_t)m * kCap;
  const float* row = S + (size_t)m * n;
  const int64_t per = ms_seg(n, G);
  const int64_t p0 = (int64_t)blockIdx.x * per, p1 = min(n, p0 + per);
  if (tid == 0) { s_sel = 0; s_cand = 0; }
  pdl_wait();
  pdl_trigger();
  MsScan scan;
  scan.start(row, (int64_t)m * n, p0, p1);  // in flight while the range is derived
  const MsRange cur = ms_range(st, H, kMsPasses, n, kk, hist, part, &bnd);
  uint64_t lo = cur.lo, hi = cur.hi;
  if (cur.count <= kCap) {
    // this CTA's keys above the range and inside it go to shared memory first
    // (at most kk and kCap: the row's lists are no longer), then to the row's
    // lists through one global reservation per list. The range's low 32 bits
    // are free, so the score bits decide.
    const uint32_t lo32 = (uint32_t)(lo >> 32), hi32 = (uint32_t)(hi >> 32);
    auto keep = [&](float x, int64_t q) {
      const uint32_t k32 = float_key(x);
      if (k32 < lo32) return;
      const int32_t id = token_ids ? __ldg(token_ids + q) : (int32_t)q;
      const uint64_t key = select_key(x, id);
      if (k32 > hi32) {
        const int i = atomicAdd(&s_sel, 1);
        if (i < kCap) keys[i] = key;
      } else {
        const int i = atomicAdd(&s_cand, 1);
        if (i < kCap) keys[kCap + i] = key;
      }
    };
    scan.run(row, keep);
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
    return;
  }
  // fallback (more than kCap keys share the histograms' 24 key bits): the
  // remaining passes over the whole row by the row's first CTA alone
  if (blockIdx.x != 0) return;
  int gt = cur.gt;
  for (int pass = kMsPasses;; ++pass) {
    const int shift = ms_shift(pass);
    for (int i = tid; i < kBins; i += kMsThreads) hist[i] = 0;
    cta_sync();
    for (int64_t q = tid; q < n; q += kMsThreads) {
      const uint64_t key = key_at(row, token_ids, q);
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
  cta_sync();
  for (int64_t q = tid; q < n; q += kMsThreads) {
    const uint64_t key = key_at(row, token_ids, q);
    if (key > hi) {
      const int i = atomicAdd(&s_sel, 1);
      if (i < kk) rsel[i] = key;
    } else if (key >= lo) {
      const int i = atomicAdd(&s_cand, 1);
      if (i < kCap) rcand[i] = key;
    }
  }
  cta_sync();
  if (tid == 0) {
    st->n_sel = min(s_sel, kk);
    st->n_cand = min(s_cand, kCap);
  }
}

// Output order of the collected keys. Every key above the range outranks
// every key inside it, so a key's place is the number of keys of its own list
// above it, plus the length of the `sel` list for a `cand` key; places below
// k are written. The keys are unique, so the places are too. grid (X, M); the
// lists' keys in chunks of 32 KPL, `sel` chunks first (its length rounded up
// to a chunk), chunk c taken by CTA c mod X. A lane holds KPL keys of the
// chunk; each warp counts over one eighth of the list (in shared memory, read
// two keys at a time) for all of the chunk's keys. KPL = 2 halves the loads
// per comparison (many rows: instruction-bound); KPL = 1 halves the work per
// CTA (a few rows: latency-bound).
constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / 32;

template <int KPL>
__global__ void __launch_bounds__(kRankThreads)
ms_rank_kernel(int64_t n, int k, const int* __restrict__ zero, const uint64_t* __restrict__ sel,
               const uint64_t* __restrict__ cand, int32_t* __restrict__ out_ids,
               float* __restrict__ out_scores) {
  constexpr int kChunk = 32 * KPL;
  __shared__ __align__(16) uint64_t list[kCap + 2];
  __shared__ uint32_t cnt[kRankWarps][kChunk];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, m = blockIdx.y;
  const MsRow* st = reinterpret_cast<const MsRow*>(zero + (size_t)m * kMsRowInts);
  const int kk = (int)min((int64_t)k, n);
  pdl_wait();
  pdl_trigger();
  const int ns = min(__ldcg(&st->n_sel), kk), nc = min(__ldcg(&st->n_cand), kCap);
  const int s0 = (ns + kChunk - 1) / kChunk * kChunk;
  const int chunks = s0 / kChunk + (nc + kChunk - 1) / kChunk;
  int loaded = -1;  // which list is in shared memory: 0 sel, 1 cand
  for (int c = blockIdx.x; c < chunks; c += gridDim.x) {
    const int which = kChunk * c < s0 ? 0 : 1;
    const int len = which ? nc : ns;
    if (which != loaded) {
      const uint64_t* src = which ? cand + (size_t)m * kCap : sel + (size_t)m * k;
      cta_sync();  // the previous chunk is done with the list
      for (int i = tid; i < len; i += kRankThreads) list[i] = __ldcg(src + i);
      if (tid == 0) list[len] = 0ull;  // pairs past an odd length count nothing
      cta_sync();
      loaded = which;
    }
    const int idx = kChunk * c - (which ? s0 : 0) + lane;
    uint64_t x[KPL];
    uint32_t above[KPL];
#pragma unroll
    for (int e = 0; e < KPL; ++e) {
      x[e] = idx + 32 * e < len ? list[idx + 32 * e] : ~0ull;
      above[e] = 0;
    }
    const int pairs = (len + 1) >> 1;
    const int per = (pairs + kRankWarps - 1) / kRankWarps;
    const int j0 = warp * per, j1 = min(pairs, j0 + per);
    const ulonglong2* lp = reinterpret_cast<const ulonglong2*>(list);
#pragma unroll 4
    for (int j = j0; j < j1; ++j) {
      const ulonglong2 y = lp[j];
#pragma unroll
      for (int e = 0; e < KPL; ++e) above[e] += (y.x > x[e] ? 1u : 0u) + (y.y > x[e] ? 1u : 0u);
    }
#pragma unroll
    for (int e = 0; e < KPL; ++e) cnt[warp][lane + 32 * e] = above[e];
    cta_sync();
    if (warp < KPL) {
      const int ie = idx + warp * 32;  // this warp publishes key `warp` of each lane
      if (ie < len) {
        uint32_t place = which ? (uint32_t)ns : 0u;
#pragma unroll
        for (int w = 0; w < kRankWarps; ++w) place += cnt[w][lane + 32 * warp];
        const uint64_t key = list[ie];
        if (place < (uint32_t)kk) {
          out_ids[(size_t)m * k + place] = key_id(key);
          if (out_scores) out_scores[(size_t)m * k + place] = key_score(key);
        }
      }
    }
    cta_sync();  // cnt is reused
  }
}

// CTAs per row: one wave in all (two 1024-thread CTAs per SM), so every CTA
// pays the range derivation and its barriers once, and at least ~2 keys per
// thread.
int ms_ctas(int64_t n, int M, int sms) {
  const int64_t want = 2 * (int64_t)sms / M;
  const int64_t cap = (n + 2047) / 2048;  // at least ~2 keys per thread
  return (int)max((int64_t)1, min(want, cap));
}

}  // namespace

bool row_select_multi(int64_t n, int M, int k) {
  return n > 2 * kCap && k <= kCap && M <= 2 * 152;
}

int row_select_multi_ints(int M) { return M * kMsRowInts; }

int row_select_multi_hist0(int m) { return m * kMsRowInts + kMsStateInts; }

size_t row_select_multi_bytes(int M, int k) {
  return (size_t)M * ((size_t)k + kCap) * sizeof(uint64_t);
}

cudaError_t launch_row_select_multi(const float* S, const int32_t* token_ids, int64_t n, int M,
                                    int k, int32_t* out_ids, float* out_scores, int* zero,
                                    void* scratch, bool hist0_filled, cudaStream_t s) {
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const dim3 grid((unsigned)ms_ctas(n, M, sms), (unsigned)M);
  for (int pass = hist0_filled ? 1 : 0; pass < kMsPasses; ++pass) {
    cudaError_t e = launch_kernel(true, ms_pass_kernel, grid, dim3(kMsThreads), 0, s, S, token_ids,
                                  n, k, zero, pass);
    if (e != cudaSuccess) return e;
  }
  uint64_t* sel = static_cast<uint64_t*>(scratch);
  uint64_t* cand = sel + (size_t)M * k;
  // 2 kCap keys of list space, then the histogram and scan space
  const size_t smem = (size_t)2 * kCap * sizeof(uint64_t) + (kBins + kMsThreads) * sizeof(uint32_t);
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(ms_collect_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  e = launch_kernel(true, ms_collect_kernel, grid, dim3(kMsThreads), smem, s, S, token_ids, n, k,
                    zero, sel, cand);
  if (e != cudaSuccess) return e;
  // one CTA per chunk of the usual lists (k + kMsDone keys); longer candidate
  // lists are taken in turns. Two keys a lane from 16 rows up: measured at
  // 64 rows, the call 2 us faster; at 8 rows, 4 us slower (half the CTAs).
  const int kk = (int)(k < n ? k : n);
  const int kpl = M >= 16 ? 2 : 1;
  const int ch = 32 * kpl;
  const dim3 rgrid((unsigned)((kk + ch - 1) / ch + (kMsDone + ch - 1) / ch), (unsigned)M);
  return launch_kernel(true, kpl == 2 ? ms_rank_kernel<2> : ms_rank_kernel<1>, rgrid,
                       dim3(kRankThreads), 0, s, n, k, (const int*)zero, (const uint64_t*)sel,
                       (const uint64_t*)cand, out_ids, out_scores);
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
