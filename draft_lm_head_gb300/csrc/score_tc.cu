// K4 on the 5th-generation tensor cores: fused low-rank tile scores + local
// top-k (EAGLE-4 notes, "A Local Top-k based variant": each program scores
// one vocabulary tile, keeps the scores on chip, picks the tile's top k_tile
// and writes tile.token_ids[local_ids]; no full-vocabulary score writeback).
//
// Design for sm_103a, one persistent CTA per SM:
//  - The vocabulary is cut into 128-row chunks; CTA b streams a contiguous
//    range of chunks (balanced over the CTAs). Chunk rows of A (n x r bf16,
//    row-major = K-major) arrive by TMA as 128-row x 64-element boxes with
//    the 128-byte swizzle into a ring of shared-memory stages.
//  - u (128 hidden vectors x r, zero-filled past M) is loaded once by TMA and
//    is the MMA's A operand; the chunk is the B operand (N = 128). One
//    elected thread issues tcgen05.mma (M=128, N=128, K=16, fp32 in TMEM)
//    into four TMEM accumulators, so the MMAs run up to four chunks ahead of
//    the epilogue.
//  - Epilogue: 4 warps; thread t owns TMEM lane t = one hidden vector and
//    reads its 128 scores with tcgen05.ld, keeping a sorted top-k_tile list
//    of (score, position) in registers. A tile boundary flushes the list:
//    ids are written through token_ids (ties: smaller vocabulary id).
//  - Tiles of a multiple of 128 rows (the usual case) are scheduled
//    dynamically, whole tiles per CTA (local_topk_tc_dyn_kernel). For tiles
//    of a multiple of 256 rows it uses 256-row chunks: 256-row boxes and
//    N = 256 MMAs into two TMEM accumulators. One tcgen05.mma (M = 128,
//    K = 16) occupies the tensor pipe about the same time at N = 128 as at
//    N = 256 (measured), so the wider MMA halves the tensor time per byte
//    of A. Otherwise
//    CTAs take balanced contiguous chunk ranges; a tile cut by a CTA boundary
//    leaves partial lists in the workspace and the last CTA to finish a part
//    (atomic ticket, no waiting) merges them.
//  - Every mbarrier wait is bounded; on timeout the CTA raises an abort flag,
//    records LMHEAD_ERR_TIMEOUT in the device error word, drains its own TMA
//    copies, frees TMEM and exits.
#include <math.h>
#include <stdlib.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace lmhead {
namespace {

constexpr int kChunk = 128;                 // vocabulary rows per chunk (MMA N)
constexpr int kHid = 128;                   // hidden vectors per CTA (MMA M, TMEM lanes)
constexpr int kKBlock = 64;                 // bf16 per 128-byte swizzled row
constexpr int kStageBytes = kChunk * 128;   // one 128-row x 64-element box
constexpr int kThreads = 192;               // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kMaxStages = 12;
constexpr int kOverlapStages = 3;           // ring depth when the gather overlaps
constexpr int kAcc = 4;                     // TMEM accumulators (the MMA runs ahead)
constexpr int kTmemCols = kAcc * 128;       // 128 fp32 columns each
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kHid, kChunk);

struct SharedCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t ufull;
  uint64_t acc_full[kAcc];
  uint64_t acc_empty[kAcc];
  uint64_t mma_drain;  // after an abort: the MMA thread's issued MMAs are done
  uint32_t tmem_base;
  int abort;
  int decision[2];
};

struct Params {
  const int32_t* token_ids;
  int64_t n;
  int r, M, T, k_tile, K;
  int64_t n_chunks, tiles;
  int G, stages;
  int lane_shift;  // R == 1 and M <= 64: hidden rows sit in TMEM lanes 64..127
  int R;           // copies of the hidden rows across the 128 TMEM lanes (1, 2, 4)
  int rows_per_rep;  // 128 / R
  int32_t* out_ids;
  float* out_scores;
  float2* partials;   // [HC][G][2][kHid][KT]
  int* tile_tickets;  // [HC][tiles]
  int* err;
  long long wait_cycles;  // budget of every role wait (drains keep tc::kWaitCycles)
  int* ready;             // dynamic kernel: the gather's ready counters, or nullptr
};

__device__ __forceinline__ int32_t vocab_id(const Params& p, int64_t pos) {
  if (pos >= p.n) return 0x7FFFFFFF;
  return p.token_ids ? __ldg(p.token_ids + pos) : (int32_t)pos;
}

// Sorted (descending) top-KT list of (score, key), kept in registers. The key
// is a position (ties resolved through token_ids) or, for merged partials, a
// vocabulary id. push() is branch-free for distinct scores: every column of
// every lane runs the same few compares and selects (32 independent lanes
// would otherwise diverge on almost every column). A NaN score is a no-op.
// Only an exact tie with a listed score takes the branch that compares
// vocabulary ids.
template <int KT, bool kPositions>
struct RegList {
  float s[KT];
  int32_t k[KT];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < KT; ++i) { s[i] = -INFINITY; k[i] = 0x7FFFFFFF; }
  }

  __device__ __forceinline__ static int32_t vocab(int32_t key, const int32_t* tok, int64_t n) {
    if (!kPositions) return key;
    if (key >= n) return 0x7FFFFFFF;
    return tok ? __ldg(tok + key) : key;
  }

  // Branch-free insertion by strict score order. A score equal to a listed
  // one is not inserted; push_fast returns true and the caller inserts it
  // later with push_exact.
  __device__ __forceinline__ bool push_fast(float x, int32_t key) {
    bool tie = false;
#pragma unroll
    for (int i = 0; i < KT; ++i) tie |= (x == s[i]);
    const float xe = tie ? __int_as_float(0x7FC00000) : x;
    bool c[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) c[i] = xe > s[i];
#pragma unroll
    for (int i = KT - 1; i > 0; --i) {
      s[i] = c[i] ? (c[i - 1] ? s[i - 1] : xe) : s[i];
      k[i] = c[i] ? (c[i - 1] ? k[i - 1] : key) : k[i];
    }
    s[0] = c[0] ? xe : s[0];
    k[0] = c[0] ? key : k[0];
    return tie;
  }

  // Merge another list into this one (exact order).
  __device__ __forceinline__ void absorb(const RegList& o, const int32_t* tok, int64_t n) {
#pragma unroll
    for (int i = 0; i < KT; ++i)
      push_exact(o.s[i] == -INFINITY ? __int_as_float(0x7FC00000) : o.s[i], o.k[i], tok, n);
  }

  // Exact insertion: score descending, then the smaller vocabulary id.
  __device__ __forceinline__ void push_exact(float x, int32_t key, const int32_t* tok, int64_t n) {
    float cs = x;
    int32_t ck = key;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      const bool wins = cs > s[i] || (cs == s[i] && vocab(ck, tok, n) < vocab(k[i], tok, n));
      if (wins) {
        const float ts = s[i]; s[i] = cs; cs = ts;
        const int32_t tk = k[i]; k[i] = ck; ck = tk;
      }
    }
  }
};

__device__ __forceinline__ int64_t chunk_start(int64_t b, int64_t nc, int G) { return b * nc / G; }
// CTA owning chunk c under the balanced split start(b) = floor(b * nc / G).
__device__ __forceinline__ int64_t cta_of_chunk(int64_t c, int64_t nc, int G) {
  return ((c + 1) * G + nc - 1) / nc - 1;
}

template <int KT, bool kPos>
__device__ __forceinline__ void write_tile(const Params& p, int m, int64_t tile, int count,
                                           const RegList<KT, kPos>& L, bool keys_are_positions) {
  int32_t* ids = p.out_ids + (size_t)m * p.K + (size_t)tile * KT;
  float* sc = p.out_scores ? p.out_scores + (size_t)m * p.K + (size_t)tile * KT : nullptr;
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    if (j < count) {
      ids[j] = keys_are_positions ? vocab_id(p, L.k[j]) : L.k[j];
      if (sc) sc[j] = L.s[j];
    }
  }
}

template <int KT>
__global__ void __launch_bounds__(kThreads, 1)
local_topk_tc_kernel(const __grid_constant__ CUtensorMap amap,
                     const __grid_constant__ CUtensorMap umap, const Params p) {
  extern __shared__ uint8_t dsmem_raw[];
  __shared__ SharedCtl ctl;
  uint8_t* dsmem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int kblocks = (p.r + kKBlock - 1) / kKBlock;
  uint8_t* u_s = dsmem;
  uint8_t* stage_s = dsmem + (size_t)kblocks * kStageBytes;
  float2* xchg = reinterpret_cast<float2*>(stage_s + (size_t)p.stages * kStageBytes);  // [128][KT]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x, y = blockIdx.y;
  const int64_t c0 = chunk_start(b, p.n_chunks, p.G);
  const int64_t c1 = chunk_start(b + 1, p.n_chunks, p.G);
  const int nch = (int)(c1 - c0);
  const int NS = p.stages;
  volatile int* abort_flag = &ctl.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&ctl.full[s], 1);
      tc::mbar_init(&ctl.empty[s], 1);
    }
    tc::mbar_init(&ctl.ufull, 1);
    for (int a = 0; a < kAcc; ++a) {
      tc::mbar_init(&ctl.acc_full[a], 1);
      tc::mbar_init(&ctl.acc_empty[a], 4);
    }
    tc::mbar_init(&ctl.mma_drain, 1);
    ctl.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&ctl.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  cta_sync();
  tc::fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&amap);
      tc::prefetch_tmap(&umap);
      uint32_t it = 0;
      bool ok = true;
      // A does not depend on the previous kernel: fill the ring first, then
      // wait for u (written by the projection kernel) and load it
      const uint32_t total_it = (uint32_t)nch * kblocks;
      const uint32_t pre = total_it < (uint32_t)NS ? total_it : (uint32_t)NS;
      for (; it < pre; ++it) {
        const int s = (int)it;
        tc::mbar_arrive_expect_tx(&ctl.full[s], kStageBytes);
        tc::tma_load_2d(stage_s + (size_t)s * kStageBytes, &amap, &ctl.full[s],
                        (int)(it % kblocks) * kKBlock, (int)((c0 + it / kblocks) * kChunk));
      }
      pdl_wait();
      tc::mbar_arrive_expect_tx(&ctl.ufull, (uint32_t)(kblocks * kStageBytes));
      for (int kb = 0; kb < kblocks; ++kb)
        for (int rep = 0; rep < p.R; ++rep)  // R copies; rows before 0 / past M are zero
          tc::tma_load_2d(u_s + (size_t)kb * kStageBytes + (size_t)rep * p.rows_per_rep * 128, &umap,
                          &ctl.ufull, kb * kKBlock, y * p.rows_per_rep - p.lane_shift);
      for (int i = (int)(it / kblocks); i < nch && ok; ++i) {
        for (int kb = (i == (int)(it / kblocks)) ? (int)(it % kblocks) : 0; kb < kblocks; ++kb, ++it) {
          const int s = (int)(it % NS);
          if (!tc::mbar_wait(&ctl.empty[s], ((it / NS) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&ctl.full[s], kStageBytes);
          tc::tma_load_2d(stage_s + (size_t)s * kStageBytes, &amap, &ctl.full[s], kb * kKBlock,
                          (int)((c0 + i) * kChunk));
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kDevErrTimeout);
      }
      if (*abort_flag) {
        // drain: wait (bounded) for the copies this thread issued last on every stage
        const uint32_t first = it > (uint32_t)NS ? it - NS : 0;
        for (uint32_t j = first; j < it; ++j) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(&ctl.full[j % NS], (j / NS) & 1) &&
                 clock64() - t0 < tc::kWaitCycles) {
          }
        }
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(&ctl.ufull, 0) && clock64() - t0 < tc::kWaitCycles) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = tc::mbar_wait(&ctl.ufull, 0, abort_flag, p.wait_cycles);
      uint32_t it = 0;
      for (int i = 0; i < nch && ok; ++i) {
        const int a = i % kAcc;
        if (!tc::mbar_wait(&ctl.acc_empty[a], ((i / kAcc) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t d = tmem + a * kChunk;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = (int)(it % NS);
          if (!tc::mbar_wait(&ctl.full[s], (it / NS) & 1, abort_flag, p.wait_cycles)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t adesc = tc::sw128_kmajor_desc(tc::smem_addr(u_s + (size_t)kb * kStageBytes));
          const uint64_t bdesc = tc::sw128_kmajor_desc(tc::smem_addr(stage_s + (size_t)s * kStageBytes));
          const int nk = min(4, (p.r - kb * kKBlock + 15) / 16);
          for (int k = 0; k < nk; ++k)
            tc::mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, kIdesc, (kb | k) != 0);
          tc::mma_commit(&ctl.empty[s]);
        }
        if (!ok) break;
        tc::mma_commit(&ctl.acc_full[a]);
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kDevErrTimeout);
        tc::mma_drain(&ctl.mma_drain);  // TMEM is freed below
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // tile tickets are zeroed by the projection kernel
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    const int ml = q * 32 + lane;
    const int rep = (q * 32) / p.rows_per_rep;  // which copy of the hidden rows
    const int m = y * p.rows_per_rep + ml % p.rows_per_rep - p.lane_shift;
    const bool valid = m >= 0 && m < p.M;
    const bool valid_out = valid && rep == 0;  // copy 0 publishes the results
    const int64_t n = p.n, T = p.T;
    const int64_t P0 = c0 * kChunk;
    const int64_t P1 = min(n, c1 * kChunk);
    int64_t tile = P0 / T;
    int64_t tile_end = min(n, tile * T + T);
    const int64_t first_tile = tile;
    const bool first_partial = P0 > tile * T;
    const float kNaN = __int_as_float(0x7FC00000);  // a pushed NaN changes nothing
    // kSub independent sub-lists (column jj goes to jj % kSub) break the
    // serial dependency between consecutive columns; merged at tile ends
    constexpr int kSub = KT <= 4 ? 4 : 2;
    RegList<KT, true> sub[kSub], cur, first;
#pragma unroll
    for (int j = 0; j < kSub; ++j) sub[j].reset();
    first.reset();
    auto merged = [&]() {
      RegList<KT, true> L = sub[0];
#pragma unroll
      for (int j = 1; j < kSub; ++j) L.absorb(sub[j], p.token_ids, n);
      return L;
    };
    bool ok = true;
    // warps whose 32 hidden rows all lie outside [0, M) only pace the ring
    const int m_lo = y * p.rows_per_rep + (q * 32) % p.rows_per_rep - p.lane_shift;
    const bool warp_live = m_lo + 31 >= 0 && m_lo < p.M;
    if (p.R > 1) {
      // T % 128 == 0: tiles end on chunk edges. Copy `rep` of the rows scans
      // columns [rep*cols, (rep+1)*cols) of every chunk; at a tile end the
      // copies' lists meet in shared memory and copy 0 combines them.
      const int cols = kChunk / p.R;
      const int jb = rep * cols;
      const int qstep = p.rows_per_rep / 32;
      for (int i = 0; i < nch; ++i) {
        const int a = i % kAcc;
        int okw = 1;
        if (lane == 0) {
          okw = ok && tc::mbar_wait(&ctl.acc_full[a], (i / kAcc) & 1, abort_flag, p.wait_cycles) ? 1 : 0;
          if (!okw) *abort_flag = 1;
        }
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        ok = ok && okw;  // keep iterating on failure: the barriers below need every warp
        tc::fence_after_sync();
        const int64_t cbase = (c0 + i) * kChunk;
        for (int j0 = jb; j0 < jb + cols && warp_live && ok; j0 += 32) {
          const int64_t base = cbase + j0;
          if (base >= P1) break;
          uint32_t v[32];
          tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * kChunk + j0), v);
          tc::tmem_ld_wait();
          const int lim = (int)min((int64_t)32, P1 - base);
          uint32_t ties = 0;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const bool t = sub[jj % kSub].push_fast(
                jj < lim && valid ? __uint_as_float(v[jj]) : kNaN, (int32_t)(base + jj));
            ties |= (t ? 1u : 0u) << jj;
          }
          if (ties != 0) {
            float rest[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) rest[jj] = __uint_as_float(v[jj]);
            for (uint32_t t = ties; t; t &= t - 1) {
              const int jj = __ffs(t) - 1;
              sub[0].push_exact(rest[jj], (int32_t)(base + jj), p.token_ids, n);
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&ctl.acc_empty[a]);
        const int64_t cend = min(P1, cbase + kChunk);
        const int64_t ctile = cbase / T;
        if (cend == min(n, ctile * T + T) || cend == P1) {  // this chunk ends a tile
          RegList<KT, true> Lst = merged();
#pragma unroll
          for (int j = 0; j < KT; ++j)
            xchg[ml * KT + j] = make_float2(Lst.s[j], __int_as_float(Lst.k[j]));
          named_sync(1, 128);
          if (rep == 0) {
            for (int r2 = 1; r2 < p.R; ++r2) {
              const int ol = (q + r2 * qstep) * 32 + lane;
#pragma unroll
              for (int j = 0; j < KT; ++j) {
                const float2 e = xchg[ol * KT + j];
                Lst.push_exact(e.x == -INFINITY ? kNaN : e.x, __float_as_int(e.y), p.token_ids, n);
              }
            }
            if (cend == P1) {
              cur = Lst;  // the range's last tile: the code below decides
            } else if (ctile == first_tile && first_partial) {
              first = Lst;  // part of a tile cut by this CTA's start
            } else if (valid_out && ok) {
              write_tile<KT>(p, m, ctile, (int)min((int64_t)KT, min(n, ctile * T + T) - ctile * T),
                             Lst, true);
            }
          }
          named_sync(1, 128);
#pragma unroll
          for (int j = 0; j < kSub; ++j) sub[j].reset();
        }
      }
    } else {
    for (int i = 0; i < nch; ++i) {
      const int a = i % kAcc;
      int okw = 1;
      if (lane == 0) okw = tc::mbar_wait(&ctl.acc_full[a], (i / kAcc) & 1, abort_flag, p.wait_cycles) ? 1 : 0;
      okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
      if (!okw) { ok = false; break; }
      tc::fence_after_sync();
      const int64_t cbase = (c0 + i) * kChunk;
      for (int j0 = 0; j0 < kChunk && warp_live; j0 += 32) {
        const int64_t base = cbase + j0;
        if (base >= P1) break;
        uint32_t v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * kChunk + j0), v);
        tc::tmem_ld_wait();
        const int lim = (int)min((int64_t)32, P1 - base);
        // columns [0, bnd) belong to the current tile; at most one boundary
        // falls inside 32 columns because T >= 32
        const int bnd = (int)min((int64_t)lim, tile_end - base);
        uint32_t ties = 0;  // columns held back by an exact tie
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const bool t = sub[jj % kSub].push_fast(
              jj < bnd && valid ? __uint_as_float(v[jj]) : kNaN, (int32_t)(base + jj));
          ties |= (t ? 1u : 0u) << jj;
        }
        if (ties != 0 || bnd < lim) {  // rare: a tie, or a tile ends inside this batch
          float rest[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) rest[jj] = __uint_as_float(v[jj]);
          for (uint32_t t = ties; t; t &= t - 1) {
            const int jj = __ffs(t) - 1;
            sub[0].push_exact(rest[jj], (int32_t)(base + jj), p.token_ids, n);
          }
          if (bnd < lim) {
            cur = merged();
            if (tile == first_tile && first_partial) {
              first = cur;  // part of a tile cut by this CTA's start
            } else if (valid) {
              write_tile<KT>(p, m, tile, (int)min((int64_t)KT, tile_end - tile * T), cur, true);
            }
#pragma unroll
            for (int j = 0; j < kSub; ++j) sub[j].reset();
            ++tile;
            tile_end = min(n, tile_end + T);
            for (int jj = bnd; jj < lim; ++jj)
              sub[0].push_exact(valid ? rest[jj] : kNaN, (int32_t)(base + jj), p.token_ids, n);
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.acc_empty[a]);
    }
    cur = merged();
    }

    // ---- tiles cut by CTA boundaries: publish parts, last part merges.
    // Which tiles are cut depends only on this CTA's range [P0, P1).
    const int64_t last_tile = (P1 - 1) / T;
    const int64_t last_end = min(n, last_tile * T + T);
    const bool first_cut = P0 > first_tile * T || P1 < min(n, first_tile * T + T);
    const bool last_cut = last_tile != first_tile && P1 < last_end;
    int64_t part_tile[2] = {first_cut ? first_tile : -1, last_cut ? last_tile : -1};
    // the running list now holds the last tile; complete unless cut
    const bool last_is_cut = (last_tile == first_tile) ? first_cut : last_cut;
    if (ok && valid_out && !last_is_cut)
      write_tile<KT>(p, m, last_tile, (int)min((int64_t)KT, last_end - last_tile * T), cur, true);
    if (ok && valid_out) {
      for (int side = 0; side < 2; ++side) {
        if (part_tile[side] < 0) continue;
        const RegList<KT, true>& src = (side == 0 && last_tile != first_tile) ? first : cur;
        float2* slot = p.partials + ((((size_t)y * p.G + b) * 2 + side) * kHid + ml) * KT;
#pragma unroll
        for (int j = 0; j < KT; ++j)
          slot[j] = make_float2(src.s[j], __int_as_float(vocab_id(p, src.k[j])));
      }
    }
    __threadfence();
    named_sync(1, 128);
    if (warp == 2 && lane == 0) {
      const bool go = !(*abort_flag);
      for (int side = 0; side < 2; ++side) {
        ctl.decision[side] = 0;
        const int64_t t = part_tile[side];
        if (!go || t < 0) continue;
        const int64_t fc = t * T / kChunk;
        const int64_t lc = (min(n, t * T + T) - 1) / kChunk;
        const int parts = (int)(cta_of_chunk(lc, p.n_chunks, p.G) - cta_of_chunk(fc, p.n_chunks, p.G) + 1);
        __threadfence();
        const int old = atomicAdd(p.tile_tickets + (size_t)y * p.tiles + t, 1);
        ctl.decision[side] = (old == parts - 1) ? 1 : 0;
      }
    }
    named_sync(1, 128);
    for (int side = 0; side < 2; ++side) {
      if (!ctl.decision[side]) continue;
      const int64_t t = part_tile[side];
      __threadfence();
      if (valid_out) {
        const int64_t fc = t * T / kChunk;
        const int64_t lc = (min(n, t * T + T) - 1) / kChunk;
        const int64_t b0 = cta_of_chunk(fc, p.n_chunks, p.G), b1 = cta_of_chunk(lc, p.n_chunks, p.G);
        RegList<KT, false> mg;
        mg.reset();
        for (int64_t bb = b0; bb <= b1; ++bb) {
          const int64_t ft = chunk_start(bb, p.n_chunks, p.G) * kChunk / T;
          const int sd = (t == ft) ? 0 : 1;
          const float2* slot = p.partials + ((((size_t)y * p.G + bb) * 2 + sd) * kHid + ml) * KT;
#pragma unroll
          for (int j = 0; j < KT; ++j) {
            const float2 e = __ldcg(slot + j);
            mg.push_exact(e.x == -INFINITY ? kNaN : e.x, __float_as_int(e.y), nullptr, n);
          }
        }
        write_tile<KT>(p, m, t, (int)min((int64_t)KT, min(n, t * T + T) - t * T), mg, false);
      }
      if (warp == 2 && lane == 0) p.tile_tickets[(size_t)y * p.tiles + t] = 0;
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) record_error(p.err, kDevErrTimeout);
    }
  }

  tc::fence_before_sync();
  cta_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- dynamic tiles
// Variant for tiles of a multiple of 128 rows (chunks of CH = 128 or 256
// rows): whole tiles are the unit of work. CTA b first takes tile b (so it can stream A before the projection
// kernel finishes), then claims tiles G, G+1, ... from a counter in the
// workspace (zeroed by the projection kernel), so SMs that get their data
// faster take more tiles. Chunk descriptors reach the MMA and epilogue
// warps through a shared ring; no tile is ever split between CTAs.
constexpr int kDescRing = 32;  // > stages + accumulators: the producer is never a ring ahead

// All 128 epilogue threads agree: true only if every one passes true.
__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

template <int KT, int CH>
__global__ void __launch_bounds__(kThreads, 1)
local_topk_tc_dyn_kernel(const __grid_constant__ CUtensorMap amap,
                         const __grid_constant__ CUtensorMap umap, const Params p) {
  extern __shared__ uint8_t dsmem_raw[];
  __shared__ SharedCtl ctl;
  __shared__ int desc_tile[kDescRing], desc_chunk[kDescRing];
  uint8_t* dsmem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kSt = CH * 128;                  // one CH-row x 64-element box of A
  constexpr int kNAcc = kTmemCols / CH;          // TMEM accumulators of CH columns
  constexpr uint32_t kIdescCH = tc::idesc_bf16_f32(kHid, CH);
  const int kblocks = (p.r + kKBlock - 1) / kKBlock;
  uint8_t* u_s = dsmem;
  uint8_t* stage_s = dsmem + (size_t)kblocks * kStageBytes;  // u: 128 rows per K-block
  float2* xchg = reinterpret_cast<float2*>(stage_s + (size_t)p.stages * kSt);  // [128][KT]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int y = blockIdx.y;
  const int NS = p.stages;
  const int64_t n = p.n, T = p.T;
  const int cpt = (int)(T / CH);  // chunks per tile
  int* counter = p.tile_tickets + y;
  volatile int* abort_flag = &ctl.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&ctl.full[s], 1);
      tc::mbar_init(&ctl.empty[s], 1);
    }
    tc::mbar_init(&ctl.ufull, 1);
    for (int a = 0; a < kAcc; ++a) {
      tc::mbar_init(&ctl.acc_full[a], 1);
      tc::mbar_init(&ctl.acc_empty[a], 4);
    }
    tc::mbar_init(&ctl.mma_drain, 1);
    ctl.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&ctl.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  cta_sync();
  tc::fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&amap);
      tc::prefetch_tmap(&umap);
      uint32_t it = 0;  // stage sequence
      int c = 0;        // chunk sequence
      // 128-row boxes go in groups of four (each row's 128-byte pieces requested
      // together); 256-row boxes, four to a small ring, one at a time
      const int grp = CH == 256 ? 1 : min(min(4, NS), kblocks);
      bool ok = true, u_loaded = false;
      // u is written by the previous kernel: wait for it, then load it once
      auto load_u = [&]() {
        pdl_wait();
        pdl_trigger();  // the projection is done (see the epilogue)
        tc::mbar_arrive_expect_tx(&ctl.ufull, (uint32_t)(kblocks * kStageBytes));
        for (int ub = 0; ub < kblocks; ++ub)
          for (int rep = 0; rep < p.R; ++rep)
            tc::tma_load_2d(u_s + (size_t)ub * kStageBytes + (size_t)rep * p.rows_per_rep * 128,
                            &umap, &ctl.ufull, ub * kKBlock, y * p.rows_per_rep - p.lane_shift);
        u_loaded = true;
      };
      int64_t tile = blockIdx.x < p.tiles ? (int64_t)blockIdx.x : -1;
      int64_t next = -1;
      while (ok) {
        if (tile >= 0 && u_loaded && next < 0) {
          // claim the tile after this one early; its value is needed later
          next = (int64_t)p.G + atomicAdd(counter, 1);
        }
        const int slot = c % kDescRing;
        if (tile < 0 || tile >= p.tiles) {  // no more work: an end marker through the ring
          const int s = (int)(it % NS);
          if (it >= (uint32_t)NS && !tc::mbar_wait(&ctl.empty[s], ((it / NS) & 1) ^ 1, abort_flag, p.wait_cycles)) {
            ok = false;
            break;
          }
          desc_tile[slot] = -1;
          tc::mbar_arrive(&ctl.full[s]);
          ++it;
          break;
        }
        for (int j = 0; j < cpt && ok; ++j) {
          const int64_t gc = tile * cpt + j;  // global chunk
          if (gc * CH >= n) break;
          const bool last = j == cpt - 1 || (gc + 1) * CH >= n;
          desc_tile[c % kDescRing] = (int)tile;
          desc_chunk[c % kDescRing] = j | (last ? (int)0x80000000 : 0);
          // a group of up to four boxes (one chunk at r = 256) is issued back to
          // back once all its stages are free, so each row's 128-byte pieces
          // are requested together (contiguous DRAM reads); one box at a time,
          // the requests scatter and the stream loses a third of its rate
          for (int kb0 = 0; kb0 < kblocks && ok; kb0 += grp) {
            const int gcount = min(grp, kblocks - kb0);
            // stages of the group that are still in use free up only once the
            // MMA runs, which needs u: load it before waiting on them
            if (!u_loaded && it + (uint32_t)gcount > (uint32_t)NS) load_u();
            for (int g2 = 0; g2 < gcount; ++g2) {
              const uint32_t itg = it + (uint32_t)g2;
              if (itg >= (uint32_t)NS &&
                  !tc::mbar_wait(&ctl.empty[itg % NS], ((itg / NS) & 1) ^ 1, abort_flag, p.wait_cycles)) {
                ok = false;
                break;
              }
            }
            if (!ok) break;
            for (int g2 = 0; g2 < gcount; ++g2, ++it) {
              const int s = (int)(it % NS);
              tc::mbar_arrive_expect_tx(&ctl.full[s], kSt);
              tc::tma_load_2d(stage_s + (size_t)s * kSt, &amap, &ctl.full[s],
                              (kb0 + g2) * kKBlock, (int)(gc * CH));
            }
            // ring filled, or the first tile fully issued: u next
            if (!u_loaded && (it >= (uint32_t)NS || (j == cpt - 1 && kb0 + gcount == kblocks)))
              load_u();
          }
          ++c;
        }
        if (!u_loaded) load_u();  // no tile at all for this CTA
        if (tile >= 0 && next < 0) next = (int64_t)p.G + atomicAdd(counter, 1);
        tile = next;
        next = -1;
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kDevErrTimeout);
      }
      if (*abort_flag) {
        const uint32_t first = it > (uint32_t)NS ? it - NS : 0;
        for (uint32_t jq = first; jq < it; ++jq) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(&ctl.full[jq % NS], (jq / NS) & 1) &&
                 clock64() - t0 < tc::kWaitCycles) {
          }
        }
        const long long t0 = clock64();
        while (u_loaded && !tc::mbar_try_wait(&ctl.ufull, 0) && clock64() - t0 < tc::kWaitCycles) {
        }
      }
    } else {
      pdl_wait();
      pdl_trigger();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = tc::mbar_wait(&ctl.ufull, 0, abort_flag, p.wait_cycles);
      if (ok) {
        pdl_wait();  // returns at once: u is loaded, so the projection is done
        pdl_trigger();
      }
      uint32_t it = 0;
      for (int c = 0; ok; ++c) {
        const int a = c % kNAcc;
        int s = (int)(it % NS);
        if (!tc::mbar_wait(&ctl.full[s], (it / NS) & 1, abort_flag, p.wait_cycles)) { ok = false; break; }
        // the slot must be free before anything, the end marker included, is
        // signalled on it: an arrival two phases ahead of the epilogue's wait
        // would hide the phase it waits for
        if (!tc::mbar_wait(&ctl.acc_empty[a], ((c / kNAcc) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
        if (desc_tile[c % kDescRing] < 0) {  // end marker: pass it on to the epilogue
          tc::mbar_arrive(&ctl.acc_full[a]);
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + a * CH;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          s = (int)(it % NS);
          if (kb > 0 && !tc::mbar_wait(&ctl.full[s], (it / NS) & 1, abort_flag, p.wait_cycles)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t adesc = tc::sw128_kmajor_desc(tc::smem_addr(u_s + (size_t)kb * kStageBytes));
          const uint64_t bdesc = tc::sw128_kmajor_desc(tc::smem_addr(stage_s + (size_t)s * kSt));
          const int nk = min(4, (p.r - kb * kKBlock + 15) / 16);
          for (int k = 0; k < nk; ++k)
            tc::mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, kIdescCH, (kb | k) != 0);
          tc::mma_commit(&ctl.empty[s]);
        }
        if (!ok) break;
        tc::mma_commit(&ctl.acc_full[a]);
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kDevErrTimeout);
        tc::mma_drain(&ctl.mma_drain);  // TMEM is freed below
      }
    } else {
      pdl_wait();
      pdl_trigger();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // The gather that follows may launch once every thread of every CTA has
    // triggered; each thread triggers only after the projection kernel has
    // completed, so the gather never sees the ready counters before the
    // projection kernel zeroed them.
    pdl_wait();
    pdl_trigger();
    const int q = warp & 3;
    const int ml = q * 32 + lane;
    const int rep = (q * 32) / p.rows_per_rep;
    const int m = y * p.rows_per_rep + ml % p.rows_per_rep - p.lane_shift;
    const bool valid = m >= 0 && m < p.M;
    const bool valid_out = valid && rep == 0;
    const int m_lo = y * p.rows_per_rep + (q * 32) % p.rows_per_rep - p.lane_shift;
    const bool warp_live = m_lo + 31 >= 0 && m_lo < p.M;
    // hidden rows of this chunk (what one finished tile adds to its ready count)
    const int rows_valid = max(0, min(p.M, (y + 1) * p.rows_per_rep - p.lane_shift) -
                                      max(0, y * p.rows_per_rep - p.lane_shift));
    const float kNaN = __int_as_float(0x7FC00000);
    const int cols = CH / p.R;
    const int jb = rep * cols;
    const int qstep = p.rows_per_rep / 32;
    constexpr int kSub = KT <= 4 ? 4 : 2;
    RegList<KT, true> sub[kSub];
#pragma unroll
    for (int j = 0; j < kSub; ++j) sub[j].reset();
    for (int c = 0;; ++c) {
      const int a = c % kNAcc;
      int okw = 1;
      if (lane == 0) okw = tc::mbar_wait(&ctl.acc_full[a], (c / kNAcc) & 1, abort_flag, p.wait_cycles) ? 1 : 0;
      okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
      if (!epilogue_all(okw != 0)) {  // uniform: every epilogue warp leaves together
        if (lane == 0) { *abort_flag = 1; record_error(p.err, kDevErrTimeout); }
        break;
      }
      tc::fence_after_sync();
      const int tile = desc_tile[c % kDescRing];
      if (tile < 0) break;  // end marker (same for every warp)
      const int dc = desc_chunk[c % kDescRing];
      const int j = dc & 0x7FFFFFFF;
      const bool last = dc < 0;
      const int64_t cbase = ((int64_t)tile * cpt + j) * CH;
      const int64_t cend = min(n, cbase + CH);
      for (int j0 = jb; j0 < jb + cols && warp_live; j0 += 32) {
        const int64_t base = cbase + j0;
        if (base >= cend) break;
        uint32_t v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * CH + j0), v);
        tc::tmem_ld_wait();
        const int lim = (int)min((int64_t)32, cend - base);
        uint32_t ties = 0;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const bool t = sub[jj % kSub].push_fast(
              jj < lim && valid ? __uint_as_float(v[jj]) : kNaN, (int32_t)(base + jj));
          ties |= (t ? 1u : 0u) << jj;
        }
        if (ties != 0) {
          float rest[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) rest[jj] = __uint_as_float(v[jj]);
          for (uint32_t t = ties; t; t &= t - 1) {
            const int jj = __ffs(t) - 1;
            sub[0].push_exact(rest[jj], (int32_t)(base + jj), p.token_ids, n);
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.acc_empty[a]);
      if (last) {  // the tile is complete: combine the copies' lists and write it
        RegList<KT, true> Lst = sub[0];
#pragma unroll
        for (int jj = 1; jj < kSub; ++jj) Lst.absorb(sub[jj], p.token_ids, n);
        if (p.R > 1) {
#pragma unroll
          for (int jj = 0; jj < KT; ++jj)
            xchg[ml * KT + jj] = make_float2(Lst.s[jj], __int_as_float(Lst.k[jj]));
          named_sync(1, 128);
          if (rep == 0) {
            for (int r2 = 1; r2 < p.R; ++r2) {
              const int ol = (q + r2 * qstep) * 32 + lane;
#pragma unroll
              for (int jj = 0; jj < KT; ++jj) {
                const float2 e = xchg[ol * KT + jj];
                Lst.push_exact(e.x == -INFINITY ? kNaN : e.x, __float_as_int(e.y), p.token_ids, n);
              }
            }
          }
          named_sync(1, 128);
        }
        if (valid_out)
          write_tile<KT>(p, m, tile, (int)min((int64_t)KT, min(n, (int64_t)(tile + 1) * T) - (int64_t)tile * T),
                         Lst, true);
        if (p.ready) {  // this tile's ids of this chunk's hidden rows are written
          __threadfence();
          named_sync(2, 128);
          if (warp == 2 && lane == 0) signal_count(p.ready + tile / kReadyTiles, rows_valid);
        }
#pragma unroll
        for (int jj = 0; jj < kSub; ++jj) sub[jj].reset();
      }
    }
  }

  tc::fence_before_sync();
  cta_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  // an aborted CTA will not publish its tiles: release the gather's waits
  if (p.ready && threadIdx.x == 0 && *abort_flag)
    atomicExch(p.ready + ready_blocks(p.tiles), 1);
}

// ---------------------------------------------------------------- host side
// LMHEAD_K4_STAGES = s caps the ring at s stages (measurements only: a
// smaller ring leaves shared memory for more gather CTAs beside each CTA).
int stage_cap() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LMHEAD_K4_STAGES");
    v = e ? atoi(e) : 0;
  }
  return v;
}

// LMHEAD_K4_CHUNK = 128 keeps 128-row MMAs for every tile (measurements only).
bool chunk256_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("LMHEAD_K4_CHUNK");
    v = (e && atoi(e) == 128) ? 0 : 1;
  }
  return v == 1;
}

template <int KT, int CH>
cudaError_t launch_dyn(const CUtensorMap& amap, const CUtensorMap& umap, const Params& p, int HC,
                       size_t smem, cudaStream_t s) {
  static int smem_set_dyn[64] = {0};
  cudaError_t e = ensure_dynamic_smem(local_topk_tc_dyn_kernel<KT, CH>, smem, smem_set_dyn);
  if (e != cudaSuccess) return e;
  return launch_kernel(true, local_topk_tc_dyn_kernel<KT, CH>, dim3(p.G, HC), dim3(kThreads), smem,
                       s, amap, umap, p);
}

template <int KT>
cudaError_t launch_kt(const CUtensorMap& amap, const CUtensorMap& umap, const Params& p, int HC,
                      size_t smem, int ch, cudaStream_t s) {
  if (p.T % kChunk == 0)
    return ch == 256 ? launch_dyn<KT, 256>(amap, umap, p, HC, smem, s)
                     : launch_dyn<KT, 128>(amap, umap, p, HC, smem, s);
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(local_topk_tc_kernel<KT>, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_kernel(true, local_topk_tc_kernel<KT>, dim3(p.G, HC), dim3(kThreads), smem, s, amap,
                       umap, p);
}

}  // namespace

bool local_topk_tc_supported(int r, int T, int k_tile) {
  return r <= kLocalTcMaxR && T >= 32 &&
         (k_tile == 1 || k_tile == 2 || k_tile == 4 || k_tile == 8);
}

size_t local_topk_tc_scratch_bytes(int64_t n, int M, int T) {
  const int64_t HC = (M + kHid - 1) / kHid;
  const int64_t tiles = (n + T - 1) / T;
  (void)tiles;
  return (size_t)HC * kLocalTcMaxCtas * 2 * kHid * 8 * sizeof(float2);
}

int local_topk_tc_tickets(int64_t n, int M, int T) {
  const int64_t HC = (M + kHid - 1) / kHid;
  if (T % kChunk == 0) return (int)HC;  // one tile counter per hidden-row chunk
  return (int)(HC * ((n + T - 1) / T));
}

cudaError_t launch_local_topk_tc(const bf16_t* A, const bf16_t* u, const int32_t* token_ids,
                                 int64_t n, int r, int M, int T, int k_tile, int32_t* out_ids,
                                 float* out_scores, void* partials, int* tile_tickets, int* err,
                                 cudaStream_t s, int* ready) {
  Params p;
  p.token_ids = token_ids;
  p.n = n;
  p.r = r;
  p.M = M;
  p.T = T;
  p.k_tile = k_tile;
  const int64_t full = n / T, tail = n - full * T;
  p.K = (int)(full * k_tile + (tail ? (tail < k_tile ? tail : k_tile) : 0));
  p.n_chunks = (n + kChunk - 1) / kChunk;
  p.tiles = (n + T - 1) / T;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  p.G = (int)min((int64_t)min(sms, kLocalTcMaxCtas), T % kChunk == 0 ? p.tiles : p.n_chunks);
  const int kblocks = (r + kKBlock - 1) / kKBlock;
  const size_t budget = 232448 - 2048;  // opt-in shared memory minus static + alignment slack
  const size_t xchg_bytes = (size_t)kHid * 8 * sizeof(float2);
  const size_t u_bytes = (size_t)kblocks * kStageBytes;
  // tiles of a multiple of 256 rows: one MMA covers 256 rows (N = 256). The
  // tensor pipe takes about the same time per MMA at N = 128 as at N = 256,
  // so the wider MMA halves the tensor time per byte of A.
  const int ch = (T % 256 == 0 && chunk256_enabled()) ? 256 : kChunk;
  const size_t st_bytes = (size_t)ch * 128;
  int stages = (int)((budget - 1024 - u_bytes - xchg_bytes) / st_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  // With the gather overlapping this kernel, three stages: the 32 KB given
  // up lets a gather CTA more sit beside each of these CTAs (four instead of
  // two, then bound by registers), worth more than the fourth stage (the
  // 128256-row head at 64 hidden vectors: 109.2 -> 98.5 us per call).
  const int cap = stage_cap() >= 2 ? stage_cap() : (ready && T % kChunk == 0 ? kOverlapStages : 0);
  if (cap >= 2 && stages > cap) stages = cap;
  if (stages < 2) return cudaErrorInvalidValue;
  p.stages = stages;
  p.R = (T % kChunk == 0) ? (M <= 32 ? 4 : (M <= 64 ? 2 : 1)) : 1;
  p.rows_per_rep = kHid / p.R;
  p.lane_shift = (p.R == 1 && M <= 64) ? 64 : 0;
  p.out_ids = out_ids;
  p.out_scores = out_scores;
  p.partials = static_cast<float2*>(partials);
  p.tile_tickets = tile_tickets;
  p.err = err;
  p.wait_cycles = role_wait_cycles();
  p.ready = (T % kChunk == 0) ? ready : nullptr;  // only the dynamic kernel signals
  CUtensorMap amap, umap;
  if (!make_bf16_map(&amap, A, (uint64_t)n, (uint64_t)r, ch, kKBlock) ||
      !make_bf16_map(&umap, u, (uint64_t)M, (uint64_t)r, p.rows_per_rep, kKBlock))
    return cudaErrorInvalidValue;
  const int HC = (M + p.rows_per_rep - 1) / p.rows_per_rep;
  const size_t smem = 1024 + u_bytes + (size_t)stages * st_bytes + xchg_bytes;
  switch (k_tile) {
    case 1: return launch_kt<1>(amap, umap, p, HC, smem, ch, s);
    case 2: return launch_kt<2>(amap, umap, p, HC, smem, ch, s);
    case 4: return launch_kt<4>(amap, umap, p, HC, smem, ch, s);
    case 8: return launch_kt<8>(amap, umap, p, HC, smem, ch, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lmhead
