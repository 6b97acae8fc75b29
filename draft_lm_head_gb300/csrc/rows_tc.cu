// Row-dot products of the head on the 5th-generation tensor cores:
// out[m, j] = X[j] . Y[m] over the contraction length, for every row j of X
// (n x kdim, streamed from HBM) and every hidden vector m of Y (M x kdim,
// streamed from L2 beside it), 128 rows x N hidden vectors per tcgen05 MMA
// with fp32 accumulators in TMEM.
//
// It serves the dense full-vocabulary head W.h that the two-stage head is
// measured against (EAGLE-4 notes, "EAGLE Efficient LM Head"), the
// frequency-pruned head on its 32000 kept rows, and the global variant's
// full score writeback S = A.u ("A Global Top-k based variant": scores of
// the whole vocabulary go back to HBM before the top-k).
//
// Work item = 128 consecutive rows of X x one block of N <= 256 hidden
// vectors; persistent CTAs (one per SM) take items round-robin. A pipeline
// stage holds ksub consecutive 64-element K-blocks of the 128 rows (ksub
// tiled TMA boxes with the 128-byte swizzle, so each row is requested
// ksub x 128 contiguous bytes at a time) and the matching boxes of Y.
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer, warps
// 2-5 epilogue (one TMEM lane quadrant each; two accumulators let the
// epilogue of one item overlap the MMAs of the next). Every mbarrier wait is
// bounded; on timeout the CTA raises an abort flag, records
// LMHEAD_ERR_TIMEOUT in the device error word, drains its own TMA copies,
// frees TMEM and exits.
#include <math.h>
#include <stdlib.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace lmhead {
namespace {

constexpr int kRows = 128;               // X rows per MMA (TMEM lanes)
constexpr int kKB = 64;                  // bf16 per 128-byte swizzled row
constexpr int kXBox = kRows * 128;       // one 128-row x 64-element box
constexpr int kThreads = 192;
constexpr int kMaxStages = 16;
constexpr size_t kSmemBudget = 232448 - 2048;

struct Ctl {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_drain;  // after an abort: the MMA thread's issued MMAs are done
  uint32_t tmem_base;
  int abort;
};

struct RowsParams {
  int64_t n;         // rows of X
  int kdim;          // contraction length
  int kblocks;       // ceil(kdim / 64)
  int ksub;          // K-blocks per pipeline stage
  int kgroups;       // ceil(kblocks / ksub)
  int M;             // rows of Y
  int N;             // MMA N: hidden vectors per item, multiple of 16, <= 256
  int acc_cols;      // TMEM columns per accumulator (power of two >= max(N, 32))
  uint32_t idesc;
  int stages;
  int G;             // CTAs
  int64_t items;
  int64_t n_chunks;  // ceil(n / 128)
  float* out;        // out[m * ldo + row]
  int64_t ldo;
  int* err;
  long long wait_cycles;  // budget of every role wait (drains keep tc::kWaitCycles)
};

__global__ void __launch_bounds__(kThreads, 1)
rows_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
               const RowsParams p) {
  extern __shared__ uint8_t dsmem_raw[];
  __shared__ Ctl ctl;
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NS = p.stages;
  const uint32_t ybox = (uint32_t)p.N * 128u;
  const size_t xstage = (size_t)p.ksub * kXBox;
  const size_t ystage = (size_t)p.ksub * ybox;
  uint8_t* x_s = base;                        // NS x xstage
  uint8_t* y_s = base + (size_t)NS * xstage;  // NS x ystage

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ctl.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&ctl.full[s], 1);
      tc::mbar_init(&ctl.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&ctl.acc_full[a], 1);
      tc::mbar_init(&ctl.acc_empty[a], 4);
    }
    tc::mbar_init(&ctl.mma_drain, 1);
    ctl.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&ctl.tmem_base, 2 * p.acc_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  cta_sync();
  tc::fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&xmap);
      tc::prefetch_tmap(&ymap);
      uint32_t it_s = 0;
      bool ok = true, y_ready = false;
      for (int64_t item = blockIdx.x; item < p.items && ok; item += p.G) {
        const int64_t row0 = (item % p.n_chunks) * kRows;
        const int y0 = (int)(item / p.n_chunks) * p.N;
        for (int kg = 0; kg < p.kgroups; ++kg, ++it_s) {
          const int s = (int)(it_s % NS);
          const int kb0 = kg * p.ksub;
          const int nsub = min(p.ksub, p.kblocks - kb0);
          if (it_s >= (uint32_t)NS &&
              !tc::mbar_wait(&ctl.empty[s], ((it_s / NS) & 1) ^ 1, abort_flag, p.wait_cycles)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&ctl.full[s], (uint32_t)nsub * ((uint32_t)kXBox + ybox));
          for (int sub = 0; sub < nsub; ++sub)
            tc::tma_load_2d(x_s + (size_t)s * xstage + (size_t)sub * kXBox, &xmap, &ctl.full[s],
                            (kb0 + sub) * kKB, (int)row0);
          if (!y_ready) {
            pdl_wait();  // Y may be written by the previous kernel (u of the global path)
            y_ready = true;
          }
          for (int sub = 0; sub < nsub; ++sub)
            tc::tma_load_2d(y_s + (size_t)s * ystage + (size_t)sub * ybox, &ymap, &ctl.full[s],
                            (kb0 + sub) * kKB, y0);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.err, kDevErrTimeout);
      }
      pdl_trigger();
      if (*abort_flag) {
        // drain (bounded) the copies issued last on every stage
        const uint32_t first = it_s > (uint32_t)NS ? it_s - NS : 0;
        for (uint32_t j = first; j < it_s; ++j) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(&ctl.full[j % NS], (j / NS) & 1) &&
                 clock64() - t0 < tc::kWaitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it_s = 0, gq = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < p.items && ok; item += p.G, ++gq) {
        const int a = (int)(gq & 1);
        if (!tc::mbar_wait(&ctl.acc_empty[a], ((gq >> 1) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(a * p.acc_cols);
        for (int kg = 0; kg < p.kgroups; ++kg, ++it_s) {
          const int s = (int)(it_s % NS);
          if (!tc::mbar_wait(&ctl.full[s], (it_s / NS) & 1, abort_flag, p.wait_cycles)) { ok = false; break; }
          tc::fence_after_sync();
          const int kb0 = kg * p.ksub;
          const int nsub = min(p.ksub, p.kblocks - kb0);
          for (int sub = 0; sub < nsub; ++sub) {
            const int kb = kb0 + sub;
            const uint64_t adesc = tc::sw128_kmajor_desc(
                tc::smem_addr(x_s + (size_t)s * xstage + (size_t)sub * kXBox));
            const uint64_t bdesc = tc::sw128_kmajor_desc(
                tc::smem_addr(y_s + (size_t)s * ystage + (size_t)sub * ybox));
            const int nk = min(4, (p.kdim - kb * kKB + 15) / 16);
            for (int k = 0; k < nk; ++k)
              tc::mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, p.idesc, (kb | k) != 0 ? 1u : 0u);
          }
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
    pdl_wait();  // the output may still be read by the previous kernel
    const int q = warp & 3;
    const int row = q * 32 + lane;  // TMEM lane
    uint32_t gq = 0;
    for (int64_t item = blockIdx.x; item < p.items; item += p.G, ++gq) {
      const int a = (int)(gq & 1);
      int okw = 1;
      if (lane == 0) okw = tc::mbar_wait(&ctl.acc_full[a], (gq >> 1) & 1, abort_flag, p.wait_cycles) ? 1 : 0;
      okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
      if (!okw) {
        if (lane == 0) {
          *abort_flag = 1;
          record_error(p.err, kDevErrTimeout);
        }
        break;
      }
      tc::fence_after_sync();
      const int64_t grow = (item % p.n_chunks) * kRows + row;
      const int m0 = (int)(item / p.n_chunks) * p.N;
      const int mcount = min(p.N, p.M - m0);
      for (int cc = 0; cc * 32 < mcount; ++cc) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * p.acc_cols + cc * 32), v);
        tc::tmem_ld_wait();
        if (grow < p.n) {
          // for a fixed column the warp's 32 lanes write 32 consecutive rows
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            if (cc * 32 + jj < mcount)
              p.out[(size_t)(m0 + cc * 32 + jj) * p.ldo + grow] = __uint_as_float(v[jj]);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&ctl.acc_empty[a]);
    }
  }

  tc::fence_before_sync();
  cta_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * p.acc_cols);
  }
}

int stages_for(int N, int ksub) {
  const size_t per = (size_t)ksub * ((size_t)kXBox + (size_t)N * 128);
  int st = (int)((kSmemBudget - 1024) / per);
  return st > kMaxStages ? kMaxStages : st;
}

// Widest stage (most contiguous bytes per row per request) that still
// leaves two stages; LMHEAD_ROWS_KSUB (1, 2 or 4) overrides it for measurements.
int ksub_for(int N) {
  static int forced = -1;
  if (forced < 0) {
    const char* e = getenv("LMHEAD_ROWS_KSUB");
    forced = e ? atoi(e) : 0;
  }
  if ((forced == 1 || forced == 2 || forced == 4) && stages_for(N, forced) >= 2) return forced;
  for (int ks = 4; ks > 1; ks >>= 1)
    if (stages_for(N, ks) >= 2) return ks;
  return 1;
}

}  // namespace

cudaError_t launch_rows_dense_tc(const bf16_t* X, int64_t n, int kdim, const bf16_t* Y, int M,
                                 float* out, int64_t ldo, int* err, cudaStream_t s) {
  RowsParams p = {};
  p.n = n;
  p.kdim = kdim;
  p.kblocks = (kdim + kKB - 1) / kKB;
  p.M = M;
  p.N = M > kRowsTcMaxN ? kRowsTcMaxN : (M + 15) / 16 * 16;
  int acc = 32;
  while (acc < p.N) acc <<= 1;
  p.acc_cols = acc;
  p.idesc = tc::idesc_bf16_f32(kRows, (uint32_t)p.N);
  p.ksub = ksub_for(p.N);
  p.kgroups = (p.kblocks + p.ksub - 1) / p.ksub;
  p.stages = stages_for(p.N, p.ksub);
  if (p.stages < 2) return cudaErrorInvalidValue;
  p.n_chunks = (n + kRows - 1) / kRows;
  p.items = p.n_chunks * ((M + p.N - 1) / p.N);
  p.out = out;
  p.ldo = ldo;
  p.err = err;
  p.wait_cycles = role_wait_cycles();
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  p.G = (int)(p.items < (int64_t)sms ? p.items : (int64_t)sms);
  CUtensorMap xmap, ymap;
  if (!make_bf16_map(&xmap, X, (uint64_t)n, (uint64_t)kdim, kRows, kKB) ||
      !make_bf16_map(&ymap, Y, (uint64_t)M, (uint64_t)kdim, (uint32_t)p.N, kKB))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)p.stages * p.ksub * ((size_t)kXBox + (size_t)p.N * 128);
  static int smem_set[64] = {0};
  cudaError_t e = ensure_dynamic_smem(rows_tc_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_kernel(true, rows_tc_kernel, dim3(p.G), dim3(kThreads), smem, s, xmap, ymap, p);
}

}  // namespace lmhead
