// K1: the skinny projection u = B h of stage 1 (EAGLE-4 notes, "A Local
// Top-k based variant": both flows start with u = B @ h).
//
// B is r x d (2-5 MB at the workloads' sizes), h is M x d, u is M x r bf16.
// One warp owns one row of B and streams it once with 16-byte loads; a CTA
// holds 8 rows and a block of up to kMB hidden vectors, whose d-chunks are
// staged in shared memory and shared by the 8 warps. fp32 accumulation, one
// bf16 rounding (nearest-even) at the end.
#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace lmhead {
namespace {

constexpr int kRowsPerCta = 8;
constexpr int kMB = 16;
constexpr int kDChunk = 1024;  // bf16 elements of h per staged chunk

__global__ void __launch_bounds__(256) project_u_kernel(const bf16_t* __restrict__ B,
                                                        const bf16_t* __restrict__ h, int d, int r,
                                                        int M, bf16_t* __restrict__ u,
                                                        int* zero_ptr, int zero_ints) {
  __shared__ uint4 hs[kMB * kDChunk / 8];
  pdl_trigger();
  if (zero_ptr) {
    const int nb = gridDim.x * gridDim.y, bid = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = bid * blockDim.x + threadIdx.x; i < zero_ints; i += nb * blockDim.x) zero_ptr[i] = 0;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = blockIdx.x * kRowsPerCta + warp;
  const int m0 = blockIdx.y * kMB;
  const int mb = min(kMB, M - m0);
  float acc[kMB];
#pragma unroll
  for (int i = 0; i < kMB; ++i) acc[i] = 0.f;

  const uint4* brow = reinterpret_cast<const uint4*>(B + (size_t)min(k, r - 1) * d);
  for (int c0 = 0; c0 < d; c0 += kDChunk) {
    const int nvec = min(kDChunk, d - c0) / 8;
    cta_sync();
    for (int i = threadIdx.x; i < mb * nvec; i += blockDim.x) {
      const int mm = i / nvec, v = i - mm * nvec;
      hs[mm * (kDChunk / 8) + v] =
          *reinterpret_cast<const uint4*>(h + (size_t)(m0 + mm) * d + c0 + v * 8);
    }
    cta_sync();
    if (k < r) {
#pragma unroll 2
      for (int v = lane; v < nvec; v += 32) {
        float bf[8];
        unpack8(ldg_nc_v4(brow + c0 / 8 + v), bf);
#pragma unroll
        for (int mm = 0; mm < kMB; ++mm) {
          if (mm < mb) {
            float hf[8];
            unpack8(hs[mm * (kDChunk / 8) + v], hf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[mm] = fmaf(bf[e], hf[e], acc[mm]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int mm = 0; mm < kMB; ++mm) {
    if (mm < mb) {
      const float s = warp_sum(acc[mm]);
      if (lane == 0 && k < r) {
        const __nv_bfloat16 b = __float2bfloat16_rn(s);
        u[(size_t)(m0 + mm) * r + k] = *reinterpret_cast<const bf16_t*>(&b);
      }
    }
  }
}


// ---------------------------------------------------------------- tensor cores
// u tile (up to 128 hidden rows x NB rows of B) = h_tile . B_tile^T, split
// over d across the KS CTAs of a thread-block cluster. Each CTA loads its
// d-slice of h (hrows = min(M, 128) rows; the MMA's other rows hold whatever
// shared memory held, and their output lanes are never read) and of B by
// TMA, runs the MMAs into TMEM, parks its fp32 partial in shared memory, and
// after a cluster barrier the CTAs reduce the partials through distributed
// shared memory in a fixed rank order (deterministic), round to bf16 and
// store u. Every CTA moves kslice x (hrows + 32) bf16 through TMA; loading
// only the M real rows of h (not 128) keeps the projection short.
constexpr int kTcHid = 128;  // MMA M
constexpr int kTcN = 32;     // rows of B per CTA (MMA N); 16 measured slower (more clusters to place)
constexpr int kRedPitch = 33;  // fp32 partial row pitch (bank-conflict padding)

__global__ void __launch_bounds__(128, 1)
project_u_tc_kernel(const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap bmap,
                    int r, int M, int kslice, int hrows, bf16_t* __restrict__ u, int* zero_ptr,
                    int zero_ints, int* err) {
  extern __shared__ uint8_t raw[];
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int nkb = kslice / 64;
  uint8_t* h_s = base;                               // nkb x (128 rows x 128 B)
  uint8_t* b_s = base + (size_t)nkb * kTcHid * 128;  // nkb x (32 rows x 128 B)
  float* red = reinterpret_cast<float*>(h_s);        // reused once the MMAs are done
  const int KS = gridDim.x;
  const int ks = blockIdx.x, rs = blockIdx.y, hc = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();  // the scoring kernel may start streaming A now

  if (zero_ptr) {
    const int nb = gridDim.x * gridDim.y * gridDim.z;
    const int bid = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    for (int i = bid * blockDim.x + threadIdx.x; i < zero_ints; i += nb * blockDim.x) zero_ptr[i] = 0;
  }
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar_load, 1);
    tc::mbar_init(&bar_mma, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 32);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  cta_sync();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (threadIdx.x == 0) {
    tc::prefetch_tmap(&hmap);
    tc::prefetch_tmap(&bmap);
    tc::mbar_arrive_expect_tx(&bar_load, (uint32_t)nkb * (hrows + kTcN) * 128);
    for (int kb = 0; kb < nkb; ++kb) {
      const int x = ks * kslice + kb * 64;
      tc::tma_load_2d(h_s + (size_t)kb * kTcHid * 128, &hmap, &bar_load, x, hc * kTcHid);
      tc::tma_load_2d(b_s + (size_t)kb * kTcN * 128, &bmap, &bar_load, x, rs * kTcN);
    }
    if (tc::mbar_wait(&bar_load, 0, &abort_flag)) {
      tc::fence_after_sync();
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTcHid, kTcN);
      for (int kb = 0; kb < nkb; ++kb) {
        const uint64_t ad = tc::sw128_kmajor_desc(tc::smem_addr(h_s + (size_t)kb * kTcHid * 128));
        const uint64_t bd = tc::sw128_kmajor_desc(tc::smem_addr(b_s + (size_t)kb * kTcN * 128));
        for (int k = 0; k < 4; ++k) tc::mma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
      }
      tc::mma_commit(&bar_mma);
    } else {
      abort_flag = 1;
      record_error(err, kDevErrTimeout);
      // drain the copies issued above before the CTA may exit
      const long long t0 = clock64();
      while (!tc::mbar_try_wait(&bar_load, 0) && clock64() - t0 < tc::kWaitCycles) {
      }
    }
  }
  int okw = 1;
  if (lane == 0) okw = tc::mbar_wait(&bar_mma, 0, &abort_flag) ? 1 : 0;
  okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
  tc::fence_after_sync();
  const int row = warp * 32 + lane;
  if (okw) {
    uint32_t v[32];
    tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), v);
    tc::tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 32; ++c) red[row * kRedPitch + c] = __uint_as_float(v[c]);
  } else {
    for (int c = 0; c < 32; ++c) red[row * kRedPitch + c] = 0.f;
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // every CTA's partial is in its shared memory
  // this CTA reduces rows [r0, r1) of the 128 x 32 tile over the KS ranks
  const int rows_per = (hrows + KS - 1) / KS;
  const int r0 = ks * rows_per, r1 = min(hrows, r0 + rows_per);
  const uint32_t red_addr = tc::smem_addr(red);
  for (int o = threadIdx.x; o < (r1 - r0) * kTcN; o += blockDim.x) {
    const int rr = r0 + o / kTcN, c = o % kTcN;
    const int m = hc * kTcHid + rr, col = rs * kTcN + c;
    if (m >= M || col >= r) continue;
    const uint32_t off = red_addr + (uint32_t)(rr * kRedPitch + c) * 4u;
    float part[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)  // all remote loads in flight, summed in rank order
      part[q] = q < KS ? tc::ld_cluster_f32(tc::map_to_rank(off, (uint32_t)q)) : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) acc += part[q];
    const __nv_bfloat16 b = __float2bfloat16_rn(acc);
    u[(size_t)m * r + col] = *reinterpret_cast<const bf16_t*>(&b);
  }
  tc::cluster_sync();  // no CTA leaves while another still reads its shared memory
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 32);
  }
}

// ---------------------------------------------------------------- small M
// GEMV form for a few hidden vectors: one CTA per row k of B; each thread
// loads its slice of B[k] and of every h[m] at once (everything in flight
// together), then one block reduction per hidden vector. Latency-bound by
// design: a single round trip to memory.
constexpr int kGemvThreads = 128;
constexpr int kGemvMaxM = 8;

// VPT 16-byte vectors per thread cover d <= VPT * 1024; up to MM hidden vectors.
template <int VPT, int MM>
__global__ void __launch_bounds__(kGemvThreads)
project_u_gemv_kernel(const bf16_t* __restrict__ B, const bf16_t* __restrict__ h, int d, int r,
                      int M, bf16_t* __restrict__ u, int* zero_ptr, int zero_ints) {
  constexpr int kGemvMaxVpt = VPT;
  __shared__ float red[kGemvMaxM][kGemvThreads / 32];
  pdl_trigger();  // the scoring kernel may start streaming A now
  if (zero_ptr) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < zero_ints; i += gridDim.x * blockDim.x)
      zero_ptr[i] = 0;
  }
  const int k = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = d >> 3;
  const uint4* brow = reinterpret_cast<const uint4*>(B + (size_t)k * d);
  uint4 bv[kGemvMaxVpt];
  uint4 hv[MM][kGemvMaxVpt];
#pragma unroll
  for (int i = 0; i < kGemvMaxVpt; ++i) {
    const int v = tid + kGemvThreads * i;
    bv[i] = v < nvec ? ldg_nc_v4(brow + v) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int mm = 0; mm < MM; ++mm) {
    const uint4* hrow = reinterpret_cast<const uint4*>(h + (size_t)mm * d);
#pragma unroll
    for (int i = 0; i < kGemvMaxVpt; ++i) {
      const int v = tid + kGemvThreads * i;
      hv[mm][i] = (mm < M && v < nvec) ? __ldg(hrow + v) : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int mm = 0; mm < MM; ++mm) {
    if (mm < M) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kGemvMaxVpt; ++i) acc += dot8(bv[i], hv[mm][i]);
      acc = warp_sum(acc);
      if (lane == 0) red[mm][warp] = acc;
    }
  }
  cta_sync();
  if (tid < M) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kGemvThreads / 32; ++w) s += red[tid][w];
    const __nv_bfloat16 b = __float2bfloat16_rn(s);
    u[(size_t)tid * r + k] = *reinterpret_cast<const bf16_t*>(&b);
  }
}

}  // namespace

cudaError_t launch_project_u(const bf16_t* B, const bf16_t* h, int d, int r, int M, bf16_t* u,
                             int* zero_ptr, int zero_ints, cudaStream_t s) {
  if (M <= kGemvMaxM && d <= 8192) {
    // templates by d (16-byte pieces per thread) and by the batch (1, 2, 4 or 8
    // hidden vectors in registers: a one-vector call keeps its register count
    // low, so the scoring kernel's CTAs fit beside it and start streaming A)
    const int vpt = (d + 1023) / 1024;
    const int mm = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
#define PG(V, MM) \
  return launch_kernel(false, project_u_gemv_kernel<V, MM>, dim3(r), dim3(kGemvThreads), 0, s, B, h, \
                       d, r, M, u, zero_ptr, zero_ints)
    if (vpt <= 1) {
      if (mm == 1) PG(1, 1);
      if (mm == 2) PG(1, 2);
      if (mm == 4) PG(1, 4);
      PG(1, 8);
    }
    if (vpt <= 2) {
      if (mm == 1) PG(2, 1);
      if (mm == 2) PG(2, 2);
      if (mm == 4) PG(2, 4);
      PG(2, 8);
    }
    if (vpt <= 4) {
      if (mm == 1) PG(4, 1);
      if (mm == 2) PG(4, 2);
      if (mm == 4) PG(4, 4);
      PG(4, 8);
    }
    if (mm <= 4) {
      if (mm == 1) PG(8, 1);
      if (mm == 2) PG(8, 2);
      PG(8, 4);
    }
#undef PG
  }
  if (d <= kProjTcMaxD) {
    // d split over a cluster of KS <= 8 CTAs, slices of a multiple of 64 columns
    const int KS = min(8, (d + 511) / 512);
    const int kslice = ((d + KS - 1) / KS + 63) / 64 * 64;
    const int nkb = kslice / 64;
    const int hrows = M < kTcHid ? M : kTcHid;
    const size_t smem = 1024 + (size_t)nkb * (kTcHid + kTcN) * 128;
    CUtensorMap hmap, bmap;
    if (!make_bf16_map(&hmap, h, (uint64_t)M, (uint64_t)d, (uint32_t)hrows, 64) ||
        !make_bf16_map(&bmap, B, (uint64_t)r, (uint64_t)d, kTcN, 64))
      return cudaErrorInvalidValue;
    static int smem_set[64] = {0};
    cudaError_t e = ensure_dynamic_smem(project_u_tc_kernel, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(KS, (r + kTcN - 1) / kTcN, (M + kTcHid - 1) / kTcHid);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = KS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, project_u_tc_kernel, hmap, bmap, r, M, kslice, hrows, u,
                              zero_ptr, zero_ints, device_error_word());
  }
  dim3 grid((r + kRowsPerCta - 1) / kRowsPerCta, (M + kMB - 1) / kMB);
  return launch_kernel(false, project_u_kernel, grid, dim3(256), 0, s, B, h, d, r, M, u, zero_ptr,
                       zero_ints);
}

}  // namespace lmhead
