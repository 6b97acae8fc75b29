// Shared device helpers of liblmhead (bf16 unpacking, order-preserving keys,
// warp reductions, the device error word).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lmhead.h"

namespace lmhead {

constexpr int kWarp = 32;

// Error word values (a kernel never traps: it records and carries on).
constexpr int kDevErrBadId = 1;
constexpr int kDevErrTimeout = 2;

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// 8 bf16 packed in a uint4 -> 8 floats (bf16 -> fp32 is exact: shift left 16).
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  float fa[8], fb[8];
  unpack8(a, fa);
  unpack8(b, fb);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = fmaf(fa[i], fb[i], s);
  return s;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// fp32 -> uint32 whose unsigned order is the float order (-0 folded into +0).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// Unique 64-bit selection key: score order first, then the smaller
// vocabulary id wins among equal scores.
__device__ __forceinline__ uint64_t select_key(float score, int32_t vocab_id) {
  return (static_cast<uint64_t>(float_key(score)) << 32) |
         static_cast<uint32_t>(~static_cast<uint32_t>(vocab_id));
}

__device__ __forceinline__ int32_t key_id(uint64_t k) {
  return static_cast<int32_t>(~static_cast<uint32_t>(k & 0xFFFFFFFFull));
}

__device__ __forceinline__ float key_score(uint64_t k) {
  return key_float(static_cast<uint32_t>(k >> 32));
}

// (score desc, id asc) "a beats b".
__device__ __forceinline__ bool beats(float sa, int32_t ia, float sb, int32_t ib) {
  return sa > sb || (sa == sb && ia < ib);
}

// Raise a kernel's dynamic shared-memory limit, once per device and size:
// the attribute call is slow enough to starve the GPU if made per launch.
template <typename Kernel>
inline cudaError_t ensure_dynamic_smem(Kernel kernel, size_t bytes, int* cache64) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if ((size_t)cache64[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cache64[dev] = (int)bytes;
  return e;
}

// Launch `kernel`; with pdl, as a programmatic dependent of the previous
// kernel on the stream: it may start while that kernel runs and must
// execute griddepcontrol.wait before reading what that kernel writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                 size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// CTA-wide barriers that count arriving threads one by one (PTX
// barrier.sync without .aligned), so they are correct when the lanes of a
// warp arrive at different times, as in the warp-specialised kernels where
// lane 0 runs a role loop while lanes 1-31 go straight to the final barrier.
// A globaltimer trace of the fused scoring kernel showed __syncthreads (the
// aligned form) releasing such a CTA before its epilogue warps had arrived.
__device__ __forceinline__ void cta_sync() { asm volatile("barrier.sync 0;" ::: "memory"); }
// Named barrier `id` over `count` threads (a multiple of 32), same counting.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- ready counters between the scoring kernel and the gather
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// A bounded wait on another kernel's progress gives up after this many SM
// clock cycles (about a second).
constexpr long long kCounterWaitCycles = 2000000000ll;

// Wait until *counter >= need. Gives up (false) when *stop is set (the
// producing kernel aborted on a timeout of its own) or after
// kCounterWaitCycles (then records a timeout in `err`).
__device__ __forceinline__ bool wait_count(const int* counter, int need, const int* stop,
                                           int* err) {
  const long long t0 = clock64();
  while (ld_acquire(counter) < need) {
    if (*reinterpret_cast<const volatile int*>(stop) != 0) return false;
    if (clock64() - t0 > kCounterWaitCycles) {
      record_error(err, kDevErrTimeout);
      return false;
    }
    __nanosleep(256);
  }
  return true;
}

// Publish `count` more ready rows on `counter`, after this thread's and (by
// a preceding CTA barrier) its CTA's earlier stores.
__device__ __forceinline__ void signal_count(int* counter, int count) {
  __threadfence();
  atomicAdd(counter, count);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace lmhead
