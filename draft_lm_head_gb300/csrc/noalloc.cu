// lmhead_two_stage_local_noalloc: the fused local two-stage head for callers
// that cannot allocate device memory and cannot hand the library a workspace.
//
// Who needs it: a serving engine that gives all free HBM to its KV-cache pool
// at start-up and allows no allocation afterwards in its decode loop, or C/C++
// code that embeds this library without any device allocator of its own. Such
// callers can still pass inputs and outputs, but not the scratch that
// lmhead_two_stage takes from its workspace (u, M x r bf16, and the
// tensor-core scoring kernel's tile counters).
//
// Here that scratch is a fixed file-scope device array. Every GPU that loads
// the library holds it (kScratchBytes) until the process exits. In host code
// the array's name is only a host-side stand-in, so its device address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on it; the address is then passed to the
// kernels. The call allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library routine.
//
// All calls share the array and it keeps the last call's contents. The tile
// counters must start at zero; the first kernel of every call zeroes them (u
// is fully overwritten). Scoring takes the routes lmhead_two_stage takes
// except where its scratch grows with M and n (tiles that are not a multiple
// of 128 rows on the tensor cores: partial lists per CTA); those score on the
// CUDA-core tile kernel. The gather never overlaps the scoring kernel here. Calls whose work overlaps on the GPU (two streams,
// two host threads) race on the array and corrupt each other's results.
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "lmhead.h"

namespace lmhead {
namespace {

constexpr int kNoAllocMaxM = 256;
constexpr int kNoAllocMaxR = 1024;
constexpr size_t kUBytes = (size_t)kNoAllocMaxM * kNoAllocMaxR * sizeof(bf16_t);  // 512 KiB
constexpr size_t kTicketsOffset = kUBytes;                                     // 256-aligned
constexpr int kTicketInts = kNoAllocMaxM;  // tile counters (one per 128 hidden vectors)
constexpr size_t kScratchBytes = kUBytes + (size_t)kTicketInts * sizeof(int);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch on the current device (set up once per
// device); nullptr if the lookup failed.
char* noalloc_scratch() {
  static char* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    addr[dev] = static_cast<char*>(p);
  }
  return addr[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace lmhead

using namespace lmhead;

extern "C" int lmhead_two_stage_local_noalloc(
    const lmhead_bf16* W, const lmhead_bf16* A, const lmhead_bf16* B, const lmhead_bf16* h,
    const int32_t* token_ids, int64_t n, int d, int r, int M, int T, int k_tile,
    float temperature, int32_t* out_ids, float* out_logits, float* out_q, lmhead_stream stream) {
  if (!W || !A || !B || !h || !out_ids || !out_logits || !out_q) return LMHEAD_ERR_NULL;
  if (n < 1 || n > INT32_MAX || d < 8 || d % 8 || d > 65536 || r < 8 || r % 8 || M < 1 ||
      T < 1 || k_tile < 1 || k_tile > T)
    return LMHEAD_ERR_SHAPE;
  if (!(temperature > 0.f) || temperature == INFINITY) return LMHEAD_ERR_SHAPE;
  // beyond the fixed scratch: refuse rather than allocate
  if (M > kNoAllocMaxM || r > kNoAllocMaxR || k_tile > kFusedMaxKTile) return LMHEAD_ERR_UNSUPPORTED;
  const int64_t full = n / T, tail = n - full * T;
  const int64_t K = full * k_tile + (tail ? (tail < k_tile ? tail : k_tile) : 0);
  if ((int64_t)M * K > INT32_MAX) return LMHEAD_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(A) || !aligned16(B) || !aligned16(h) ||
      (token_ids && !aligned16(token_ids)) || !aligned16(out_ids))
    return LMHEAD_ERR_ALIGN;
  char* scratch = noalloc_scratch();
  if (!scratch) return LMHEAD_ERR_CUDA;
  bf16_t* u = reinterpret_cast<bf16_t*>(scratch);
  int* tickets = reinterpret_cast<int*>(scratch + kTicketsOffset);
  cudaStream_t s = (cudaStream_t)stream;
  // tensor-core scoring where its scratch is only the tile counters (tiles
  // of a multiple of 128 rows, more than the GEMV kernel's two vectors)
  const bool tc = local_topk_tc_supported(r, T, k_tile) && T % 128 == 0 &&
                  !local_topk_gemv_supported(M, r, T, k_tile);
  const int counters = tc ? local_topk_tc_tickets(n, M, T) : 0;
  if (counters > kTicketInts) return LMHEAD_ERR_UNSUPPORTED;
  if (launch_project_u(B, h, d, r, M, u, counters ? tickets : nullptr, counters, s) != cudaSuccess)
    return LMHEAD_ERR_CUDA;
  const cudaError_t e =
      tc ? launch_local_topk_tc(A, u, token_ids, n, r, M, T, k_tile, out_ids, nullptr, nullptr,
                                tickets, device_error_word(), s)
         : launch_local_topk_fma(A, u, token_ids, n, r, M, T, k_tile, out_ids, nullptr, s);
  if (e != cudaSuccess) return LMHEAD_ERR_CUDA;
  // the candidates in blocks of 16 tiles (all hidden vectors of a block
  // together, so repeated W rows hit L2), then the softmax launch
  if (launch_gather_logits(W, h, out_ids, n, d, M, (int)K, out_logits, nullptr, 1.f / temperature,
                           nullptr, device_error_word(), s, kReadyTiles * k_tile) != cudaSuccess)
    return LMHEAD_ERR_CUDA;
  if (launch_row_softmax(out_logits, M, K, 1.f / temperature, out_q, s) != cudaSuccess)
    return LMHEAD_ERR_CUDA;
  return LMHEAD_OK;
}
