// Candidate expansion of the cluster-level two-stage head (EAGLE-4 notes,
// "EAGLE Efficient LM Head", the third route: select a few groups of tokens,
// then compute the logits of every token inside them).
//
// A group is `group` consecutive rows of the head, so group g contributes
// rows g*group .. g*group + group - 1. Row m's candidate list is its G
// selected groups in selection order, each expanded to its rows in ascending
// order: ids[m, j*group + t] = groups[m, j]*group + t.
#include "common.cuh"
#include "kernels.h"

namespace lmhead {
namespace {

__global__ void __launch_bounds__(256)
expand_groups_kernel(const int32_t* __restrict__ groups, int M, int G, int group,
                     int64_t ngroups, int32_t* __restrict__ ids, int* __restrict__ err) {
  pdl_trigger();
  pdl_wait();  // the groups come from the selection kernel
  const int64_t K = (int64_t)G * group;
  const int64_t total = (int64_t)M * K;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / K;
    const int64_t c = i - m * K;
    const int j = (int)(c / group);
    const int t = (int)(c - (int64_t)j * group);
    const int32_t g = __ldg(groups + m * G + j);
    if (g < 0 || (int64_t)g >= ngroups) {
      record_error(err, kDevErrBadId);
      ids[i] = -1;
    } else {
      ids[i] = g * group + t;
    }
  }
}

}  // namespace

cudaError_t launch_expand_groups(const int32_t* groups, int M, int G, int group, int64_t ngroups,
                                 int32_t* ids, int* err, cudaStream_t s) {
  const int64_t total = (int64_t)M * G * group;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = 8LL * sm_count();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel(true, expand_groups_kernel, dim3((unsigned)blocks), dim3(256), 0, s, groups,
                       M, G, group, ngroups, ids, err);
}

}  // namespace lmhead
