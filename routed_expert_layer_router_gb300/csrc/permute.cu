// permute.cu - K-perm: histogram, exclusive scan and stable permutation of the
// routes by expert (the grouping behind the Strata-GLM blog's "one batched
// matrix multiply per expert" and the dev.to page's grouped prefill).
// One CTA of 1024 threads per 1024 routes; ranks are computed from warp match
// masks and per-warp counts, so the permutation is deterministic without
// atomics on positions.
#include "permute_body.cuh"

namespace moe {

// K-perm: one CTA per 1024-route chunk (see permute_body)
__global__ void __launch_bounds__(kPermThreads) k_permute(const int32_t* __restrict__ ids, int n,
                                                          int E, int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ perm,
                                                          int32_t* __restrict__ inv,
                                                          int32_t* __restrict__ pad_offsets,
                                                          int pad_align, int32_t* status,
                                                          LookupArgs lk) {
  extern __shared__ int sm[];
  pdl_wait();
  pdl_launch_dependents();
  permute_body(ids, n, E, counts, offsets, perm, inv, pad_offsets, pad_align, status, lk, sm,
               blockIdx.x);
}

// K-lookup: one CTA of 1024 threads, one expert per thread
__global__ void __launch_bounds__(kPermThreads) k_lookup(LookupArgs a, int E,
                                                         const int32_t* __restrict__ counts,
                                                         int32_t* status) {
  __shared__ int s_scan[33];
  const int e = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  lookup_body(a, E, e < E ? counts[e] : 0, s_scan, status);
}

}  // namespace moe

namespace moe {
// opt in to more than 48 KiB of dynamic shared memory (E > 340); idempotent
moe_status permute_setup() {
  static int done = 0;
  if (done) return MOE_OK;
  if (cudaFuncSetAttribute(k_permute, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  done = 1;
  return MOE_OK;
}
}  // namespace moe

using namespace moe;

namespace moe {
// K-perm, followed in the same launch by the expert-cache lookup when lk.table
// is set (the layer's path: one launch instead of two)
moe_status launch_permute(const int32_t* ids, int T, int k, int E, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* pad_offsets,
                          int pad_align, int32_t* status, const LookupArgs& lk, cudaStream_t s) {
  if (T < 0 || k <= 0 || E <= 0 || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !perm || !inv)) return MOE_ERR_INVALID_ARG;
  if (pad_offsets && pad_align <= 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || (long long)T * k > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  size_t smem = sizeof(int) * ((size_t)E * (3 + kPermWarps) + 33);
  if (smem > 48 * 1024 && permute_setup() != MOE_OK) return MOE_ERR_CUDA;
  const int n = T * k;
  const int grid = n > 0 ? (n + kPermThreads - 1) / kPermThreads : 1;
  if (launch_pdl(k_permute, grid, kPermThreads, smem, s, ids, T * k, E, counts, offsets, perm, inv,
                 pad_offsets, pad_align, status, lk) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
}  // namespace moe

MOE_API moe_status moe_permute(const int32_t* ids, int T, int k, int E, int32_t* counts,
                               int32_t* offsets, int32_t* perm, int32_t* inv,
                               int32_t* pad_offsets, int pad_align, int32_t* status,
                               void* stream) {
  LookupArgs none = {};
  return launch_permute(ids, T, k, E, counts, offsets, perm, inv, pad_offsets, pad_align, status,
                        none, (cudaStream_t)stream);
}

namespace moe {
moe_status launch_lookup(const LookupArgs& a, int E, const int32_t* counts, int32_t* status,
                         cudaStream_t s) {
  if (launch_pdl(k_lookup, 1, kPermThreads, 0, s, a, E, counts, status) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
}  // namespace moe
