// permute.cu - K-perm: histogram, exclusive scan and stable permutation of the
// routes by expert (the grouping behind the Strata-GLM blog's "one batched
// matrix multiply per expert" and the dev.to page's grouped prefill).
// One CTA of 1024 threads per 1024 routes; ranks are computed from warp match
// masks and per-warp counts, so the permutation is deterministic without
// atomics on positions.
#include "common.cuh"

namespace moe {

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// block-wide exclusive scan of one int per thread (returns the total)
__device__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += n;
    }
    s_warp[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  int r = s_warp[wid] + incl - v;
  total = s_warp[32];
  __syncthreads();
  return r;
}

// one expert per thread (E <= 1024 = blockDim); c = routes to expert e
__device__ void lookup_body(const LookupArgs& a, int E, int c, int* s_scan, int32_t* status) {
  const int e = threadIdx.x;
  bool active = (e < E) && c > 0;
  int slot = active ? a.table[e] : -1;
  if (active && slot >= 0 && (slot < a.slot_lo || slot >= a.slot_hi)) {
    set_status(status, MOE_ERR_DEVICE);  // stale or foreign slot: treat as a miss
    slot = -1;
  }
  bool hit = active && slot >= 0;
  bool miss = active && slot < 0;
  int nh, nm;
  int ph = block_exclusive_scan(hit ? 1 : 0, s_scan, nh);
  int pm = block_exclusive_scan(miss ? 1 : 0, s_scan, nm);
  if (e < E) {
    int s = -1;
    if (hit) {
      s = slot;
      a.act_list[ph] = e;
    } else if (miss) {
      a.act_list[nh + pm] = e;
      a.miss_ids[pm] = e;
      if (a.n_stage > 0) s = a.n_cache + (pm % a.n_stage);
      else set_status(status, MOE_ERR_DEVICE);
    }
    a.src_slot[e] = s;
  }
  if (e == 0) {
    a.n_act[0] = nh + nm;
    a.n_act[1] = nh;
    *a.n_miss = nm;
  }
}

// One CTA per 1024-route chunk.  Every CTA histograms all n routes (split into
// those before its chunk and the rest), so each knows both the global offsets
// and its chunk's starting rank per expert without any exchange between CTAs;
// CTA 0 alone writes counts/offsets/pad_offsets and runs the lookup.
// smem: counts[E] | before[E] | base[E] | wcnt[32][E] | scan scratch[33]
__global__ void __launch_bounds__(kPermThreads) k_permute(const int32_t* __restrict__ ids, int n,
                                                          int E, int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ perm,
                                                          int32_t* __restrict__ inv,
                                                          int32_t* __restrict__ pad_offsets,
                                                          int pad_align, int32_t* status,
                                                          LookupArgs lk) {
  extern __shared__ int sm[];
  int* s_cnt = sm;
  int* s_pre = s_cnt + E;
  int* s_base = s_pre + E;
  int* s_w = s_base + E;  // [32][E]
  int* s_scan = s_w + kPermWarps * E;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool lead = blockIdx.x == 0;
  pdl_wait();
  pdl_launch_dependents();
  const int r0 = blockIdx.x * kPermThreads;

  for (int e = tid; e < E; e += kPermThreads) {
    s_cnt[e] = 0;
    s_pre[e] = 0;
  }
  __syncthreads();
  // routes before this chunk count into s_pre, the rest into s_cnt
#pragma unroll 4
  for (int r = tid; r < n; r += kPermThreads) {
    const int e = __ldg(ids + r);
    if (e >= 0 && e < E) atomicAdd(r < r0 ? &s_pre[e] : &s_cnt[e], 1);
    else if (lead) set_status(status, MOE_ERR_DEVICE);
  }
  __syncthreads();
  // exclusive scans of counts (and of padded counts); E <= 1024 = one per thread
  const int pre = (tid < E) ? s_pre[tid] : 0;
  const int c = (tid < E) ? s_cnt[tid] + pre : 0;
  int tot;
  const int off = block_exclusive_scan(c, s_scan, tot);
  if (tid < E) s_base[tid] = off + pre;
  if (lead) {
    if (tid < E) {
      counts[tid] = c;
      offsets[tid] = off;
    }
    if (tid == 0) offsets[E] = tot;
    if (pad_offsets) {
      int cp = (tid < E) ? ((c + pad_align - 1) / pad_align) * pad_align : 0;
      int ptot;
      int poff = block_exclusive_scan(cp, s_scan, ptot);
      if (tid < E) pad_offsets[tid] = poff;
      if (tid == 0) pad_offsets[E] = ptot;
    }
    if (lk.table) lookup_body(lk, E, c, s_scan, status);
  }
  for (int i = tid; i < kPermWarps * E; i += kPermThreads) s_w[i] = 0;
  __syncthreads();

  // stable positions of this chunk's routes: rank within the warp from the
  // match mask, then the per-expert prefix over the warps
  const int r = r0 + tid;
  const int e = (r < n) ? __ldg(ids + r) : -1;
  const bool ok = (e >= 0 && e < E);
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, ok ? e : -1);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (ok && rank == 0) s_w[wid * E + e] = __popc(peers);
  __syncthreads();
  for (int x = tid; x < E; x += kPermThreads) {
    int run = s_base[x];
#pragma unroll 8
    for (int w = 0; w < kPermWarps; ++w) {
      const int cw = s_w[w * E + x];
      s_w[w * E + x] = run;
      run += cw;
    }
  }
  __syncthreads();
  if (ok) {
    const int p = s_w[wid * E + e] + rank;
    perm[p] = r;
    inv[r] = p;
  } else if (r < n) {
    inv[r] = -1;
  }
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
