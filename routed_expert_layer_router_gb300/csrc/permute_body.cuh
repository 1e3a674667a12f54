// permute_body.cuh - the body of K-perm (histogram, exclusive scans, stable
// permutation of the routes by expert, optional cache lookup), shared by the
// permutation kernel and the few-token router kernel that ends with it.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// outputs of the permutation (see moe_permute) and the optional lookup
// an id of -1 is a dropped route (the renorm-skip): not listed, inv = -1, no error
constexpr int kDroppedRoute = -1;

// The renorm-skip (Strata-GLM blog, "Uncensoring without touching the
// weights"), token t by one thread: route r = t*k + j (expert ids[r], weight
// w[r]) is dropped when its expert is not resident in the layer's slot run
// and w[r] < tau: ids_eff[r] = kDroppedRoute, w_eff[r] = 0; the kept routes
// keep their expert and get their weight divided by the token's kept sum.
// ids and w are read through L2 (the caller may have written them in the same
// kernel).
struct SkipArgs {
  const int32_t* table;  // the layer's row of the slot table
  int slot_lo, slot_hi;
  float tau;             // 0: off
  int32_t* ids_eff;
  float* w_eff;
};

__device__ __forceinline__ void skip_token(const SkipArgs& sk, const int32_t* ids, const float* w,
                                           int t, int k, int E) {
  float sum = 0.f;
  unsigned keep = 0u;  // k <= 32
  for (int j = 0; j < k; ++j) {
    const int r = t * k + j;
    const int e = __ldcg(ids + r);
    const float wr = __ldcg(w + r);
    int slot = -1;
    if (e >= 0 && e < E) slot = sk.table[e];
    const bool resident = slot >= sk.slot_lo && slot < sk.slot_hi;
    if (resident || !(wr < sk.tau)) {
      keep |= 1u << j;
      sum += wr;
    }
  }
  for (int j = 0; j < k; ++j) {
    const int r = t * k + j;
    const bool kept = (keep >> j) & 1u;
    sk.ids_eff[r] = kept ? __ldcg(ids + r) : kDroppedRoute;
    sk.w_eff[r] = kept ? __ldcg(w + r) / sum : 0.f;
  }
}

struct PermArgs {
  int32_t *counts, *offsets, *perm, *inv, *pad_offsets;
  int pad_align;
  int32_t* status;
  LookupArgs lk;
};

// the bf16 shared expert's gate/up for one token, run beside the router
// (Is == 0: none): h_shared[i] = silu(gate_i . x) * (up_i . x)
struct SharedGuArgs {
  const uint16_t *s_gate, *s_up;  // [Is][H]
  int Is;
  float* h_shared;  // [Is]
};

// shared-memory bytes of permute_body for E experts
__host__ __device__ constexpr size_t permute_smem_bytes(int E) {
  return sizeof(int) * ((size_t)E * (3 + kPermWarps) + 33);
}

// block-wide exclusive scan of one int per thread (returns the total)
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
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
__device__ __forceinline__ void lookup_body(const LookupArgs& a, int E, int c, int* s_scan, int32_t* status) {
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
// `chunk` is the CTA's 1024-route chunk; `sm` holds (3 + 32) * E + 33 ints.
// ids are read through L2 (ld.global.cg): the caller may have written them
// in the same kernel.
__device__ __forceinline__ void permute_body(const int32_t* ids, int n, int E,
                                             int32_t* __restrict__ counts,
                                             int32_t* __restrict__ offsets,
                                             int32_t* __restrict__ perm,
                                             int32_t* __restrict__ inv,
                                             int32_t* __restrict__ pad_offsets, int pad_align,
                                             int32_t* status, const LookupArgs& lk, int* sm,
                                             int chunk) {
  int* s_cnt = sm;
  int* s_pre = s_cnt + E;
  int* s_base = s_pre + E;
  int* s_w = s_base + E;  // [32][E]
  int* s_scan = s_w + kPermWarps * E;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool lead = chunk == 0;
  const int r0 = chunk * kPermThreads;

  for (int e = tid; e < E; e += kPermThreads) {
    s_cnt[e] = 0;
    s_pre[e] = 0;
  }
  __syncthreads();
  // routes before this chunk count into s_pre, the rest into s_cnt
#pragma unroll 4
  for (int r = tid; r < n; r += kPermThreads) {
    const int e = __ldcg(ids + r);
    if (e >= 0 && e < E) atomicAdd(r < r0 ? &s_pre[e] : &s_cnt[e], 1);
    else if (lead && e != kDroppedRoute) set_status(status, MOE_ERR_DEVICE);
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
  const int e = (r < n) ? __ldcg(ids + r) : -1;
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


// The same results as permute_body (and lookup_body) for n <= 32 routes and
// no padded offsets, without block-wide scans: warp 0 ranks the routes by
// (expert, route) with shuffles and runs the lookup over the distinct
// experts (at most 32); every thread writes the counts/offsets of its
// experts by counting the staged ids.  `s_ids` holds 32 ints of shared
// memory.  Called by all threads of the CTA.
__device__ __forceinline__ void permute_small(const int32_t* ids, int n, int E,
                                              int32_t* __restrict__ counts,
                                              int32_t* __restrict__ offsets,
                                              int32_t* __restrict__ perm,
                                              int32_t* __restrict__ inv, int32_t* status,
                                              const LookupArgs& lk, int* s_ids) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    const int r = lane;
    int e = r < n ? __ldcg(ids + r) : -1;
    const bool valid = r < n && e >= 0 && e < E;
    if (r < n && !valid && e != kDroppedRoute) set_status(status, MOE_ERR_DEVICE);
    if (!valid) e = -1;
    s_ids[r] = e;
    // rank among the valid routes by (expert, route), and whether this route
    // is the first of its expert
    int rank = 0, cnt = 0;
    bool first = valid;
    for (int j = 0; j < 32; ++j) {
      const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
      if (ej >= 0 && valid && (ej < e || (ej == e && j < r))) ++rank;
      if (ej == e && j < r) first = false;
      cnt += valid && ej == e;
    }
    if (valid) {
      perm[rank] = r;
      inv[r] = rank;
    } else if (r < n) {
      inv[r] = -1;
    }
    if (lk.table) {
      // lookup over the distinct experts, in expert order: hits, then misses
      int slot = first ? lk.table[e] : -1;
      if (first && slot >= 0 && (slot < lk.slot_lo || slot >= lk.slot_hi)) {
        set_status(status, MOE_ERR_DEVICE);  // stale or foreign slot: treat as a miss
        slot = -1;
      }
      const bool hit = first && slot >= 0, miss = first && slot < 0;
      const unsigned hb = __ballot_sync(0xFFFFFFFFu, hit), mb = __ballot_sync(0xFFFFFFFFu, miss);
      int ph = 0, pm = 0;  // hits / misses among the distinct experts below e
      for (int j = 0; j < 32; ++j) {
        const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
        if (ej < e) {
          ph += (hb >> j) & 1u;
          pm += (mb >> j) & 1u;
        }
      }
      const int nh = __popc(hb), nm = __popc(mb);
      int pos = -1, fslot = -1;
      if (hit) {
        pos = ph;
        fslot = slot;
        lk.act_list[ph] = e;
        lk.src_slot[e] = slot;
      } else if (miss) {
        pos = nh + pm;
        lk.act_list[nh + pm] = e;
        lk.miss_ids[pm] = e;
        if (lk.n_stage > 0) fslot = lk.n_cache + (pm % lk.n_stage);
        else set_status(status, MOE_ERR_DEVICE);
        lk.src_slot[e] = fslot;
      }
      if (lk.meta && pos >= 0) {  // the first route of expert e is at rank
        lk.meta[2 * pos] = make_int4(e, fslot, rank, cnt);
        lk.meta[2 * pos + 1] = make_int4(__float_as_int(lk.gscale[e * 3 + 0]),
                                         __float_as_int(lk.gscale[e * 3 + 1]),
                                         __float_as_int(lk.gscale[e * 3 + 2]), 0);
      }
      if (lane == 0) {
        lk.n_act[0] = nh + nm;
        lk.n_act[1] = nh;
        *lk.n_miss = nm;
      }
    }
  }
  __syncthreads();
  int nv = 0;  // valid routes
  for (int j = 0; j < n; ++j) nv += s_ids[j] >= 0;
  for (int x = tid; x < E; x += blockDim.x) {
    int c = 0, below = 0;
    for (int j = 0; j < n; ++j) {
      const int ej = s_ids[j];
      c += ej == x;
      below += ej >= 0 && ej < x;
    }
    counts[x] = c;
    offsets[x] = below;
    if (lk.table && c == 0) lk.src_slot[x] = -1;  // the active experts' slots: warp 0
  }
  if (tid == 0) offsets[E] = nv;
}

}  // namespace moe
