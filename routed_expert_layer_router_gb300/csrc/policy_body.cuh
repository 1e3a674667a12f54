// policy_body.cuh - the adaptive expert cache's policy step ("Project Maya"
// page: "How 'most-used' is measured", "Promotion on every miss, eviction at
// the boundary"), shared by the cache's own kernel and the fused router
// kernel of the layer's few-token path.
#pragma once
#include "common.cuh"

namespace moe {

// One layer forward, after the lookup (one CTA, a thread per expert):
//   1. promotion: the lookup's misses, in ascending id, take the layer's free
//      slots in ascending order and are resident from then on; the others keep
//      their staging slot (miss_dst[i] = where miss i is gathered);
//   2. counts: +1 per route, capped at 2^24; last = this forward's number;
//      every 32,768 route events (all layers) every count is halved;
//   3. boundary: while fewer than `spares` slots are free, the resident with
//      the smallest (count, last, id) is evicted.
struct PolicyArgs {
  int L, E, layer, slot_lo, slot_hi, spares;
  int32_t* table_row;
  uint32_t *cnt, *last, *stamp;  // stamp[L] = route events
  int32_t* freeslot;
  const int32_t* counts;
  int32_t* src_slot;
  const int32_t *n_act, *miss_ids, *n_miss;
  int32_t* miss_dst;
  int4* meta;  // the layer's compact expert records, or nullptr
};

constexpr int kPolicyThreads = 1024;
constexpr int kPolicyMaxRun = 8192;  // slots of one layer's run
constexpr uint32_t kCountCap = 1u << 24;
constexpr uint32_t kHalveEvents = 32768;

// (key, id) minimum over the CTA; every thread gets the winner's id (-1: none)
__device__ __forceinline__ int block_argmin(uint64_t key, int id, uint64_t* s_key, int* s_id) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t k2 = __shfl_down_sync(0xFFFFFFFFu, key, o);
    const int i2 = __shfl_down_sync(0xFFFFFFFFu, id, o);
    if (k2 < key || (k2 == key && (unsigned)i2 < (unsigned)id)) { key = k2; id = i2; }
  }
  if (lane == 0) { s_key[wid] = key; s_id[wid] = id; }
  __syncthreads();
  if (wid == 0) {
    key = lane < (int)(blockDim.x >> 5) ? s_key[lane] : ~0ull;
    id = lane < (int)(blockDim.x >> 5) ? s_id[lane] : -1;
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t k2 = __shfl_down_sync(0xFFFFFFFFu, key, o);
      const int i2 = __shfl_down_sync(0xFFFFFFFFu, id, o);
      if (k2 < key || (k2 == key && (unsigned)i2 < (unsigned)id)) { key = k2; id = i2; }
    }
    if (lane == 0) s_id[32] = key == ~0ull ? -1 : id;
  }
  __syncthreads();
  const int w = s_id[32];
  __syncthreads();
  return w;
}

// The layer's row of the table and counts, and its slot run's free flags, are
// staged in shared memory (`sm`, policy_smem_bytes(E, run) bytes, 16-byte
// aligned), so that the serial parts (promotions, evictions) run on shared
// memory and the whole step costs a few global round trips.  Called by all
// threads of one CTA (E <= blockDim.x <= 1024); on the caller's stream order
// after the lookup, or in the same CTA after a __syncthreads.
// layout: argmin scratch (32 keys, 33 ids), then table row, misses, slots,
// counts, latest forwards (E each), then the run's free flags
constexpr int kPolicyScratch = 32 * 8 + 36 * 4;  // 400 bytes, keeps what follows 16-byte aligned
__host__ __device__ __forceinline__ size_t policy_smem_bytes(int E, int run) {
  return (size_t)kPolicyScratch + (size_t)5 * E * 4 + (size_t)run;
}

__device__ __forceinline__ void policy_body(const PolicyArgs& a, unsigned char* sm) {
  const int t = threadIdx.x, E = a.E, P = a.slot_hi - a.slot_lo;
  uint64_t* s_key = reinterpret_cast<uint64_t*>(sm);
  int* s_id = reinterpret_cast<int*>(sm + 32 * 8);
  int* s_tab = reinterpret_cast<int*>(sm + kPolicyScratch);
  int* s_miss = s_tab + E;
  int* s_src = s_miss + E;
  uint32_t* s_cnt = reinterpret_cast<uint32_t*>(s_src + E);
  uint32_t* s_last = s_cnt + E;
  unsigned char* s_free = reinterpret_cast<unsigned char*>(s_last + E);
  __shared__ unsigned long long s_routes;
  __shared__ uint32_t s_now;
  __shared__ int s_halve, s_nfree;
  const size_t row = (size_t)a.layer * E;
  // stage (one round trip)
  int c = 0;
  if (t < E) {
    s_tab[t] = a.table_row[t];
    s_cnt[t] = a.cnt[row + t];
    s_last[t] = a.last[row + t];
    s_miss[t] = a.miss_ids[t];
    s_src[t] = a.src_slot[t];
    c = a.counts[t];
  }
  for (int j = t; j < P; j += blockDim.x) s_free[j] = a.freeslot[a.slot_lo + j] != 0;
  if (t == 0) {
    s_routes = 0;
    s_now = a.stamp[a.layer] + 1;
  }
  __syncthreads();
  // 1. promotion: misses and free slots in ascending order (one thread)
  if (t == 0) {
    const int nm = *a.n_miss, nh = a.n_act[1];
    int f = 0;
    for (int i = 0; i < nm; ++i) {
      const int e = s_miss[i];
      if (e < 0 || e >= E) {  // reported by the lookup's checks
        a.miss_dst[i] = -1;
        continue;
      }
      while (f < P && !s_free[f]) ++f;
      int dst = s_src[e];  // its staging slot
      if (f < P) {
        dst = a.slot_lo + f;
        s_free[f++] = 0;
        s_tab[e] = dst;
        a.src_slot[e] = dst;
        if (a.meta) a.meta[2 * (nh + i)].y = dst;
      }
      a.miss_dst[i] = dst;
    }
  }
  // 2. counts
  if (c > 0) {
    const uint64_t v = (uint64_t)s_cnt[t] + (uint64_t)c;
    s_cnt[t] = v > kCountCap ? kCountCap : (uint32_t)v;
    s_last[t] = s_now;
    atomicAdd(&s_routes, (unsigned long long)c);
  }
  __syncthreads();
  if (t == 0) {
    const uint64_t ev = (uint64_t)a.stamp[a.L] + s_routes;
    s_halve = ev >= kHalveEvents;
    a.stamp[a.L] = s_halve ? 0u : (uint32_t)ev;
    a.stamp[a.layer] = s_now;
  }
  __syncthreads();
  if (s_halve) {
    if (t < E) s_cnt[t] >>= 1;
    for (size_t i = t; i < (size_t)a.L * E; i += blockDim.x)
      if (i < row || i >= row + E) a.cnt[i] >>= 1;  // the other layers
  }
  // 3. boundary: evict down to the spares
  if (t == 0) {
    int nf = 0;
    for (int j = 0; j < P; ++j) nf += s_free[j];
    s_nfree = nf;
  }
  __syncthreads();
  while (s_nfree < a.spares) {
    const bool res = t < E && s_tab[t] >= 0;
    const uint64_t key = res ? ((uint64_t)s_cnt[t] << 32) | s_last[t] : ~0ull;
    const int victim = block_argmin(key, res ? t : -1, s_key, s_id);
    if (victim < 0) break;
    if (t == 0) {
      const int f = s_tab[victim] - a.slot_lo;  // a slot outside the run: the lookup reports it
      if (f >= 0 && f < P) {
        s_free[f] = 1;
        ++s_nfree;
      }
      s_tab[victim] = -1;
    }
    __syncthreads();
  }
  __syncthreads();
  // write back
  if (t < E) {
    a.table_row[t] = s_tab[t];
    a.cnt[row + t] = s_cnt[t];
    a.last[row + t] = s_last[t];
  }
  for (int j = t; j < P; j += blockDim.x) a.freeslot[a.slot_lo + j] = s_free[j];
}

}  // namespace moe
