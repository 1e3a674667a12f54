// cache.cu - the per-layer HBM hot-expert cache and K-gather.
//
// Slot arena: n_cache slots followed by n_stage staging slots, one fixed-stride
// record each ("Project Maya": a device table layer x expert -> VRAM slot, each
// layer owning its own run of slots so no slot is overwritten while another
// layer reads it; Strata-GLM blog: exclusive tiers, byte-sized slots).
// K-gather copies records of missing experts from the pinned, mapped host
// arena with 16-byte loads issued by many thread blocks at once (the "Project
// Maya" GPU pull of RAM-tier experts; the dev.to page's wide-read gather over a
// GPU-resident list, which keeps CUDA graphs replayable).
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "policy_body.cuh"

struct expcache {
  int L, E, H, I, fmt;
  int n_cache, n_stage;
  uint64_t rec_bytes;
  uint8_t* arena;            // device, (n_cache + n_stage) * rec_bytes
  int32_t* table;            // device [L][E]
  int32_t* slot_lo;          // host [L]: layer l owns cache slots [slot_lo[l], slot_hi[l])
  int32_t* slot_hi;
  const uint8_t* host_dev;   // device-side address of the host arena (or NULL)
  uint64_t host_records;
  int64_t* host_index_dev;   // device [L][E] (or NULL)
  bool partitioned;          // created with per-layer slot runs
  // adaptive policy (expcache_set_policy), all device; spares < 0: off
  int spares;
  uint32_t* cnt;             // [L][E] decayed route counts
  uint32_t* last;            // [L][E] layer-forward number of the latest route
  uint32_t* stamp;           // [L] forwards of each layer, then [L] = route events
  int32_t* freeslot;         // [n_cache] 1 = free (a spare)
};

namespace moe {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 8;                       // 16-byte loads in flight per thread
constexpr uint64_t kGatherChunk = (uint64_t)kGatherThreads * kGatherUnroll * 16 * 4;  // 128 KiB

__global__ void __launch_bounds__(kGatherThreads) k_gather(
    const uint8_t* __restrict__ host, const int64_t* __restrict__ host_index, uint64_t host_records,
    uint8_t* __restrict__ arena, int32_t* __restrict__ table_row, int E, uint64_t rec_bytes,
    int n_cache, int n_stage, const int32_t* __restrict__ ids, const int32_t* __restrict__ d_n,
    int first, const int32_t* __restrict__ dst_slots, int slot_lo, int slot_hi, int32_t* status) {
  // The next kernel (the FFN, which waits for this one anyway) is let launch
  // only when a CTA has done its copying: launched early, its CTAs would sit
  // on the SMs that this grid's later CTAs need to keep the link busy.
  pdl_wait();
  const int i = first + blockIdx.y;
  if (i >= *d_n) return;
  const int e = ids[i];
  if (e < 0 || e >= E) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MOE_ERR_DEVICE);
    return;
  }
  const int64_t hr = host_index ? host_index[e] : -1;
  int slot;
  if (dst_slots) {
    // a cache slot of this layer, or a staging slot (a miss the adaptive
    // policy could not promote)
    slot = dst_slots[i];
    const bool staging = n_stage > 0 && slot >= n_cache && slot < n_cache + n_stage;
    if (!staging && (slot < slot_lo || slot >= slot_hi)) slot = -1;
  } else {
    slot = n_stage > 0 ? n_cache + (i % n_stage) : -1;
  }
  if (hr < 0 || (uint64_t)hr >= host_records || !host || slot < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MOE_ERR_DEVICE);
    return;
  }
  const uint8_t* src = host + (uint64_t)hr * rec_bytes;
  uint8_t* dst = arena + (uint64_t)slot * rec_bytes;
  const uint64_t n16 = rec_bytes / 16;
  // grid-stride over 16-byte words of this record, kGatherUnroll loads in flight
  const uint64_t stride = (uint64_t)gridDim.x * kGatherThreads;
  uint64_t w = (uint64_t)blockIdx.x * kGatherThreads + threadIdx.x;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (; w + (kGatherUnroll - 1) * stride < n16; w += kGatherUnroll * stride) {
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) v[u] = ldg_stream(s4 + w + u * stride);
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) d4[w + u * stride] = v[u];
  }
  for (; w < n16; w += stride) d4[w] = ldg_stream(s4 + w);
  if (dst_slots && table_row && slot < n_cache && blockIdx.x == 0 && threadIdx.x == 0)
    table_row[e] = slot;
  pdl_launch_dependents();
}

__global__ void k_set_table(int32_t* table_entry, int slot) { *table_entry = slot; }

// K-policy: one CTA running policy_body (policy_body.cuh)
__global__ void __launch_bounds__(kPolicyThreads) k_cache_policy(PolicyArgs a) {
  extern __shared__ __align__(16) unsigned char smem_pol[];
  pdl_wait();
  pdl_launch_dependents();
  policy_body(a, smem_pol);
}

// One 16-byte read per 4 KiB page of the mapped host arena.  The device's
// first read of a host page is slow: on the 16-layer stack a step whose misses
// read records never read before took up to ten times as long as the same
// step repeated.  The cache pays that once, at creation.
constexpr uint64_t kTouchStride = 4096;
__global__ void __launch_bounds__(256) k_touch_host(const uint8_t* __restrict__ host,
                                                    uint64_t pages) {
  for (uint64_t i = (uint64_t)blockIdx.x * 256 + threadIdx.x; i < pages;
       i += (uint64_t)gridDim.x * 256)
    (void)ldg_stream(host + i * kTouchStride);
}

moe_status launch_lookup(const LookupArgs& a, int E, const int32_t* counts, int32_t* status,
                         cudaStream_t s);

}  // namespace moe

using namespace moe;

MOE_API uint64_t moe_record_bytes(int H, int I, int format) {
  if (H <= 0 || I <= 0) return 0;
  if (format != MOE_FMT_NVFP4 && format != MOE_FMT_MXFP4) return 0;
  return RecordLayout(H, I, format).bytes;
}

namespace moe {
moe_status ensure_setup();
}

MOE_API moe_status expcache_create(const expcache_desc* d, expcache** out) {
  if (!d || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (d->L <= 0 || d->E <= 0 || d->H <= 0 || d->I <= 0 || d->n_cache_slots < 0 || d->n_stage < 0)
    return MOE_ERR_INVALID_ARG;
  if (d->H % 256 || d->I % 128 || d->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (d->format != MOE_FMT_NVFP4 && d->format != MOE_FMT_MXFP4) return MOE_ERR_UNSUPPORTED;
  if (d->host_arena && !d->host_index) return MOE_ERR_INVALID_ARG;
  if (d->layer_slots) {
    if (d->layer_slots[0] < 0) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < d->L; ++l)
      if (d->layer_slots[l + 1] < d->layer_slots[l]) return MOE_ERR_INVALID_ARG;
    if (d->layer_slots[d->L] > d->n_cache_slots) return MOE_ERR_INVALID_ARG;
  }
  if (moe_status st = moe::ensure_setup()) return st;
  expcache* c = (expcache*)calloc(1, sizeof(expcache));
  if (!c) return MOE_ERR_OOM;
  c->L = d->L; c->E = d->E; c->H = d->H; c->I = d->I;
  c->n_cache = d->n_cache_slots; c->n_stage = d->n_stage;
  c->partitioned = d->layer_slots != nullptr;
  c->spares = -1;
  c->fmt = d->format;
  c->rec_bytes = RecordLayout(d->H, d->I, d->format).bytes;
  c->slot_lo = (int32_t*)malloc(sizeof(int32_t) * d->L);
  c->slot_hi = (int32_t*)malloc(sizeof(int32_t) * d->L);
  if (!c->slot_lo || !c->slot_hi) {
    free(c->slot_lo); free(c->slot_hi); free(c);
    return MOE_ERR_OOM;
  }
  for (int l = 0; l < d->L; ++l) {
    c->slot_lo[l] = d->layer_slots ? d->layer_slots[l] : 0;
    c->slot_hi[l] = d->layer_slots ? d->layer_slots[l + 1] : d->n_cache_slots;
  }
  uint64_t slots = (uint64_t)d->n_cache_slots + (uint64_t)d->n_stage;
  moe_status st = MOE_OK;
  if (slots && cudaMalloc((void**)&c->arena, slots * c->rec_bytes) != cudaSuccess) st = MOE_ERR_OOM;
  if (st == MOE_OK &&
      cudaMalloc((void**)&c->table, sizeof(int32_t) * (size_t)d->L * d->E) != cudaSuccess)
    st = MOE_ERR_OOM;
  if (st == MOE_OK && cudaMemset(c->table, 0xFF, sizeof(int32_t) * (size_t)d->L * d->E) != cudaSuccess)
    st = MOE_ERR_CUDA;
  if (st == MOE_OK && d->host_arena) {
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, (void*)d->host_arena, 0) != cudaSuccess) st = MOE_ERR_CUDA;
    c->host_dev = (const uint8_t*)dp;
    c->host_records = d->host_arena_records;
    if (st == MOE_OK &&
        cudaMalloc((void**)&c->host_index_dev, sizeof(int64_t) * (size_t)d->L * d->E) != cudaSuccess)
      st = MOE_ERR_OOM;
    if (st == MOE_OK && cudaMemcpy(c->host_index_dev, d->host_index,
                                   sizeof(int64_t) * (size_t)d->L * d->E,
                                   cudaMemcpyHostToDevice) != cudaSuccess)
      st = MOE_ERR_CUDA;
    // the records are multiples of 16 bytes, so every read below ends inside the arena
    const uint64_t bytes = c->host_records * c->rec_bytes;
    if (st == MOE_OK && bytes > 0) {
      k_touch_host<<<kSMs * 8, 256>>>(c->host_dev, (bytes + kTouchStride - 1) / kTouchStride);
      if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        st = MOE_ERR_CUDA;
    }
  }
  if (st != MOE_OK) {
    cudaGetLastError();
    expcache_destroy(c);
    return st;
  }
  *out = c;
  return MOE_OK;
}

MOE_API moe_status expcache_destroy(expcache* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  if (c->arena) cudaFree(c->arena);
  if (c->table) cudaFree(c->table);
  if (c->host_index_dev) cudaFree(c->host_index_dev);
  if (c->cnt) cudaFree(c->cnt);
  if (c->last) cudaFree(c->last);
  if (c->stamp) cudaFree(c->stamp);
  if (c->freeslot) cudaFree(c->freeslot);
  free(c->slot_lo);
  free(c->slot_hi);
  free(c);
  return MOE_OK;
}

MOE_API void* expcache_slot_ptr(const expcache* c, int s) {
  if (!c || s < 0 || s >= c->n_cache + c->n_stage) return nullptr;
  return c->arena + (uint64_t)s * c->rec_bytes;
}

MOE_API const int32_t* expcache_slot_table(const expcache* c) { return c ? c->table : nullptr; }

MOE_API moe_status expcache_set_resident(expcache* c, int layer, int expert, int slot,
                                         void* stream) {
  if (!c || layer < 0 || layer >= c->L || expert < 0 || expert >= c->E) return MOE_ERR_INVALID_ARG;
  if (slot != -1 && (slot < c->slot_lo[layer] || slot >= c->slot_hi[layer]))
    return MOE_ERR_INVALID_ARG;
  if (c->spares >= 0) return MOE_ERR_UNSUPPORTED;  // the adaptive policy owns the table
  k_set_table<<<1, 1, 0, (cudaStream_t)stream>>>(c->table + (size_t)layer * c->E + expert, slot);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

namespace moe {
// grid width for one record: enough blocks to keep the link busy
static int gather_blocks_per_record(uint64_t rec_bytes, int max_count) {
  uint64_t chunks = (rec_bytes + kGatherChunk - 1) / kGatherChunk;
  int want = (int)((2 * kSMs + max_count - 1) / max_count);  // ~2 blocks per SM overall
  if (want < 1) want = 1;
  return (int)(chunks < (uint64_t)want ? chunks : (uint64_t)want);
}
}  // namespace moe

MOE_API moe_status expcache_fill(expcache* c, int layer, const int32_t* d_expert_ids,
                                 const int32_t* d_n, int first, int max_count,
                                 const int32_t* d_dst_slots, int32_t* status, void* stream) {
  if (!c || !d_expert_ids || !d_n || layer < 0 || layer >= c->L || first < 0 || max_count < 0)
    return MOE_ERR_INVALID_ARG;
  if (max_count == 0) return MOE_OK;
  if (!d_dst_slots && c->n_stage == 0) return MOE_ERR_INVALID_ARG;
  if (max_count > 65535) return MOE_ERR_UNSUPPORTED;
  dim3 grid(gather_blocks_per_record(c->rec_bytes, max_count), max_count);
  if (launch_pdl(k_gather, grid, kGatherThreads, 0, (cudaStream_t)stream, c->host_dev,
                 c->host_index_dev ? c->host_index_dev + (size_t)layer * c->E : nullptr,
                 c->host_records, c->arena,
                 c->spares >= 0 ? nullptr : c->table + (size_t)layer * c->E,  // the policy's table
                 c->E, c->rec_bytes,
                 c->n_cache, c->n_stage, d_expert_ids, d_n, first, d_dst_slots,
                 c->slot_lo[layer], c->slot_hi[layer], status) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

namespace moe {
void cache_gather_args(const expcache* c, int layer, GatherArgs* out) {
  out->host = c->host_dev;
  out->host_index = c->host_index_dev ? c->host_index_dev + (size_t)layer * c->E : nullptr;
  out->host_records = c->host_records;
  out->n_cache = c->n_cache;
  out->n_stage = c->n_stage;
  out->slot_lo = c->slot_lo[layer];
  out->slot_hi = c->slot_hi[layer];
}

void cache_lookup_args(const expcache* c, int layer, int32_t* src_slot, int32_t* act_list,
                       int32_t* n_act, int32_t* miss_ids, int32_t* n_miss, LookupArgs* out) {
  out->table = c->table + (size_t)layer * c->E;
  out->slot_lo = c->slot_lo[layer];
  out->slot_hi = c->slot_hi[layer];
  out->n_cache = c->n_cache;
  out->n_stage = c->n_stage;
  out->src_slot = src_slot;
  out->act_list = act_list;
  out->n_act = n_act;
  out->miss_ids = miss_ids;
  out->n_miss = n_miss;
  out->meta = nullptr;
  out->gscale = nullptr;
}
}  // namespace moe

MOE_API moe_status expcache_lookup(const expcache* c, int layer, const int32_t* counts,
                                   int32_t* src_slot, int32_t* act_list, int32_t* n_act,
                                   int32_t* miss_ids, int32_t* n_miss, int32_t* status,
                                   void* stream) {
  if (!c || !counts || !src_slot || !act_list || !n_act || !miss_ids || !n_miss || layer < 0 ||
      layer >= c->L)
    return MOE_ERR_INVALID_ARG;
  LookupArgs la;
  cache_lookup_args(c, layer, src_slot, act_list, n_act, miss_ids, n_miss, &la);
  return launch_lookup(la, c->E, counts, status, (cudaStream_t)stream);
}

// internal accessors for the FFN and the layer
namespace moe {
const uint8_t* cache_arena(const expcache* c) { return c->arena; }
uint64_t cache_rec_bytes(const expcache* c) { return c->rec_bytes; }
int cache_format(const expcache* c) { return c->fmt; }
int cache_n_cache(const expcache* c) { return c->n_cache; }
int cache_n_stage(const expcache* c) { return c->n_stage; }
int cache_E(const expcache* c) { return c->E; }
int cache_L(const expcache* c) { return c->L; }
int cache_H(const expcache* c) { return c->H; }
int cache_I(const expcache* c) { return c->I; }
}  // namespace moe

// ---- adaptive policy: host entry points -------------------------------------
namespace moe {
// the cache-owned fields of one layer's policy step (false: the policy is off)
bool cache_policy_args(const expcache* c, int layer, PolicyArgs* a) {
  if (c->spares < 0) return false;
  memset(a, 0, sizeof(*a));
  a->L = c->L; a->E = c->E; a->layer = layer;
  a->slot_lo = c->slot_lo[layer]; a->slot_hi = c->slot_hi[layer]; a->spares = c->spares;
  a->table_row = c->table + (size_t)layer * c->E;
  a->cnt = c->cnt; a->last = c->last; a->stamp = c->stamp; a->freeslot = c->freeslot;
  return true;
}
}  // namespace moe

MOE_API moe_status expcache_set_policy(expcache* c, int spares_per_layer) {
  if (!c || spares_per_layer < 0) return MOE_ERR_INVALID_ARG;
  if (!c->partitioned || c->E > kPolicyThreads) return MOE_ERR_UNSUPPORTED;
  for (int l = 0; l < c->L; ++l)
    if (c->slot_hi[l] - c->slot_lo[l] > kPolicyMaxRun) return MOE_ERR_UNSUPPORTED;
  const size_t le = (size_t)c->L * c->E;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (!c->cnt) {
    if (cudaMalloc((void**)&c->cnt, le * 4) != cudaSuccess ||
        cudaMalloc((void**)&c->last, le * 4) != cudaSuccess ||
        cudaMalloc((void**)&c->stamp, ((size_t)c->L + 1) * 4) != cudaSuccess ||
        cudaMalloc((void**)&c->freeslot, ((size_t)c->n_cache + 1) * 4) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_OOM;
    }
  }
  // free slots: those of each layer's run that its table row does not use
  int32_t* tab = (int32_t*)malloc(le * 4);
  int32_t* fr = (int32_t*)calloc((size_t)c->n_cache + 1, 4);
  if (!tab || !fr) {
    free(tab);
    free(fr);
    return MOE_ERR_OOM;
  }
  moe_status st = MOE_OK;
  if (cudaMemcpy(tab, c->table, le * 4, cudaMemcpyDeviceToHost) != cudaSuccess) st = MOE_ERR_CUDA;
  for (int l = 0; st == MOE_OK && l < c->L; ++l) {
    for (int s = c->slot_lo[l]; s < c->slot_hi[l]; ++s) fr[s] = 1;
    for (int e = 0; e < c->E; ++e) {
      const int s = tab[(size_t)l * c->E + e];
      if (s >= c->slot_lo[l] && s < c->slot_hi[l]) fr[s] = 0;
    }
  }
  if (st == MOE_OK &&
      (cudaMemset(c->cnt, 0, le * 4) != cudaSuccess || cudaMemset(c->last, 0, le * 4) != cudaSuccess ||
       cudaMemset(c->stamp, 0, ((size_t)c->L + 1) * 4) != cudaSuccess ||
       cudaMemcpy(c->freeslot, fr, ((size_t)c->n_cache + 1) * 4, cudaMemcpyHostToDevice) !=
           cudaSuccess))
    st = MOE_ERR_CUDA;
  free(tab);
  free(fr);
  if (st != MOE_OK) {
    cudaGetLastError();
    return st;
  }
  c->spares = spares_per_layer;
  return MOE_OK;
}

MOE_API moe_status expcache_policy_step(expcache* c, int layer, const int32_t* counts,
                                        int32_t* src_slot, const int32_t* n_act,
                                        const int32_t* miss_ids, const int32_t* n_miss,
                                        int32_t* miss_dst, void* meta, void* stream) {
  if (!c || !counts || !src_slot || !n_act || !miss_ids || !n_miss || !miss_dst || layer < 0 ||
      layer >= c->L)
    return MOE_ERR_INVALID_ARG;
  PolicyArgs a;
  if (!cache_policy_args(c, layer, &a)) return MOE_ERR_UNSUPPORTED;
  a.counts = counts; a.src_slot = src_slot; a.n_act = n_act; a.miss_ids = miss_ids;
  a.n_miss = n_miss; a.miss_dst = miss_dst; a.meta = (int4*)meta;
  if (launch_pdl(k_cache_policy, 1, kPolicyThreads, policy_smem_bytes(a.E, a.slot_hi - a.slot_lo),
                 (cudaStream_t)stream, a) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

MOE_API moe_status expcache_policy_state(const expcache* c, int* spares, const uint32_t** cnt,
                                         const uint32_t** last, const uint32_t** stamp,
                                         const int32_t** freeslot) {
  if (!c || !spares || !cnt || !last || !stamp || !freeslot) return MOE_ERR_INVALID_ARG;
  *spares = c->spares;
  *cnt = c->cnt;
  *last = c->last;
  *stamp = c->stamp;
  *freeslot = c->freeslot;
  return MOE_OK;
}

// ---- per-layer slot budgets ------------------------------------------------
// "Project Maya" page, section "VRAM: one partition per layer, sized by what
// the layer routes": a floor per layer, then each further slot to the layer
// whose next-most-routed expert serves the largest share of its lookups.
// Within a layer the shares of successive experts (by count, descending) never
// grow, so handing out slots one at a time in that way takes the candidates
// (layer l, rank r >= floor) in one global order - share descending, then
// layer ascending, then rank ascending - and keeps the first N of them.  Here
// each candidate finds its place in that order directly: in its own layer r -
// floor candidates precede it, and in every other layer a prefix of the ranks
// (found by binary search, since the shares there never grow).
namespace moe {

constexpr int kPlanThreads = 1024;

// c1 / s1 > c2 / s2 for counts c < 2^32 and sums s < 2^64, exactly (128-bit
// products); a layer without routes (s == 0) has share 0
__device__ __forceinline__ int share_cmp(uint32_t c1, uint64_t s1, uint32_t c2, uint64_t s2) {
  const uint64_t a = s1 ? c1 : 0, b = s2 ? c2 : 0;
  const uint64_t t1 = s1 ? s1 : 1, t2 = s2 ? s2 : 1;
  // compare a * t2 with b * t1
  const uint64_t hi1 = __umul64hi(a, t2), lo1 = a * t2;
  const uint64_t hi2 = __umul64hi(b, t1), lo2 = b * t1;
  if (hi1 != hi2) return hi1 > hi2 ? 1 : -1;
  if (lo1 != lo2) return lo1 > lo2 ? 1 : -1;
  return 0;
}

__global__ void __launch_bounds__(kPlanThreads) k_plan_slots(
    const uint32_t* __restrict__ counts, int L, int E, int floor, int n_extra,
    int32_t* __restrict__ layer_slots, int32_t* __restrict__ order) {
  extern __shared__ unsigned long long s_sum[];  // [L] route sums, then [L] slot counts
  int* s_n = reinterpret_cast<int*>(s_sum + L);
  for (int l = threadIdx.x; l < L; l += blockDim.x) {
    s_sum[l] = 0ull;
    s_n[l] = floor;
  }
  __syncthreads();
  // 1. per layer: rank of every expert (count descending, id ascending) and the sums
  for (int i = threadIdx.x; i < L * E; i += blockDim.x) {
    const int l = i / E, e = i % E;
    const uint32_t* c = counts + (size_t)l * E;
    const uint32_t v = c[e];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const uint32_t u = c[f];
      rank += (u > v) || (u == v && f < e);
    }
    order[(size_t)l * E + rank] = e;
    atomicAdd(&s_sum[l], (unsigned long long)v);
  }
  __syncthreads();
  // 2. every candidate (l, r >= floor): its position in the global order
  const int per = E - floor;
  for (int i = threadIdx.x; i < L * per; i += blockDim.x) {
    const int l = i / per, r = floor + i % per;
    const uint32_t cv = counts[(size_t)l * E + order[(size_t)l * E + r]];
    const uint64_t sv = s_sum[l];
    long long pos = r - floor;
    for (int m = 0; m < L; ++m) {
      if (m == l) continue;
      // ranks of layer m that come first: share greater, or equal and m < l
      const uint64_t sm = s_sum[m];
      int lo = floor, hi = E;  // first rank of m that does not come first
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int c = share_cmp(counts[(size_t)m * E + order[(size_t)m * E + mid]], sm, cv, sv);
        if (c > 0 || (c == 0 && m < l)) lo = mid + 1;
        else hi = mid;
      }
      pos += lo - floor;
    }
    if (pos < n_extra) atomicAdd(&s_n[l], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    layer_slots[0] = 0;
    for (int l = 0; l < L; ++l) {
      acc += s_n[l];
      layer_slots[l + 1] = acc;
    }
  }
}

}  // namespace moe

MOE_API moe_status expcache_plan_slots(const uint32_t* d_counts, int L, int E, int total_slots,
                                       int floor, int32_t* d_layer_slots, int32_t* d_order,
                                       void* stream) {
  if (!d_counts || !d_layer_slots || !d_order || L <= 0 || E <= 0 || floor < 0 || total_slots < 0)
    return MOE_ERR_INVALID_ARG;
  if (floor > E || (long long)total_slots < (long long)L * floor) return MOE_ERR_INVALID_ARG;
  if (L > 4096 || E > 1024) return MOE_ERR_UNSUPPORTED;
  long long all = (long long)L * E;
  const int n_extra = (int)((total_slots < all ? total_slots : all) - (long long)L * floor);
  const size_t smem = (size_t)L * (sizeof(unsigned long long) + sizeof(int));
  moe::k_plan_slots<<<1, moe::kPlanThreads, smem, (cudaStream_t)stream>>>(
      d_counts, L, E, floor, n_extra, d_layer_slots, d_order);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
