// api.cu - C-ABI entry points that tie the kernels together: status strings,
// moe_expert_ffn dispatch and the moe_layer (route -> permute -> lookup ->
// gather/FFN per expert group -> combine on one stream).
#include <stdlib.h>
#include <string.h>

#include "permute_body.cuh"
#include "policy_body.cuh"

namespace moe {
const uint8_t* cache_arena(const expcache* c);
int cache_n_cache(const expcache* c);
int cache_n_stage(const expcache* c);
int cache_E(const expcache* c);
int cache_L(const expcache* c);
int cache_H(const expcache* c);
int cache_I(const expcache* c);
size_t decode_workspace_bytes(int T, int I, int k, int Is);
moe_status decode_ffn(const moe_ffn_args* a, cudaStream_t s, const DecodeFuse& fz);
moe_status decode_setup();
size_t prefill_workspace_bytes(int T, int H, int I, int E, int k, int Is);
const float* prefill_h_rows(const void* workspace, int T, int H, int I, int E, int k, int Is);
moe_status prefill_ffn(const moe_ffn_args* a, cudaStream_t s, int part, void (*mark)(void*),
                       void* mark_ctx, bool zero_y, uint16_t* y);
moe_status prefill_setup();
moe_status nvfp4_quantize(const void* x, int dtype, int T, int K, uint8_t* codes,
                          uint8_t* scales, float* G, cudaStream_t s);
moe_status permute_setup();
moe_status noalloc_setup();
moe_status launch_permute(const int32_t* ids, int T, int k, int E, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* pad_offsets,
                          int pad_align, int32_t* status, const LookupArgs& lk, cudaStream_t s);
void cache_lookup_args(const expcache* c, int layer, int32_t* src_slot, int32_t* act_list,
                       int32_t* n_act, int32_t* miss_ids, int32_t* n_miss, LookupArgs* out);
moe_status route_permute_small(const moe_route_args* a, const PermArgs& pa,
                               const SharedGuArgs& sg, const PolicyArgs* pol,
                               const SkipArgs* sk, cudaStream_t s);
moe_status launch_route_skip(const SkipArgs& sk, const int32_t* ids, const float* w, int T, int k,
                             int E, cudaStream_t s);
bool cache_policy_args(const expcache* c, int layer, PolicyArgs* a);
size_t route_split_bytes(int E, int H);
}  // namespace moe

using namespace moe;

// the layer's control area: the few-token router's counter, then one counter
// per 128-row tile for the combine in the decode down kernel (H <= 16384),
// then the one-launch decode FFN's control words (4 + one per act position)
// moe_route's tensor-core logits serve more than this many tokens
constexpr int kRouteTcMinT = 1024;
constexpr size_t kRouteCtlBytes = 256, kTileCtlBytes = 128 * 4,
                 kFfnCtlBytes = (4 + 2 * 1024) * 4;  // + h-ready and landed counts

MOE_API const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    default: return "MOE_ERR_UNKNOWN";
  }
}

MOE_API int moe_abi_version(void) { return 6; }

namespace moe {
moe_status ensure_setup() {
  static int done = 0;
  if (done) return MOE_OK;
  moe_status s = decode_setup();
  if (s != MOE_OK) return s;
  s = permute_setup();
  if (s != MOE_OK) return s;
  s = prefill_setup();
  if (s != MOE_OK) return s;
  s = noalloc_setup();
  if (s != MOE_OK) return s;
  done = 1;
  return MOE_OK;
}
}  // namespace moe

MOE_API size_t moe_ffn_workspace_bytes(int mode, int T, int H, int I, int E, int k, int Is) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || Is < 0) return 0;
  if (mode == MOE_MODE_PREFILL) return prefill_workspace_bytes(T, H, I, E, k, Is);
  return decode_workspace_bytes(T, I, k, Is);
}

// fz: what the layer's own sequence allows beyond the public call (DecodeFuse);
// part: the prefill split of group 0 (prefill_ffn)
static moe_status expert_ffn(const moe_ffn_args* a, void* stream, const DecodeFuse& fz,
                             int part = 0) {
  if (!a || !a->cache || !a->gscale || !a->src_slot || !a->act_list || !a->n_act || !a->offsets ||
      !a->perm || !a->w || !a->x)
    return MOE_ERR_INVALID_ARG;
  if (a->T < 0 || a->k <= 0 || a->k > a->E || a->group < 0 || a->n_stage < 0 || a->Is < 0)
    return MOE_ERR_INVALID_ARG;
  if (a->H != cache_H(a->cache) || a->I != cache_I(a->cache) || a->E != cache_E(a->cache))
    return MOE_ERR_INVALID_ARG;
  if (a->H % 256 || a->I % 128 || a->Is % 128 || a->H > 16384 || a->I > 16384 || a->Is > 16384)
    return MOE_ERR_UNSUPPORTED;
  if (a->Is > 0 && (!a->s_gate || !a->s_up || !a->s_down || !a->o_shared))
    return MOE_ERR_INVALID_ARG;
  if (a->T == 0) return MOE_OK;
  if (!a->workspace ||
      a->workspace_bytes < moe_ffn_workspace_bytes(a->mode, a->T, a->H, a->I, a->E, a->k, a->Is))
    return MOE_ERR_INVALID_ARG;
  moe_status st = ensure_setup();
  if (st != MOE_OK) return st;
  if (a->mode == MOE_MODE_DECODE) {
    if (!a->o_route || a->stages < 1 || a->stages > 3) return MOE_ERR_INVALID_ARG;
    return decode_ffn(a, (cudaStream_t)stream, fz);
  }
  if (a->mode == MOE_MODE_PREFILL) {
    if (!a->y_acc || !a->pad_offsets) return MOE_ERR_INVALID_ARG;
    return prefill_ffn(a, (cudaStream_t)stream, part, fz.mark, fz.mark_ctx, fz.pf_zero_y, fz.pf_y);
  }
  return MOE_ERR_INVALID_ARG;
}

MOE_API moe_status moe_expert_ffn(const moe_ffn_args* a, void* stream) {
  const DecodeFuse none = {nullptr, nullptr, nullptr, false, false, nullptr, nullptr,
                           nullptr, nullptr, nullptr, 0,       nullptr, nullptr, nullptr,
                           false,   nullptr, nullptr};
  return expert_ffn(a, stream, none);
}

// ------------------------------------------------------------------- layer
struct moe_layer {
  moe_layer_desc d;
  void* ws;
  size_t ws_bytes;
  float* logits;
  int32_t *ids, *counts, *offsets, *pad_offsets, *perm, *inv;
  float *w, *p_sel;
  int32_t *src_slot, *act_list, *n_act, *miss_ids, *n_miss, *status;
  float *o_route, *o_shared, *y_acc;
  void* route_ctl;
  int4* act_meta;  // compact per-expert records of the small-route path
  int32_t* miss_dst;  // adaptive cache: the slot each miss is gathered into
  int32_t* ids_eff;   // renorm-skip: the kept routes' experts (-1: dropped)
  float* w_eff;       // renorm-skip: the kept routes' renormalised weights
  void* w_split;      // the router weights' bf16 pieces (tensor-core router), or null
  size_t w_split_bytes;
  uint16_t* x_dev;    // the tokens, when the caller passes them in pinned host memory
  void* ffn_ws;
  size_t ffn_ws_bytes;
  int last_T;
  // timing hook: events recorded at the forward's launch boundaries
  cudaEvent_t ev[32];
  int n_ev, ev_i;
  cudaStream_t ev_stream;
  // prefill over a partly cached layer: the misses are gathered on a second
  // stream into the two halves of the staging slots while the first stream
  // runs the GEMMs of the hits and of the misses already landed
  cudaStream_t side;
  cudaEvent_t ev_lookup, ev_gathered[2], ev_used[2];
};

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

MOE_API moe_status moe_layer_create(const moe_layer_desc* d, moe_layer** out) {
  if (!d || !out || !d->cache || !d->w_router || !d->gscale) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (d->T_max <= 0 || d->k <= 0 || d->k > d->E || d->k > 32 || d->Is < 0 || d->layer < 0 ||
      d->layer >= cache_L(d->cache) || d->prefill_min_tokens < 0)
    return MOE_ERR_INVALID_ARG;
  if (d->H != cache_H(d->cache) || d->I != cache_I(d->cache) || d->E != cache_E(d->cache))
    return MOE_ERR_INVALID_ARG;
  if (d->Is > 0 && (!d->s_gate || !d->s_up || !d->s_down)) return MOE_ERR_INVALID_ARG;
  if (!(d->skip_tau >= 0.f) || d->skip_tau * (float)d->k >= 1.f) return MOE_ERR_INVALID_ARG;
  if (d->H % 256 || d->I % 128 || d->Is % 128 || d->E > 1024) return MOE_ERR_UNSUPPORTED;
  moe_status st = ensure_setup();
  if (st != MOE_OK) return st;
  moe_layer* l = (moe_layer*)calloc(1, sizeof(moe_layer));
  if (!l) return MOE_ERR_OOM;
  l->d = *d;
  const int T = d->T_max, k = d->k, E = d->E, H = d->H;
  const bool prefill = d->prefill_min_tokens > 0 && T >= d->prefill_min_tokens;
  size_t ffn_dec = decode_workspace_bytes(T, d->I, k, d->Is);
  size_t ffn_pre = prefill ? prefill_workspace_bytes(T, H, d->I, E, k, d->Is) : 0;
  l->ffn_ws_bytes = ffn_dec > ffn_pre ? ffn_dec : ffn_pre;
  size_t sizes[] = {
      (size_t)T * E * 4,  /* logits */
      (size_t)T * k * 4,  /* ids */
      (size_t)T * k * 4,  /* w */
      (size_t)T * k * 4,  /* p_sel */
      (size_t)E * 4,      /* counts */
      (size_t)(E + 1) * 4, /* offsets */
      (size_t)(E + 1) * 4, /* pad_offsets */
      (size_t)T * k * 4,  /* perm */
      (size_t)T * k * 4,  /* inv */
      (size_t)E * 4,      /* src_slot */
      (size_t)E * 4,      /* act_list */
      8,                  /* n_act */
      (size_t)E * 4,      /* miss_ids */
      4,                  /* n_miss */
      4,                  /* status */
      (size_t)T * k * H * 4, /* o_route */
      (size_t)T * H * 4,  /* o_shared */
      (size_t)E * 32,     /* act_meta */
      prefill ? (size_t)T * H * 4 : 0, /* y_acc */
      l->ffn_ws_bytes,
      kRouteCtlBytes + kTileCtlBytes + kFfnCtlBytes, /* route_ctl, tile counters, FFN */
      (size_t)E * 4,      /* miss_dst */
      (size_t)T * k * 4,  /* ids_eff */
      (size_t)T * k * 4,  /* w_eff */
      T > kRouteTcMinT ? route_split_bytes(E, H) : 0, /* router weight pieces */
      (size_t)T * H * 2   /* x copied in from pinned host memory */};
  const int n = (int)(sizeof(sizes) / sizeof(sizes[0]));
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += align256(sizes[i]);
  if (cudaMalloc(&l->ws, total) != cudaSuccess) {
    cudaGetLastError();
    free(l);
    return MOE_ERR_OOM;
  }
  l->ws_bytes = total;
  uint8_t* p = (uint8_t*)l->ws;
  void* ptrs[26];
  for (int i = 0; i < n; ++i) {
    ptrs[i] = sizes[i] ? p : nullptr;
    p += align256(sizes[i]);
  }
  l->logits = (float*)ptrs[0];
  l->ids = (int32_t*)ptrs[1];
  l->w = (float*)ptrs[2];
  l->p_sel = (float*)ptrs[3];
  l->counts = (int32_t*)ptrs[4];
  l->offsets = (int32_t*)ptrs[5];
  l->pad_offsets = (int32_t*)ptrs[6];
  l->perm = (int32_t*)ptrs[7];
  l->inv = (int32_t*)ptrs[8];
  l->src_slot = (int32_t*)ptrs[9];
  l->act_list = (int32_t*)ptrs[10];
  l->n_act = (int32_t*)ptrs[11];
  l->miss_ids = (int32_t*)ptrs[12];
  l->n_miss = (int32_t*)ptrs[13];
  l->status = (int32_t*)ptrs[14];
  l->o_route = (float*)ptrs[15];
  l->o_shared = (float*)ptrs[16];
  l->act_meta = (int4*)ptrs[17];
  l->y_acc = (float*)ptrs[18];
  l->ffn_ws = ptrs[19];
  l->route_ctl = ptrs[20];
  l->miss_dst = (int32_t*)ptrs[21];
  l->ids_eff = (int32_t*)ptrs[22];
  l->w_eff = (float*)ptrs[23];
  l->w_split = ptrs[24];
  l->w_split_bytes = sizes[24];
  l->x_dev = (uint16_t*)ptrs[25];
  bool ok = cudaMemset(l->ws, 0, total) == cudaSuccess &&
            cudaStreamCreateWithFlags(&l->side, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&l->ev_lookup, cudaEventDisableTiming) == cudaSuccess;
  for (int h = 0; h < 2 && ok; ++h)
    ok = cudaEventCreateWithFlags(&l->ev_gathered[h], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&l->ev_used[h], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    moe_layer_destroy(l);
    return MOE_ERR_CUDA;
  }
  *out = l;
  return MOE_OK;
}

MOE_API moe_status moe_layer_destroy(moe_layer* l) {
  if (!l) return MOE_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  cudaFree(l->ws);
  if (l->side) cudaStreamDestroy(l->side);
  if (l->ev_lookup) cudaEventDestroy(l->ev_lookup);
  for (int h = 0; h < 2; ++h) {
    if (l->ev_gathered[h]) cudaEventDestroy(l->ev_gathered[h]);
    if (l->ev_used[h]) cudaEventDestroy(l->ev_used[h]);
  }
  free(l);
  return MOE_OK;
}

// the timing hook: record the next event, if any, on the forward's stream
static void layer_mark(moe_layer* l) {
  if (l->ev_i < l->n_ev) cudaEventRecord(l->ev[l->ev_i++], l->ev_stream);
}
static void layer_mark_cb(void* ctx) { layer_mark((moe_layer*)ctx); }

// The prefill FFN over a partly cached layer with a staging ring of S >= 2
// slots (hot-cache page, "Prefill in groups of 64 experts": the experts walk
// through a staging buffer).  The misses go in groups of S/2, alternating
// between the two halves of the ring (the lookup gives miss i the staging
// slot i mod S).  The second stream gathers group g + 2 into a half once the
// GEMMs of group g are done with it; the first stream runs the GEMMs of each
// group once its records have landed, and the hits' GEMMs (and the shared
// expert) while the first group lands.  Every wait is an event, none a spin.
static moe_status prefill_streamed(moe_layer* l, moe_ffn_args* fa, cudaStream_t s, bool policy) {
  const moe_layer_desc& d = l->d;
  const int S = cache_n_stage(d.cache), S2 = S / 2;
  const int max_miss = fa->T * d.k < d.E ? fa->T * d.k : d.E;
  const int groups = (max_miss + S2 - 1) / S2;
  const int32_t* dst = policy ? l->miss_dst : nullptr;
  // the token quantisation (first call) clears y_acc; the shared expert runs
  // with the hits, before the misses' GEMMs, so a separate combine writes y
  const DecodeFuse marks = {layer_mark_cb, l, nullptr, false, false, nullptr, nullptr,
                            nullptr, nullptr, nullptr, 0,       nullptr, nullptr, nullptr,
                            true,          nullptr, nullptr};
  moe_status st;
  auto gather = [&](int g) -> moe_status {
    const int h = g & 1, cnt = S2 < max_miss - g * S2 ? S2 : max_miss - g * S2;
    if (g >= 2 && cudaStreamWaitEvent(l->side, l->ev_used[h], 0) != cudaSuccess) return MOE_ERR_CUDA;
    moe_status r = expcache_fill(d.cache, d.layer, l->miss_ids, l->n_miss, g * S2, cnt, dst,
                                 l->status, l->side);
    if (r != MOE_OK) return r;
    return cudaEventRecord(l->ev_gathered[h], l->side) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  };
  if (cudaEventRecord(l->ev_lookup, s) != cudaSuccess ||
      cudaStreamWaitEvent(l->side, l->ev_lookup, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int g = 0; g < 2 && g < groups; ++g)
    if ((st = gather(g)) != MOE_OK) return st;
  fa->n_stage = S2;  // misses per FFN group
  fa->group = 0;
  if ((st = expert_ffn(fa, s, marks, 1)) != MOE_OK) return st;  // quantisation, hits, shared
  for (int g = 0; g < groups; ++g) {
    const int h = g & 1;
    if (cudaStreamWaitEvent(s, l->ev_gathered[h], 0) != cudaSuccess) return MOE_ERR_CUDA;
    fa->group = g;
    if ((st = expert_ffn(fa, s, marks, g == 0 ? 2 : 0)) != MOE_OK) return st;
    if (g + 2 < groups) {
      if (cudaEventRecord(l->ev_used[h], s) != cudaSuccess) return MOE_ERR_CUDA;
      if ((st = gather(g + 2)) != MOE_OK) return st;
    }
  }
  return MOE_OK;
}

// `bytes` of tokens from pinned host memory into device memory: one kernel of
// 16-byte loads (the copy engine's setup costs more than this for a token or
// a few), or the copy engine when an address is not 16-byte aligned
__global__ void __launch_bounds__(256) k_copy_rows(const uint4* __restrict__ src,
                                                   uint4* __restrict__ dst, size_t n) {
  pdl_wait();  // the previous forward's kernels may still read dst
  for (size_t i = blockIdx.x * (size_t)256 + threadIdx.x; i < n; i += (size_t)gridDim.x * 256)
    dst[i] = src[i];
  pdl_launch_dependents();
}
static moe_status copy_rows_in(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  if (((uintptr_t)src & 15) || ((uintptr_t)dst & 15) || (bytes & 15))
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
  const size_t n = bytes / 16;
  const size_t blocks = (n + 255) / 256;
  const int grid = (int)(blocks < (size_t)kSMs * 4 ? blocks : (size_t)kSMs * 4);
  return launch_pdl(k_copy_rows, grid, 256, 0, s, (const uint4*)src, (uint4*)dst, n) ==
                 cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// y = bf16(y_acc): the prefill path's combine (its down GEMMs added into y_acc),
// unless the shared expert's down GEMM already wrote y (y_written)
static moe_status finish_prefill(moe_layer* l, int T, void* y, void* stream,
                                 bool y_written = false) {
  l->last_T = T;
  if (y_written) return MOE_OK;
  moe_combine_args ca;
  memset(&ca, 0, sizeof(ca));
  ca.T = T; ca.H = l->d.H; ca.k = l->d.k;
  ca.y_acc = l->y_acc;
  ca.inv = l->inv;
  ca.y = y;
  moe_status st = moe_combine(&ca, stream);
  if (st != MOE_OK) return st;
  layer_mark(l);
  return MOE_OK;
}

MOE_API moe_status moe_layer_forward(moe_layer* l, const void* x_in, int T, void* y,
                                     void* stream) {
  if (!l || !x_in || !y || T < 0 || T > l->d.T_max) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const moe_layer_desc& d = l->d;
  cudaStream_t s = (cudaStream_t)stream;
  const bool prefill = d.prefill_min_tokens > 0 && T >= d.prefill_min_tokens;
  moe_status st;
  l->ev_i = 0;
  l->ev_stream = s;
  layer_mark(l);
  // tokens in pinned host memory: copied once into the layer's buffer by the
  // forward's first kernel (the later kernels read them many times)
  const void* x = x_in;
  cudaPointerAttributes pat;
  if (cudaPointerGetAttributes(&pat, x_in) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_INVALID_ARG;
  }
  if (pat.type == cudaMemoryTypeUnregistered) return MOE_ERR_INVALID_ARG;
  // y is written by a kernel: device memory, managed memory or pinned host
  // memory (pageable host memory would fault the kernel that stores it)
  cudaPointerAttributes yat;
  if (cudaPointerGetAttributes(&yat, y) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_INVALID_ARG;
  }
  if (yat.type == cudaMemoryTypeUnregistered) return MOE_ERR_INVALID_ARG;
  if (pat.type == cudaMemoryTypeHost) {
    if ((st = copy_rows_in(x_in, l->x_dev, (size_t)T * d.H * 2, s)) != MOE_OK) return st;
    x = l->x_dev;
  }

  moe_route_args ra;
  memset(&ra, 0, sizeof(ra));
  ra.x = x; ra.w_router = d.w_router; ra.bias = d.bias;
  ra.T = T; ra.H = d.H; ra.E = d.E; ra.k = d.k;
  ra.ids = l->ids; ra.w = l->w; ra.p_sel = l->p_sel; ra.logits = l->logits;
  ra.workspace = l->route_ctl; ra.workspace_bytes = 256;
  ra.status = l->status;
  ra.w_split = l->w_split; ra.w_split_bytes = l->w_split_bytes;
  LookupArgs lk;
  cache_lookup_args(d.cache, d.layer, l->src_slot, l->act_list, l->n_act, l->miss_ids, l->n_miss,
                    &lk);
  // up to 8 tokens: router, permutation and slot lookup in one launch;
  // otherwise the router, then the permutation with the lookup as its tail
  PermArgs pa;
  pa.counts = l->counts; pa.offsets = l->offsets; pa.perm = l->perm; pa.inv = l->inv;
  pa.pad_offsets = prefill ? l->pad_offsets : nullptr; pa.pad_align = 128;
  pa.status = l->status; pa.lk = lk;
  // few routes and no padding: the fused kernel's permutation also writes the
  // compact per-expert records that the decode FFN reads
  const bool small_routes = T * d.k <= 32 && !prefill;
  if (small_routes) {
    pa.lk.meta = l->act_meta;
    pa.lk.gscale = d.gscale;
  }
  // one decode token: the shared expert's gate/up runs beside the router,
  // into the FFN workspace's h_shared (after the routes' h)
  SharedGuArgs sg = {nullptr, nullptr, 0, nullptr};
  if (!prefill && T == 1 && d.Is > 0) {
    sg.s_gate = (const uint16_t*)d.s_gate;
    sg.s_up = (const uint16_t*)d.s_up;
    sg.Is = d.Is;
    sg.h_shared = (float*)l->ffn_ws + (size_t)T * d.k * d.I;
  }
  // adaptive cache: its step (promotions, counts, the boundary's evictions)
  // runs in the same kernel, on the lookup's results, when that kernel is used
  PolicyArgs pol;
  const bool policy = cache_policy_args(d.cache, d.layer, &pol);
  if (policy) {
    pol.counts = l->counts; pol.src_slot = l->src_slot; pol.n_act = l->n_act;
    pol.miss_ids = l->miss_ids; pol.n_miss = l->n_miss; pol.miss_dst = l->miss_dst;
    pol.meta = small_routes ? l->act_meta : nullptr;
  }
  // renorm-skip: low-weight misses dropped before the permutation
  const bool skip = d.skip_tau > 0.f;
  SkipArgs sk = {lk.table, lk.slot_lo, lk.slot_hi, d.skip_tau, l->ids_eff, l->w_eff};
  st = route_permute_small(&ra, pa, sg, policy ? &pol : nullptr, skip ? &sk : nullptr, s);
  const bool policy_done = policy && st == MOE_OK;
  const bool shared_gu_done = st == MOE_OK && sg.Is > 0;
  const int4* act_meta = (st == MOE_OK && small_routes) ? l->act_meta : nullptr;
  if (st == MOE_ERR_UNSUPPORTED) {
    if ((st = moe_route(&ra, stream)) != MOE_OK) return st;
    layer_mark(l);
    if (skip && (st = launch_route_skip(sk, l->ids, l->w, T, d.k, d.E, s)) != MOE_OK) return st;
    st = launch_permute(skip ? l->ids_eff : l->ids, T, d.k, d.E, l->counts, l->offsets, l->perm,
                        l->inv, pa.pad_offsets, 128, l->status, lk, s);
  }
  if (st != MOE_OK) return st;
  layer_mark(l);
  // otherwise the adaptive cache's step as a kernel of its own, before the
  // misses are gathered (into their promoted or staging slots)
  if (policy && !policy_done) {
    if ((st = expcache_policy_step(d.cache, d.layer, l->counts, l->src_slot, l->n_act, l->miss_ids,
                                   l->n_miss, l->miss_dst, (void*)act_meta, stream)) != MOE_OK)
      return st;
    layer_mark(l);
  }

  const int n_stage = cache_n_stage(d.cache);
  const int max_miss = T * d.k < d.E ? T * d.k : d.E;
  const int S = n_stage > 0 ? n_stage : 1;
  const int groups = n_stage > 0 ? (max_miss + S - 1) / S : 1;

  moe_ffn_args fa;
  memset(&fa, 0, sizeof(fa));
  fa.mode = prefill ? MOE_MODE_PREFILL : MOE_MODE_DECODE;
  fa.stages = MOE_STAGE_ALL;
  fa.T = T; fa.H = d.H; fa.I = d.I; fa.E = d.E; fa.k = d.k;
  fa.x = x; fa.cache = d.cache; fa.gscale = d.gscale;
  fa.src_slot = l->src_slot; fa.act_list = l->act_list; fa.n_act = l->n_act;
  fa.offsets = l->offsets; fa.pad_offsets = l->pad_offsets; fa.perm = l->perm; fa.inv = l->inv;
  fa.w = skip ? l->w_eff : l->w;
  fa.n_stage = n_stage;
  fa.prefill_group = d.prefill_group;
  fa.Is = d.Is; fa.s_gate = d.s_gate; fa.s_up = d.s_up; fa.s_down = d.s_down;
  fa.o_route = l->o_route; fa.o_shared = d.Is > 0 ? l->o_shared : nullptr;
  fa.y_acc = l->y_acc;
  fa.workspace = l->ffn_ws; fa.workspace_bytes = l->ffn_ws_bytes;
  fa.status = l->status;
  if (prefill && n_stage >= 2) {
    if ((st = prefill_streamed(l, &fa, s, policy)) != MOE_OK) return st;
    return finish_prefill(l, T, y, stream);
  }
  // decode with every miss in one staging group: the FFN kernel gathers the
  // misses itself, computing the hits while their records land
  const bool ffn_gathers = !prefill && groups == 1 && n_stage > 0;
  for (int g = 0; g < groups; ++g) {
    if (n_stage > 0 && !ffn_gathers) {
      int cnt = S < max_miss - g * S ? S : max_miss - g * S;
      if ((st = expcache_fill(d.cache, d.layer, l->miss_ids, l->n_miss, g * S, cnt,
                              policy ? l->miss_dst : nullptr, l->status, stream)) != MOE_OK)
        return st;
      layer_mark(l);
    }
    fa.group = g;
    // the kernel before this call is the permutation or the gather; a single
    // decode group's down kernel also writes y (no separate combine)
    // the one-launch FFN only where it also gathers the misses: with every
    // expert resident the gate/up and down kernels of their own are faster
    // (13.8k against 11.9k tokens/s on the decode layer, one box)
    DecodeFuse fz = {layer_mark_cb, l, act_meta, true, shared_gu_done && g == 0,
                     nullptr, nullptr, nullptr,
                     ffn_gathers ? (unsigned int*)((char*)l->route_ctl + kRouteCtlBytes +
                                                   kTileCtlBytes)
                                 : nullptr,
                     ffn_gathers ? d.cache : nullptr, d.layer, l->miss_ids, l->n_miss,
                     policy ? l->miss_dst : nullptr, false, nullptr, nullptr};
    if (!prefill && groups == 1) {
      fz.comb_ctl = (unsigned int*)((char*)l->route_ctl + kRouteCtlBytes);
      fz.inv = l->inv;
      fz.y = (uint16_t*)y;
      // the one-launch FFN's per-position counts, unused by the two launches
      if (!ffn_gathers)
        fz.h_counts = (unsigned int*)((char*)l->route_ctl + kRouteCtlBytes + kTileCtlBytes) + 4;
    }
    // prefill: the token quantisation clears y_acc; with one FFN call its
    // shared-expert down GEMM is the last writer of y_acc and writes y
    fz.pf_zero_y = prefill;
    fz.pf_y = (prefill && groups == 1 && d.Is > 0) ? (uint16_t*)y : nullptr;
    if ((st = expert_ffn(&fa, stream, fz)) != MOE_OK) return st;
  }
  if (!prefill && groups == 1) {
    l->last_T = T;
    return MOE_OK;
  }

  if (prefill) return finish_prefill(l, T, y, stream, groups == 1 && d.Is > 0);
  moe_combine_args ca;
  memset(&ca, 0, sizeof(ca));
  ca.T = T; ca.H = d.H; ca.k = d.k;
  ca.y_acc = prefill ? l->y_acc : nullptr;
  ca.o_route = prefill ? nullptr : l->o_route;
  ca.inv = l->inv;
  ca.o_shared = (d.Is > 0 && !prefill) ? l->o_shared : nullptr;  // prefill adds it into y_acc
  ca.y = y;
  if ((st = moe_combine(&ca, stream)) != MOE_OK) return st;
  layer_mark(l);
  l->last_T = T;
  return MOE_OK;
}

MOE_API moe_status moe_layer_debug_ptrs(const moe_layer* l, const int32_t** ids, const float** w,
                                        const float** p_sel, const int32_t** perm,
                                        const int32_t** src_slot, const int32_t** n_act) {
  if (!l) return MOE_ERR_INVALID_ARG;
  if (ids) *ids = l->ids;
  if (w) *w = l->w;
  if (p_sel) *p_sel = l->p_sel;
  if (perm) *perm = l->perm;
  if (src_slot) *src_slot = l->src_slot;
  if (n_act) *n_act = l->n_act;
  return MOE_OK;
}

MOE_API moe_status moe_layer_debug_prefill(const moe_layer* l, const float** h_rows,
                                           const int32_t** offsets,
                                           const int32_t** pad_offsets) {
  if (!l || !h_rows || !offsets || !pad_offsets) return MOE_ERR_INVALID_ARG;
  const moe_layer_desc& d = l->d;
  if (!(d.prefill_min_tokens > 0 && l->last_T >= d.prefill_min_tokens)) return MOE_ERR_INVALID_ARG;
  *h_rows = prefill_h_rows(l->ffn_ws, l->last_T, d.H, d.I, d.E, d.k, d.Is);
  *offsets = l->offsets;
  *pad_offsets = l->pad_offsets;
  return MOE_OK;
}

MOE_API moe_status moe_layer_set_timing(moe_layer* l, void* const* events, int n) {
  if (!l || n < 0 || n > 32 || (n > 0 && !events)) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) l->ev[i] = (cudaEvent_t)events[i];
  l->n_ev = n;
  return MOE_OK;
}

MOE_API moe_status moe_read_device_status(moe_layer* l, void* stream, int32_t* status_out) {
  if (!l || !status_out) return MOE_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, l->status, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
          cudaSuccess ||
      cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  *status_out = v;
  if (cudaMemsetAsync(l->status, 0, 4, (cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

MOE_API moe_status moe_nvfp4_quantize(const void* x, int dtype, int T, int K, uint8_t* codes,
                                      uint8_t* scales, float* G, void* stream) {
  return nvfp4_quantize(x, dtype, T, K, codes, scales, G, (cudaStream_t)stream);
}
