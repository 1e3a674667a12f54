/*
 * moe.h - C ABI of the routed mixture-of-experts layer library (libmoe.so)
 * for one GB300 GPU (sm_103a).
 *
 * The layer (GLM-5.3-Flash style: 288 routed experts, top-8 per token, one
 * shared expert) runs in these steps, each a hand-written CUDA kernel:
 *   moe_route        router GEMV/GEMM + softmax + top-k + renormalisation
 *   moe_permute      token->expert histogram, scan and stable permutation
 *   expcache_lookup  per-layer HBM hot-expert cache: hit slot or staged miss
 *   expcache_fill    wide-read gather of records from pinned host memory
 *   moe_expert_ffn   NVFP4 gate/up -> SiLU*mul -> down per selected expert
 *   moe_combine      weighted sum of the experts' outputs (+ shared) -> bf16
 *   moe_layer_forward  all of the above in order on one stream.
 * Sources of the operations: "Project Maya" page, sections "What is in the
 * 96.5 GB" (an expert blob is gate+up+down; top-8 of 288; fp32 router) and
 * "Three tiers and the rules between them" (device router, device table
 * layer x expert -> VRAM slot, per-layer slot partitions, GPU pull of
 * RAM-tier experts from host-mapped memory with 16-byte loads); dev.to page
 * "A hot expert cache made a 181 GiB model faster", sections "The wall"
 * (NVFP4 experts, 8 of 288 per token), "A gather kernel that reads wide"
 * (wide-read gather driven by a GPU-resident expert list, no host sync, CUDA
 * graph replay), "Offload more, cache the hot experts" (per-layer cache of
 * the 66 most-used experts) and "Prefill in groups of 64 experts"; the
 * Strata-GLM blog "Day one" list (exclusive tiers, byte-sized slots, chunked
 * prefill as one batched matmul per expert).
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented "device" are device addresses; the
 *     caller owns every buffer it passes and every stream.  The library owns
 *     only its opaque handles (expcache, moe_layer) and what they allocate.
 *   - Every call is stream-ordered and asynchronous: it enqueues work on
 *     `stream` (a cudaStream_t, NULL = legacy default stream) and returns
 *     without synchronising, except where documented.
 *   - Argument errors are detected on the host and returned at once, before
 *     anything is enqueued.  Errors only visible on the device (an expert id
 *     out of range, a slot outside its layer's partition, a miss with no host
 *     record, a bounded wait that ran out) are written to a sticky device
 *     status word (int32, first error wins) when the caller passes one; no
 *     kernel traps.  The kernel that sees such an error skips the bad item.
 *   - Shapes: H % 256 == 0, I % 128 == 0, 1 <= k <= min(E, 32), E <= 1024.
 *
 * Expert record (the storage and transfer unit; fixed stride per (H, I) and
 * format), in one of two 4-bit formats:
 *   NVFP4 (MOE_FMT_NVFP4; dev.to page, "The wall"): E4M3 block scale per 16
 *     values (B = 16);
 *   MXFP4 (MOE_FMT_MXFP4; windlass README: GLM-5.2 in MXFP4): E8M0 block
 *     scale (2^(b-127), OCP Microscaling Formats v1.0) per 32 values (B = 32).
 *   [gate codes I x H/2][up codes I x H/2][down codes H x I/2]
 *   [gate scales I x H/B][up scales I x H/B][down scales H x I/B]
 *   Codes: E2M1 (sign bit 3; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6), two per
 *   byte, element 2j in the low nibble, rows contiguous (K-major).
 *   Scales: one byte per B consecutive elements of a row, stored in 512-byte
 *   atoms: for row r and block kb of a matrix with KB = K/B blocks per row,
 *   byte ((r/128)*(KB/4) + kb/4)*512 + (r%32)*16 + ((r%128)/32)*4 + kb%4.
 *   weight(r, c) = e2m1(code) * scale(r, c/B) * g[expert][matrix], g an
 *   fp32 per-(expert, matrix) global scale held outside the record (for
 *   MXFP4 g = 1 is the format as published).
 *   Size: 3*I*H/2 + 3*I*H/B bytes (H = 6144, I = 2048: 21,233,664 NVFP4,
 *   20,054,016 MXFP4).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int moe_status;
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* NULL where required, negative size, k > E, ...      */
  MOE_ERR_UNSUPPORTED = 2, /* shape or alignment outside what the kernels handle  */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, copy, ...)      */
  MOE_ERR_OOM = 4,         /* device allocation failed                            */
  MOE_ERR_TIMEOUT = 5,     /* a bounded device wait ran out (device status only)  */
  MOE_ERR_DEVICE = 6       /* bad id / slot / record seen on the device           */
};

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status s);

/* ABI version of this header (bumped on any incompatible change). */
int moe_abi_version(void);

/* Record formats. */
enum { MOE_FMT_NVFP4 = 0, MOE_FMT_MXFP4 = 1 };

/* Bytes of one expert record for hidden size H, expert intermediate I and
 * format (0 for an unknown format). */
uint64_t moe_record_bytes(int H, int I, int format);

/* ------------------------------------------------------------------ route
 * Router of the "Project Maya" page (device-side router, fp32 router
 * weights): logits[t][e] = sum_h W_r[e][h] * x[t][h] + bias[e] (fp32); the
 * k largest logits in (logit desc, id asc) order give ids[t][0..k); p_sel is
 * the full-softmax probability of each selected expert; w is the softmax over
 * the selected logits only (renormalised top-k, sums to 1 per token).
 * moe_route_workspace_bytes(T, E) = 256 + T*E*4.
 */
typedef struct {
  const void* x;        /* device [T][H] bf16, row-major                        */
  const float* w_router;/* device [E][H] fp32                                   */
  const float* bias;    /* device [E] fp32, or NULL for none                     */
  int T, H, E, k;
  int32_t* ids;         /* device out [T][k]                                     */
  float* w;             /* device out [T][k] renormalised weights                */
  float* p_sel;         /* device out [T][k] full-softmax probabilities, or NULL */
  float* logits;        /* device [T][E] fp32: output if non-NULL; else the call
                           needs workspace of moe_route_workspace_bytes(T, E)   */
  void* workspace;      /* device scratch, may be NULL when logits != NULL: its
                           first 256 bytes are a control area that must be zero
                           before the first call on it (every call leaves it
                           zero); the logits follow it when logits == NULL.
                           With T <= 8 and a workspace the router runs as one
                           kernel (per-expert logits, then softmax/top-k in the
                           CTA that finishes last); calls that share a
                           workspace must not overlap on the GPU.           */
  size_t workspace_bytes;
  int32_t* status;      /* device sticky status word, or NULL                    */
  void* w_split;        /* device scratch of moe_route_split_bytes(E, H) bytes,
                           16-byte aligned, or NULL.  With T > 1024, H a
                           multiple of 64 and x and w_router 16-byte aligned,
                           the call rewrites it with w_router as three bf16
                           pieces (W = W1 + W2 + W3 exactly, rows padded to a
                           multiple of 32 with zeros) and computes the logits
                           on the tensor cores from them: every product exact,
                           each 64-deep partial sum read out and added in fp32
                           with compensation.  Otherwise (or NULL) the logits
                           run on the CUDA cores in fp32.  Calls that share it
                           must not overlap on the GPU.                      */
  size_t w_split_bytes;
} moe_route_args;

size_t moe_route_workspace_bytes(int T, int E);
/* 3 * ceil(E/32)*32 * H * 2: the bf16 pieces of the router weights (w_split). */
size_t moe_route_split_bytes(int E, int H);
moe_status moe_route(const moe_route_args* a, void* stream);

/* ---------------------------------------------------------------- permute
 * Groups the T*k routes r = t*k + j by expert (the batched-matmul-per-expert
 * grouping of the Strata-GLM blog's chunked prefill): counts[e] = routes to
 * e; offsets = exclusive scan of counts (E+1 entries); perm[p] = r for the
 * p-th route in (expert asc, r asc) order - a stable sort, so the result is
 * unique; inv[r] = p.  pad_offsets (optional) is the exclusive scan of the
 * counts rounded up to multiples of pad_align (the prefill staging layout).
 * Out-of-range ids set MOE_ERR_DEVICE in *status and are dropped; an id of
 * -1 is a dropped route (the renorm-skip) and is left out without an error.
 * A route left out is not counted and gets inv[r] = -1.
 * One thread block per 1024 routes (each block histograms all routes, so
 * the blocks never wait on one another); T*k <= 1<<20.
 */
moe_status moe_permute(const int32_t* ids, int T, int k, int E, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* pad_offsets,
                       int pad_align, int32_t* status, void* stream);

/* ---------------------------------------------------------- expert cache
 * Per-layer HBM hot-expert cache ("Project Maya": a device table layer x
 * expert -> VRAM slot, each layer owning its own run of slots; dev.to: a
 * per-layer cache of the most-used experts, misses pulled from host RAM by
 * a wide-read gather driven by a device-resident list).  Device memory holds
 * n_cache_slots cache slots followed by n_stage staging slots, one record
 * each; slot s is at expcache_slot_ptr(c, s).  Records that are not resident
 * live in a pinned host arena owned by the caller (allocated with
 * cudaHostAlloc(..., cudaHostAllocMapped) or registered with
 * cudaHostRegister(..., cudaHostRegisterMapped)); the cache maps it with
 * cudaHostGetDevicePointer and never frees it; it must stay valid and
 * unchanged while the cache exists.
 */
typedef struct expcache expcache;

typedef struct {
  int L, E;                     /* layers, experts per layer                        */
  int H, I;                     /* dims (record size = moe_record_bytes(H, I))      */
  int n_cache_slots;            /* HBM cache slots, all layers                      */
  const int32_t* layer_slots;   /* host [L+1]: layer l owns slots
                                   [layer_slots[l], layer_slots[l+1]); NULL = every
                                   layer may use every cache slot                   */
  int n_stage;                  /* HBM staging slots for misses (>= 0)              */
  const void* host_arena;       /* pinned host records, or NULL if none             */
  uint64_t host_arena_records;  /* records in the host arena                        */
  const int64_t* host_index;    /* host [L][E]: record index in the host arena of
                                   (layer, expert), -1 = not there; NULL = none     */
  int format;                   /* MOE_FMT_NVFP4 or MOE_FMT_MXFP4: every record of
                                   the cache (the layers' FFN kernels follow it)    */
} expcache_desc;

/* Allocates the slot arenas and the device slot table (all entries -1 = not
 * resident) and maps the host arena.  Synchronous.  MOE_ERR_OOM if the
 * arenas do not fit. */
moe_status expcache_create(const expcache_desc* d, expcache** out);
/* Frees what create allocated (the host arena is the caller's).  Synchronous. */
moe_status expcache_destroy(expcache* c);
/* Device address of slot s (cache slots first, then staging), NULL if out of range. */
void* expcache_slot_ptr(const expcache* c, int s);
/* Device [L][E] int32 slot table (-1 = not resident). */
const int32_t* expcache_slot_table(const expcache* c);
/* Marks (layer, expert) resident in cache slot `slot` (the caller has written
 * the record there, e.g. with cudaMemcpyAsync on the same stream), or not
 * resident when slot == -1.  Stream-ordered table write.  MOE_ERR_UNSUPPORTED
 * once the adaptive policy is on (it owns the table). */
moe_status expcache_set_resident(expcache* c, int layer, int expert, int slot, void* stream);

/* Wide-read gather: for list entries i in [first, first + max_count) with
 * i < *d_n, copies the host record of (layer, d_expert_ids[i]) into slot
 * d_dst_slots[i] - a cache slot of the layer (which it marks resident, unless
 * the adaptive policy is on: that owns the table) or a staging slot (no table
 * change) - or, when d_dst_slots is NULL, into staging
 * slot n_cache_slots + (i mod n_stage).  Any other destination sets
 * MOE_ERR_DEVICE in *status.  The copy is done by
 * thread blocks reading the mapped host memory with 16-byte loads.  The list
 * and its length stay on the device (no host synchronisation), so the call
 * can be captured in a CUDA graph. */
moe_status expcache_fill(expcache* c, int layer, const int32_t* d_expert_ids, const int32_t* d_n,
                         int first, int max_count, const int32_t* d_dst_slots, int32_t* status,
                         void* stream);

/* Lookup for one layer: for every expert e with counts[e] > 0 (active),
 * src_slot[e] = its cache slot (a hit) or, for the i-th miss in ascending
 * expert id, the staging slot n_cache_slots + (i mod n_stage); -1 when not
 * active.  act_list lists the active experts, hits first (ascending id), then
 * misses (ascending id); n_act[0] = active count, n_act[1] = hit count.
 * miss_ids / n_miss list the misses (ascending id), ready for expcache_fill.
 * A miss with n_stage == 0, or a table slot outside the layer's partition,
 * sets MOE_ERR_DEVICE in *status. */
moe_status expcache_lookup(const expcache* c, int layer, const int32_t* counts, int32_t* src_slot,
                           int32_t* act_list, int32_t* n_act, int32_t* miss_ids, int32_t* n_miss,
                           int32_t* status, void* stream);

/* Adaptive cache ("Project Maya" page, sections "How 'most-used' is
 * measured" and "Promotion on every miss, eviction at the boundary").
 * expcache_set_policy turns it on for every layer: a decayed route count and
 * the number of its latest forward per (layer, expert), all zero, and as free
 * ("spare") slots those of each layer's run that its table row does not use.
 * Needs per-layer slot runs (layer_slots) and spares_per_layer >= 0, else
 * MOE_ERR_UNSUPPORTED / MOE_ERR_INVALID_ARG.  Synchronous; calling it again
 * resets the state from the current table.
 *
 * expcache_policy_step, for one forward of `layer`, after expcache_lookup on
 * the same stream (its counts, src_slot, n_act, miss_ids, n_miss are the
 * lookup's arrays):
 *   1. promotion: the misses, in ascending id, take the layer's free slots in
 *      ascending slot order and are resident from then on (table, src_slot
 *      and, when meta is given, the slot field of the compact expert records
 *      meta[2 a] = {expert, slot, first route, routes}, a = n_act[1] + i);
 *      miss_dst[i] (device, >= E entries) = the slot miss i is to be gathered
 *      into: its cache slot, or the staging slot the lookup gave it;
 *   2. counts: each route adds 1 to its expert's count, capped at 2^24, and
 *      sets its latest forward; every 32,768 route events (over all layers,
 *      checked once per step) every count of every layer is halved;
 *   3. boundary: while the layer has fewer than spares_per_layer free slots,
 *      its resident with the smallest (count, latest forward, id) is evicted
 *      (its slot is free; the record stays until a promotion overwrites it,
 *      which the stream orders after this forward's reads).
 * Then expcache_fill(..., d_dst_slots = miss_dst, ...) gathers the misses.
 * One CTA; MOE_ERR_UNSUPPORTED when the policy is off. */
moe_status expcache_set_policy(expcache* c, int spares_per_layer);
moe_status expcache_policy_step(expcache* c, int layer, const int32_t* counts, int32_t* src_slot,
                                const int32_t* n_act, const int32_t* miss_ids,
                                const int32_t* n_miss, int32_t* miss_dst, void* meta,
                                void* stream);
/* The policy's device state (read only; NULL before expcache_set_policy):
 * cnt and last [L][E] uint32, stamp [L + 1] uint32 (forwards per layer, then
 * the route events since the last halving), freeslot [n_cache_slots] int32
 * (1 = free); *spares = spares_per_layer, or -1 when the policy is off. */
moe_status expcache_policy_state(const expcache* c, int* spares, const uint32_t** cnt,
                                 const uint32_t** last, const uint32_t** stamp,
                                 const int32_t** freeslot);

/* Per-layer slot budgets ("Project Maya" page, section "VRAM: one partition
 * per layer, sized by what the layer routes"): splits total_slots cache slots
 * over L layers from route counts per (layer, expert) - for instance the
 * moe_permute counts of a calibration batch summed per layer, or the
 * adaptive policy's decayed counts.  Each layer's experts are ordered by
 * count, descending, ties to the lower id (d_order [L][E]); every layer gets
 * `floor` slots; each further slot goes to the layer whose next expert in
 * that order serves the largest share of that layer's lookups (count / the
 * layer's total; 0 for a layer without routes), ties to the lower layer; a
 * full layer (E slots) takes no more, and slots beyond L*E stay unassigned.
 * d_layer_slots [L+1] receives the partition's prefix sums, ready for
 * expcache_desc.layer_slots (copied to the host); layer l's residents are
 * d_order[l][0 .. layer_slots[l+1] - layer_slots[l]).
 *   d_counts device [L][E] uint32; outputs device.  floor > E or total_slots <
 *   L*floor: MOE_ERR_INVALID_ARG; L > 4096 or E > 1024: MOE_ERR_UNSUPPORTED.
 *   One thread block; stream-ordered. */
moe_status expcache_plan_slots(const uint32_t* d_counts, int L, int E, int total_slots, int floor,
                               int32_t* d_layer_slots, int32_t* d_order, void* stream);

/* ------------------------------------------------------------- expert FFN
 * For each route p (p-th route of the expert-sorted order) of the active
 * experts of group `group` (group 0 = all hits and misses [0, n_stage);
 * group g > 0 = misses [g*n_stage, (g+1)*n_stage)), with e its expert and t
 * its token: g = Wg x_t, u = Wu x_t, h = silu(g) * u, o = Wd h, all weights
 * read from the record in slot src_slot[e] (SiLU-gated FFN without biases).
 * DECODE mode: weights dequantised in registers; the activations (x, then h)
 *   are held in f16 and every product is an exact f16 x f16 product summed
 *   in fp32 (x is bf16: exact in f16 for magnitudes in [2^-14, 65504];
 *   smaller ones are rounded to f16's subnormal grid, an absolute error of at
 *   most 2^-25; h is fp32 rounded to f16, relative error 2^-11).  A value
 *   of x or h beyond 65504 (or inf or NaN) is outside the decode path: the
 *   kernel sets MOE_ERR_UNSUPPORTED in *status (its outputs are then not
 *   defined).  Writes o_route[p] = w[t][j] * o (fp32).  For routes whose
 *   expert is not in the group nothing is written.
 * PREFILL mode: activations quantised to the records' format (NVFP4 records:
 *   per token, and h per route, G = amax/(6*448), block scale
 *   e4m3_rne(amax_b/(6 G)), codes e2m1_rne(v/(s G)); MXFP4 records: per block
 *   of 32 the OCP MX rule, scale 2^(floor(log2 amax_b) - 2), codes
 *   e2m1_rne(v / scale)) and multiplied on the tcgen05 tensor cores (FP4 x
 *   FP4, fp32 accumulation in tensor memory); adds w[t][j] * o into y_acc[t]
 *   (fp32, caller-zeroed).  Each expert is read from the slot src_slot gives
 *   it: a hit's cache slot, or the staging slot a miss's record was gathered
 *   into (expcache_fill) before this call.  The group-0 call also quantises
 *   the tokens and plans the tiles of every active expert; the calls of the
 *   later groups reuse that plan (same arguments and workspace, in group
 *   order on one stream).  Experts are taken prefill_group at a time; H and
 *   I must be multiples of 256 (else MOE_ERR_UNSUPPORTED).
 * Shared expert (Is > 0, group 0 only): bf16 gate/up [Is][H], down [H][Is];
 *   DECODE writes o_shared[t] = shared(x_t) (fp32); PREFILL adds it into
 *   y_acc[t] (bf16 tensor-core GEMMs, h rounded to bf16).
 * stages (DECODE only): MOE_STAGE_GATE_UP computes h into the workspace,
 *   MOE_STAGE_DOWN consumes it; MOE_STAGE_ALL does both.
 */
enum { MOE_MODE_DECODE = 0, MOE_MODE_PREFILL = 1 };
enum { MOE_STAGE_GATE_UP = 1, MOE_STAGE_DOWN = 2, MOE_STAGE_ALL = 3 };

typedef struct {
  int mode, stages;
  int T, H, I, E, k;
  const void* x;             /* device [T][H] bf16                                  */
  const expcache* cache;     /* weights come from its slots                          */
  const float* gscale;       /* device [E][3] fp32 global scales (gate, up, down)    */
  const int32_t* src_slot;   /* device [E]  (expcache_lookup)                        */
  const int32_t* act_list;   /* device [E]  (expcache_lookup)                        */
  const int32_t* n_act;      /* device [2]  (expcache_lookup)                        */
  const int32_t* offsets;    /* device [E+1] (moe_permute)                            */
  const int32_t* pad_offsets;/* device [E+1] (moe_permute, pad_align 128; PREFILL)    */
  const int32_t* perm;       /* device [T*k] (moe_permute)                            */
  const int32_t* inv;        /* device [T*k] (moe_permute; PREFILL)                   */
  const float* w;            /* device [T][k] routing weights (moe_route)            */
  int group, n_stage;        /* expert group walked by this call                     */
  int prefill_group;         /* PREFILL: experts per launch group (0 = all at once)  */
  int Is;                    /* shared expert intermediate size, 0 = none            */
  const void* s_gate;        /* device bf16 [Is][H]                                   */
  const void* s_up;          /* device bf16 [Is][H]                                   */
  const void* s_down;        /* device bf16 [H][Is]                                   */
  float* o_route;            /* DECODE: device out [T*k][H] fp32                      */
  float* y_acc;              /* PREFILL: device in/out [T][H] fp32                    */
  float* o_shared;           /* device out [T][H] fp32 (Is > 0)                       */
  void* workspace;           /* device scratch of moe_ffn_workspace_bytes(...)        */
  size_t workspace_bytes;
  int32_t* status;           /* device sticky status word, or NULL                   */
} moe_ffn_args;

size_t moe_ffn_workspace_bytes(int mode, int T, int H, int I, int E, int k, int Is);
moe_status moe_expert_ffn(const moe_ffn_args* a, void* stream);

/* moe_expert_ffn_noalloc - the DECODE expert FFN for callers that cannot
 * allocate device memory.  The pages have no counterpart to this call; it
 * exists for code that must not allocate on its own: an engine whose device
 * memory is fully reserved up front by an outer framework or pool (so a
 * cudaMalloc would fail or fragment it), a latency-critical serving loop
 * where an allocation could block on the driver, or a plugin that is only
 * handed input and output buffers.
 *
 * Same arguments and results as moe_expert_ffn in MOE_MODE_DECODE, except
 * that a->workspace and a->workspace_bytes are ignored: the scratch between
 * the gate/up and down kernels (T*k*I + T*Is floats) lives in one fixed
 * array in the library's device memory, MOE_NOALLOC_SCRATCH_BYTES large,
 * which every GPU that loads the library holds until the process exits.
 * The caller still passes inputs and outputs.  Nothing is allocated.
 *   - Returns MOE_ERR_UNSUPPORTED when mode is not MOE_MODE_DECODE or when
 *     moe_ffn_workspace_bytes(MOE_MODE_DECODE, T, H, I, E, k, Is) exceeds
 *     MOE_NOALLOC_SCRATCH_BYTES (use moe_expert_ffn for such sizes).
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress).  CUDA loads the library's array lazily, and
 *     loading it reserves its MOE_NOALLOC_SCRATCH_BYTES of device memory:
 *     the library's first expcache_create, moe_layer_create or FFN call in
 *     the process does that on its current device.  On any other device the
 *     first moe_expert_ffn_noalloc loads it, so a caller that reserves all
 *     device memory up front makes one call on each device first, before
 *     any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     no part of it needs to start at zero.  Calls that overlap on the GPU
 *     (different streams, no ordering between them) race on it and give
 *     wrong results: order them on one stream or with events. */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
moe_status moe_expert_ffn_noalloc(const moe_ffn_args* a, void* stream);

/* moe_nvfp4_quantize - the prefill path's activation quantiser on its own:
 * NVFP4 codes of T rows of K values, written in the tensor-core operand
 * layout that the prefill GEMMs read (dev.to page, "The wall": NVFP4 is E2M1
 * values with an E4M3 scale per 16 and a global fp32 scale).  Per row t:
 * G[t] = amax_t / 2688 (1 for a row of zeros); per 16-value block b the scale
 * byte s = e4m3_rne(amax_b / (6 G)); each value v gets the E2M1 code of
 * v / (e4m3_value(s) * G), round to nearest even, saturating at 6 (every
 * step fp32, quotients correctly rounded; a block whose scale byte is 0 gets
 * codes 0).
 *   x       device [T][K], bf16 (dtype 0) or fp32 (dtype 1)
 *   codes   device [T][K/2]: value 2j of a row in the low nibble of byte j
 *   scales  device, ceil(T/128)*128*K/16 bytes: the scale of block b of row t
 *           at byte ((t/128)*(K/64) + b/4)*512 + (t%32)*16 + ((t%128)/32)*4
 *           + b%4 (512-byte atoms of 128 rows x 4 blocks); bytes of rows >= T
 *           are left as they were
 *   G       device [T] fp32
 * K % 256 == 0 and K <= 8192 (bf16) or 4096 (fp32), else
 * MOE_ERR_UNSUPPORTED; T == 0 is a no-op.  Stream-ordered.
 */
moe_status moe_nvfp4_quantize(const void* x, int dtype, int T, int K, uint8_t* codes,
                              uint8_t* scales, float* G, void* stream);

/* ---------------------------------------------------------------- combine
 * y[t] = bf16_rne( y_acc[t] + sum_{j<k} o_route[inv[t*k+j]] + o_shared[t] ),
 * each term skipped when its pointer is NULL; the k-term sum is taken in
 * j order (deterministic).  No residual is added. */
typedef struct {
  int T, H, k;
  const float* y_acc;     /* device [T][H] or NULL            */
  const float* o_route;   /* device [T*k][H] or NULL          */
  const int32_t* inv;     /* device [T*k] (with o_route)      */
  const float* o_shared;  /* device [T][H] or NULL            */
  void* y;                /* device out [T][H] bf16           */
} moe_combine_args;

moe_status moe_combine(const moe_combine_args* a, void* stream);

/* ------------------------------------------------------------------ layer
 * One MoE layer: owns a workspace for up to T_max tokens and runs route ->
 * permute -> lookup -> (fill group g -> ffn group g, for every group) ->
 * combine on one stream.  T >= prefill_min_tokens (> 0) takes the PREFILL
 * path (experts walked in groups of prefill_group through the staging
 * layout), otherwise DECODE.  Neither path synchronises with the host, and
 * the decode path can be captured in a CUDA graph.
 * Misses: decode gathers them into the staging slots group by group, or,
 * when every miss fits in them, inside the FFN kernel itself (copy units run
 * beside the hits' units; a miss's units wait for its record, bounded).  With
 * every active expert resident and one group, the decode down kernel's units
 * of an expert start as soon as that expert's gate/up units have written h
 * (counts in the layer's workspace, a bounded wait each).  A wait that runs
 * out sets MOE_ERR_TIMEOUT in the status word; the layer's counts are then
 * undefined and the layer should be destroyed.  A
 * prefill with at least 2 staging slots gathers its misses on a second
 * stream of the layer, in groups of n_stage/2 into alternating halves of the
 * staging slots, while the first stream runs the GEMMs of the hits and of
 * the groups already landed (the "groups of 64 experts through a staging
 * buffer" of the dev.to page); the streams are joined before the forward's
 * last kernel.  The prefill path clears its fp32 sum of the experts'
 * outputs inside the token quantisation; with a shared expert and one FFN
 * call (every active expert resident, or no staging slots) the shared
 * expert's down GEMM, the last to add into that sum, writes y = bf16(sum +
 * shared) itself and no separate combine runs.
 *
 * skip_tau > 0 turns on the renorm-skip (Strata-GLM blog, section
 * "Uncensoring without touching the weights"): a route whose expert is not
 * resident in the layer's cache when the forward looks it up and whose
 * combine weight w is below skip_tau is dropped - never gathered or computed
 * - and its token's remaining weights are renormalised to sum to 1.  An
 * approximation of the layer; the routing outputs (ids, w, p_sel) stay the
 * router's.  0 <= skip_tau < 1/k (the top route is always kept), else
 * MOE_ERR_INVALID_ARG.
 */
typedef struct moe_layer moe_layer;

typedef struct {
  int H, I, E, k, Is;
  const float* w_router;   /* device [E][H] fp32                          */
  const float* bias;       /* device [E] fp32 or NULL                     */
  const float* gscale;     /* device [E][3] fp32                          */
  const void* s_gate;      /* device bf16 shared expert (NULL if Is == 0) */
  const void* s_up;
  const void* s_down;
  expcache* cache;         /* weights of this layer: layer index `layer` */
  int layer;
  int T_max;
  int prefill_min_tokens;  /* 0 = always DECODE                           */
  int prefill_group;       /* experts per prefill group (e.g. 64)         */
  float skip_tau;          /* renorm-skip threshold, 0 = exact (below)    */
} moe_layer_desc;

moe_status moe_layer_create(const moe_layer_desc* d, moe_layer** out);
moe_status moe_layer_destroy(moe_layer* l);
/* x: [T][H] bf16, device memory or pinned host memory (cudaHostAlloc /
 * cudaHostRegister); a host x is copied into the layer's own buffer by the
 * forward's first kernel (16-byte loads; the copy engine when x is not
 * 16-byte aligned), since the later kernels read it many times.  y: [T][H]
 * bf16, device memory or pinned host memory, which the kernels address
 * directly under unified addressing: the forward's last kernel writes it with
 * plain stores, so a host y is the device->host transfer of the result.
 * Pageable (unregistered) host memory is MOE_ERR_INVALID_ARG. */
moe_status moe_layer_forward(moe_layer* l, const void* x, int T, void* y, void* stream);
/* Device pointers (inside the layer's workspace) to the last forward's router
 * outputs: ids [T][k] int32, w [T][k] fp32, p_sel [T][k] fp32; and the
 * expert-sorted permutation perm [T*k] and lookup results src_slot [E],
 * n_act [2]. */
moe_status moe_layer_debug_ptrs(const moe_layer* l, const int32_t** ids, const float** w,
                                const float** p_sel, const int32_t** perm,
                                const int32_t** src_slot, const int32_t** n_act);
/* After a forward that took the PREFILL path: device pointers to its fp32
 * h = silu(g) * u rows before their NVFP4 quantisation (I values per padded
 * route row: the route at expert-sorted position p of expert e is row
 * pad_offsets[e] + p - offsets[e]), and to offsets [E+1] and pad_offsets
 * [E+1].  Valid until the next forward.  MOE_ERR_INVALID_ARG when the last
 * forward took the DECODE path.  (For tests; the pages have no
 * counterpart.) */
moe_status moe_layer_debug_prefill(const moe_layer* l, const float** h_rows,
                                   const int32_t** offsets, const int32_t** pad_offsets);
/* Timing hook (the pages have no counterpart; it serves measurement):
 * events[0..n) are cudaEvent_t handles owned by the caller.  While set, every
 * moe_layer_forward records events[0] before its first kernel and events[i]
 * (i < n) after its i-th launch step: the router (with the permutation and
 * lookup when they share its kernel: up to 8 tokens), the permutation, the
 * adaptive cache's step (when a kernel of its own), then per expert group the
 * gather (unless the FFN gathers itself or a second stream does) and the FFN:
 * decode one kernel, prefill each of its kernels (token quantisation, tile
 * tables, per launch group the gate/up GEMM, h quantisation and down GEMM,
 * then the shared expert's two GEMMs), then the combine (when it is a kernel
 * of its own: not in a prefill whose shared-expert down GEMM writes y).  So
 * the caller can time each kernel of the layer's own
 * sequence.
 * n = 0 clears the hook.  n > 32 is MOE_ERR_INVALID_ARG. */
moe_status moe_layer_set_timing(moe_layer* l, void* const* events, int n);
/* Synchronises `stream`, returns the layer's sticky device status in
 * *status_out and clears it. */
moe_status moe_read_device_status(moe_layer* l, void* stream, int32_t* status_out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
