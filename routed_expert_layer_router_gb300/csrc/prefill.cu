// prefill.cu - the prefill path: many tokens per expert, so the expert FFN is
// a grouped GEMM on the tcgen05 tensor cores.
//
//   K-actq   each route's token quantised to NVFP4 (E2M1 codes, E4M3 scale per
//            16 values, fp32 global per row) into an expert-sorted staging
//            layout whose segments are padded to 128 rows;
//   K-gemm   per (expert, 128 weight rows, 128 routes) tile:
//            D[rows, routes] = W[rows, K] . Xq[routes, K]^T with
//            tcgen05.mma kind::mxf4nvf4 (block scale, 16-value E4M3 scales in
//            tensor memory), fp32 accumulators in tensor memory; TMA tile loads
//            of both operands (one 3-D tensor map spans the whole slot arena, so
//            every expert record is addressed by its slot), an mbarrier ring
//            (gate/up: 4 stages of one 128-byte K chunk; down: 3 stages of
//            two), one warp loading, one warp
//            issuing MMAs, eight warps in the epilogue.  Gate and up share the
//            activation tile and accumulate into two TMEM accumulators; the
//            epilogue forms silu(g)*u.
//   K-hq     h quantised to NVFP4 per route, same layout as K-actq, with each
//            route's down-epilogue data (weight x G x down scale, token);
//   K-gemm   down projection, tiles in row-tile-major order; the epilogue
//            scales by the routing weight and adds each route's 128-value row
//            segment into y_acc[token] with L2 reductions (the weighted combine).
// The bf16 shared expert runs through the same GEMM with kind::f16.
// Experts are walked in act_list order in launch groups of prefill_group
// experts (0: every expert in one launch per GEMM).
// Sources: Strata-GLM blog, "Day one" list (chunked prefill: each layer's
// experts run as one batched matrix multiply per chunk); dev.to page,
// "Prefill in groups of 64 experts"; "Project Maya" page, "440 tokens a
// second of prefill" (a prompt chunk touches nearly every expert).
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <string.h>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

const uint8_t* cache_arena(const expcache* c);
uint64_t cache_rec_bytes(const expcache* c);
int cache_format(const expcache* c);
int cache_n_cache(const expcache* c);
int cache_n_stage(const expcache* c);

namespace pf {

constexpr int kTileM = 128, kTileN = 128, kStageKB = 128;  // K bytes per stage and operand row
// tokens per tile of the bf16 shared-expert GEMMs: 256 halves the weight
// tiles loaded per token against 128 (bf16 needs no scale-factor columns, so
// two 256-column accumulators fit in tensor memory)
constexpr int kSharedN = 256;
constexpr int kMaxN = 256;
constexpr int kThreads = 320;  // warp 0: TMA, warp 1: MMA, warps 2..9: epilogue
constexpr int kEpiWarps = 8;   // two per tensor-memory lane quarter, each half of the columns
constexpr uint64_t kWaitNs = 2000000000ull;  // no wait lasts longer than 2 s
constexpr uint32_t kTmemCols = 512;
constexpr int kSingleChunks = 2;
constexpr int kDualChunks = 1;

enum Epi { EPI_GU_ROUTED = 0, EPI_GU_SHARED = 1, EPI_DOWN_ROUTED = 2, EPI_DOWN_SHARED = 3 };

struct GemmParams {
  int mtiles;   // 128-row weight tiles per expert
  int kstages;  // K / (128 bytes of each operand row)
  // routed experts of this launch: planned experts (act_list order) [lo + g0,
  // min(lo + g1, hi)) where [lo, hi) is the FFN call's expert group
  // (pf_group_range), their tiles tiles[plan_begin[g0]*mtiles ..
  // plan_begin[g1]*mtiles)
  const uint32_t* tiles;     // gate/up: packed (expert index j, m tile, n tile)
  const int4* ctab;          // down: column tiles {expert, slot, padded row of column 0, routes}
  const float2* dcol;        // down: per padded row {weight x G x down scale, token bits}
  const int32_t* plan_e;     // expert id of index j
  const int32_t* plan_slot;  // its cache slot
  const int32_t* plan_begin; // prefix of its 128-route column tiles
  const int32_t* plan_n;     // [0]: planned experts, [1]: of them hits (act_list first)
  int g0, g1;
  int group, gsize;          // the FFN call's expert group and misses per group
  int part;                  // group 0 only: 0 all of it, 1 its hits, 2 its misses
  const int32_t* offsets;
  const int32_t* pad_offsets;
  const int32_t* perm;
  const float* gscale;
  const float* w;
  int k;
  int n_slots;
  // shared expert: T activation rows
  int T;
  // block scales
  const uint8_t* arena;
  uint64_t rec_bytes;
  uint64_t sfa_off0, sfa_off1;  // offsets of the A matrices' scales in a record
  int kgroups;                  // K / 64 (scale atoms per 128-row tile row)
  const uint8_t* b_scales;      // activation scale atoms
  const float* b_gscale;        // activation per-row global scales
  // outputs
  float* h32;       int h_ld;   // routed gate/up: h [rows][I]
  uint16_t* hs;     int hs_ld;  // shared gate/up: h [T][Is] bf16
  float* y_acc;     int H;      // down: y_acc [T][H]
  uint16_t* y;                  // shared down only: write y = bf16(y_acc + shared) instead of
                                // adding into y_acc (it is then the last writer of y_acc)
  int32_t* status;
};

// ---- tile schedule ------------------------------------------------------------
// packed tile entry: expert index j (11 bits) | m tile (8 bits) | n tile (13 bits)
__host__ __device__ __forceinline__ uint32_t tile_pack(int j, int mt, int nt) {
  return ((uint32_t)j << 21) | ((uint32_t)mt << 13) | (uint32_t)nt;
}

// Tile orders.  Gate/up: an expert-major table (the 16 row tiles of an expert
// run side by side and share its activation tile in L2), decoded by tile_info.
// Down: a tile is a pair of adjacent 128-row tiles (m = 0 .. mtiles/2 - 1,
// rows 256 m .. 256 m + 255) and one column tile, row-pair-major over the
// launch's ncols column tiles, t = m * ncols + c, each column tile a record
// {expert, slot, padded row of column 0, routes} (ctab); so at any time the
// CTAs add into a few 256-row bands of every token's y_acc row, which stay in
// L2, instead of into all of y_acc.  A CTA's shared-memory fill rate, not
// HBM, limited the down GEMM with one row tile per activation tile (its
// activations were half of every stage); two row tiles per activation tile
// measured 441 -> 412 us for the 4096-token layer.

// act_list range [lo, hi) of FFN group `group` among the planned experts:
// group 0 = the hits and misses [0, S), group g > 0 = misses [g S, (g+1) S)
// (S misses per group, all of them when S == 0)
__device__ __forceinline__ void pf_group_range(const int32_t* plan_n, int group, int S, int part,
                                               int& lo, int& hi) {
  const int n = plan_n[0], n_hit = plan_n[1], n_miss = n - n_hit;
  const int sz = S > 0 ? S : (n_miss > 0 ? n_miss : 1);
  if (group == 0) {
    lo = part == 2 ? n_hit : 0;
    hi = part == 1 ? n_hit : n_hit + min(sz, n_miss);
  } else {
    lo = n_hit + group * sz;
    hi = n_hit + min((group + 1) * sz, n_miss);
  }
  if (hi < lo) hi = lo;
}

// gate/up or shared tile t of a launch -> (m tile, n tile, expert id, slot);
// N columns per shared tile
template <bool ROUTED, int N>
__device__ __forceinline__ void tile_info(const GemmParams& p, int t, int& mt, int& nt, int& e,
                                          int& slot) {
  if (ROUTED) {
    const uint32_t v = p.tiles[t];
    const int j = (int)(v >> 21);
    mt = (int)((v >> 13) & 0xFFu);
    nt = (int)(v & 0x1FFFu);
    e = p.plan_e[j];
    slot = p.plan_slot[j];
  } else {
    const int ntn = (p.T + N - 1) / N;
    mt = t / ntn;
    nt = t % ntn;
    e = 0;
    slot = 0;
  }
}

// K-plan: the active experts in act_list order (hits, then the misses, which
// the FFN reads from the staging slots the lookup gave them), their 128-route
// column tiles, the gate/up tile table (mt_gu row tiles per column tile,
// expert-major) and the column-tile table of the down GEMM.
// One CTA of 1024 threads, one expert per thread.
__global__ void __launch_bounds__(1024) k_tile_plan(
    const int32_t* __restrict__ act_list, const int32_t* __restrict__ n_act,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pad_offsets,
    const int32_t* __restrict__ src_slot, int n_slots, int E, int mt_gu,
    uint32_t* __restrict__ tiles_gu, int4* __restrict__ ctab,
    int32_t* __restrict__ plan_e, int32_t* __restrict__ plan_slot,
    int32_t* __restrict__ plan_begin, int32_t* __restrict__ plan_n, int32_t* status) {
  __shared__ int s_w[33];
  const int j = threadIdx.x, lane = j & 31, wid = j >> 5;
  const int act = n_act[0];
  int e = -1, slot = -1, nt = 0, cnt = 0;
  if (j < act && j < E) {
    e = act_list[j];
    slot = src_slot[e];
    cnt = offsets[e + 1] - offsets[e];
    if (slot < 0 || slot >= n_slots) set_status(status, MOE_ERR_DEVICE);
    else nt = (cnt + kTileN - 1) / kTileN;
  }
  // block-wide exclusive scan of nt
  int incl = nt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_w[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int w = lane < (int)(blockDim.x >> 5) ? s_w[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += v;
    }
    s_w[lane] = wi - w;
    if (lane == 31) s_w[32] = wi;
  }
  __syncthreads();
  const int begin = s_w[wid] + incl - nt;
  const int n = act < E ? act : E;
  if (j < n) {
    plan_e[j] = e;
    plan_slot[j] = slot;
    plan_begin[j] = begin;
    for (int m = 0; m < mt_gu; ++m)
      for (int c = 0; c < nt; ++c) tiles_gu[(size_t)begin * mt_gu + m * nt + c] = tile_pack(j, m, c);
    for (int c = 0; c < nt; ++c)
      ctab[begin + c] = make_int4(e, slot, pad_offsets[e] + c * kTileN, min(kTileN, cnt - c * kTileN));
  }
  if (j == 0) {
    plan_begin[n] = s_w[32];
    plan_n[0] = n;
    plan_n[1] = min(n_act[1], n);
  }
}

template <int KIND, int EPI>
struct Cfg {
  // two A operands against one B, two accumulators: gate/up takes the gate
  // and up rows of one row tile, the routed down two adjacent row tiles (so
  // each activation tile loaded serves 256 weight rows)
  static constexpr bool kDual = (EPI == EPI_GU_ROUTED || EPI == EPI_GU_SHARED || EPI == EPI_DOWN_ROUTED);
  static constexpr bool kRouted = (EPI == EPI_GU_ROUTED || EPI == EPI_DOWN_ROUTED);
  // routed down: row-tile-major order over a table of column tiles (ctab)
  static constexpr bool kMMajor = (EPI == EPI_DOWN_ROUTED);
  static constexpr bool kNvf4 = (KIND == 0);
  static constexpr bool kMxf4 = (KIND == 2);
  static constexpr bool kFp4 = kNvf4 || kMxf4;
  static constexpr int kTileBytes = kTileM * kStageKB;  // 16 KiB (an A tile)
  // B rows (routes or tokens) per tile and their bytes per 128-byte K chunk
  static constexpr int kN = (KIND == 1) ? kSharedN : kTileN;
  static constexpr int kBBytes = kN * kStageKB;
  // scale atoms (512 B: 128 rows x 4 blocks) per operand and 128-byte K chunk
  // (256 values): blocks of 16 (NVFP4) take 4 atoms, blocks of 32 (MXFP4) 2
  static constexpr int kAtoms = kNvf4 ? 4 : (kMxf4 ? 2 : 0);
  static constexpr int kSfBytes = kAtoms * 512;
  // one 128-byte K chunk of every operand (A tiles, B tile, their scale atoms)
  static constexpr int kChunkBytes =
      kTileBytes * (kDual ? 2 : 1) + kBBytes + kSfBytes * (kDual ? 3 : 2);
  // several chunks per stage: fewer stages per tile, so fewer barrier round
  // trips and commits for the same bytes in flight (4 dual or 6 single
  // chunks fill the shared memory)
  static constexpr int kChunks = kDual ? kDualChunks : (kN > kTileN ? 1 : kSingleChunks);
  static constexpr int kStageBytes = kChunks * kChunkBytes;
  static constexpr int kStagesFit = (226 * 1024) / kStageBytes;
  static constexpr int kStages =
      (kDual ? 4 : 6) / kChunks < kStagesFit ? (kDual ? 4 : 6) / kChunks : kStagesFit;
  static constexpr int kSmem = 1024 + kStages * kStageBytes;
  // tensor memory: accumulators, then per-stage scale-factor columns
  static constexpr uint32_t kAccCols = (uint32_t)kN * (kDual ? 2 : 1);
  static constexpr uint32_t kOpSfCols = kAtoms * 4;  // tensor-memory columns per operand
  static constexpr uint32_t kSfColsPerChunk = kOpSfCols * (kDual ? 3 : 2);
  static constexpr uint32_t kSfColsPerStage = kChunks * kSfColsPerChunk;
  // two accumulators where they fit beside the scale factors, so that a tile's
  // MMAs never wait for the previous tile's epilogue to read its accumulator
  static constexpr int kAccBufs = (2 * kAccCols + kStages * kSfColsPerStage <= kTmemCols) ? 2 : 1;
  static constexpr uint32_t kSfCol0 = kAccCols * kAccBufs;
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// SiLU with the fast exponential and division (a few ulp: far below the
// tolerance and the rounding-boundary slack of the quantised h)
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Down epilogue of one thread: its accumulator row of 64 columns (routes or
// tokens, ra then rb), each weighted by cs[j] and added into y_acc row cr[j]
// at yb; a warp instruction adds 32 consecutive rows (one 128-byte reduction
// in L2).  Columns from nv on are padding.
__device__ __forceinline__ void add_columns(const uint32_t (&ra)[32], const uint32_t (&rb)[32],
                                            float* yb, const float* cs, const int* cr, int H,
                                            int nv) {
#pragma unroll
  for (int jj = 0; jj < 32; ++jj)
    if (jj < nv) ptx::red_add_f32(yb + (size_t)cr[jj] * H, __uint_as_float(ra[jj]) * cs[jj]);
#pragma unroll
  for (int jj = 0; jj < 32; ++jj)
    if (32 + jj < nv)
      ptx::red_add_f32(yb + (size_t)cr[32 + jj] * H, __uint_as_float(rb[jj]) * cs[32 + jj]);
}

// The same columns as add_columns, as the layer's last contribution: each
// y_acc element plus the column's value, rounded to bf16 into y (one 128-byte
// read and one 64-byte write per warp instruction); no other CTA writes them.
// All 32 reads of a register set are issued before the first write.
__device__ __forceinline__ void write_col32(const uint32_t (&r)[32], const float* ya,
                                            uint16_t* yb, const int* cr, int H, int nv) {
  float v[32];
#pragma unroll
  for (int jj = 0; jj < 32; ++jj) v[jj] = jj < nv ? __ldcg(ya + (size_t)cr[jj] * H) : 0.f;
#pragma unroll
  for (int jj = 0; jj < 32; ++jj)
    if (jj < nv) yb[(size_t)cr[jj] * H] = f32_to_bf16_rne(v[jj] + __uint_as_float(r[jj]));
}
__device__ __forceinline__ void write_columns(const uint32_t (&ra)[32], const uint32_t (&rb)[32],
                                              const float* ya, uint16_t* yb, const int* cr,
                                              int H, int nv) {
  write_col32(ra, ya, yb, cr, H, nv);
  write_col32(rb, ya, yb, cr + 32, H, nv - 32);
}

template <int KIND, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
           const __grid_constant__ CUtensorMap tmB, GemmParams p) {
  using C = Cfg<KIND, EPI>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full_bar[C::kStages], empty_bar[C::kStages];
  __shared__ uint64_t acc_full[C::kAccBufs], acc_empty[C::kAccBufs];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int s_tlo, s_thi, s_cbase, s_ncols;
  __shared__ float col_scale[kMaxN];
  __shared__ int col_row[kMaxN];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the tiles of this launch
  if (threadIdx.x == 0) {
    abort_flag = 0;
    if (C::kRouted) {
      int lo, hi;
      pf_group_range(p.plan_n, p.group, p.gsize, p.part, lo, hi);
      const int g0 = min(lo + p.g0, hi), g1 = min(lo + p.g1, hi);
      s_cbase = p.plan_begin[g0];
      s_ncols = p.plan_begin[g1] - s_cbase;
      s_tlo = C::kMMajor ? 0 : s_cbase * p.mtiles;
      s_thi = C::kMMajor ? s_ncols * (C::kDual ? p.mtiles / 2 : p.mtiles) : p.plan_begin[g1] * p.mtiles;
    } else {
      s_cbase = 0;
      s_ncols = 1;
      s_tlo = 0;
      s_thi = ((p.T + C::kN - 1) / C::kN) * p.mtiles;
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      ptx::mbar_init(&acc_full[b], 1);
      ptx::mbar_init(&acc_empty[b], kEpiWarps);
    }
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int tlo = s_tlo, thi = s_thi, cbase = s_cbase, ncols = s_ncols;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      uint32_t g = 0;
      // The next tile's info is loaded during this tile's stages: for the
      // gate/up table a chain of three dependent loads (table entry, plan
      // entry, padded row offset), one link per stage; for the down GEMM one
      // column-tile record.  Either would otherwise stall the ring at every
      // tile boundary.
      int mt = 0, nt = 0, e = 0, slot = 0, brow = 0;
      const int t0 = tlo + blockIdx.x;
      if (t0 < thi) {
        if (C::kMMajor) {
          const int4 r = p.ctab[cbase + t0 % ncols];
          mt = t0 / ncols;
          slot = r.y;
          brow = r.z;
        } else {
          tile_info<C::kRouted, C::kN>(p, t0, mt, nt, e, slot);
          brow = nt * C::kN + (C::kRouted ? p.pad_offsets[e] : 0);
        }
      }
      for (int t = t0; t < thi && !abort_flag; t += gridDim.x) {
        const int tn = t + gridDim.x;
        uint32_t vn = 0;
        int mtn = 0, ntn = 0, en = 0, sn = 0, pn = 0;
        int4 rn = make_int4(0, 0, 0, 0);
        const int kst = (p.kstages + C::kChunks - 1) / C::kChunks;  // stages per tile
        const int arow = mt * kTileM * (C::kMMajor && C::kDual ? 2 : 1);  // weight rows
        for (int kb = 0; kb < kst; ++kb, ++g) {
          if (C::kMMajor && tn < thi && kb == 0) rn = p.ctab[cbase + tn % ncols];
          if (C::kRouted && !C::kMMajor && tn < thi) {  // one link per stage
            if (kb == 0) vn = p.tiles[tn];
            if (kb == min(1, kst - 1)) {
              mtn = (int)((vn >> 13) & 0xFFu);
              ntn = (int)(vn & 0x1FFFu);
              en = p.plan_e[vn >> 21];
              sn = p.plan_slot[vn >> 21];
            }
            if (kb == min(2, kst - 1)) pn = p.pad_offsets[en];
          }
          const int s = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          if (!ptx::mbar_wait(&empty_bar[s], ph ^ 1, kWaitNs)) {
            set_status(p.status, MOE_ERR_TIMEOUT);
            abort_flag = 1;
            break;
          }
          unsigned char* const st0 = smem + (size_t)s * C::kStageBytes;
          const int ncs = min(C::kChunks, p.kstages - kb * C::kChunks);  // chunks in this stage
          ptx::mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(ncs * C::kChunkBytes));
          for (int c = 0; c < ncs; ++c) {
            unsigned char* st = st0 + (size_t)c * C::kChunkBytes;
            const int kq = kb * C::kChunks + c;  // 128-byte K chunk
            const int kc = C::kFp4 ? kq * kStageKB : kq * (kStageKB / 2);  // bytes or bf16s
            // Down: the weights are read once, the activation tiles by every row
            // tile of their column, and y_acc is added into meanwhile; the cache
            // policies keep the activations and y_acc in L2 ahead of the weights.
            const uint64_t pol_w = ptx::l2_evict_first(), pol_a = ptx::l2_evict_last();
            if (C::kMMajor) {
              ptx::tma_load_3d_hint(st, &tmA0, kc, arow, slot, &full_bar[s], pol_w);
              if (C::kDual)
                ptx::tma_load_3d_hint(st + C::kTileBytes, &tmA0, kc, arow + kTileM, slot,
                                      &full_bar[s], pol_w);
            } else if (C::kRouted) {
              ptx::tma_load_3d(st, &tmA0, kc, arow, slot, &full_bar[s]);
              if (C::kDual) ptx::tma_load_3d(st + C::kTileBytes, &tmA1, kc, arow, slot, &full_bar[s]);
            } else {
              ptx::tma_load_2d(st, &tmA0, kc, arow, &full_bar[s]);
              if (C::kDual) ptx::tma_load_2d(st + C::kTileBytes, &tmA1, kc, arow, &full_bar[s]);
            }
            unsigned char* bdst = st + C::kTileBytes * (C::kDual ? 2 : 1);
            if (C::kMMajor) ptx::tma_load_2d_hint(bdst, &tmB, kc, brow, &full_bar[s], pol_a);
            else ptx::tma_load_2d(bdst, &tmB, kc, brow, &full_bar[s]);
            if (C::kFp4) {
              // kAtoms scale atoms (512 B each) per operand: atom columns
              // kq*kAtoms .. (kq+1)*kAtoms-1 of the row tile
              unsigned char* sf = bdst + C::kBBytes;
              const uint8_t* rec = p.arena + (uint64_t)slot * p.rec_bytes;
              const uint64_t aoff =
                  ((uint64_t)(arow / kTileM) * p.kgroups + (uint64_t)kq * C::kAtoms) * 512;
              const uint64_t boff =
                  ((uint64_t)(brow / kTileN) * p.kgroups + (uint64_t)kq * C::kAtoms) * 512;
              unsigned char* sfb = sf + C::kSfBytes * (C::kDual ? 2 : 1);
              if (C::kMMajor) {
                ptx::bulk_load_hint(sf, rec + p.sfa_off0 + aoff, C::kSfBytes, &full_bar[s], pol_w);
                if (C::kDual)
                  ptx::bulk_load_hint(sf + C::kSfBytes,
                                      rec + p.sfa_off0 + aoff + (uint64_t)p.kgroups * 512,
                                      C::kSfBytes, &full_bar[s], pol_w);
                ptx::bulk_load_hint(sfb, p.b_scales + boff, C::kSfBytes, &full_bar[s], pol_a);
              } else {
                ptx::bulk_load(sf, rec + p.sfa_off0 + aoff, C::kSfBytes, &full_bar[s]);
                if (C::kDual)
                  ptx::bulk_load(sf + C::kSfBytes, rec + p.sfa_off1 + aoff, C::kSfBytes, &full_bar[s]);
                ptx::bulk_load(sfb, p.b_scales + boff, C::kSfBytes, &full_bar[s]);
              }
            }
          }
        }
        if (C::kMMajor) {
          mt = tn / ncols;
          slot = rn.y;
          brow = rn.z;
        } else if (C::kRouted) {
          mt = mtn;
          nt = ntn;
          e = en;
          slot = sn;
          brow = ntn * kTileN + pn;
        } else if (tn < thi) {
          tile_info<false, C::kN>(p, tn, mt, nt, e, slot);
          brow = nt * C::kN;
        }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      // instruction descriptor: M = 128, N = 128, K-major A and B
      uint32_t idesc = ((uint32_t)(C::kN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
      if (C::kNvf4) idesc |= (1u << 7) | (1u << 10);               // E2M1 x E2M1, UE4M3 scales
      else if (C::kMxf4) idesc |= (1u << 7) | (1u << 10) | (1u << 23);  // E2M1 x E2M1, UE8M0
      else idesc |= (1u << 4) | (1u << 7) | (1u << 10);            // fp32 D, bf16 A and B
      uint32_t g = 0, it = 0;
      for (int t = tlo + blockIdx.x; t < thi && !abort_flag; t += gridDim.x, ++it) {
        const int ab = (int)(it % C::kAccBufs);           // accumulator of this tile
        const uint32_t au = it / C::kAccBufs;              // its earlier uses
        const uint32_t acc = tmem + (uint32_t)ab * C::kAccCols;
        if (!ptx::mbar_wait(&acc_empty[ab], (au & 1) ^ 1, kWaitNs)) {
          set_status(p.status, MOE_ERR_TIMEOUT);
          abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb * C::kChunks < p.kstages; ++kb, ++g) {
          const int s = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          if (!ptx::mbar_wait(&full_bar[s], ph, kWaitNs)) {
            set_status(p.status, MOE_ERR_TIMEOUT);
            abort_flag = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int ncs = min(C::kChunks, p.kstages - kb * C::kChunks);
          for (int c = 0; c < ncs; ++c) {
            unsigned char* st = smem + (size_t)s * C::kStageBytes + (size_t)c * C::kChunkBytes;
            const uint32_t a0 = ptx::smem_u32(st);
            const uint32_t a1 = a0 + C::kTileBytes;
            const uint32_t b = a0 + C::kTileBytes * (C::kDual ? 2 : 1);
            const uint32_t sf = b + C::kBBytes;
            const uint32_t sfcol =
                C::kSfCol0 + (uint32_t)s * C::kSfColsPerStage + (uint32_t)c * C::kSfColsPerChunk;
            if (C::kFp4) {
              // scale atoms -> tensor memory (4 columns each)
              for (int kk = 0; kk < C::kAtoms; ++kk) {
                const int nops = C::kDual ? 3 : 2;
                for (int o = 0; o < nops; ++o) {
                  const uint64_t d = ptx::smem_desc(sf + o * C::kSfBytes + kk * 512, 128, 128, 0);
                  ptx::tmem_cp_32x128b_x4(tmem + sfcol + o * C::kOpSfCols + kk * 4, d);
                }
              }
            }
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t da0 = ptx::smem_desc(a0 + kk * 32, 16, 1024, 2);
              const uint64_t db = ptx::smem_desc(b + kk * 32, 16, 1024, 2);
              const bool accum = (kb > 0) || (c > 0) || (kk > 0);
              if (C::kNvf4) {
                const uint32_t sfb = tmem + sfcol + (C::kDual ? 32 : 16) + kk * 4;
                ptx::mma_nvf4(acc, da0, db, idesc, tmem + sfcol + kk * 4, sfb, accum);
                if (C::kDual) {
                  const uint64_t da1 = ptx::smem_desc(a1 + kk * 32, 16, 1024, 2);
                  ptx::mma_nvf4(acc + C::kN, da1, db, idesc, tmem + sfcol + 16 + kk * 4, sfb, accum);
                }
              } else if (C::kMxf4) {
                // this K = 64 step's scales: atom kk / 2, bytes 0-1 (kk even)
                // or 2-3 (kk odd) of each row's word
                const uint32_t at = (uint32_t)(kk >> 1) * 4;
                const uint32_t id = (kk & 1) ? ((2u << 29) | (2u << 4)) : 0u;
                const uint32_t sfb = tmem + sfcol + C::kOpSfCols * (C::kDual ? 2 : 1) + at;
                ptx::mma_mxf4(acc, da0, db, idesc | id, tmem + sfcol + at, sfb, accum);
                if (C::kDual) {
                  const uint64_t da1 = ptx::smem_desc(a1 + kk * 32, 16, 1024, 2);
                  ptx::mma_mxf4(acc + C::kN, da1, db, idesc | id, tmem + sfcol + C::kOpSfCols + at,
                                sfb, accum);
                }
              } else {
                ptx::mma_bf16(acc, da0, db, idesc, accum);
                if (C::kDual) {
                  const uint64_t da1 = ptx::smem_desc(a1 + kk * 32, 16, 1024, 2);
                  ptx::mma_bf16(acc + C::kN, da1, db, idesc, accum);
                }
              }
            }
          }
          ptx::tc_commit(&empty_bar[s]);  // stage reusable once these MMAs finish
        }
        if (!ok) break;
        ptx::tc_commit(&acc_full[ab]);
      }
    }
  } else {
    // ================= epilogue (warps 2..9) =================
    // A warp reads the tensor-memory lanes of its quarter (warp id mod 4) and
    // half of the columns; it copies its accumulator columns to registers and
    // releases the accumulator before any arithmetic or store, so that the
    // next tile's MMAs run while this tile's outputs are formed and written.
    const int q = warp & 3;             // tensor-memory lane quarter of this warp
    const int ch = (warp - 2) >> 2;     // column half
    const int row = q * 32 + lane;      // weight row within the tile
    const int et = threadIdx.x - 64;    // 0..255
    constexpr int kHalf = kTileN / 2;

    if (C::kMMajor) {
      // Routed down.  The column data of a tile (combine weight x activation
      // scale x expert scale, and token, per route) comes precomputed per
      // padded row (dcol); the next tile's record and column data are loaded
      // while this tile waits and is reduced, so no chain of loads sits
      // between two tiles.
      const int t0 = tlo + blockIdx.x;
      int4 r = make_int4(0, 0, 0, 0);
      float2 dc = make_float2(0.f, 0.f);
      if (t0 < thi) {
        r = p.ctab[cbase + t0 % ncols];
        if (et < kTileN) dc = p.dcol[r.z + et];
      }
      uint32_t it = 0;
      for (int t = t0; t < thi; t += gridDim.x, ++it) {
        const int mt = t / ncols, n_valid = r.w;
        if (et < kTileN) {
          col_scale[et] = et < n_valid ? dc.x : 0.f;
          col_row[et] = __float_as_int(dc.y);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        const int tn = t + gridDim.x;
        int4 rn = r;
        if (tn < thi) rn = p.ctab[cbase + tn % ncols];
        const int ab = (int)(it % C::kAccBufs);
        if (!ptx::mbar_wait(&acc_full[ab], (it / C::kAccBufs) & 1, kWaitNs)) {
          set_status(p.status, MOE_ERR_TIMEOUT);
          abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) +
                                   (uint32_t)ab * C::kAccCols + (uint32_t)(ch * kHalf);
        uint32_t ra[32], rb[32], ra2[32], rb2[32];
        ptx::tmem_ld_32x32b_x32(lane_addr, ra);
        ptx::tmem_ld_32x32b_x32(lane_addr + 32, rb);
        ptx::tmem_ld_32x32b_x32(lane_addr + 128, ra2);
        ptx::tmem_ld_32x32b_x32(lane_addr + 160, rb2);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);  // the accumulator is free
        float2 dn = dc;
        if (tn < thi && et < kTileN) dn = p.dcol[rn.z + et];
        add_columns(ra, rb, p.y_acc + 2 * mt * kTileM + row, col_scale + ch * kHalf,
                    col_row + ch * kHalf, p.H, n_valid - ch * kHalf);
        add_columns(ra2, rb2, p.y_acc + (2 * mt + 1) * kTileM + row, col_scale + ch * kHalf,
                    col_row + ch * kHalf, p.H, n_valid - ch * kHalf);
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        r = rn;
        dc = dn;
      }
    } else {
      constexpr int kHalfN = C::kN / 2;  // columns per thread (the warp's column half)
      uint32_t it = 0;
      for (int t = tlo + blockIdx.x; t < thi; t += gridDim.x, ++it) {
        int mt, nt, e, slot;
        tile_info<C::kRouted, C::kN>(p, t, mt, nt, e, slot);
        int n_valid, col0;
        if (C::kRouted) {
          const int cnt = p.offsets[e + 1] - p.offsets[e];
          n_valid = min(C::kN, cnt - nt * C::kN);
          col0 = p.pad_offsets[e] + nt * C::kN;  // padded activation row of column 0
        } else {
          n_valid = min(C::kN, p.T - nt * C::kN);
          col0 = nt * C::kN;
        }
        // per-column data (column = route or token)
        if (et < C::kN) {
          float sc = 1.f;
          int rr = col0 + et;
          if (et < n_valid) {
            if (EPI == EPI_GU_ROUTED) sc = p.b_gscale[col0 + et];
          }
          col_scale[et] = sc;
          col_row[et] = rr;
        }
        float gg = 1.f, gu = 1.f;
        if (EPI == EPI_GU_ROUTED) {
          gg = p.gscale[e * 3 + 0];
          gu = p.gscale[e * 3 + 1];
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        const int ab = (int)(it % C::kAccBufs);
        if (!ptx::mbar_wait(&acc_full[ab], (it / C::kAccBufs) & 1, kWaitNs)) {
          set_status(p.status, MOE_ERR_TIMEOUT);
          abort_flag = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)ab * C::kAccCols +
                                   (uint32_t)(ch * kHalfN);
        if (EPI == EPI_GU_ROUTED) {
          // routed gate/up: h = silu(g) * u formed chunk by chunk (64 values
          // kept), then the accumulator is released and h is written
          float hv[kHalfN];
#pragma unroll
          for (int c = 0; c < kHalfN; c += 16) {
            uint32_t ga[16], ua[16];
            ptx::tmem_ld_32x32b_x16(lane_addr + c, ga);
            ptx::tmem_ld_32x32b_x16(lane_addr + C::kN + c, ua);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float g = __uint_as_float(ga[jj]), u = __uint_as_float(ua[jj]);
              const float G = col_scale[ch * kHalfN + c + jj];
              hv[c + jj] = silu_f(g * gg * G) * (u * gu * G);
            }
          }
          ptx::tc_fence_before();
          if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);  // the accumulator is free
#pragma unroll
          for (int jj = 0; jj < kHalfN; ++jj) {
            const int n = ch * kHalfN + jj;
            if (n < n_valid) p.h32[(size_t)(col0 + n) * p.h_ld + mt * kTileM + row] = hv[jj];
          }
        } else if (C::kDual) {
          // shared gate/up: h = silu(g) * u written as bf16 16 columns at a
          // time; the (single) accumulator is released after the last read
#pragma unroll 2
          for (int c = 0; c < kHalfN; c += 16) {
            uint32_t ga[16], ua[16];
            ptx::tmem_ld_32x32b_x16(lane_addr + c, ga);
            ptx::tmem_ld_32x32b_x16(lane_addr + C::kN + c, ua);
            ptx::tmem_ld_wait();
            if (c + 16 >= kHalfN) {
              ptx::tc_fence_before();
              if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);  // the accumulator is free
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int n = ch * kHalfN + c + jj;
              const float h = silu_f(__uint_as_float(ga[jj])) * __uint_as_float(ua[jj]);
              if (n < n_valid)
                p.hs[(size_t)(col0 + n) * p.hs_ld + mt * kTileM + row] = f32_to_bf16_rne(h);
            }
          }
        } else {
          // shared down: the token columns added into y_acc, 64 at a time
#pragma unroll 1
          for (int c0 = 0; c0 < kHalfN; c0 += 64) {
            uint32_t ra[32], rb[32];
            ptx::tmem_ld_32x32b_x32(lane_addr + c0, ra);
            ptx::tmem_ld_32x32b_x32(lane_addr + c0 + 32, rb);
            ptx::tmem_ld_wait();
            if (c0 + 64 >= kHalfN) {
              ptx::tc_fence_before();
              if (lane == 0) ptx::mbar_arrive(&acc_empty[ab]);  // the accumulator is free
            }
            if (p.y)
              write_columns(ra, rb, p.y_acc + mt * kTileM + row, p.y + mt * kTileM + row,
                            col_row + ch * kHalfN + c0, p.H, n_valid - ch * kHalfN - c0);
            else
              add_columns(ra, rb, p.y_acc + mt * kTileM + row, col_scale + ch * kHalfN + c0,
                          col_row + ch * kHalfN + c0, p.H, n_valid - ch * kHalfN - c0);
          }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- NVFP4 activation quantisation -------------------------------------------------
// The prefill reading of the activation quantiser, for a row of K values: G =
// amax/2688 (1 for a zero row), block scale s = e4m3_rne(amax_b / (6 G)),
// dequantised scale sdq = s * G, codes e2m1_rne_sat(v / sdq); every step fp32,
// the quotients correctly rounded.

// two values to E2M1 codes, round to nearest even, saturating at +-6 (lo in
// bits 0-3, hi in bits 4-7; the sign bit follows the value's sign)
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// E4M3 (round to nearest even, saturating to 448) of t >= 0, and its value
__device__ __forceinline__ uint32_t e4m3_rne(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(t));
  return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  return f16_lo(e4m3x2_to_f16x2(b & 0xFFu));
}

// v / s rounded to nearest even, given y = RN(1/s): the product v*y refined
// by two residual steps (r = v - s*q is exact under an FMA, then q = RN(q +
// r*y)).  Markstein's theorem (IBM J. Res. Dev. 34(1), 1990) makes the last
// step correctly rounded once q is within one ulp of v/s, which the first
// step ensures.  Valid while s, y and the quotient stay in the normal range:
// callers keep s in [2^-56, 2^48] (|v/s| < 16 there) and divide otherwise.
__device__ __forceinline__ float quot_rn(float v, float s, float y) {
  float q = __fmul_rn(v, y);
  q = __fmaf_rn(__fmaf_rn(-s, q, v), y, q);
  return __fmaf_rn(__fmaf_rn(-s, q, v), y, q);
}

// block scale byte and dequantised scale of a block with max |v| = ab
__device__ __forceinline__ uint32_t block_scale(float ab, float sixG, float G, float& sdq) {
  const uint32_t sc = e4m3_rne(__fdiv_rn(ab, sixG));
  sdq = __fmul_rn(e4m3_value(sc), G);
  return sc;
}

// codes of n consecutive values of one block (n even), packed 2 per byte
template <int N>
__device__ __forceinline__ uint32_t block_codes(const float* v, uint32_t sc, float sdq) {
  if (sc == 0) return 0u;  // the whole block quantises to +-0; written as +0
  float q[N];
  if (sdq >= 0x1p-56f && sdq <= 0x1p48f) {
    const float y = __frcp_rn(sdq);
#pragma unroll
    for (int i = 0; i < N; ++i) q[i] = quot_rn(v[i], sdq, y);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) q[i] = __fdiv_rn(v[i], sdq);
  }
  uint32_t c = 0;
#pragma unroll
  for (int i = 0; i < N; i += 2) c |= e2m1x2_rn(q[i], q[i + 1]) << (4 * i);
  return c;
}

__device__ __forceinline__ float absmax4(float a, float b, float c, float d) {
  return fmaxf(fmaxf(fabsf(a), fabsf(b)), fmaxf(fabsf(c), fabsf(d)));
}

// ---- MXFP4 activation quantisation (records in MXFP4: the tensor cores take
// both operands' scales in one format).  OCP Microscaling Formats v1.0: a
// block of 32 values shares X = floor(log2 max|v|) - 2, kept in E8M0's range
// [-127, 127] (scale byte X + 127); each code is E2M1(v / 2^X), round to
// nearest even, saturating at 6; an all-zero block gets byte 0 and codes 0.
// v / 2^X is a multiplication by an exact power of two.
__device__ __forceinline__ uint32_t mx_scale(float ab, float& inv) {
  if (!(ab > 0.f)) {
    inv = 0.f;
    return 0u;
  }
  const int X = max(ilogbf(ab) - 2, -127);
  inv = __uint_as_float((uint32_t)(127 - X) << 23);  // 2^-X (X <= 125)
  return (uint32_t)(X + 127);
}
template <int N>
__device__ __forceinline__ uint32_t mx_codes(const float* v, float ab, float inv) {
  if (!(ab > 0.f)) return 0u;
  uint32_t c = 0;
#pragma unroll
  for (int i = 0; i < N; i += 2) c |= e2m1x2_rn(v[i] * inv, v[i + 1] * inv) << (4 * i);
  return c;
}

// byte offset of the scale word (4 blocks, kg = block / 4) of padded row `row`
// in the 512-byte scale atoms of a K-wide operand
__device__ __forceinline__ size_t scale_word(int row, int kg, int KG) {
  return ((size_t)(row >> 7) * KG + kg) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4;
}

// codes of N consecutive values (N % 8 == 0) of one NVFP4 block with scale
// byte sc and dequantised scale sdq, 8 codes per word (one reciprocal)
template <int N>
__device__ __forceinline__ void block_codes_w(const float* v, uint32_t sc, float sdq,
                                              uint32_t* out) {
  if (sc == 0) {  // the whole block quantises to +-0; written as +0
#pragma unroll
    for (int w = 0; w < N / 8; ++w) out[w] = 0u;
    return;
  }
  float q[N];
  if (sdq >= 0x1p-56f && sdq <= 0x1p48f) {
    const float y = __frcp_rn(sdq);
#pragma unroll
    for (int i = 0; i < N; ++i) q[i] = quot_rn(v[i], sdq, y);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) q[i] = __fdiv_rn(v[i], sdq);
  }
#pragma unroll
  for (int w = 0; w < N / 8; ++w) {
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < 8; i += 2) c |= e2m1x2_rn(q[8 * w + i], q[8 * w + i + 1]) << (4 * i);
    out[w] = c;
  }
}

// One fp32 row of K values (K % 256 == 0, K <= KMAX) by one warp into padded
// row `row` of the tcgen05 layout.  Lane l owns the 64 consecutive values
// 64 (l + 32 p) .. + 63 of each pass p over 2048 values: four NVFP4 blocks
// (one scale word) or two MXFP4 blocks, so no block spans lanes and a lane
// writes its 32 code bytes and its scale word (half word for MX) itself.  The
// row is read once (through L1: consecutive loads of a lane share sectors)
// and held in registers.  The block scales' quotients amax_b / (6 G) use one
// correctly rounded reciprocal of 6 G per row and two residual steps (as the
// codes do), dividing when 6 G is outside [2^-56, 2^48].  Returns the row's
// global scale G (on every lane; 1 for MX).
template <int KMAX, int FMT>
__device__ __forceinline__ float quant_row_f32(const float* __restrict__ hr, int K, int row,
                                              uint8_t* __restrict__ codes,
                                              uint8_t* __restrict__ scales,
                                              float* __restrict__ Gr) {
  constexpr int kNP = (KMAX + 2047) / 2048;
  const int lane = threadIdx.x & 31;
  const int KG = K / (4 * fmt_block(FMT));
  float4 v[kNP][16];
  float amax = 0.f;
#pragma unroll
  for (int p = 0; p < kNP; ++p) {
    const int c0 = 64 * (lane + 32 * p);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      v[p][q] = c0 < K ? __ldg(reinterpret_cast<const float4*>(hr + c0) + q)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      amax = fmaxf(amax, absmax4(v[p][q].x, v[p][q].y, v[p][q].z, v[p][q].w));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const float G = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  const float sixG = __fmul_rn(6.0f, G);
  const bool fast = sixG >= 0x1p-56f && sixG <= 0x1p48f;
  const float y6 = fast ? __frcp_rn(sixG) : 0.f;
#pragma unroll
  for (int p = 0; p < kNP; ++p) {
    const int u = lane + 32 * p;  // 64-value unit of the row
    if (64 * u >= K) break;
    uint32_t cw[8];
    uint32_t sw = 0;
    if (FMT == MOE_FMT_MXFP4) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        float f[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          f[4 * q] = v[p][8 * b + q].x;
          f[4 * q + 1] = v[p][8 * b + q].y;
          f[4 * q + 2] = v[p][8 * b + q].z;
          f[4 * q + 3] = v[p][8 * b + q].w;
        }
        float ab = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) ab = fmaxf(ab, fabsf(f[i]));
        float inv;
        const uint32_t sc = mx_scale(ab, inv);
#pragma unroll
        for (int w = 0; w < 4; ++w) cw[4 * b + w] = mx_codes<8>(f + 8 * w, ab, inv);
        sw |= sc << (8 * b);
      }
      *reinterpret_cast<uint16_t*>(scales + scale_word(row, u >> 1, KG) + 2 * (u & 1)) =
          (uint16_t)sw;
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float f[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[4 * q] = v[p][4 * b + q].x;
          f[4 * q + 1] = v[p][4 * b + q].y;
          f[4 * q + 2] = v[p][4 * b + q].z;
          f[4 * q + 3] = v[p][4 * b + q].w;
        }
        float ab = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(f[i]));
        const uint32_t sc = e4m3_rne(fast ? quot_rn(ab, sixG, y6) : __fdiv_rn(ab, sixG));
        const float sdq = __fmul_rn(e4m3_value(sc), G);
        block_codes_w<16>(f, sc, sdq, cw + 2 * b);
        sw |= sc << (8 * b);
      }
      *reinterpret_cast<uint32_t*>(scales + scale_word(row, u, KG)) = sw;
    }
    uint4* crow = reinterpret_cast<uint4*>(codes + (size_t)row * (K / 2) + 32 * (size_t)u);
    crow[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    crow[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
  }
  const float Gout = FMT == MOE_FMT_MXFP4 ? 1.0f : G;
  if (lane == 0) Gr[row] = Gout;
  return Gout;
}

// zero padded rows [r0, r1) of a K-wide operand (codes, scale words, G) with
// the threads of one CTA; blk = values per block scale
__device__ __forceinline__ void zero_rows(int r0, int r1, int K, int blk,
                                          uint8_t* __restrict__ codes,
                                          uint8_t* __restrict__ scales, float* __restrict__ G) {
  const int n = r1 - r0;
  if (n <= 0) return;
  const int n16 = K / 32, KG = K / (4 * blk);  // 16-byte chunks of a codes row; scale words
  uint4* c = reinterpret_cast<uint4*>(codes + (size_t)r0 * (K / 2));
  for (int i = threadIdx.x; i < n * n16; i += blockDim.x) c[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < n * KG; i += blockDim.x)
    *reinterpret_cast<uint32_t*>(scales + scale_word(r0 + i / KG, i % KG, KG)) = 0u;
  for (int i = threadIdx.x; i < n; i += blockDim.x) G[r0 + i] = 0.f;
}

constexpr int kQuantHMaxK = 4096;  // I up to 4096 (the prefill path checks)
constexpr int kQuantXMaxK = 8192;  // H up to 8192

// K-hq: h -> NVFP4 for the padded rows of planned experts [g0, g1): CTA
// (j - g0, part) takes an eighth of expert plan_e[j]'s rows, one warp per
// row; padding rows are zeroed.  Three CTAs per SM for rows up to 2048 values
// (80 registers, a few bytes spilled).  The kernel is bound by latency, not
// by HBM: for the 4096-token layer's h, lane-owned blocks (no shuffles) took
// 95 -> 90 us, eighths instead of quarters and the next-row prefetch 85 us.
template <int KMAX, int FMT>
__global__ void __launch_bounds__(256, KMAX <= 2048 ? 3 : 1) k_quant_h(
    const float* __restrict__ h32, int K, int g0, int g1, int group, int gsize, int part,
    const int32_t* __restrict__ plan_e,
    const int32_t* __restrict__ plan_n, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ pad_offsets, const int32_t* __restrict__ perm,
    const float* __restrict__ w, const float* __restrict__ gscale, int k,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ G,
    float2* __restrict__ dcol) {
  int glo, ghi;
  pf_group_range(plan_n, group, gsize, part, glo, ghi);
  const int j = glo + g0 + (int)blockIdx.x;
  if (j >= min(glo + g1, ghi)) return;
  const int e = plan_e[j];
  const int cnt = offsets[e + 1] - offsets[e];
  const int r0 = pad_offsets[e], nrow = pad_offsets[e + 1] - r0;
  const int per = (nrow + gridDim.y - 1) / gridDim.y;
  const int lo = blockIdx.y * per, hi = min(nrow, lo + per);
  const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float gsd = gscale[e * 3 + 2];
  for (int i = lo + wid; i < min(hi, cnt); i += nw) {
    // the warp's next row is fetched into L2 while this one is quantised
    if ((threadIdx.x & 31) == 0 && i + nw < min(hi, cnt))
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   ::"l"(h32 + (size_t)(r0 + i + nw) * K), "r"((uint32_t)K * 4u) : "memory");
    const float Gi =
        quant_row_f32<KMAX, FMT>(h32 + (size_t)(r0 + i) * K, K, r0 + i, codes, scales, G);
    if ((threadIdx.x & 31) == 0) {
      // the down GEMM's column data of this route: combine weight x G x the
      // expert's down scale (in that order), and the token
      const int route = perm[offsets[e] + i];
      dcol[r0 + i] = make_float2(Gi * w[route] * gsd, __int_as_float(route / k));
    }
  }
  zero_rows(r0 + max(lo, cnt), r0 + hi, K, fmt_block(FMT), codes, scales, G);
  for (int i = max(lo, cnt) + threadIdx.x; i < hi; i += blockDim.x)
    dcol[r0 + i] = make_float2(0.f, 0.f);
}

// K-hq over plain rows: row t of x (fp32, T rows) -> row t, one warp per row
template <int KMAX>
__global__ void __launch_bounds__(256) k_quant_rows_f32(const float* __restrict__ x, int T, int K,
                                                        uint8_t* __restrict__ codes,
                                                        uint8_t* __restrict__ scales,
                                                        float* __restrict__ G) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t < T) quant_row_f32<KMAX, MOE_FMT_NVFP4>(x + (size_t)t * K, K, t, codes, scales, G);
}

// K-actq: the tokens quantised once each and written straight into the
// padded rows of their k routes (route t*k + j at position p = inv[t*k + j]
// of expert e goes to row pad_offsets[e] + p - offsets[e]).  CTA t < T takes
// token t: 256 threads, thread i holding 16-byte chunks i + 256 m (8 values;
// two threads per block).  CTA T + e zeroes expert e's padding rows.  With
// inv == NULL (k = 1) token t goes to row t and no rows are padded.  With
// y_zero, CTA t also zeroes row t of y_zero (K floats): the down GEMMs' sum,
// cleared inside this latency-bound kernel instead of by a separate pass.
template <int KMAX, int FMT>
__global__ void __launch_bounds__(256) k_quant_routes(
    const uint16_t* __restrict__ x, int T, int K, int E, int k, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pad_offsets,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ G,
    float* __restrict__ y_zero) {
  constexpr int kNJ = KMAX / 2048;
  __shared__ int s_row[32];
  __shared__ float s_max[8];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if ((int)blockIdx.x >= T) {
    const int e = blockIdx.x - T;
    if (inv && e < E)
      zero_rows(pad_offsets[e] + offsets[e + 1] - offsets[e], pad_offsets[e + 1], K,
                fmt_block(FMT), codes, scales, G);
    return;
  }
  const int t = blockIdx.x;
  const int NC = K / 8, KG = K / (4 * fmt_block(FMT));
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * K);
  uint4 v[kNJ];
#pragma unroll
  for (int m = 0; m < kNJ; ++m) {
    const int c = tid + 256 * m;
    v[m] = c < NC ? __ldg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (y_zero) {
    float4* yz = reinterpret_cast<float4*>(y_zero + (size_t)t * K);
    for (int c = tid; c < K / 4; c += 256) yz[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (tid < k) {
    int row = -1;
    if (!inv) {
      row = t;
    } else {
      const int p = inv[(size_t)t * k + tid];
      if (p >= 0) {  // expert of position p: the last e with offsets[e] <= p
        int lo = 0, hi = E;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (__ldg(offsets + mid) <= p) lo = mid;
          else hi = mid;
        }
        row = pad_offsets[lo] + p - offsets[lo];
      }
    }
    s_row[tid] = row;
  }
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < kNJ; ++m) {
    const uint32_t w[4] = {v[m].x, v[m].y, v[m].z, v[m].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (lane == 0) s_max[wid] = amax;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, s_max[i]);
  const float Gt = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
  const float sixG = __fmul_rn(6.0f, Gt);
  uint32_t cw[kNJ], sw[kNJ];
#pragma unroll
  for (int m = 0; m < kNJ; ++m) {
    cw[m] = 0u;
    sw[m] = 0u;
    if (tid + 256 * m >= NC) break;  // uniform per warp: NC is a multiple of 32
    const uint32_t w[4] = {v[m].x, v[m].y, v[m].z, v[m].w};
    float f[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = bf16_lo(w[q]);
      f[2 * q + 1] = bf16_hi(w[q]);
    }
    float ab = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) ab = fmaxf(ab, fabsf(f[q]));
    ab = fmaxf(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, 1));  // the other half of the block
    if (FMT == MOE_FMT_MXFP4) {
      ab = fmaxf(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, 2));  // four threads per block of 32
      float inv;
      const uint32_t sc = mx_scale(ab, inv);
      cw[m] = mx_codes<8>(f, ab, inv);
      // block (tid + 256 m) / 4; lanes 16i gather the scale word of blocks 4i..4i+3
      const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sc, 4);
      const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sc, 8);
      const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sc, 12);
      sw[m] = sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
      continue;
    }
    float sdq;
    const uint32_t sc = block_scale(ab, sixG, Gt, sdq);
    cw[m] = block_codes<8>(f, sc, sdq);
    // block (tid + 256 m) / 2; lanes 8i gather the scale word of blocks 4i..4i+3
    const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sc, 2);
    const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sc, 4);
    const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sc, 6);
    sw[m] = sc | (s1 << 8) | (s2 << 16) | (s3 << 24);
  }
  for (int j = 0; j < k; ++j) {
    const int row = s_row[j];
    if (row < 0) continue;
    uint32_t* crow = reinterpret_cast<uint32_t*>(codes + (size_t)row * (K / 2));
#pragma unroll
    for (int m = 0; m < kNJ; ++m) {
      const int c = tid + 256 * m;
      if (c >= NC) break;
      crow[c] = cw[m];
      if (FMT == MOE_FMT_MXFP4) {
        if ((lane & 15) == 0)
          *reinterpret_cast<uint32_t*>(scales + scale_word(row, c >> 4, KG)) = sw[m];
      } else if ((lane & 7) == 0) {
        *reinterpret_cast<uint32_t*>(scales + scale_word(row, c >> 3, KG)) = sw[m];
      }
    }
    if (tid == 0) G[row] = FMT == MOE_FMT_MXFP4 ? 1.0f : Gt;
  }
}

// ---- host side ---------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static moe_status load_encoder() {
  if (g_encode) return MOE_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return MOE_ERR_CUDA;
  g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  return MOE_OK;
}

// rows of `inner` elements (uint8 codes or bf16), box = 128 bytes x box_rows rows,
// 128-byte swizzle; optional third dimension (slots)
static moe_status make_map(CUtensorMap* m, const void* base, bool bf16, uint64_t inner,
                           uint64_t rows, uint64_t row_stride_bytes, uint64_t slots,
                           uint64_t slot_stride_bytes, uint32_t box_rows = 128) {
  cuuint64_t dims[3] = {inner, rows, slots};
  cuuint64_t strides[2] = {row_stride_bytes, slot_stride_bytes};
  cuuint32_t box[3] = {bf16 ? 64u : 128u, box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const cuuint32_t rank = slots > 0 ? 3 : 2;
  CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// workspace layout for a prefill call on T tokens
struct PrefillWs {
  size_t rows;  // padded rows
  size_t xq_codes, xq_scales, xq_G, h32, hq_codes, hq_scales, hq_G, dcol, hs, tiles_gu, ctab, plan,
      total;
  size_t max_ntiles;  // 128-route column tiles of all experts, at most
  PrefillWs(int T, int H, int I, int E, int k, int Is) {
    rows = (((size_t)T * k + (size_t)E * (kTileN - 1)) + kTileN - 1) / kTileN * kTileN;
    size_t o = 0;
    auto take = [&](size_t b) { size_t r = o; o += (b + 1023) & ~(size_t)1023; return r; };
    xq_codes = take(rows * H / 2);
    xq_scales = take(rows * H / 16);
    xq_G = take(rows * 4);
    h32 = take(rows * I * 4);
    hq_codes = take(rows * I / 2);
    hq_scales = take(rows * I / 16);
    hq_G = take(rows * 4);
    hs = take((size_t)T * Is * 2);
    max_ntiles = ((size_t)T * k + kTileN - 1) / kTileN + (size_t)E;
    tiles_gu = take(max_ntiles * (I / kTileM) * 4);
    ctab = take(max_ntiles * 16);  // down: column-tile records
    dcol = take(rows * 8);
    plan = take(((size_t)3 * (E + 1) + 2) * 4);  // plan_e | plan_slot | plan_begin | plan_n
    total = o + 1024;
  }
};

template <int KIND, int EPI>
static moe_status launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                              const GemmParams& p, cudaStream_t s) {
  using C = Cfg<KIND, EPI>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(k_gemm<KIND, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmem) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr = true;
  }
  k_gemm<KIND, EPI><<<kSMs, kThreads, C::kSmem, s>>>(a0, a1, b, p);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

}  // namespace pf

moe_status nvfp4_quantize(const void* x, int dtype, int T, int K, uint8_t* codes,
                          uint8_t* scales, float* G, cudaStream_t s) {
  using namespace pf;
  if (T < 0 || K <= 0 || (dtype != 0 && dtype != 1)) return MOE_ERR_INVALID_ARG;
  if (K % 256 || K > (dtype == 0 ? kQuantXMaxK : kQuantHMaxK)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !codes || !scales || !G) return MOE_ERR_INVALID_ARG;
  if (dtype == 0) {
    auto* kx = K <= 4096 ? k_quant_routes<4096, MOE_FMT_NVFP4>
                         : k_quant_routes<kQuantXMaxK, MOE_FMT_NVFP4>;
    kx<<<T, 256, 0, s>>>((const uint16_t*)x, T, K, 1, 1, nullptr, nullptr, nullptr, codes, scales,
                         G, nullptr);
  } else {
    auto* kq = K <= 2048 ? k_quant_rows_f32<2048> : k_quant_rows_f32<kQuantHMaxK>;
    kq<<<(T + 7) / 8, 256, 0, s>>>((const float*)x, T, K, codes, scales, G);
  }
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}

size_t prefill_workspace_bytes(int T, int H, int I, int E, int k, int Is) {
  return pf::PrefillWs(T, H, I, E, k, Is).total;
}

// the fp32 h rows (one per padded route row, I values) inside a prefill
// call's workspace
const float* prefill_h_rows(const void* workspace, int T, int H, int I, int E, int k, int Is) {
  const uint8_t* ws = (const uint8_t*)(((uintptr_t)workspace + 1023) & ~(uintptr_t)1023);
  return (const float*)(ws + pf::PrefillWs(T, H, I, E, k, Is).h32);
}

moe_status prefill_setup() { return pf::load_encoder(); }

// 2-D bf16 tensor map (rows of `inner` values, `rows` rows), box 64 values x
// box_rows rows, 128-byte swizzle, zero fill outside the rows
moe_status tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                        uint64_t row_stride_bytes, uint32_t box_rows) {
  moe_status st = pf::load_encoder();
  if (st != MOE_OK) return st;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = pf::g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// part (the layer's own sequence): 0 = the call's whole group; for group 0, 1 =
// the token quantisation, tile tables, hits and shared expert, 2 = the first
// misses (whose records the layer gathers meanwhile).  Also the layer's own:
// zero_y clears y_acc in the token quantisation (instead of the caller); y,
// when this call's shared-expert down is the last writer of y_acc, makes it
// write y = bf16(y_acc + shared) itself (no separate combine).
moe_status prefill_ffn(const moe_ffn_args* a, cudaStream_t s, int part, void (*mark)(void*),
                       void* mark_ctx, bool zero_y, uint16_t* y) {
  // the timing hook: a mark after every kernel of the FFN
  auto marked = [&]() {
    if (mark) mark(mark_ctx);
  };
  using namespace pf;
  if (!a->inv || !a->pad_offsets) return MOE_ERR_INVALID_ARG;
  if (a->H % 256 || a->I % 256 || a->Is % 128 || a->I > kQuantHMaxK || a->H > kQuantXMaxK ||
      a->k > 32)
    return MOE_ERR_UNSUPPORTED;
  moe_status st = load_encoder();
  if (st != MOE_OK) return st;
  const PrefillWs W(a->T, a->H, a->I, a->E, a->k, a->Is);
  uint8_t* ws = (uint8_t*)(((uintptr_t)a->workspace + 1023) & ~(uintptr_t)1023);
  const int fmt = cache_format(a->cache);
  const bool is_mx = fmt == MOE_FMT_MXFP4;
  const int blk = fmt_block(fmt);
  const RecordLayout L(a->H, a->I, fmt);
  const uint8_t* arena = cache_arena(a->cache);
  const uint64_t rb = cache_rec_bytes(a->cache);
  const int n_slots = cache_n_cache(a->cache) + cache_n_stage(a->cache);
  const int H = a->H, I = a->I;

  // tensor maps: weights of every slot; staged activations; shared expert
  CUtensorMap mg, mu, md, mxq, mhq, msg, msu, msd, mx, mhs;
  if ((st = make_map(&mg, arena + L.gate_codes, false, H / 2, I, H / 2, n_slots, rb)) ||
      (st = make_map(&mu, arena + L.up_codes, false, H / 2, I, H / 2, n_slots, rb)) ||
      (st = make_map(&md, arena + L.down_codes, false, I / 2, H, I / 2, n_slots, rb)) ||
      (st = make_map(&mxq, ws + W.xq_codes, false, H / 2, W.rows, H / 2, 0, 0)) ||
      (st = make_map(&mhq, ws + W.hq_codes, false, I / 2, W.rows, I / 2, 0, 0)))
    return st;
  const bool shared = a->Is > 0 && a->group == 0 && part != 2;
  if (shared) {
    if ((st = make_map(&msg, a->s_gate, true, H, a->Is, (uint64_t)H * 2, 0, 0)) ||
        (st = make_map(&msu, a->s_up, true, H, a->Is, (uint64_t)H * 2, 0, 0)) ||
        (st = make_map(&msd, a->s_down, true, a->Is, H, (uint64_t)a->Is * 2, 0, 0)) ||
        (st = make_map(&mx, a->x, true, H, a->T, (uint64_t)H * 2, 0, 0, kSharedN)) ||
        (st = make_map(&mhs, ws + W.hs, true, a->Is, a->T, (uint64_t)a->Is * 2, 0, 0, kSharedN)))
      return st;
  }

  // the call's expert group (group 0: hits and the first misses; group g: the
  // next n_stage misses), walked in launch groups of `grp` (act_list order);
  // 0 = all at once
  const int grp = a->prefill_group > 0 ? a->prefill_group : a->E;
  const int max_act = a->T * a->k < a->E ? a->T * a->k : a->E;
  const int gmax = (a->group == 0 || a->n_stage == 0) ? max_act
                   : (a->n_stage < max_act ? a->n_stage : max_act);  // experts in the group, at most
  int32_t* plan = (int32_t*)(ws + W.plan);
  int32_t *plan_e = plan, *plan_slot = plan + (a->E + 1), *plan_begin = plan + 2 * (a->E + 1),
          *plan_n = plan + 3 * (a->E + 1);
  uint32_t* tiles_gu = (uint32_t*)(ws + W.tiles_gu);
  int4* ctab = (int4*)(ws + W.ctab);
  // group 0: the tokens, quantised once each into their routes' padded rows;
  // the tile tables of both GEMMs for every active expert (the later groups'
  // calls reuse them: same workspace, same stream)
  if (a->group == 0 && part != 2) {
    auto* kx = is_mx ? (H <= 4096 ? k_quant_routes<4096, MOE_FMT_MXFP4>
                               : k_quant_routes<kQuantXMaxK, MOE_FMT_MXFP4>)
                  : (H <= 4096 ? k_quant_routes<4096, MOE_FMT_NVFP4>
                               : k_quant_routes<kQuantXMaxK, MOE_FMT_NVFP4>);
    kx<<<a->T + a->E, 256, 0, s>>>((const uint16_t*)a->x, a->T, H, a->E, a->k, a->inv, a->offsets,
                                   a->pad_offsets, ws + W.xq_codes, ws + W.xq_scales,
                                   (float*)(ws + W.xq_G), zero_y ? a->y_acc : nullptr);
    MOE_CHECK_LAUNCH();
    marked();
    k_tile_plan<<<1, 1024, 0, s>>>(a->act_list, a->n_act, a->offsets, a->pad_offsets, a->src_slot,
                                  n_slots, a->E, I / kTileM, tiles_gu, ctab, plan_e, plan_slot,
                                  plan_begin, plan_n, a->status);
    MOE_CHECK_LAUNCH();
    marked();
  }
  for (int g0 = 0; g0 < gmax; g0 += grp) {
    const int g1 = g0 + grp;
    GemmParams gp;
    memset(&gp, 0, sizeof(gp));
    gp.plan_e = plan_e; gp.plan_slot = plan_slot; gp.plan_begin = plan_begin;
    gp.plan_n = plan_n; gp.g0 = g0; gp.g1 = g1;
    gp.group = a->group; gp.gsize = a->n_stage; gp.part = part;
    gp.offsets = a->offsets; gp.pad_offsets = a->pad_offsets;
    gp.perm = a->perm; gp.gscale = a->gscale; gp.w = a->w; gp.k = a->k; gp.n_slots = n_slots;
    gp.arena = arena; gp.rec_bytes = rb; gp.H = H; gp.status = a->status;
    // gate/up
    gp.tiles = tiles_gu;
    gp.mtiles = I / kTileM;
    gp.kstages = (H / 2) / kStageKB;
    gp.kgroups = H / (4 * blk);  // scale atoms per 128-row tile
    gp.sfa_off0 = L.gate_scales; gp.sfa_off1 = L.up_scales;
    gp.b_scales = ws + W.xq_scales; gp.b_gscale = (const float*)(ws + W.xq_G);
    gp.h32 = (float*)(ws + W.h32); gp.h_ld = I;
    st = is_mx ? launch_gemm<2, EPI_GU_ROUTED>(mg, mu, mxq, gp, s)
               : launch_gemm<0, EPI_GU_ROUTED>(mg, mu, mxq, gp, s);
    if (st != MOE_OK) return st;
    marked();
    // h -> NVFP4
    const int ng = (g1 < gmax ? g1 : gmax) - g0;
    auto* kq = is_mx ? (I <= 2048 ? k_quant_h<2048, MOE_FMT_MXFP4>
                               : k_quant_h<kQuantHMaxK, MOE_FMT_MXFP4>)
                  : (I <= 2048 ? k_quant_h<2048, MOE_FMT_NVFP4>
                               : k_quant_h<kQuantHMaxK, MOE_FMT_NVFP4>);
    kq<<<dim3(ng, 8), 256, 0, s>>>((const float*)(ws + W.h32), I, g0, g1, a->group, a->n_stage,
                                  part, plan_e, plan_n,
                                  a->offsets, a->pad_offsets, a->perm, a->w, a->gscale, a->k,
                                  ws + W.hq_codes, ws + W.hq_scales, (float*)(ws + W.hq_G),
                                  (float2*)(ws + W.dcol));
    MOE_CHECK_LAUNCH();
    marked();
    // down, weighted, added into y_acc
    gp.ctab = ctab;
    gp.dcol = (const float2*)(ws + W.dcol);
    gp.mtiles = H / kTileM;
    gp.kstages = (I / 2) / kStageKB;
    gp.kgroups = I / (4 * blk);
    gp.sfa_off0 = L.down_scales; gp.sfa_off1 = 0;
    gp.b_scales = ws + W.hq_scales; gp.b_gscale = (const float*)(ws + W.hq_G);
    gp.y_acc = a->y_acc;
    st = is_mx ? launch_gemm<2, EPI_DOWN_ROUTED>(md, md, mhq, gp, s)
               : launch_gemm<0, EPI_DOWN_ROUTED>(md, md, mhq, gp, s);
    if (st != MOE_OK) return st;
    marked();
  }

  // shared expert (bf16): y_acc += Wd (silu(Wg x) * Wu x)
  if (shared) {
    GemmParams gp;
    memset(&gp, 0, sizeof(gp));
    gp.T = a->T; gp.H = H; gp.status = a->status;
    gp.mtiles = a->Is / kTileM;
    gp.kstages = (H * 2) / kStageKB;
    gp.hs = (uint16_t*)(ws + W.hs); gp.hs_ld = a->Is;
    if ((st = launch_gemm<1, EPI_GU_SHARED>(msg, msu, mx, gp, s)) != MOE_OK) return st;
    marked();
    gp.mtiles = H / kTileM;
    gp.kstages = (a->Is * 2) / kStageKB;
    gp.y_acc = a->y_acc;
    gp.y = y;
    if ((st = launch_gemm<1, EPI_DOWN_SHARED>(msd, msd, mhs, gp, s)) != MOE_OK) return st;
    marked();
  }
  return MOE_OK;
}

}  // namespace moe
