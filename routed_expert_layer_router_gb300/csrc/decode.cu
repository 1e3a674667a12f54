// decode.cu - K-decode-gu, K-decode-down and K-combine: the expert FFN for few
// tokens per expert, HBM-bound.  Weights stream from their cache or staging
// slot with 128-bit loads (the next step's loads are issued before the current
// step is computed); the NVFP4 dequant happens in registers: the E2M1 codes go
// through the hardware e2m1x2 -> f16x2 conversion and meet the activations in
// mixed-precision FMAs (f16 x f16 products, exact, accumulated in fp32); each
// 16-element partial sum is scaled once by its E4M3 block scale and the fp32
// global scale at the end.  One warp owns the rows {m0 + 32*m1 : m1 < 4} of a
// 128-row tile, which share one 16-byte row of every 512-byte scale atom, and
// every activation it reads from shared memory is reused across those rows.
// Sources: "Project Maya" page, section "A V100 has no BF16 and no FP8" (decode
// is a matrix-vector product where the bytes, not the arithmetic, set the
// speed); dev.to page, section "The wall" (NVFP4 experts).
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

const uint8_t* cache_arena(const expcache* c);
uint64_t cache_rec_bytes(const expcache* c);
int cache_format(const expcache* c);
int cache_n_cache(const expcache* c);
int cache_n_stage(const expcache* c);

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kXPad = 36;  // fp32 staging: floats per 32 values (bank spread)
constexpr int kHPad = 40;  // f16 staging: halves per 32 values (80-byte stride, conflict-free)
constexpr int kSharedKSplit = kDecWarps;  // shared gate/up: warps splitting the row length
// routed gate/up units: a warp takes kGuRows rows of the gate and of the up
// matrix, rows m0 + 32 (mo + m1) (m1 < kGuRows) of a 128-row tile; a tile is
// kGuParts units (4 quarters of m0 times the row groups mo)
constexpr int kGuRows = 4;
constexpr int kGuParts = 4 * (4 / kGuRows);
constexpr int kGuMinBlocks = 2;  // CTAs per SM the gate/up kernel is compiled for

struct DecodeParams {
  int T, H, I, E, k, Is;
  const uint16_t* x;
  const uint8_t* arena;
  uint64_t rec_bytes;
  int n_slots;  // cache + staging slots in the arena
  const float* gscale;
  const int32_t* src_slot;
  const int32_t* act_list;
  const int32_t* n_act;
  const int32_t* offsets;
  const int32_t* perm;
  const float* w;
  int group, n_stage;
  int n_shared_units;  // shared-expert grid units (down: leading; gate/up: trailing)
  int n_routed_units;  // gate/up: leading routed grid units
  // gate/up: shared-expert down units after the routed ones (one token, when
  // h_shared is already in the workspace: the down kernel then has none)
  int n_sdown_units;
  const uint16_t* s_gate;
  const uint16_t* s_up;
  const uint16_t* s_down;
  float* h_route;   // [T*k][I]
  float* h_shared;  // [T][Is]
  float* o_route;   // [T*k][H]
  float* o_shared;  // [T][H]
  int32_t* status;
  int maxm;  // tokens staged per pass (1; the kernels also take 2)
  // the shared-expert units of K-decode-gu may start before the previous
  // kernel on the stream completes: set only when that kernel neither reads
  // nor writes h_shared (the layer's own sequence, where it is the
  // permutation or the gather)
  int shared_early;
  // combine in K-decode-down: per 128-row tile a counter (zero before the
  // launch, reset by the tile's last CTA) and the CTAs that count into it;
  // the last one writes y's columns of that tile.  comb_ctl == nullptr: off.
  unsigned int* comb_ctl;
  int comb_target;
  const int4* act_meta;  // per act_list position: {expert, slot, route, routes}, gscale row
  const int32_t* inv;
  uint16_t* y;
  // two launches, the down kernel's routed units started early: per act
  // position the gate/up units' count (h_ready, gu_units per expert) and the
  // count of down units that waited on it (h_seen, H/128 per expert; the last
  // one zeroes both).  nullptr: the down kernel waits for the whole gate/up
  // kernel.
  unsigned int* h_ready;
  unsigned int* h_seen;
  int gu_units;
  // K-decode-ffn (one launch): routed down units after the gate/up and
  // shared-down units, and its control words (ticket, done, shared h ready,
  // then one h-ready count per act position), zero before and after a launch
  int n_rdown_units;
  unsigned int* ffn_ctl;
  // the misses' records gathered inside K-decode-ffn (n_gather_workers > 0):
  // the leading tickets copy them from the mapped host arena, chunk by chunk
  // in miss order, and count the chunks of each miss as they land
  int n_gather_workers;
  const uint8_t* g_host;          // device address of the mapped host arena
  const int64_t* g_host_index;    // this layer's row: expert -> host record
  uint64_t g_host_records;
  const int32_t* g_miss_ids;      // the lookup's misses (ascending id)
  const int32_t* g_n_miss;
  const int32_t* g_dst_slots;     // adaptive cache: each miss's slot; nullptr: staging i mod S
  int g_n_cache, g_n_stage, g_slot_lo, g_slot_hi;
  int g_chunks;                   // chunks per record
};

constexpr int kFfnMaxPos = 1024;             // act positions (E <= 1024)
constexpr uint64_t kGatherChunkBytes = 256 * 1024;
constexpr int kGatherWorkers = 96;           // CTAs copying at once: the link, not the SMs, bounds them
constexpr int kGatherUnroll = 8;             // 16-byte loads in flight per worker thread

// An active expert of this group: its id, slot, first route position,
// number of routes and global scales.  From the compact record when the
// routing wrote one (a single round trip), else from act_list, src_slot,
// offsets and gscale.  False: position a is past the group's end.
struct ActExpert {
  int e, slot, pb, cnt;
  float g[3];
};
__device__ __forceinline__ void group_range(const DecodeParams& p, int& a0, int& a1);
__device__ __forceinline__ bool act_expert(const DecodeParams& p, int a, ActExpert& x) {
  int4 m0 = make_int4(0, 0, 0, 0), m1 = m0;
  if (p.act_meta && p.group == 0) {  // issued before the group's bounds are known
    m0 = p.act_meta[2 * a];
    m1 = p.act_meta[2 * a + 1];
  }
  int a0, a1;
  group_range(p, a0, a1);
  if (a0 + a >= a1) return false;
  if (p.act_meta) {
    if (p.group != 0) {
      m0 = p.act_meta[2 * (a0 + a)];
      m1 = p.act_meta[2 * (a0 + a) + 1];
    }
    x.e = m0.x; x.slot = m0.y; x.pb = m0.z; x.cnt = m0.w;
    x.g[0] = __int_as_float(m1.x); x.g[1] = __int_as_float(m1.y); x.g[2] = __int_as_float(m1.z);
    return true;
  }
  x.e = p.act_list[a0 + a];
  x.slot = (x.e >= 0 && x.e < p.E) ? p.src_slot[x.e] : -1;
  if (x.e >= 0 && x.e < p.E) {
    x.pb = p.offsets[x.e];
    x.cnt = p.offsets[x.e + 1] - x.pb;
    x.g[0] = p.gscale[x.e * 3 + 0];
    x.g[1] = p.gscale[x.e * 3 + 1];
    x.g[2] = p.gscale[x.e * 3 + 2];
  } else {
    x.pb = x.cnt = 0;
    x.g[0] = x.g[1] = x.g[2] = 0.f;
  }
  return true;
}

// act_list index range of this group
__device__ __forceinline__ void group_range(const DecodeParams& p, int& a0, int& a1) {
  const int n_act = p.n_act[0], n_hit = p.n_act[1], n_miss = n_act - n_hit;
  const int S = p.n_stage > 0 ? p.n_stage : (n_miss > 0 ? n_miss : 1);
  if (p.group == 0) {
    a0 = 0;
    a1 = n_hit + min(S, n_miss);
  } else {
    a0 = n_hit + p.group * S;
    a1 = n_hit + min((p.group + 1) * S, n_miss);
  }
}

// ---- staging ---------------------------------------------------------------
// Each thread issues the loads of up to kStageBatch of its elements before
// storing any of them, so that a CTA's staging costs about one round trip.
constexpr int kStageBatch = 8;

// Largest magnitude the f16 staging holds (f16's largest finite value): the
// decode FFN's products are f16 x f16, so an activation beyond it (or inf or
// NaN) is outside what the decode path computes.  The staging functions
// return true when a thread saw such a value; the kernel then sets
// MOE_ERR_UNSUPPORTED in the status word.
constexpr float kF16Max = 65504.f;
__device__ __forceinline__ bool f16_out_of_range(float a, float b) {
  return !(fabsf(a) <= kF16Max) || !(fabsf(b) <= kF16Max);
}

// f16 layout: row j, half-k-group hk (32 values) at (j*nhk + hk)*kHPad halves
__device__ __forceinline__ bool stage_bf16_to_f16(__half* xs, const uint16_t* const* rows, int m,
                                                  int K) {
  const int nhk = K / 32, n = K / 2;
  bool bad = false;
  for (int j = 0; j < m; ++j) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(rows[j]);
    __half* dst = xs + (size_t)j * nhk * kHPad;
    for (int i0 = threadIdx.x; i0 < n; i0 += kStageBatch * blockDim.x) {
      uint32_t v[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        v[u] = i < n ? __ldg(src + i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int e = 2 * (i0 + u * blockDim.x);
        if (e < K) {
          bad |= f16_out_of_range(bf16_lo(v[u]), bf16_hi(v[u]));
          *reinterpret_cast<__half2*>(dst + (e >> 5) * kHPad + (e & 31)) =
              __floats2half2_rn(bf16_lo(v[u]), bf16_hi(v[u]));
        }
      }
    }
  }
  return bad;
}

__device__ __forceinline__ bool stage_f32_to_f16(__half* xs, const float* const* rows, int m,
                                                 int K) {
  const int nhk = K / 32, n = K / 2;
  bool bad = false;
  for (int j = 0; j < m; ++j) {
    const float2* src = reinterpret_cast<const float2*>(rows[j]);
    __half* dst = xs + (size_t)j * nhk * kHPad;
    for (int i0 = threadIdx.x; i0 < n; i0 += kStageBatch * blockDim.x) {
      float2 v[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        v[u] = i < n ? src[i] : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int e = 2 * (i0 + u * blockDim.x);
        if (e < K) {
          bad |= f16_out_of_range(v[u].x, v[u].y);
          *reinterpret_cast<__half2*>(dst + (e >> 5) * kHPad + (e & 31)) =
              __floats2half2_rn(v[u].x, v[u].y);
        }
      }
    }
  }
  return bad;
}

// fp32 layout: row j, half-k-group hk at (j*nhk + hk)*kXPad floats
__device__ __forceinline__ void stage_bf16_to_f32(float* xs, const uint16_t* const* rows, int m,
                                                  int K) {
  const int nhk = K / 32, n = K / 2;
  for (int j = 0; j < m; ++j) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(rows[j]);
    float* dst = xs + (size_t)j * nhk * kXPad;
    for (int i0 = threadIdx.x; i0 < n; i0 += kStageBatch * blockDim.x) {
      uint32_t v[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        v[u] = i < n ? __ldg(src + i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int e = 2 * (i0 + u * blockDim.x);
        if (e < K) {
          dst[(e >> 5) * kXPad + (e & 31)] = bf16_lo(v[u]);
          dst[(e >> 5) * kXPad + (e & 31) + 1] = bf16_hi(v[u]);
        }
      }
    }
  }
}

__device__ __forceinline__ void stage_f32_to_f32(float* xs, const float* const* rows, int m,
                                                 int K) {
  const int nhk = K / 32, n = K / 4;
  for (int j = 0; j < m; ++j) {
    const float4* src = reinterpret_cast<const float4*>(rows[j]);
    float* dst = xs + (size_t)j * nhk * kXPad;
    for (int i0 = threadIdx.x; i0 < n; i0 += kStageBatch * blockDim.x) {
      float4 v[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * blockDim.x;
        v[u] = i < n ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int e = 4 * (i0 + u * blockDim.x);
        if (e < K) *reinterpret_cast<float4*>(dst + (e >> 5) * kXPad + (e & 31)) = v[u];
      }
    }
  }
}

// ---- FP4 x f16 dot products -------------------------------------------------
// a += w.lo * x.lo, b += w.hi * x.hi : f16 operands, exact products, fp32 sums
__device__ __forceinline__ void fma_h2(float& a, float& b, uint32_t w2, uint32_t x2) {
  asm("{\n .reg .b16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %2;\n mov.b32 {xl, xh}, %3;\n"
      " fma.rn.f32.f16 %0, wl, xl, %0;\n fma.rn.f32.f16 %1, wh, xh, %1;\n}"
      : "+f"(a), "+f"(b) : "r"(w2), "r"(x2));
}

// 32 E2M1 codes (16 bytes) of one row against M staged f16 vectors (16 f16x2
// registers each).  Codes 0..15 form the block with scale s0, 16..31 with s1.
template <int M>
__device__ __forceinline__ void fp4_dot32h(const uint4& c, float s0, float s1, const uint32_t* xh,
                                           float* acc) {
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    float pa[M], pb[M];
#pragma unroll
    for (int j = 0; j < M; ++j) pa[j] = pb[j] = 0.f;
#pragma unroll
    for (int q = 2 * blk; q < 2 * blk + 2; ++q) {
      uint32_t h[4];
      e2m1x8_to_f16x2x4(cw[q], h);
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int j = 0; j < M; ++j) fma_h2(pa[j], pb[j], h[b], xh[j * 16 + q * 4 + b]);
    }
    const float s = blk ? s1 : s0;
#pragma unroll
    for (int j = 0; j < M; ++j) acc[j] = fmaf(s, pa[j] + pb[j], acc[j]);
  }
}

// The two E4M3 scales of a lane's 32-value NVFP4 step hk of row m0 + 32 m1,
// from the 16-byte atom row a (the 4-byte word m1 holds that row's four block
// scales; the step's blocks of 16 are bytes 2 (hk & 1) and 2 (hk & 1) + 1).
// An MXFP4 step is one block of 32 whose E8M0 scale is byte hk & 3 (row_step).
__device__ __forceinline__ void scales_of(const uint4& a, int m1, int hk, float& s0, float& s1) {
  uint32_t wd = (m1 == 0) ? a.x : (m1 == 1) ? a.y : (m1 == 2) ? a.z : a.w;
  uint32_t h2 = e4m3x2_to_f16x2((wd >> (16 * (hk & 1))) & 0xFFFFu);
  s0 = f16_lo(h2);
  s1 = f16_hi(h2);
}

// byte offset, within a matrix's scales, of the atom row holding step hk of
// row tile rt, row m0 (K values per row)
template <int FMT>
__device__ __forceinline__ uint64_t step_atom_row(int rt, int hk, int m0, int K) {
  return FMT == MOE_FMT_MXFP4 ? atom_offset(rt, hk >> 2, K / 32) + (uint64_t)m0 * 16
                              : atom_offset(rt, hk >> 1, K / 16) + (uint64_t)m0 * 16;
}

// The same for an MXFP4 step: the 32 codes share one scale, applied once.
template <int M>
__device__ __forceinline__ void fp4_dot32h_mx(const uint4& c, float sc, const uint32_t* xh,
                                              float* acc) {
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  float pa[M], pb[M];
#pragma unroll
  for (int j = 0; j < M; ++j) pa[j] = pb[j] = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x2x4(cw[q], h);
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int j = 0; j < M; ++j) fma_h2(pa[j], pb[j], h[b], xh[j * 16 + q * 4 + b]);
  }
#pragma unroll
  for (int j = 0; j < M; ++j) acc[j] = fmaf(sc, pa[j] + pb[j], acc[j]);
}

// one row's step: dot products against the staged vectors, scaled per block
template <int M, int FMT>
__device__ __forceinline__ void row_step(const uint4& c, const uint4& atom_row, int m1, int hk,
                                         const uint32_t* xh, float* acc) {
  if (FMT == MOE_FMT_MXFP4) {
    const uint32_t wd = (m1 == 0) ? atom_row.x : (m1 == 1) ? atom_row.y
                      : (m1 == 2) ? atom_row.z : atom_row.w;
    fp4_dot32h_mx<M>(c, e8m0_value((wd >> (8 * (hk & 3))) & 0xFFu), xh, acc);
  } else {
    float s0, s1;
    scales_of(atom_row, m1, hk, s0, s1);
    fp4_dot32h<M>(c, s0, s1, xh, acc);
  }
}

template <int M>
__device__ __forceinline__ void load_xh(const __half* xs, int nhk, int hk, uint32_t* xh) {
#pragma unroll
  for (int j = 0; j < M; ++j) {
    const uint4* src = reinterpret_cast<const uint4*>(xs + ((size_t)j * nhk + hk) * kHPad);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 v = src[i];
      xh[j * 16 + 4 * i + 0] = v.x;
      xh[j * 16 + 4 * i + 1] = v.y;
      xh[j * 16 + 4 * i + 2] = v.z;
      xh[j * 16 + 4 * i + 3] = v.w;
    }
  }
}

// gate+up of the kGuRows rows {rt*128 + m0 + 32*(mo + m1)} of one expert, M
// staged tokens.  Returns warp-reduced sums (all lanes).
// One lane's 32-value step of a warp's gate and up rows: codes and the two
// scale atom rows (an atom row holds the scales of rows m0 + 32 i, i < 4).
struct GuRegs {
  uint4 g[kGuRows], u[kGuRows], sg, su;
};
template <int FMT>
__device__ __forceinline__ void gu_fetch(const uint8_t* rec, const RecordLayout& L, int H, int rt,
                                         int m0, int mo, int hk, GuRegs& r) {
  const uint8_t* gc = rec + L.gate_codes + (uint64_t)(rt * 128 + m0 + 32 * mo) * (H / 2);
  const uint8_t* uc = rec + L.up_codes + (uint64_t)(rt * 128 + m0 + 32 * mo) * (H / 2);
  const uint64_t rstride = (uint64_t)32 * (H / 2);
  const uint64_t aoff = step_atom_row<FMT>(rt, hk, m0, H);
  r.sg = ldg_stream(rec + L.gate_scales + aoff);
  r.su = ldg_stream(rec + L.up_scales + aoff);
#pragma unroll
  for (int m1 = 0; m1 < kGuRows; ++m1) {
    r.g[m1] = ldg_stream(gc + m1 * rstride + (uint64_t)hk * 16);
    r.u[m1] = ldg_stream(uc + m1 * rstride + (uint64_t)hk * 16);
  }
}

// `first` holds the step hk = lane, fetched by the caller (before it staged
// the tokens, so that those loads were already in flight).  The next step's
// loads are issued after this step's arithmetic, into the same registers: a
// second register set (loads issued before the arithmetic) needed more than
// the 128 registers a thread has at two CTAs per SM and spilled.
template <int M, int FMT>
__device__ void warp_gu_fp4(const uint8_t* rec, const RecordLayout& L, int H, int rt, int m0,
                            int mo, const __half* xs, float accg[kGuRows][M],
                            float accu[kGuRows][M], const GuRegs& first) {
  const int lane = threadIdx.x & 31;
  const int nhk = H / 32;
#pragma unroll
  for (int m1 = 0; m1 < kGuRows; ++m1)
#pragma unroll
    for (int j = 0; j < M; ++j) accg[m1][j] = accu[m1][j] = 0.f;
  uint4 cg[kGuRows], cu[kGuRows], sg = first.sg, su = first.su;
#pragma unroll
  for (int m1 = 0; m1 < kGuRows; ++m1) {
    cg[m1] = first.g[m1];
    cu[m1] = first.u[m1];
  }
  auto fetch = [&](int hk, uint4* g4, uint4* u4, uint4& sgv, uint4& suv) {
    GuRegs r;
    gu_fetch<FMT>(rec, L, H, rt, m0, mo, hk, r);
    sgv = r.sg;
    suv = r.su;
#pragma unroll
    for (int m1 = 0; m1 < kGuRows; ++m1) {
      g4[m1] = r.g[m1];
      u4[m1] = r.u[m1];
    }
  };
  for (int hk = lane; hk < nhk; hk += 32) {
    const bool more = hk + 32 < nhk;
    uint32_t xh[M * 16];
    load_xh<M>(xs, nhk, hk, xh);
#pragma unroll
    for (int m1 = 0; m1 < kGuRows; ++m1) {
      row_step<M, FMT>(cg[m1], sg, mo + m1, hk, xh, accg[m1]);
      row_step<M, FMT>(cu[m1], su, mo + m1, hk, xh, accu[m1]);
    }
    if (more) fetch(hk + 32, cg, cu, sg, su);
  }
#pragma unroll
  for (int m1 = 0; m1 < kGuRows; ++m1)
#pragma unroll
    for (int j = 0; j < M; ++j) {
      accg[m1][j] = warp_sum(accg[m1][j]);
      accu[m1][j] = warp_sum(accu[m1][j]);
    }
}

// ---- bf16 rows (shared expert) against fp32 staged vectors -----------------
template <int M>
__device__ __forceinline__ void bf16_dot8(const uint4& c, const float* xv, float* acc) {
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int j = 0; j < M; ++j) {
      acc[j] = fmaf(bf16_lo(cw[q]), xv[j * 8 + 2 * q], acc[j]);
      acc[j] = fmaf(bf16_hi(cw[q]), xv[j * 8 + 2 * q + 1], acc[j]);
    }
}

// NR rows over elements [k0, k1) of length-K rows: per-lane partial sums
template <int M, int NR>
__device__ void warp_rows_bf16(const uint16_t* const* rows, int K, int k0, int k1, const float* xs,
                               float acc[NR][M]) {
  const int lane = threadIdx.x & 31;
  const int nhk = K / 32;
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int j = 0; j < M; ++j) acc[r][j] = 0.f;
  for (int i0 = k0 + lane * 8; i0 < k1; i0 += 256) {
    uint4 c[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) c[r] = ldg_stream(rows[r] + i0);
    float xv[M * 8];
#pragma unroll
    for (int j = 0; j < M; ++j) {
      const float* src = xs + ((size_t)j * nhk + (i0 >> 5)) * kXPad + (i0 & 31);
      *reinterpret_cast<float4*>(xv + j * 8) = *reinterpret_cast<const float4*>(src);
      *reinterpret_cast<float4*>(xv + j * 8 + 4) = *reinterpret_cast<const float4*>(src + 4);
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) bf16_dot8<M>(c[r], xv, acc[r]);
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

// shared expert down: warp = 4 rows of s_down (r0..r0+3) over all of Is
template <int M>
__device__ void down_shared_pass(const DecodeParams& p, int r0, int t0, int mm, const float* hs) {
  const uint16_t* rows[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) rows[r] = p.s_down + (size_t)(r0 + r) * p.Is;
  float acc[4][M];
  warp_rows_bf16<M, 4>(rows, p.Is, 0, p.Is, hs, acc);
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int j = 0; j < M; ++j) {
      const float v = warp_sum(acc[r][j]);
      if (lane == r * M + j && j < mm) p.o_shared[(size_t)(t0 + j) * p.H + r0 + r] = v;
    }
}

// ---- bounded waits on counts that other CTAs raise ------------------------------
// Every wait is bounded (MOE_ERR_TIMEOUT in the status word).
constexpr uint64_t kFfnWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t gtimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// thread 0 waits for *c >= target, bounded; the CTA then reads what the
// counted units wrote (through L2)
__device__ __forceinline__ void cta_wait_count(const unsigned int* c, unsigned int target,
                                               int32_t* status) {
  if (threadIdx.x == 0) {
    const uint64_t t0 = gtimer_ns();
    while (ld_acquire(c) < target) {
      if (gtimer_ns() - t0 > kFfnWaitNs) {
        set_status(status, MOE_ERR_TIMEOUT);
        break;
      }
      __nanosleep(100);
    }
    __threadfence();
  }
  __syncthreads();
}
// the CTA's writes are visible before the count (called by every thread:
// each fences its own writes, then one thread counts)
__device__ __forceinline__ void cta_signal(unsigned int* c) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(c, 1u);
}


// ---- K-decode-gu -------------------------------------------------------------
template <int M, int FMT>
__device__ void gu_routed_pass(const DecodeParams& p, const RecordLayout& L, const uint8_t* rec,
                               int rt, int m0, int mo, int q0, int mm, const __half* xs,
                               float gg, float gu, const GuRegs& first) {
  float accg[kGuRows][M], accu[kGuRows][M];
  warp_gu_fp4<M, FMT>(rec, L, p.H, rt, m0, mo, xs, accg, accu, first);
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m1 = 0; m1 < kGuRows; ++m1)
#pragma unroll
    for (int j = 0; j < M; ++j)
      if (lane == m1 * M + j && j < mm) {
        const float g = accg[m1][j] * gg, u = accu[m1][j] * gu;
        p.h_route[(size_t)(q0 + j) * p.I + rt * 128 + m0 + 32 * (mo + m1)] = silu_f(g) * u;
      }
}

// shared expert: CTA = 4 row pairs (gate row i and up row i); warp = 1/8 of H
template <int M>
__device__ void gu_shared_pass(const DecodeParams& p, int i0, int t0, int mm, const float* xs,
                               float* red) {
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* rows[8];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    rows[r] = p.s_gate + (size_t)(i0 + r) * p.H;
    rows[4 + r] = p.s_up + (size_t)(i0 + r) * p.H;
  }
  const int kq = p.H / kSharedKSplit;
  float acc[8][M];
  warp_rows_bf16<M, 8>(rows, p.H, wid * kq, (wid + 1) * kq, xs, acc);
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int j = 0; j < M; ++j) {
      float v = warp_sum(acc[r][j]);
      if (lane == 0) red[(wid * 8 + r) * 2 + j] = v;
    }
  __syncthreads();
  // 4 pairs x mm tokens: thread -> (r, j); the 8 warps' parts in a fixed order
  const int t = threadIdx.x;
  if (t < 4 * 2) {
    const int r = t / 2, j = t % 2;
    if (j < mm) {
      float g = 0.f, u = 0.f;
      for (int w = 0; w < kSharedKSplit; ++w) {
        g += red[(w * 8 + r) * 2 + j];
        u += red[(w * 8 + 4 + r) * 2 + j];
      }
      p.h_shared[(size_t)(t0 + j) * p.Is + i0 + r] = silu_f(g) * u;
    }
  }
  __syncthreads();
}

// Grid: the routed units (one expert x one 128-row tile x a quarter of its
// 32 atom rows) first, then the shared-expert units (4 row pairs each), which
// are half as large and so fill the last wave.
template <int MAXM, int FMT>
__global__ void __launch_bounds__(kDecThreads, MAXM == 1 ? kGuMinBlocks : 1) k_decode_gu(DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ float red[kDecWarps * 8 * 2];
  const int wid = threadIdx.x >> 5;
  const int u = blockIdx.x;
  if (u >= p.n_routed_units && p.n_sdown_units > 0) {
    // shared down: h_shared was written by the kernel before this one
    pdl_wait();
    pdl_launch_dependents();
    float* hs = reinterpret_cast<float*>(smem_raw);
    const int r0 = (u - p.n_routed_units) * (kDecWarps * 4) + wid * 4;
    const float* row = p.h_shared;
    __syncthreads();
    stage_f32_to_f32(hs, &row, 1, p.Is);
    __syncthreads();
    if (r0 < p.H) down_shared_pass<1>(p, r0, 0, 1, hs);
    return;
  }
  if (u >= p.n_routed_units) {
    // the shared expert reads only x and its weights: in the layer's own
    // sequence it runs without waiting for the routing
    if (!p.shared_early) pdl_wait();
    pdl_launch_dependents();
    float* xs = reinterpret_cast<float*>(smem_raw);
    const int i0 = (u - p.n_routed_units) * 4;
    for (int t0 = 0; t0 < p.T; t0 += p.maxm) {
      const int mm = min(p.maxm, p.T - t0);
      const uint16_t* rows[2];
      for (int j = 0; j < mm; ++j) rows[j] = p.x + (size_t)(t0 + j) * p.H;
      __syncthreads();
      stage_bf16_to_f32(xs, rows, mm, p.H);
      __syncthreads();
      if (MAXM == 2 && mm == 2) gu_shared_pass<MAXM>(p, i0, t0, mm, xs, red);
      else gu_shared_pass<1>(p, i0, t0, mm, xs, red);
    }
    return;
  }
  pdl_wait();
  pdl_launch_dependents();
  __half* xs = reinterpret_cast<__half*>(smem_raw);
  const int ur = u;
  const int tiles = p.I / 128;
  const int a = ur / (tiles * kGuParts), rem = ur % (tiles * kGuParts);
  const int rt = rem / kGuParts, part = rem % kGuParts;
  const int m0 = (part & 3) * kDecWarps + wid, mo = (part >> 2) * kGuRows;
  ActExpert ax;
  if (!act_expert(p, a, ax)) return;
  const int slot = ax.slot;
  if (slot < 0 || slot >= p.n_slots) {
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }
  const uint8_t* rec = p.arena + (uint64_t)slot * p.rec_bytes;
  const RecordLayout L(p.H, p.I, FMT);
  const float gg = ax.g[0], gu = ax.g[1];
  const int pb = ax.pb, pe = ax.pb + ax.cnt;
  const int lane = threadIdx.x & 31;
  for (int q0 = pb; q0 < pe; q0 += p.maxm) {
    const int mm = min(p.maxm, pe - q0);
    GuRegs first;  // the weights' first step, in flight while the tokens are staged
    if (lane < p.H / 32) gu_fetch<FMT>(rec, L, p.H, rt, m0, mo, lane, first);
    const uint16_t* rows[2];
    for (int j = 0; j < mm; ++j) rows[j] = p.x + (size_t)(p.perm[q0 + j] / p.k) * p.H;
    __syncthreads();
    const bool bad = stage_bf16_to_f16(xs, rows, mm, p.H);
    if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(p.status, MOE_ERR_UNSUPPORTED);
    if (MAXM == 2 && mm == 2)
      gu_routed_pass<MAXM, FMT>(p, L, rec, rt, m0, mo, q0, mm, xs, gg, gu, first);
    else
      gu_routed_pass<1, FMT>(p, L, rec, rt, m0, mo, q0, mm, xs, gg, gu, first);
  }
  if (p.h_ready) cta_signal(&p.h_ready[a]);  // this unit's h rows are written
}

// ---- K-decode-down -----------------------------------------------------------
// routed: CTA = one 128-row tile of one expert; warp w owns m0 in {w, w+8, w+16, w+24}
template <int M, int FMT>
__device__ void down_routed_pass(const DecodeParams& p, const RecordLayout& L, const uint8_t* rec,
                                 int rt, int q0, int mm, const __half* hs, float gd) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nhk = p.I / 32;
  const uint8_t* dc = rec + L.down_codes;
  float acc[4][4][M];
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1)
#pragma unroll
      for (int j = 0; j < M; ++j) acc[g][m1][j] = 0.f;
  for (int hk = lane; hk < nhk; hk += 32) {
    uint4 cd[4][4], sd[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int m0 = wid + 8 * g;
      sd[g] = ldg_stream(rec + L.down_scales + step_atom_row<FMT>(rt, hk, m0, p.I));
#pragma unroll
      for (int m1 = 0; m1 < 4; ++m1)
        cd[g][m1] = ldg_stream(dc + (uint64_t)(rt * 128 + m0 + 32 * m1) * (p.I / 2) +
                               (uint64_t)hk * 16);
    }
    uint32_t xh[M * 16];
    load_xh<M>(hs, nhk, hk, xh);
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int m1 = 0; m1 < 4; ++m1) {
        row_step<M, FMT>(cd[g][m1], sd[g], m1, hk, xh, acc[g][m1]);
      }
  }
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1)
#pragma unroll
      for (int j = 0; j < M; ++j) {
        const float v = warp_sum(acc[g][m1][j]);
        if (lane == (g * 4 + m1) * M + j && j < mm) {
          const int r = p.perm[q0 + j];  // route t*k + j' -> its weight w[r]
          p.o_route[(size_t)(q0 + j) * p.H + rt * 128 + wid + 8 * g + 32 * m1] = p.w[r] * gd * v;
        }
      }
}

// y[t] for the columns of tile rt, summed in K-combine's order (routes j <
// k, then the shared expert) from the other CTAs' outputs, read through L2
__device__ void combine_tile(const DecodeParams& p, int rt) {
  const int c0 = rt * 128;
  for (int i = threadIdx.x; i < p.T * 32; i += blockDim.x) {
    const int t = i >> 5, c = c0 + (i & 31) * 4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < p.k; ++j) {
      const int pp = p.inv[t * p.k + j];
      if (pp < 0) continue;
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p.o_route + (size_t)pp * p.H + c));
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    if (p.o_shared) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p.o_shared + (size_t)t * p.H + c));
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    uint2 out;
    out.x = (uint32_t)f32_to_bf16_rne(s.x) | ((uint32_t)f32_to_bf16_rne(s.y) << 16);
    out.y = (uint32_t)f32_to_bf16_rne(s.z) | ((uint32_t)f32_to_bf16_rne(s.w) << 16);
    *reinterpret_cast<uint2*>(p.y + (size_t)t * p.H + c) = out;
  }
}

template <int MAXM, int FMT>
__device__ __forceinline__ void down_unit(const DecodeParams& p, unsigned char* smem_raw) {
  const int wid = threadIdx.x >> 5;
  const int u = blockIdx.x;
  if (u < p.n_shared_units) {
    float* hs = reinterpret_cast<float*>(smem_raw);
    const int r0 = u * (kDecWarps * 4) + wid * 4;
    for (int t0 = 0; t0 < p.T; t0 += p.maxm) {
      const int mm = min(p.maxm, p.T - t0);
      const float* rows[2];
      for (int j = 0; j < mm; ++j) rows[j] = p.h_shared + (size_t)(t0 + j) * p.Is;
      __syncthreads();
      stage_f32_to_f32(hs, rows, mm, p.Is);
      __syncthreads();
      if (r0 < p.H) {
        if (MAXM == 2 && mm == 2) down_shared_pass<MAXM>(p, r0, t0, mm, hs);
        else down_shared_pass<1>(p, r0, t0, mm, hs);
      }
    }
    return;
  }
  __half* hs = reinterpret_cast<__half*>(smem_raw);
  const int ur = u - p.n_shared_units;
  const int tiles = p.H / 128;
  const int a = ur / tiles, rt = ur % tiles;
  ActExpert ax;
  if (!act_expert(p, a, ax)) return;
  const int slot = ax.slot;
  if (slot < 0 || slot >= p.n_slots) return;  // reported by K-decode-gu
  if (p.h_ready) {
    // started before the gate/up kernel completed: wait for this expert's h
    cta_wait_count(&p.h_ready[a], (unsigned int)p.gu_units, p.status);
    if (threadIdx.x == 0 && atomicAdd(&p.h_seen[a], 1u) == (unsigned int)tiles - 1) {
      p.h_ready[a] = 0u;  // every unit of this expert is past its wait
      p.h_seen[a] = 0u;
    }
  }
  const uint8_t* rec = p.arena + (uint64_t)slot * p.rec_bytes;
  const RecordLayout L(p.H, p.I, FMT);
  const float gd = ax.g[2];
  const int pb = ax.pb, pe = ax.pb + ax.cnt;
  for (int q0 = pb; q0 < pe; q0 += p.maxm) {
    const int mm = min(p.maxm, pe - q0);
    const float* rows[2];
    for (int j = 0; j < mm; ++j) rows[j] = p.h_route + (size_t)(q0 + j) * p.I;
    __syncthreads();
    const bool bad = stage_f32_to_f16(hs, rows, mm, p.I);
    if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(p.status, MOE_ERR_UNSUPPORTED);
    if (MAXM == 2 && mm == 2) down_routed_pass<MAXM, FMT>(p, L, rec, rt, q0, mm, hs, gd);
    else down_routed_pass<1, FMT>(p, L, rec, rt, q0, mm, hs, gd);
  }
}

// one token: three CTAs per SM (at most 85 registers), so that the routed
// units (8 experts x 48 tiles) run in one wave
//
// With p.h_ready set, the routed units do not wait for the gate/up kernel as a
// whole: each waits for its own expert's h, and the grid waits for the kernel
// before it only ahead of the combine (which reads the shared expert's output
// from that kernel).  The routing they read first is complete: this kernel
// launches only when every CTA of the gate/up kernel has passed its own wait
// for the kernel before that (the host sets h_ready only when the gate/up
// kernel has no unit that skips that wait and this kernel has no shared units).
template <int MAXM, int FMT>
__global__ void __launch_bounds__(kDecThreads, MAXM == 1 ? 3 : 2) k_decode_down(DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_last;
  if (!p.h_ready) {
    pdl_wait();
    pdl_launch_dependents();
  }
  down_unit<MAXM, FMT>(p, smem_raw);
  if (p.h_ready) {
    pdl_wait();
    pdl_launch_dependents();
  }
  if (!p.comb_ctl) return;
  // shared units cover 32 rows each (4 per tile); routed units one tile
  const int u = blockIdx.x;
  const int rt = u < p.n_shared_units ? u / 4 : (u - p.n_shared_units) % (p.H / 128);
  __threadfence();  // this CTA's outputs are visible before it is counted
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.comb_ctl[rt], 1u) == (unsigned)p.comb_target - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  combine_tile(p, rt);
  if (threadIdx.x == 0) p.comb_ctl[rt] = 0u;  // ready for the next launch
}

// ---- K-combine ---------------------------------------------------------------
__global__ void k_combine(int T, int H, int k, const float* __restrict__ y_acc,
                          const float* __restrict__ o_route, const int32_t* __restrict__ inv,
                          const float* __restrict__ o_shared, uint16_t* __restrict__ y) {
  const int n4 = H / 4;
  pdl_wait();
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * n4; i += gridDim.x * blockDim.x) {
    const int t = i / n4, c = (i % n4) * 4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (y_acc) s = *reinterpret_cast<const float4*>(y_acc + (size_t)t * H + c);
    if (o_route) {
      for (int j = 0; j < k; ++j) {
        const int pp = inv[t * k + j];
        if (pp < 0) continue;
        float4 v = *reinterpret_cast<const float4*>(o_route + (size_t)pp * H + c);
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
      }
    }
    if (o_shared) {
      float4 v = *reinterpret_cast<const float4*>(o_shared + (size_t)t * H + c);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    uint2 out;
    out.x = (uint32_t)f32_to_bf16_rne(s.x) | ((uint32_t)f32_to_bf16_rne(s.y) << 16);
    out.y = (uint32_t)f32_to_bf16_rne(s.z) | ((uint32_t)f32_to_bf16_rne(s.w) << 16);
    *reinterpret_cast<uint2*>(y + (size_t)t * H + c) = out;
  }
}

// ---- K-decode-ffn: gate/up, down and the combine in one launch ----------------
// The units of both steps run as one grid.  A CTA takes its unit from a ticket
// counter, not from blockIdx: tickets are handed out in order, so a unit that
// waits only ever waits for units with earlier tickets, which CTAs already
// running hold - every wait ends.  Ticket order: the shared expert's gate/up
// units (when its h is not ready yet), the routed gate/up units expert by
// expert, the shared expert's down units, the routed down units expert by
// expert.  A routed down unit of act position a starts when all gate/up units
// of a have written their h (a count per position); a shared down unit when
// the shared gate/up units have.  So the down units of the first experts
// stream their weights while the gate/up units of the last ones still run,
// and the grid has one tail instead of two.  The combine is done by the last
// CTA of each 128-row tile, as in K-decode-down.  The last CTA to finish
// resets the control words for the next launch.
// one routed down unit (expert at act position a, 128-row tile rt), after
// its h is complete
template <int FMT>
__device__ __forceinline__ void ffn_down_routed(const DecodeParams& p, int a, int rt,
                                                unsigned char* smem_raw, int gu_units) {
  ActExpert ax;
  if (!act_expert(p, a, ax)) return;
  const int slot = ax.slot;
  if (slot < 0 || slot >= p.n_slots) return;  // reported by its gate/up units
  cta_wait_count(p.ffn_ctl + 4 + a, (unsigned int)gu_units, p.status);
  __half* hs = reinterpret_cast<__half*>(smem_raw);
  const uint8_t* rec = p.arena + (uint64_t)slot * p.rec_bytes;
  const RecordLayout L(p.H, p.I, FMT);
  for (int q0 = ax.pb; q0 < ax.pb + ax.cnt; ++q0) {
    const float* row = p.h_route + (size_t)q0 * p.I;
    __syncthreads();
    const bool bad = stage_f32_to_f16(hs, &row, 1, p.I);
    if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(p.status, MOE_ERR_UNSUPPORTED);
    down_routed_pass<1, FMT>(p, L, rec, rt, q0, 1, hs, ax.g[2]);
  }
}

// One gather worker: takes chunks (miss i, part c) from a counter in miss
// order and copies each with 16-byte loads of the mapped host record, then
// counts it in landed[i].  A miss whose record or slot is missing sets
// MOE_ERR_DEVICE and is counted as landed (its experts' outputs are then
// undefined), so that no unit waits for it.
__device__ void ffn_gather_worker(const DecodeParams& p, unsigned int* ctl, unsigned int* landed) {
  __shared__ unsigned int s_c;
  const int n_miss = *p.g_n_miss;
  const uint64_t total = (uint64_t)n_miss * (uint64_t)p.g_chunks;
  const uint64_t rb = p.rec_bytes;
  for (;;) {
    __syncthreads();
    if (threadIdx.x == 0) s_c = atomicAdd(&ctl[3], 1u);
    __syncthreads();
    const uint64_t c = s_c;
    if (c >= total) break;
    const int i = (int)(c / (uint64_t)p.g_chunks);
    const uint64_t part = c % (uint64_t)p.g_chunks;
    const int e = p.g_miss_ids[i];
    const int64_t hr = (e >= 0 && e < p.E && p.g_host_index) ? p.g_host_index[e] : -1;
    int slot;
    if (p.g_dst_slots) {
      slot = p.g_dst_slots[i];
      const bool staging = p.g_n_stage > 0 && slot >= p.g_n_cache && slot < p.g_n_cache + p.g_n_stage;
      if (!staging && (slot < p.g_slot_lo || slot >= p.g_slot_hi)) slot = -1;
    } else {
      slot = p.g_n_stage > 0 ? p.g_n_cache + (i % p.g_n_stage) : -1;
    }
    if (hr < 0 || (uint64_t)hr >= p.g_host_records || !p.g_host || slot < 0) {
      if (threadIdx.x == 0 && part == 0) set_status(p.status, MOE_ERR_DEVICE);
    } else {
      const uint64_t b0 = part * kGatherChunkBytes;
      const uint64_t b1 = min(rb, b0 + kGatherChunkBytes);
      const uint4* s4 = reinterpret_cast<const uint4*>(p.g_host + (uint64_t)hr * rb + b0);
      uint4* d4 = reinterpret_cast<uint4*>(const_cast<uint8_t*>(p.arena) + (uint64_t)slot * rb + b0);
      const uint64_t n16 = (b1 - b0) / 16;
      constexpr int kU = kGatherUnroll;  // 16-byte loads in flight per thread
      uint64_t w = threadIdx.x;
      for (; w + (kU - 1) * kDecThreads < n16; w += kU * kDecThreads) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = ldg_stream(s4 + w + u * kDecThreads);
#pragma unroll
        for (int u = 0; u < kU; ++u) d4[w + u * kDecThreads] = v[u];
      }
      for (; w < n16; w += kDecThreads) d4[w] = ldg_stream(s4 + w);
    }
    cta_signal(&landed[i]);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kDecThreads, 2) k_decode_ffn(DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ float red[kDecWarps * 8 * 2];
  __shared__ unsigned int s_ticket;
  __shared__ int s_last;
  unsigned int* ctl = p.ffn_ctl;
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) s_ticket = atomicAdd(&ctl[0], 1u);
  __syncthreads();
  const int wid = threadIdx.x >> 5;
  const int n_gw = p.n_gather_workers;
  const int n_sgu = p.n_shared_units, n_rgu = p.n_routed_units;
  const int n_sd = p.n_sdown_units, n_rd = p.n_rdown_units;
  const int gu_units = (p.I / 128) * kGuParts;  // gate/up units of one expert
  const int tiles = p.H / 128;           // down units of one expert
  unsigned int* h_ready = ctl + 4;
  unsigned int* landed = ctl + 4 + kFfnMaxPos;
  int tile = -1;                         // the 128-row tile a down unit adds to
  // With the gather inside, the hits' whole FFN comes before the misses':
  // gate/up (hits) | shared down | down (hits) | gate/up (misses) | down
  // (misses), so that no unit waiting for a record holds an SM the hits need.
  // Unit (phase, position) of this ticket:
  int t = (int)s_ticket - n_gw;
  int gu_a = -1, gu_r = 0, dn_a = -1, dn_rt = 0, sd_u = -1;
  if ((int)s_ticket < n_gw) {
    ffn_gather_worker(p, ctl, landed);
  } else if (t < n_sgu) {
    // handled below
  } else if (n_gw > 0) {
    const int n_hit = p.n_act[1];
    const int max_act = n_rgu / gu_units;
    t -= n_sgu;
    if (t < n_hit * gu_units) {
      gu_a = t / gu_units;
      gu_r = t % gu_units;
    } else if ((t -= n_hit * gu_units) < n_sd) {
      sd_u = t;
    } else if ((t -= n_sd) < n_hit * tiles) {
      dn_a = t / tiles;
      dn_rt = t % tiles;
    } else if ((t -= n_hit * tiles) < (max_act - n_hit) * gu_units) {
      gu_a = n_hit + t / gu_units;
      gu_r = t % gu_units;
    } else {
      t -= (max_act - n_hit) * gu_units;
      dn_a = n_hit + t / tiles;
      dn_rt = t % tiles;
    }
    t = -1;
  } else {
    t -= n_sgu;
    if (t < n_rgu) {
      gu_a = t / gu_units;
      gu_r = t % gu_units;
    } else if ((t -= n_rgu) < n_sd) sd_u = t;
    else if ((t -= n_sd) < n_rd) {
      dn_a = t / tiles;
      dn_rt = t % tiles;
    }
    t = -1;
  }
  if (t >= 0 && t < n_sgu) {
    // shared gate/up: 4 row pairs
    float* xs = reinterpret_cast<float*>(smem_raw);
    for (int t0 = 0; t0 < p.T; ++t0) {
      const uint16_t* row = p.x + (size_t)t0 * p.H;
      __syncthreads();
      stage_bf16_to_f32(xs, &row, 1, p.H);
      __syncthreads();
      gu_shared_pass<1>(p, t * 4, t0, 1, xs, red);
    }
    cta_signal(&ctl[2]);
  } else if (gu_a >= 0) {
    // routed gate/up: expert at act position a, tile rt, part of its rows
    const int a = gu_a;
    const int rt = gu_r / kGuParts, part = gu_r % kGuParts;
    const int m0 = (part & 3) * kDecWarps + wid, mo = (part >> 2) * kGuRows;
    ActExpert ax;
    if (act_expert(p, a, ax)) {
      // a miss gathered by this launch: wait until its record has landed
      if (n_gw > 0 && a >= p.n_act[1])
        cta_wait_count(&landed[a - p.n_act[1]], (unsigned int)p.g_chunks, p.status);
      const int slot = ax.slot;
      if (slot < 0 || slot >= p.n_slots) {
        if (threadIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
      } else {
        __half* xs = reinterpret_cast<__half*>(smem_raw);
        const uint8_t* rec = p.arena + (uint64_t)slot * p.rec_bytes;
        const RecordLayout L(p.H, p.I, FMT);
        const int lane = threadIdx.x & 31;
        for (int q0 = ax.pb; q0 < ax.pb + ax.cnt; ++q0) {
          GuRegs first;  // the weights' first step, in flight while the token is staged
          if (lane < p.H / 32) gu_fetch<FMT>(rec, L, p.H, rt, m0, mo, lane, first);
          const uint16_t* row = p.x + (size_t)(p.perm[q0] / p.k) * p.H;
          __syncthreads();
          const bool bad = stage_bf16_to_f16(xs, &row, 1, p.H);
          if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(p.status, MOE_ERR_UNSUPPORTED);
          gu_routed_pass<1, FMT>(p, L, rec, rt, m0, mo, q0, 1, xs, ax.g[0], ax.g[1], first);
        }
      }
    }
    cta_signal(&h_ready[a]);
  } else if (sd_u >= 0) {
    // shared down: 32 rows of H over all of Is
    const int u = sd_u;
    if (n_sgu > 0) cta_wait_count(&ctl[2], (unsigned int)n_sgu, p.status);
    float* hs = reinterpret_cast<float*>(smem_raw);
    const int r0 = u * (kDecWarps * 4) + wid * 4;
    for (int t0 = 0; t0 < p.T; ++t0) {
      const float* row = p.h_shared + (size_t)t0 * p.Is;
      __syncthreads();
      stage_f32_to_f32(hs, &row, 1, p.Is);
      __syncthreads();
      if (r0 < p.H) down_shared_pass<1>(p, r0, t0, 1, hs);
    }
    tile = u / 4;
  } else if (dn_a >= 0) {
    tile = dn_rt;
    ffn_down_routed<FMT>(p, dn_a, tile, smem_raw, gu_units);
  }
  // combine: the last CTA of a 128-row tile sums its columns into y
  if (p.comb_ctl && tile >= 0) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      s_last = atomicAdd(&p.comb_ctl[tile], 1u) == (unsigned)p.comb_target - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      combine_tile(p, tile);
      if (threadIdx.x == 0) p.comb_ctl[tile] = 0u;
    }
  }
  // the last CTA resets the control words (every other CTA is done with them)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&ctl[1], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last) {
    const int n_pos = n_rgu / gu_units;
    for (int i = threadIdx.x; i < 4 + n_pos; i += blockDim.x) ctl[i] = 0u;
    if (n_gw > 0)
      for (int i = threadIdx.x; i < n_pos; i += blockDim.x) landed[i] = 0u;
  }
}

// ---- host launchers -----------------------------------------------------------
size_t decode_workspace_bytes(int T, int I, int k, int Is) {
  return ((size_t)T * k * I + (size_t)T * Is) * sizeof(float) + 256;
}

static size_t smem_f16(int maxm, int K) { return (size_t)maxm * (K / 32) * kHPad * sizeof(__half); }
static size_t smem_f32(int maxm, int K) { return (size_t)maxm * (K / 32) * kXPad * sizeof(float); }

moe_status decode_ffn(const moe_ffn_args* a, cudaStream_t s, const DecodeFuse& fz) {
  DecodeParams p;
  p.n_rdown_units = 0;
  p.ffn_ctl = nullptr;
  p.h_ready = p.h_seen = nullptr;
  p.gu_units = (a->I / 128) * kGuParts;
  p.n_gather_workers = 0;
  p.g_host = nullptr;
  p.g_host_index = nullptr;
  p.g_host_records = 0;
  p.g_miss_ids = p.g_n_miss = p.g_dst_slots = nullptr;
  p.g_n_cache = p.g_n_stage = p.g_slot_lo = p.g_slot_hi = p.g_chunks = 0;
  p.shared_early = fz.shared_early ? 1 : 0;
  p.comb_ctl = nullptr;
  p.comb_target = 0;
  p.act_meta = fz.act_meta;
  p.inv = fz.inv;
  p.y = fz.y;
  p.T = a->T; p.H = a->H; p.I = a->I; p.E = a->E; p.k = a->k; p.Is = a->Is;
  p.x = (const uint16_t*)a->x;
  p.arena = cache_arena(a->cache);
  p.rec_bytes = cache_rec_bytes(a->cache);
  const bool mx = cache_format(a->cache) == MOE_FMT_MXFP4;
  p.n_slots = cache_n_cache(a->cache) + cache_n_stage(a->cache);
  p.gscale = a->gscale; p.src_slot = a->src_slot; p.act_list = a->act_list; p.n_act = a->n_act;
  p.offsets = a->offsets; p.perm = a->perm; p.w = a->w;
  p.n_sdown_units = 0;
  p.group = a->group;
  p.n_stage = a->n_stage;
  p.s_gate = (const uint16_t*)a->s_gate; p.s_up = (const uint16_t*)a->s_up;
  p.s_down = (const uint16_t*)a->s_down;
  float* ws = (float*)a->workspace;
  p.h_route = ws;
  p.h_shared = ws + (size_t)a->T * a->k * a->I;
  p.o_route = a->o_route;
  p.o_shared = a->o_shared;
  p.status = a->status;
  // One token per pass: a unit with several routes reads its weight rows again
  // for each, from L2, at two CTAs per SM.  Two tokens per pass needed 255
  // registers (one CTA per SM) and measured slower at every token count on an
  // all-resident 6144 x 2048 layer: 2 tokens 157 against 134 us, 8 tokens 499
  // against 382 us, 64 tokens 3.36 against 2.88 ms.
  p.maxm = 1;
  // experts this group can hold at most
  int max_act = a->T * a->k < a->E ? a->T * a->k : a->E;
  if (a->group > 0) max_act = a->n_stage < max_act ? a->n_stage : max_act;
  bool shared = a->group == 0 && a->Is > 0;
  if (fz.ffn_ctl && a->stages == MOE_STAGE_ALL) {
    // one launch: gate/up, down and (one group) the combine
    p.ffn_ctl = fz.ffn_ctl;
    p.n_shared_units = (shared && !fz.shared_gu_done) ? a->Is / 4 : 0;
    p.n_routed_units = max_act * (a->I / 128) * kGuParts;
    p.n_sdown_units = shared ? (a->H + kDecWarps * 4 - 1) / (kDecWarps * 4) : 0;
    p.n_rdown_units = max_act * (a->H / 128);
    if (fz.g_cache && a->group == 0) {
      GatherArgs ga;
      cache_gather_args(fz.g_cache, fz.g_layer, &ga);
      p.n_gather_workers = kGatherWorkers;
      p.g_host = ga.host;
      p.g_host_index = ga.host_index;
      p.g_host_records = ga.host_records;
      p.g_miss_ids = fz.g_miss_ids;
      p.g_n_miss = fz.g_n_miss;
      p.g_dst_slots = fz.g_dst_slots;
      p.g_n_cache = ga.n_cache;
      p.g_n_stage = ga.n_stage;
      p.g_slot_lo = ga.slot_lo;
      p.g_slot_hi = ga.slot_hi;
      p.g_chunks = (int)((p.rec_bytes + kGatherChunkBytes - 1) / kGatherChunkBytes);
    }
    size_t smem = smem_f16(1, a->H);
    if (p.n_shared_units && smem_f32(1, a->H) > smem) smem = smem_f32(1, a->H);
    if (shared && smem_f32(1, a->Is) > smem) smem = smem_f32(1, a->Is);
    if (fz.comb_ctl && fz.inv && fz.y && (!a->Is || a->o_shared)) {
      p.comb_ctl = fz.comb_ctl;
      p.comb_target = max_act + (shared ? 4 : 0);  // CTAs per 128-row tile
    }
    const int grid = p.n_gather_workers + p.n_shared_units + p.n_routed_units + p.n_sdown_units +
                     p.n_rdown_units;
    if (grid > 0) {
      auto* kern = mx ? k_decode_ffn<MOE_FMT_MXFP4> : k_decode_ffn<MOE_FMT_NVFP4>;
      if (launch_pdl(kern, grid, kDecThreads, smem, s, p) != cudaSuccess) return MOE_ERR_CUDA;
      if (fz.mark) fz.mark(fz.mark_ctx);
    }
    return MOE_OK;
  }
  // down units started per expert: both steps in this call, no shared-expert
  // gate/up units in the gate/up kernel (they may skip its wait), and the
  // shared down (if any) in the gate/up kernel, not in the down kernel
  if (fz.h_counts && (a->stages & MOE_STAGE_GATE_UP) && (a->stages & MOE_STAGE_DOWN) &&
      max_act <= kFfnMaxPos &&
      (!shared || (fz.shared_gu_done && a->T == 1))) {
    p.h_ready = fz.h_counts;
    p.h_seen = fz.h_counts + kFfnMaxPos;
  }
  if (a->stages & MOE_STAGE_GATE_UP) {
    p.n_shared_units = (shared && !fz.shared_gu_done) ? a->Is / 4 : 0;
    p.n_sdown_units = (shared && fz.shared_gu_done && a->T == 1 && (a->stages & MOE_STAGE_DOWN))
                          ? (a->H + kDecWarps * 4 - 1) / (kDecWarps * 4) : 0;
    const int routed = max_act * (a->I / 128) * kGuParts;
    p.n_routed_units = routed;
    size_t smem = smem_f16(p.maxm, a->H);
    if (p.n_shared_units && smem_f32(p.maxm, a->H) > smem) smem = smem_f32(p.maxm, a->H);
    if (p.n_sdown_units && smem_f32(1, a->Is) > smem) smem = smem_f32(1, a->Is);
    const int grid = p.n_shared_units + p.n_sdown_units + routed;
    if (grid > 0) {
      auto* kern = mx ? k_decode_gu<1, MOE_FMT_MXFP4> : k_decode_gu<1, MOE_FMT_NVFP4>;
      if (launch_pdl(kern, grid, kDecThreads, smem, s, p) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (fz.mark) fz.mark(fz.mark_ctx);
    }
  }
  if (a->stages & MOE_STAGE_DOWN) {
    const bool sdown_done = p.n_sdown_units > 0;  // in the gate/up kernel above
    if (sdown_done) shared = false;
    p.n_shared_units = shared ? (a->H + kDecWarps * 4 - 1) / (kDecWarps * 4) : 0;
    const int routed = max_act * (a->H / 128);
    size_t smem = smem_f16(p.maxm, a->I);
    if (shared && smem_f32(p.maxm, a->Is) > smem) smem = smem_f32(p.maxm, a->Is);
    const int grid = p.n_shared_units + routed;
    if (fz.comb_ctl && fz.inv && fz.y && (!a->Is || a->o_shared)) {
      p.comb_ctl = fz.comb_ctl;
      p.comb_target = max_act + (shared ? 4 : 0);  // CTAs per 128-row tile
    }
    if (grid > 0) {
      auto* kern = mx ? k_decode_down<1, MOE_FMT_MXFP4> : k_decode_down<1, MOE_FMT_NVFP4>;
      if (launch_pdl(kern, grid, kDecThreads, smem, s, p) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (fz.mark) fz.mark(fz.mark_ctx);
    }
  }
  return MOE_OK;
}

moe_status decode_setup() {
  // H up to 16384 with two staged tokens in fp32: 2 * 512 * 36 * 4 bytes
  const void* fns[6] = {(const void*)k_decode_gu<1, MOE_FMT_NVFP4>,
                        (const void*)k_decode_down<1, MOE_FMT_NVFP4>,
                        (const void*)k_decode_gu<1, MOE_FMT_MXFP4>,
                        (const void*)k_decode_down<1, MOE_FMT_MXFP4>,
                        (const void*)k_decode_ffn<MOE_FMT_NVFP4>,
                        (const void*)k_decode_ffn<MOE_FMT_MXFP4>};
  for (const void* f : fns)
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

MOE_API moe_status moe_combine(const moe_combine_args* a, void* stream) {
  if (!a || !a->y || a->T < 0 || a->H <= 0 || a->k <= 0) return MOE_ERR_INVALID_ARG;
  if (a->o_route && !a->inv) return MOE_ERR_INVALID_ARG;
  if (a->H % 4) return MOE_ERR_UNSUPPORTED;
  if (a->T == 0) return MOE_OK;
  long long n = (long long)a->T * (a->H / 4);
  int grid = (int)((n + 255) / 256);
  if (grid > kSMs * 16) grid = kSMs * 16;
  if (launch_pdl(k_combine, grid, 256, 0, (cudaStream_t)stream, a->T, a->H, a->k, a->y_acc,
                 a->o_route, a->inv, a->o_shared, (uint16_t*)a->y) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
