// route.cu - K-route: router logits (fp32), softmax, top-k and renormalised
// weights.  The router is the device-side router of the "Project Maya" page
// ("Three tiers and the rules between them"): fp32 router weights, top-8 of
// 288 experts per token, selection kept on the device.
#include "permute_body.cuh"
#include "policy_body.cuh"

namespace moe {

// ---- logits for few tokens: one CTA per expert row -------------------------
// Each thread accumulates its strided slice of the row (fixed order), then a
// fixed-shape tree reduction: deterministic.
constexpr int kGemvMaxT = 8;

__device__ __forceinline__ void logits_of_expert(const uint16_t* __restrict__ x,
                                                 const float* __restrict__ wr,
                                                 const float* __restrict__ bias, int T, int H,
                                                 int E, int e, float* __restrict__ logits) {
  const float4* wrow = reinterpret_cast<const float4*>(wr + (size_t)e * H);
  float acc[kGemvMaxT];
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) acc[t] = 0.f;
  for (int i = threadIdx.x; i < H / 4; i += blockDim.x) {
    float4 w = __ldg(wrow + i);
#pragma unroll
    for (int t = 0; t < kGemvMaxT; ++t) {
      if (t < T) {
        uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)t * H) + i);
        float a = acc[t];
        a = fmaf(w.x, bf16_lo(xv.x), a);
        a = fmaf(w.y, bf16_hi(xv.x), a);
        a = fmaf(w.z, bf16_lo(xv.y), a);
        a = fmaf(w.w, bf16_hi(xv.y), a);
        acc[t] = a;
      }
    }
  }
  __shared__ float red[kGemvMaxT][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) {
    if (t < T) {
      float v = warp_sum(acc[t]);
      if (lane == 0) red[t][wid] = v;
    }
  }
  __syncthreads();
  if (threadIdx.x < T) {
    const int t = threadIdx.x;
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[t][w];
    if (bias) s += bias[e];
    logits[(size_t)t * E + e] = s;
  }
}

// CTA (e, g): expert e's logits of tokens [8 g, 8 g + 8), its router row
// read once per token group (from L2 after the first group)
__global__ void __launch_bounds__(256) k_logits_gemv(const uint16_t* __restrict__ x,
                                                     const float* __restrict__ wr,
                                                     const float* __restrict__ bias, int T,
                                                     int H, int E, float* __restrict__ logits) {
  pdl_wait();
  pdl_launch_dependents();
  const int t0 = blockIdx.y * kGemvMaxT;
  logits_of_expert(x + (size_t)t0 * H, wr, bias, min(kGemvMaxT, T - t0), H, E, blockIdx.x,
                   logits + (size_t)t0 * E);
}

// Up to this many tokens the router runs as token groups of the GEMV above
// (E x T/8 CTAs); the tiled GEMM below has only E/32 x T/128 tiles, under one
// wave of the 152 SMs until about 2048 tokens (64 tokens: 9 CTAs, 291 us;
// the GEMV reads x from L2 once per expert, which costs more from about 1024)
constexpr int kGemvGroupsMaxT = 1024;

// ---- logits for many tokens: SIMT tiled GEMM --------------------------------
// Tile 128 tokens x 32 experts, 128 threads, 8 tokens x 4 experts each, K
// chunks of 32.  The FMAs are packed pairs (fma.rn.f32x2 over two tokens and
// one weight; each lane rounds as a scalar fmaf would).  Shared memory holds
// x as bf16 words of two tokens at one k and W as fp32, so one 16-byte load
// gives a thread its 8 tokens (the same address across each quarter-warp)
// and one its 4 weights: six shared-memory wavefronts per 1024 FMAs of a
// warp.  Each chunk's partial sum is added to the running total with Kahan
// compensation (packed adds), keeping the fp32 error of the 6144-term dot
// products near that of the chunk sums (the router probabilities are
// compared at 1e-5).  Shared memory is double-buffered: the next chunk's
// global loads are issued before the current chunk's FMAs and stored into
// the other buffer after them, one barrier per chunk.  288 experts = 9 tiles:
// 288 CTAs for 4096 tokens, two per SM on most SMs, all resident at once.
constexpr int kTM = 128, kTN = 32, kTK = 32, kGemmThreads = 128;
constexpr int kXsLd = kTM / 2 + 4, kWsLd = kTN + 4;  // 32-bit words per shared row

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}
// shared-tile column swizzles of the router GEMM: multiples of 8 (x words)
// and of 4 (weights) keep each thread's 16-byte group contiguous
__device__ __forceinline__ int xs_swz(int kk) { return ((kk >> 3) & 3) << 3; }
__device__ __forceinline__ int ws_swz(int kk) { return ((kk >> 3) & 3) << 2; }
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  return (uint64_t)lo | ((uint64_t)hi << 32);
}

__global__ void __launch_bounds__(kGemmThreads) k_logits_gemm(const uint16_t* __restrict__ x,
                                                              const float* __restrict__ wr,
                                                              const float* __restrict__ bias,
                                                              int T, int H, int E,
                                                              float* __restrict__ logits) {
  // xs[b][kk][p] = x[t0 + 2p][k0 + kk] | x[t0 + 2p + 1][k0 + kk] << 16 (bf16 bits)
  __shared__ __align__(16) uint32_t xs[2][kTK][kXsLd];
  __shared__ __align__(16) float ws[2][kTK][kWsLd];  // ws[b][kk][c] = w[e0 + c][k0 + kk]
  pdl_wait();
  pdl_launch_dependents();
  const int t0 = blockIdx.y * kTM, e0 = blockIdx.x * kTN;
  const int tid = threadIdx.x;
  const int tx = tid & 7, ty = tid >> 3;  // tokens ty*8.., experts tx*4..
  // Load roles, each warp instruction reading whole 64- or 128-byte row
  // pieces: x: row pair q = tid/4 (+32), 16-byte piece xc = tid % 4 (k =
  // 8 xc..); W: expert we = tid/8 (+16), piece wc = tid % 8 (k = 4 wc..).
  // The next chunk's loads are ordered before this chunk's shared-memory
  // reads (a memory clobber), so they are in flight during its FMAs; rows past
  // T and experts past E read row 0 and are zeroed when staged.  Stores are
  // swizzled (columns XORed by a function of k) so that they hit 32 banks.
  const int xq = tid >> 2, xc = tid & 3, we = tid >> 3, wc = tid & 7;
  const uint4* xsrc[4];
  bool xok[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {  // rows 2(xq + 32(r/2)) + r%2
    const int t = t0 + 2 * (xq + 32 * (r >> 1)) + (r & 1);
    xok[r] = t < T;
    xsrc[r] = reinterpret_cast<const uint4*>(x + (size_t)(xok[r] ? t : 0) * H + xc * 8);
  }
  const uint4* wsrc[2];
  bool wok[2];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int e = e0 + we + 16 * m;
    wok[m] = e < E;
    wsrc[m] = reinterpret_cast<const uint4*>(wr + (size_t)(wok[m] ? e : 0) * H + wc * 4);
  }
  uint4 xv4[4], wv4[2];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) xv4[r] = ldg_nc_v4(xsrc[r] + k0 / 8);
#pragma unroll
    for (int m = 0; m < 2; ++m) wv4[m] = ldg_nc_v4(wsrc[m] + k0 / 4);
  };
  auto stage = [&](int buf) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const uint4 lo4 = xv4[2 * g], hi4 = xv4[2 * g + 1];
      const bool ok0 = xok[2 * g], ok1 = xok[2 * g + 1];
      const uint32_t a[4] = {ok0 ? lo4.x : 0u, ok0 ? lo4.y : 0u, ok0 ? lo4.z : 0u,
                             ok0 ? lo4.w : 0u};
      const uint32_t c[4] = {ok1 ? hi4.x : 0u, ok1 ? hi4.y : 0u, ok1 ? hi4.z : 0u,
                             ok1 ? hi4.w : 0u};
      const int q = xq + 32 * g;
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // word j holds k = 2j (low half), 2j + 1
        const int kk = xc * 8 + 2 * j;
        xs[buf][kk][q ^ xs_swz(kk)] = __byte_perm(a[j], c[j], 0x5410);
        xs[buf][kk + 1][q ^ xs_swz(kk + 1)] = __byte_perm(a[j], c[j], 0x7632);
      }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t w4[4] = {wv4[m].x, wv4[m].y, wv4[m].z, wv4[m].w};
      const int e = we + 16 * m;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kk = wc * 4 + i;
        ws[buf][kk][e ^ ws_swz(kk)] = __uint_as_float(wok[m] ? w4[i] : 0u);
      }
    }
  };
  // pairs: [q][j] = tokens ty*8 + 2q (low) and + 2q + 1 (high), expert tx*4 + j
  uint64_t acc[4][4], cmp[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = cmp[i][j] = 0ull;
  const int nch = H / kTK;
  fetch(0);
  stage(0);
  __syncthreads();
  for (int c = 0; c < nch; ++c) {
    const int buf = c & 1;
    if (c + 1 < nch) fetch((c + 1) * kTK);  // in flight during this chunk's FMAs
    uint64_t part[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) part[i][j] = 0ull;
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      const uint4 xv = *reinterpret_cast<const uint4*>(&xs[buf][kk][(ty * 4) ^ xs_swz(kk)]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[buf][kk][(tx * 4) ^ ws_swz(kk)]);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint64_t A[4], B[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) A[i] = f2_pack(xw[i] << 16, xw[i] & 0xFFFF0000u);
      B[0] = f2_pack(__float_as_uint(wv.x), __float_as_uint(wv.x));
      B[1] = f2_pack(__float_as_uint(wv.y), __float_as_uint(wv.y));
      B[2] = f2_pack(__float_as_uint(wv.z), __float_as_uint(wv.z));
      B[3] = f2_pack(__float_as_uint(wv.w), __float_as_uint(wv.w));
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = f2_fma(A[i], B[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // Kahan: acc += part
        const uint64_t y = f2_sub(part[i][j], cmp[i][j]);
        const uint64_t s2 = f2_add(acc[i][j], y);
        cmp[i][j] = f2_sub(f2_sub(s2, acc[i][j]), y);
        acc[i][j] = s2;
      }
    if (c + 1 < nch) stage(buf ^ 1);  // that buffer's last reads were in chunk c - 1
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + ty * 8 + 2 * i + h;
      if (t >= T) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = e0 + tx * 4 + j;
        const float v = __uint_as_float((uint32_t)(acc[i][j] >> (32 * h)));
        if (e < E) logits[(size_t)t * E + e] = v + (bias ? bias[e] : 0.f);
      }
    }
  }
}

// ---- softmax + top-k + renormalisation: one warp per token ------------------
// `src` holds the token's E logits (read once, through L2), `l` is the warp's
// shared-memory copy of them.  Ties go to the lower expert id.
// Softmax over the E logits of token t (staged in shared memory `l`), then the
// top-k by (logit desc, id asc), renormalised; one warp.  Lane j holds the
// logits of experts j, j + 32, ... in registers (PER of them, PER >= E/32),
// so that each of the k selection rounds is a register scan plus one warp
// argmax, with no memory access.
template <int PER>
__device__ __forceinline__ void topk_token_r(const float* l, int t, int E, int k,
                                             int32_t* __restrict__ ids, float* __restrict__ w,
                                             float* __restrict__ p_sel) {
  const int lane = threadIdx.x & 31;
  float v[PER];
  float lmax = -INFINITY;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? l[e] : -INFINITY;
    lmax = fmaxf(lmax, v[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
  float z = 0.f;
#pragma unroll
  for (int j = 0; j < PER; ++j)
    if (lane + 32 * j < E) z += expf(v[j] - lmax);
  z = warp_sum(z);
  float sel_sum = 0.f, my_v = 0.f;
  int my_id = -1;
  for (int s = 0; s < k; ++s) {
    float bv = -INFINITY;
    int bid = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < PER; ++j) {  // ids ascend with j: strict > keeps the lower id
      const int e = lane + 32 * j;
      if (e < E && v[j] > bv) {
        bv = v[j];
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oid = __shfl_xor_sync(0xFFFFFFFFu, bid, o);
      if (ov > bv || (ov == bv && oid < bid)) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) {  // taken: out of the later rounds
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (j == (bid >> 5)) v[j] = -INFINITY;
    }
    const float pe = expf(bv - lmax);
    sel_sum += pe;  // same value and order in every lane
    if (lane == s) {
      my_v = pe;
      my_id = bid;
    }
  }
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = my_v / sel_sum;
    if (p_sel) p_sel[(size_t)t * k + lane] = my_v / z;
  }
}

__device__ __forceinline__ void topk_token(const float* l, int t, int E, int k,
                                           int32_t* __restrict__ ids, float* __restrict__ w,
                                           float* __restrict__ p_sel) {
  if (E <= 4 * 32) topk_token_r<4>(l, t, E, k, ids, w, p_sel);
  else if (E <= 9 * 32) topk_token_r<9>(l, t, E, k, ids, w, p_sel);
  else if (E <= 16 * 32) topk_token_r<16>(l, t, E, k, ids, w, p_sel);
  else topk_token_r<32>(l, t, E, k, ids, w, p_sel);
}

// the logits of tokens [t0, t0 + nt) into shared memory, read through L2 by
// every thread of the CTA (coalesced)
__device__ __forceinline__ void stage_logits(const float* logits, int t0, int nt, int E,
                                             float* sl) {
  for (int i = threadIdx.x; i < nt * E; i += blockDim.x) sl[i] = __ldcg(logits + (size_t)t0 * E + i);
  __syncthreads();
}

__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E,
                                              int k, int32_t* __restrict__ ids,
                                              float* __restrict__ w, float* __restrict__ p_sel) {
  extern __shared__ float sl[];  // [8 tokens][E]
  pdl_wait();
  pdl_launch_dependents();
  const int wid = threadIdx.x >> 5;
  const int t0 = blockIdx.x * 8, t = t0 + wid;
  stage_logits(logits, t0, min(8, T - t0), E, sl);
  if (t >= T) return;
  topk_token(sl + (size_t)wid * E, t, E, k, ids, w, p_sel);
}

// ---- few tokens: logits and top-k in one kernel -----------------------------
// One CTA per expert computes that expert's logit for every token (as
// k_logits_gemv); the CTA that finishes last (a counter in the caller's
// workspace, zero before the launch and reset by that CTA) then runs the
// softmax/top-k, one warp per token, on the logits the others wrote.
__global__ void __launch_bounds__(256) k_route_small(const uint16_t* __restrict__ x,
                                                     const float* __restrict__ wr,
                                                     const float* __restrict__ bias, int T,
                                                     int H, int E, int k,
                                                     float* __restrict__ logits,
                                                     int32_t* __restrict__ ids,
                                                     float* __restrict__ w,
                                                     float* __restrict__ p_sel,
                                                     unsigned int* __restrict__ done) {
  extern __shared__ float sl[];  // [8 warps][E]
  __shared__ int s_last;
  pdl_wait();
  pdl_launch_dependents();
  logits_of_expert(x, wr, bias, T, H, E, blockIdx.x, logits);
  __threadfence();  // this CTA's logits are visible before it is counted
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int wid = threadIdx.x >> 5;
  stage_logits(logits, 0, T, E, sl);
  if (wid < T) topk_token(sl + (size_t)wid * E, wid, E, k, ids, w, p_sel);
  if (threadIdx.x == 0) *done = 0u;  // ready for the next call
}

// One token's shared-expert gate/up by one CTA of 1024 threads: 8 row pairs
// (gate row i, up row i), each split over 4 warps by quarters of H, 8 bf16 per
// lane and load, two loads of each row in flight (two CTAs of 1024 threads fit
// an SM at 32 registers); x is staged once in fp32.  The quarters' sums are
// added in a fixed order.
constexpr int kShSplit = 4, kShRows = (kPermThreads / 32) / kShSplit;
__device__ void shared_gu_cta(const uint16_t* __restrict__ x, int H, const SharedGuArgs& sg,
                              int cta, float* xs) {
  __shared__ float red[kPermThreads / 32][2];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < H / 2; i += blockDim.x) {
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(x) + i);
    xs[2 * i] = bf16_lo(v);
    xs[2 * i + 1] = bf16_hi(v);
  }
  __syncthreads();
  const int i = cta * kShRows + wid / kShSplit, qt = wid % kShSplit;
  float ag = 0.f, au = 0.f;
  if (i < sg.Is) {
    const int np = H / 8, nq = np / kShSplit;  // 16-byte pieces per row, per quarter
    const uint4* g = reinterpret_cast<const uint4*>(sg.s_gate + (size_t)i * H) + qt * nq;
    const uint4* u = reinterpret_cast<const uint4*>(sg.s_up + (size_t)i * H) + qt * nq;
    const float* xq = xs + qt * nq * 8;
    for (int p0 = lane; p0 < nq; p0 += 2 * 32) {
      uint4 gv[2], uv[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int pp = p0 + 32 * j;
        gv[j] = pp < nq ? ldg_stream(g + pp) : make_uint4(0u, 0u, 0u, 0u);
        uv[j] = pp < nq ? ldg_stream(u + pp) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int pp = p0 + 32 * j;
        if (pp >= nq) break;
        const float4 x0 = *reinterpret_cast<const float4*>(xq + pp * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(xq + pp * 8 + 4);
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t gw[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
        const uint32_t uw[4] = {uv[j].x, uv[j].y, uv[j].z, uv[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ag = fmaf(bf16_lo(gw[q]), xv[2 * q], ag);
          ag = fmaf(bf16_hi(gw[q]), xv[2 * q + 1], ag);
          au = fmaf(bf16_lo(uw[q]), xv[2 * q], au);
          au = fmaf(bf16_hi(uw[q]), xv[2 * q + 1], au);
        }
      }
    }
  }
  ag = warp_sum(ag);
  au = warp_sum(au);
  if (lane == 0) {
    red[wid][0] = ag;
    red[wid][1] = au;
  }
  __syncthreads();
  if (threadIdx.x < kShRows) {
    const int r = cta * kShRows + threadIdx.x;
    if (r < sg.Is) {
      float g = 0.f, uu = 0.f;
#pragma unroll
      for (int q = 0; q < kShSplit; ++q) {
        g += red[threadIdx.x * kShSplit + q][0];
        uu += red[threadIdx.x * kShSplit + q][1];
      }
      sg.h_shared[r] = g / (1.f + expf(-g)) * uu;
    }
  }
}

// The same, with the permutation of the routes by expert and the cache
// lookup (permute_body) run by that last CTA as well: one launch from the
// token to the FFN's expert list.  1024 threads per CTA.  CTAs E.. run the
// shared expert's gate/up for one token (sg.Is > 0): HBM work that needs no
// routing, streaming while the last router CTA selects and permutes.
__global__ void __launch_bounds__(kPermThreads, 2) k_route_permute_small(
    const uint16_t* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
    int T, int H, int E, int k, float* __restrict__ logits, int32_t* __restrict__ ids,
    float* __restrict__ w, float* __restrict__ p_sel, unsigned int* __restrict__ done,
    PermArgs pa, SharedGuArgs sg, PolicyArgs pol, SkipArgs sk) {
  extern __shared__ float sl[];  // top-k: [8 warps][E] floats; then the permutation's ints
  __shared__ int s_last;
  pdl_wait();
  pdl_launch_dependents();
  if ((int)blockIdx.x >= E) {
    shared_gu_cta(x, H, sg, blockIdx.x - E, sl);
    return;
  }
  logits_of_expert(x, wr, bias, T, H, E, blockIdx.x, logits);
  __threadfence();  // this CTA's logits are visible before it is counted
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == (unsigned)E - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int wid = threadIdx.x >> 5;
  stage_logits(logits, 0, T, E, sl);
  if (wid < T) topk_token(sl + (size_t)wid * E, wid, E, k, ids, w, p_sel);
  __syncthreads();  // ids written by this CTA: read back through L2 below
  const int32_t* pids = ids;
  if (sk.tau > 0.f) {  // the renorm-skip: the permutation takes the kept routes
    if ((int)threadIdx.x < T) skip_token(sk, ids, w, threadIdx.x, k, E);
    __syncthreads();
    pids = sk.ids_eff;
  }
  if (T * k <= 32 && !pa.pad_offsets)
    permute_small(pids, T * k, E, pa.counts, pa.offsets, pa.perm, pa.inv, pa.status, pa.lk,
                  reinterpret_cast<int*>(sl));
  else
    permute_body(pids, T * k, E, pa.counts, pa.offsets, pa.perm, pa.inv, pa.pad_offsets,
                 pa.pad_align, pa.status, pa.lk, reinterpret_cast<int*>(sl), 0);
  if (pol.table_row) {  // the adaptive cache's step, on this CTA's lookup results
    __syncthreads();
    policy_body(pol, reinterpret_cast<unsigned char*>(sl));
  }
  if (threadIdx.x == 0) *done = 0u;  // ready for the next call
}

}  // namespace moe

using namespace moe;

// workspace: a 256-byte control area (the few-token kernel's completion
// counter), then the logits when the caller passes none
constexpr size_t kRouteCtl = 256;

MOE_API size_t moe_route_workspace_bytes(int T, int E) {
  return (T > 0 && E > 0) ? kRouteCtl + (size_t)T * E * sizeof(float) : 0;
}

static moe_status route_check(const moe_route_args* a) {
  if (!a || !a->x || !a->w_router || !a->ids || !a->w) return MOE_ERR_INVALID_ARG;
  if (a->T < 0 || a->H <= 0 || a->E <= 0 || a->k <= 0 || a->k > a->E || a->k > 32)
    return MOE_ERR_INVALID_ARG;
  if (a->H % 256 || a->E > 1024) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

namespace moe {
// the tensor-core logits for many tokens (route_tc.cu)
bool route_tc_ok(const moe_route_args* a);
moe_status route_logits_tc(const moe_route_args* a, float* logits, cudaStream_t s);

// Router, permutation and lookup in one launch for T <= 8 tokens (the layer's
// decode sequence).  Needs a->workspace (the control area) and a->logits.
// Returns MOE_ERR_UNSUPPORTED when the shape does not qualify (the caller then
// runs moe_route and the permutation separately).
moe_status route_permute_small(const moe_route_args* a, const PermArgs& pa,
                               const SharedGuArgs& sg, const PolicyArgs* pol,
                               const SkipArgs* sk, cudaStream_t s) {
  moe_status st = route_check(a);
  if (st != MOE_OK) return st;
  if (a->T < 1 || a->T > kGemvMaxT || !a->logits || !a->workspace ||
      a->workspace_bytes < kRouteCtl)
    return MOE_ERR_UNSUPPORTED;
  if (!pa.counts || !pa.offsets || !pa.perm || !pa.inv || (pa.pad_offsets && pa.pad_align <= 0))
    return MOE_ERR_INVALID_ARG;
  if (sg.Is > 0 && (a->T != 1 || !sg.s_gate || !sg.s_up || !sg.h_shared))
    return MOE_ERR_INVALID_ARG;
  size_t smem = (size_t)8 * a->E * sizeof(float);
  if (permute_smem_bytes(a->E) > smem) smem = permute_smem_bytes(a->E);
  if (sg.Is > 0 && (size_t)a->H * sizeof(float) > smem) smem = (size_t)a->H * sizeof(float);
  if (pol && policy_smem_bytes(a->E, pol->slot_hi - pol->slot_lo) > smem)
    smem = policy_smem_bytes(a->E, pol->slot_hi - pol->slot_lo);
  static bool attr = false;
  if (smem > 48 * 1024 && !attr) {
    if (cudaFuncSetAttribute(k_route_permute_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(64 * 1024 > permute_smem_bytes(1024)
                                       ? 64 * 1024 : permute_smem_bytes(1024))) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr = true;
  }
  if (smem > 64 * 1024 && smem > permute_smem_bytes(1024)) return MOE_ERR_UNSUPPORTED;
  if (sg.Is > 0 && (a->H / 8) % kShSplit) return MOE_ERR_UNSUPPORTED;
  const int sh_ctas = sg.Is > 0 ? (sg.Is + kShRows - 1) / kShRows : 0;
  if (launch_pdl(k_route_permute_small, a->E + sh_ctas, kPermThreads, smem, s,
                 (const uint16_t*)a->x, a->w_router, a->bias, a->T, a->H, a->E, a->k, a->logits,
                 a->ids, a->w, a->p_sel, (unsigned int*)a->workspace, pa, sg,
                 pol ? *pol : PolicyArgs{}, sk ? *sk : SkipArgs{}) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// the renorm-skip alone (more than 8 tokens: after moe_route, before the permutation)
__global__ void __launch_bounds__(256) k_route_skip(SkipArgs sk, const int32_t* ids,
                                                    const float* w, int T, int k, int E) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) skip_token(sk, ids, w, t, k, E);
}

moe_status launch_route_skip(const SkipArgs& sk, const int32_t* ids, const float* w, int T, int k,
                             int E, cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  if (launch_pdl(k_route_skip, (T + 255) / 256, 256, 0, s, sk, ids, w, T, k, E) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
}  // namespace moe

MOE_API moe_status moe_route(const moe_route_args* a, void* stream) {
  moe_status st0 = route_check(a);
  if (st0 != MOE_OK) return st0;
  if (a->T == 0) return MOE_OK;
  float* logits = a->logits;
  if (!logits) {
    if (!a->workspace || a->workspace_bytes < moe_route_workspace_bytes(a->T, a->E))
      return MOE_ERR_INVALID_ARG;
    logits = (float*)((char*)a->workspace + kRouteCtl);
  }
  cudaStream_t s = (cudaStream_t)stream;
  const uint16_t* x = (const uint16_t*)a->x;
  size_t smem = (size_t)8 * a->E * sizeof(float);
  if (a->T <= kGemvMaxT && a->workspace && a->workspace_bytes >= kRouteCtl) {
    if (launch_pdl(k_route_small, a->E, 256, smem, s, x, a->w_router, a->bias, a->T, a->H, a->E,
                   a->k, logits, a->ids, a->w, a->p_sel, (unsigned int*)a->workspace) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (a->T <= kGemvGroupsMaxT) {
    const dim3 grid(a->E, (a->T + kGemvMaxT - 1) / kGemvMaxT);
    if (launch_pdl(k_logits_gemv, grid, 256, 0, s, x, a->w_router, a->bias, a->T, a->H, a->E,
                   logits) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (route_tc_ok(a)) {
    moe_status st = route_logits_tc(a, logits, s);
    if (st != MOE_OK) return st;
  } else {
    dim3 grid((a->E + kTN - 1) / kTN, (a->T + kTM - 1) / kTM);
    if (launch_pdl(k_logits_gemm, grid, kGemmThreads, 0, s, x, a->w_router, a->bias, a->T, a->H,
                   a->E, logits) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  MOE_CHECK_LAUNCH();
  if (launch_pdl(k_topk, (a->T + 7) / 8, 256, smem, s, logits, a->T, a->E, a->k, a->ids, a->w,
                 a->p_sel) != cudaSuccess)
    return MOE_ERR_CUDA;
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
