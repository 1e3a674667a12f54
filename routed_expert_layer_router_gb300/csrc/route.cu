// route.cu - K-route: router logits (fp32), softmax, top-k and renormalised
// weights.  The router is the device-side router of the "Project Maya" page
// ("Three tiers and the rules between them"): fp32 router weights, top-8 of
// 288 experts per token, selection kept on the device.
#include "common.cuh"

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
  __shared__ float red[kGemvMaxT][8];
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

__global__ void __launch_bounds__(256) k_logits_gemv(const uint16_t* __restrict__ x,
                                                     const float* __restrict__ wr,
                                                     const float* __restrict__ bias, int T,
                                                     int H, int E, float* __restrict__ logits) {
  logits_of_expert(x, wr, bias, T, H, E, blockIdx.x, logits);
}

// ---- logits for many tokens: SIMT tiled GEMM --------------------------------
// Tile 128 tokens x 32 experts, 128 threads, 8 tokens x 4 experts each (32
// FMAs per three 16-byte shared loads), K chunks of 32.  Each chunk's partial
// sum is added to the running total with Kahan compensation, keeping the fp32
// error of the 6144-term dot products near that of the chunk sums (the router
// probabilities are compared at 1e-5).  The next chunk's global loads are
// issued before the current chunk is computed; the x tile is stored
// transposed (k-major).  288 experts = 9 tiles: 288 CTAs for 4096 tokens, two
// per SM on most SMs, all resident at once.
constexpr int kTM = 128, kTN = 32, kTK = 32, kGemmThreads = 128;

__global__ void __launch_bounds__(kGemmThreads) k_logits_gemm(const uint16_t* __restrict__ x,
                                                              const float* __restrict__ wr,
                                                              const float* __restrict__ bias,
                                                              int T, int H, int E,
                                                              float* __restrict__ logits) {
  __shared__ __align__(16) float xs[kTK][kTM + 4];
  __shared__ __align__(16) float ws[kTK][kTN + 4];
  const int t0 = blockIdx.y * kTM, e0 = blockIdx.x * kTN;
  const int tid = threadIdx.x;
  const int tx = tid & 7, ty = tid >> 3;  // 8 x 16 threads; tokens ty*8.., experts tx*4..
  // load roles: x: token tid, all 32 k of the chunk; W: expert ln = tid % 32,
  // k quarter lkq = tid / 32 (8 values)
  const int ln = tid & 31, lkq = tid >> 5;
  const bool xok = t0 + tid < T, wok = e0 + ln < E;
  const uint4* xsrc = reinterpret_cast<const uint4*>(x + (size_t)(xok ? t0 + tid : 0) * H);
  const float4* wsrc = reinterpret_cast<const float4*>(wr + (size_t)(wok ? e0 + ln : 0) * H + lkq * 8);
  uint4 xv[4];
  float4 wa, wb;
  auto fetch = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) xv[i] = xok ? __ldg(xsrc + k0 / 8 + i) : make_uint4(0u, 0u, 0u, 0u);
    if (wok) {
      wa = __ldg(wsrc + k0 / 4);
      wb = __ldg(wsrc + k0 / 4 + 1);
    } else {
      wa = wb = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  float acc[8][4], cmp[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = cmp[i][j] = 0.f;
  fetch(0);
  for (int k0 = 0; k0 < H; k0 += kTK) {
    __syncthreads();  // the previous chunk's reads of xs / ws are done
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[i * 8 + 2 * q][tid] = bf16_lo(v[q]);
        xs[i * 8 + 2 * q + 1][tid] = bf16_hi(v[q]);
      }
    }
    {
      const float w8[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) ws[lkq * 8 + i][ln] = w8[i];
    }
    __syncthreads();
    if (k0 + kTK < H) fetch(k0 + kTK);  // in flight during this chunk's FMAs
    float part[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) part[i][j] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < kTK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&xs[kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&xs[kk][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // Kahan: acc += part
        float y = part[i][j] - cmp[i][j];
        float s = acc[i][j] + y;
        cmp[i][j] = (s - acc[i][j]) - y;
        acc[i][j] = s;
      }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
    }
  }
}

// ---- softmax + top-k + renormalisation: one warp per token ------------------
// `src` holds the token's E logits (read once, through L2), `l` is the warp's
// shared-memory copy of them.  Ties go to the lower expert id.
__device__ __forceinline__ void topk_token(const float* src, float* l, int t, int E, int k,
                                           int32_t* __restrict__ ids, float* __restrict__ w,
                                           float* __restrict__ p_sel) {
  const int lane = threadIdx.x & 31;
  const int per = (E + 31) / 32;
  float lmax = -INFINITY;
  for (int j = 0; j < per; ++j) {
    int e = lane + 32 * j;
    float v = (e < E) ? __ldcg(src + e) : -INFINITY;
    if (e < E) l[e] = v;
    lmax = fmaxf(lmax, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
  float z = 0.f;
  for (int j = 0; j < per; ++j) {
    int e = lane + 32 * j;
    if (e < E) z += expf(l[e] - lmax);
  }
  z = warp_sum(z);
  uint32_t taken = 0;  // bit j: element lane + 32 j selected
  float sel_sum = 0.f;
  float my_v = 0.f;
  int my_id = -1;
  for (int s = 0; s < k; ++s) {
    float bv = -INFINITY;
    int bid = 0x7FFFFFFF;
    for (int j = 0; j < per; ++j) {
      int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u)) {
        float v = l[e];
        if (v > bv || (v == bv && e < bid)) { bv = v; bid = e; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      int oid = __shfl_xor_sync(0xFFFFFFFFu, bid, o);
      if (ov > bv || (ov == bv && oid < bid)) { bv = ov; bid = oid; }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    float pe = expf(bv - lmax);
    sel_sum += pe;  // same value and order in every lane
    if (lane == s) { my_v = pe; my_id = bid; }
  }
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = my_v / sel_sum;
    if (p_sel) p_sel[(size_t)t * k + lane] = my_v / z;
  }
}

__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E,
                                              int k, int32_t* __restrict__ ids,
                                              float* __restrict__ w, float* __restrict__ p_sel) {
  extern __shared__ float sl[];  // [8 warps][E]
  const int wid = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + wid;
  if (t >= T) return;
  topk_token(logits + (size_t)t * E, sl + (size_t)wid * E, t, E, k, ids, w, p_sel);
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
  logits_of_expert(x, wr, bias, T, H, E, blockIdx.x, logits);
  __threadfence();  // this CTA's logits are visible before it is counted
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int wid = threadIdx.x >> 5;
  if (wid < T) topk_token(logits + (size_t)wid * E, sl + (size_t)wid * E, wid, E, k, ids, w, p_sel);
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

MOE_API moe_status moe_route(const moe_route_args* a, void* stream) {
  if (!a || !a->x || !a->w_router || !a->ids || !a->w) return MOE_ERR_INVALID_ARG;
  if (a->T < 0 || a->H <= 0 || a->E <= 0 || a->k <= 0 || a->k > a->E || a->k > 32)
    return MOE_ERR_INVALID_ARG;
  if (a->H % 256 || a->E > 1024) return MOE_ERR_UNSUPPORTED;
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
    k_route_small<<<a->E, 256, smem, s>>>(x, a->w_router, a->bias, a->T, a->H, a->E, a->k,
                                          logits, a->ids, a->w, a->p_sel,
                                          (unsigned int*)a->workspace);
    MOE_CHECK_LAUNCH();
    return MOE_OK;
  }
  if (a->T <= kGemvMaxT) {
    k_logits_gemv<<<a->E, 256, 0, s>>>(x, a->w_router, a->bias, a->T, a->H, a->E, logits);
  } else {
    dim3 grid((a->E + kTN - 1) / kTN, (a->T + kTM - 1) / kTM);
    k_logits_gemm<<<grid, kGemmThreads, 0, s>>>(x, a->w_router, a->bias, a->T, a->H, a->E,
                                                logits);
  }
  MOE_CHECK_LAUNCH();
  k_topk<<<(a->T + 7) / 8, 256, smem, s>>>(logits, a->T, a->E, a->k, a->ids, a->w, a->p_sel);
  MOE_CHECK_LAUNCH();
  return MOE_OK;
}
