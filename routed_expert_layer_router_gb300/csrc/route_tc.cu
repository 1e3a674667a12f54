// route_tc.cu - the router's logits for many tokens on the tcgen05 tensor
// cores, at fp32 accuracy.
//
// The router ("Project Maya" page: device-side router with fp32 weights)
// computes logits[t][e] = sum_h x[t][h] W[e][h] + bias[e] with bf16 tokens
// and fp32 weights.  A bf16 x bf16 product is exact in fp32, and an fp32
// weight is the exact sum of three bf16 values,
//   W1 = bf16(W), W2 = bf16(W - W1), W3 = W - W1 - W2
// (W - W1 keeps at most 16 significant bits and W - W1 - W2 at most 8, each
// exact in fp32; bf16 has fp32's exponent range, so the split is exact for
// |W| >= 2^-110, below which the third piece can lose low bits).  So x.W =
// x.W1 + x.W2 + x.W3 with every product exact, and only the sums round.
//
//   k_router_split  W [E][H] fp32 -> pieces [3][E_pad][H] bf16 (rows E..E_pad-1
//                   zero), rewritten by every call (the weights may change
//                   between calls; the split reads 4 and writes 6 bytes per
//                   weight, a few microseconds);
//   k_logits_tc     per tile of 128 tokens x 32 experts, one MMA per 16-deep K
//                   step with M = 128 tokens (A = x) and N = 96 columns: the
//                   three pieces of the tile's 32 experts (B), so columns
//                   0-31, 32-63, 64-95 accumulate x.W1, x.W2, x.W3.
//
// Accuracy.  The tensor cores' fp32 accumulation need not round to nearest,
// and over a 6144-deep sum its error could reach 1e-4 of a logit.  So an
// accumulator only ever sums one 64-deep K chunk (4 MMAs, a fresh accumulator
// per chunk): the epilogue warps read each chunk's 96 columns from tensor
// memory and add them into registers, the W1 column with compensated
// (Kahan) summation and the W2 + W3 columns (2^-8 smaller) plainly.  Two
// accumulators alternate, so the MMAs of chunk c + 1 run while chunk c is
// read.
//
// One warp issues TMA loads (x tile 128 x 64 bf16 and the three 32 x 64 piece
// tiles per chunk, 128-byte swizzle) into a ring of stages, one warp issues
// the MMAs, eight warps read the accumulators (warp w reads the tensor-memory
// lanes of quarter w mod 4 and 16 of the 32 experts).  Tiles are walked
// experts-fastest so that CTAs working at the same time share x tiles in L2.
#include <cudaTypedefs.h>
#include <string.h>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

moe_status tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                        uint64_t row_stride_bytes, uint32_t box_rows);

namespace rt {

constexpr int kNE = 32;                 // experts per tile
constexpr int kN = 3 * kNE;             // MMA N: three pieces of kNE experts
constexpr int kM = 128;                 // tokens per tile
constexpr int kKC = 64;                 // bf16 values per K chunk (128 bytes a row)
constexpr int kABytes = kM * 128;       // 16 KiB
constexpr int kPieceBytes = kNE * 128;  // 4 KiB
constexpr int kBBytes = 3 * kPieceBytes;
// TP token tiles of 128 per CTA share each stage's weight-piece tile: a
// stage holds TP x tiles and the pieces
template <int TP> struct TC {
  static constexpr int kStageBytes = TP * kABytes + kBBytes;  // 28 or 44 KiB
  static constexpr int kStages = TP == 1 ? 6 : 5;
  static constexpr int kSmem = 1024 + kStages * kStageBytes;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};
constexpr int kThreads = 320;           // warp 0: TMA, warp 1: MMA, warps 2..9: epilogue
constexpr int kEpiWarps = 8;
constexpr uint32_t kAccStride = 128;    // tensor-memory columns per accumulator
constexpr uint32_t kAccBufs = 2;        // accumulators (per token tile) in rotation
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;  // no wait lasts longer than 2 s
static_assert(kN <= (int)kAccStride, "accumulator columns");

struct Params {
  int T, E, E_pad, H;
  int n_nt;      // expert tiles (E_pad / kNE)
  int n_tiles;   // tiles (TP token tiles of 128 each) x expert tiles
  const float* bias;
  float* logits;
  int32_t* status;
};

__global__ void __launch_bounds__(256) k_router_split(const float* __restrict__ w, int E, int H,
                                                      int E_pad, uint16_t* __restrict__ out) {
  pdl_wait();  // the previous call's tensor-core router may still read `out`
  const size_t n4 = (size_t)E_pad * H / 4, plane = (size_t)E_pad * H;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t e = i * 4 / H;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e < (size_t)E) v = __ldg(reinterpret_cast<const float4*>(w) + i);
    const float a[4] = {v.x, v.y, v.z, v.w};
    uint16_t p1[4], p2[4], p3[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      p1[j] = f32_to_bf16_rne(a[j]);
      const float r1 = __fsub_rn(a[j], bf16_lo(p1[j]));  // exact
      p2[j] = f32_to_bf16_rne(r1);
      const float r2 = __fsub_rn(r1, bf16_lo(p2[j]));   // exact, 8 bits
      p3[j] = f32_to_bf16_rne(r2);
    }
    auto pack = [](const uint16_t* p) {
      return make_uint2((uint32_t)p[0] | ((uint32_t)p[1] << 16),
                        (uint32_t)p[2] | ((uint32_t)p[3] << 16));
    };
    reinterpret_cast<uint2*>(out)[i] = pack(p1);
    reinterpret_cast<uint2*>(out + plane)[i] = pack(p2);
    reinterpret_cast<uint2*>(out + 2 * plane)[i] = pack(p3);
  }
  pdl_launch_dependents();
}

template <int TP>
__global__ void __launch_bounds__(kThreads, 1)
    k_logits_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                Params p) {
  constexpr int kStages = TC<TP>::kStages, kStageBytes = TC<TP>::kStageBytes;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.H / kKC;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (uint32_t b = 0; b < kAccBufs; ++b) {
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
  pdl_wait();  // x and the weight pieces are written by earlier kernels
  pdl_launch_dependents();

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      uint32_t g = 0;
      for (int t = blockIdx.x; t < p.n_tiles && !abort_flag; t += gridDim.x) {
        const int mt = t / p.n_nt, nt = t % p.n_nt;
        for (int kc = 0; kc < nk; ++kc, ++g) {
          const int s = (int)(g % kStages);
          if (!ptx::mbar_wait(&empty_bar[s], ((g / kStages) & 1) ^ 1, kWaitNs)) {
            set_status(p.status, MOE_ERR_TIMEOUT);
            abort_flag = 1;
            break;
          }
          unsigned char* st = smem + (size_t)s * kStageBytes;
          ptx::mbar_arrive_expect_tx(&full_bar[s], (uint32_t)kStageBytes);
#pragma unroll
          for (int tp = 0; tp < TP; ++tp)
            ptx::tma_load_2d(st + tp * kABytes, &tmX, kc * kKC, (mt * TP + tp) * kM, &full_bar[s]);
#pragma unroll
          for (int pc = 0; pc < 3; ++pc)
            ptx::tma_load_2d(st + TP * kABytes + pc * kPieceBytes, &tmW, kc * kKC,
                             pc * p.E_pad + nt * kNE, &full_bar[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      // M = 128, N = 96, K-major A and B, bf16 inputs, fp32 accumulator
      const uint32_t idesc = ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24) |
                             (1u << 4) | (1u << 7) | (1u << 10);
      uint32_t g = 0, d = 0;
      for (int t = blockIdx.x; t < p.n_tiles && !abort_flag; t += gridDim.x) {
        for (int kc = 0; kc < nk; ++kc, ++g, ++d) {
          const uint32_t b = d % kAccBufs, u = d / kAccBufs;
          if (!ptx::mbar_wait(&acc_empty[b], (u & 1) ^ 1, kWaitNs)) {
            set_status(p.status, MOE_ERR_TIMEOUT);
            abort_flag = 1;
            break;
          }
          ptx::tc_fence_after();
          const int s = (int)(g % kStages);
          if (!ptx::mbar_wait(&full_bar[s], (g / kStages) & 1, kWaitNs)) {
            set_status(p.status, MOE_ERR_TIMEOUT);
            abort_flag = 1;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(smem + (size_t)s * kStageBytes);
          const uint32_t b0 = a0 + TP * kABytes;
#pragma unroll
          for (int tp = 0; tp < TP; ++tp)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_bf16(tmem + (b * TP + tp) * kAccStride,
                            ptx::smem_desc(a0 + tp * kABytes + kk * 32, 16, 1024, 2),
                            ptx::smem_desc(b0 + kk * 32, 16, 1024, 2), idesc, kk > 0);
          ptx::tc_commit(&empty_bar[s]);  // the stage is free once these MMAs finish
          ptx::tc_commit(&acc_full[b]);   // and the chunk's sums are ready
        }
      }
    }
  } else {
    // ================= epilogue (warps 2..9) =================
    const int q = warp & 3;          // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;  // experts [16 half, 16 half + 16) of the tile
    uint32_t d = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
      const int mt = t / p.n_nt, nt = t % p.n_nt;
      float sum[TP][16], comp[TP][16], lo[TP][16];
#pragma unroll
      for (int tp = 0; tp < TP; ++tp)
#pragma unroll
        for (int j = 0; j < 16; ++j) sum[tp][j] = comp[tp][j] = lo[tp][j] = 0.f;
      for (int kc = 0; kc < nk; ++kc, ++d) {
        const uint32_t b = d % kAccBufs, u = d / kAccBufs;
        if (!ptx::mbar_wait(&acc_full[b], u & 1, kWaitNs)) {
          set_status(p.status, MOE_ERR_TIMEOUT);
          abort_flag = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int tp = 0; tp < TP; ++tp) {
          const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (b * TP + tp) * kAccStride +
                                (uint32_t)(half * 16);
          uint32_t r1[16], r2[16], r3[16];
          ptx::tmem_ld_32x32b_x16(base, r1);
          ptx::tmem_ld_32x32b_x16(base + kNE, r2);
          ptx::tmem_ld_32x32b_x16(base + 2 * kNE, r3);
          ptx::tmem_ld_wait();
          if (tp == TP - 1) {
            ptx::tc_fence_before();
            if (lane == 0) ptx::mbar_arrive(&acc_empty[b]);  // the accumulators are free
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float y = __fsub_rn(__uint_as_float(r1[j]), comp[tp][j]);
            const float s = __fadd_rn(sum[tp][j], y);
            comp[tp][j] = __fsub_rn(__fsub_rn(s, sum[tp][j]), y);
            sum[tp][j] = s;
            lo[tp][j] =
                __fadd_rn(lo[tp][j], __fadd_rn(__uint_as_float(r2[j]), __uint_as_float(r3[j])));
          }
        }
      }
      if (!ok) break;
      const int e0 = nt * kNE + half * 16;
#pragma unroll
      for (int tp = 0; tp < TP; ++tp) {
        const int tok = (mt * TP + tp) * kM + q * 32 + lane;
        if (tok < p.T) {
          float* out = p.logits + (size_t)tok * p.E;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int e = e0 + j;
            if (e < p.E) {
              const float v = __fadd_rn(sum[tp][j], __fsub_rn(lo[tp][j], comp[tp][j]));
              out[e] = p.bias ? __fadd_rn(v, p.bias[e]) : v;
            }
          }
        }
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

}  // namespace rt

size_t route_split_bytes(int E, int H) {
  if (E <= 0 || H <= 0) return 0;
  const size_t E_pad = (size_t)(E + rt::kNE - 1) / rt::kNE * rt::kNE;
  return 3 * E_pad * (size_t)H * 2;
}

// Whether moe_route can take the tensor-core path for these arguments.
bool route_tc_ok(const moe_route_args* a) {
  return a->w_split && a->w_split_bytes >= route_split_bytes(a->E, a->H) && a->H % rt::kKC == 0 &&
         ((uintptr_t)a->x & 15) == 0 && ((uintptr_t)a->w_split & 15) == 0 &&
         ((uintptr_t)a->w_router & 15) == 0;
}

// The logits of a->T tokens into `logits` (the split, then the GEMM).
moe_status route_logits_tc(const moe_route_args* a, float* logits, cudaStream_t s) {
  using namespace rt;
  const int E_pad = (a->E + kNE - 1) / kNE * kNE;
  const size_t n4 = (size_t)E_pad * a->H / 4;
  const int sgrid = (int)((n4 + 255) / 256 < (size_t)kSMs * 8 ? (n4 + 255) / 256 : kSMs * 8);
  if (launch_pdl(k_router_split, sgrid, 256, 0, s, a->w_router, a->E, a->H, E_pad,
                 (uint16_t*)a->w_split) != cudaSuccess)
    return MOE_ERR_CUDA;
  CUtensorMap tx, tw;
  moe_status st;
  if ((st = tmap_bf16_2d(&tx, a->x, (uint64_t)a->H, (uint64_t)a->T, (uint64_t)a->H * 2, kM)) !=
          MOE_OK ||
      (st = tmap_bf16_2d(&tw, a->w_split, (uint64_t)a->H, (uint64_t)3 * E_pad,
                         (uint64_t)a->H * 2, kNE)) != MOE_OK)
    return st;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(k_logits_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TC<1>::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(k_logits_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TC<2>::kSmem) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr = true;
  }
  Params p;
  p.T = a->T;
  p.E = a->E;
  p.E_pad = E_pad;
  p.H = a->H;
  p.n_nt = E_pad / kNE;
  // two token tiles per CTA (each weight-piece tile loaded once for both)
  // once the 128-token tiles would need more than one wave
  const int tiles1 = (a->T + kM - 1) / kM * p.n_nt;
  const bool two = tiles1 > kSMs;
  p.n_tiles = two ? (a->T + 2 * kM - 1) / (2 * kM) * p.n_nt : tiles1;
  p.bias = a->bias;
  p.logits = logits;
  p.status = a->status;
  const int grid = p.n_tiles < kSMs ? p.n_tiles : kSMs;
  if ((two ? launch_pdl(k_logits_tc<2>, grid, kThreads, (size_t)TC<2>::kSmem, s, tx, tw, p)
           : launch_pdl(k_logits_tc<1>, grid, kThreads, (size_t)TC<1>::kSmem, s, tx, tw, p)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe

MOE_API size_t moe_route_split_bytes(int E, int H) { return moe::route_split_bytes(E, H); }
