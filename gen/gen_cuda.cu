// gen_cuda.cu - device implementation of the seeded synthetic input generator.
// Same definitions as gen.c (gen_core.h), so the bytes it writes into device
// memory equal the bytes gen.c writes on the host.  It fills large inputs
// (hundreds of expert records) in HBM quickly; it holds no arithmetic of the
// MoE layer.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gen_core.h"

#define GEN_API extern "C" __attribute__((visibility("default")))

static const double kSd = GEN_IH_SD;

__global__ void k_gen_expert(uint64_t seed, int layer, int expert, int H, int I, int fmt,
                             uint8_t* rec) {
  const int bl = gen_block_len(fmt);
  const uint64_t nb_gu = (uint64_t)I * (uint64_t)(H / bl);
  const uint64_t nb_total = 3 * nb_gu;
  for (uint64_t b = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; b < nb_total;
       b += (uint64_t)gridDim.x * blockDim.x) {
    int m, r, kb, K;
    if (b < 2 * nb_gu) {
      m = (int)(b / nb_gu);
      uint64_t w = b % nb_gu;
      K = H;
      r = (int)(w / (H / bl));
      kb = (int)(w % (H / bl));
    } else {
      m = 2;
      uint64_t w = b - 2 * nb_gu;
      K = I;
      r = (int)(w / (I / bl));
      kb = (int)(w % (I / bl));
    }
    uint64_t key = gen_key(seed, GEN_KIND_EXPERT, (uint64_t)layer, (uint64_t)(expert * 4 + m));
    uint8_t c[16];
    int sb = fmt ? gen_expert_block_mx(key, r, kb, K, c) : gen_expert_block(key, r, kb, K, c);
    uint8_t* dst = rec + gen_codes_off(H, I, m) + (uint64_t)r * (K / 2) + (uint64_t)kb * (bl / 2);
    for (int h = 0; h < bl / 16; ++h) {
      uint64_t packed = 0;
      for (int j = 0; j < 8; ++j) packed |= (uint64_t)c[8 * h + j] << (8 * j);
      *reinterpret_cast<uint64_t*>(dst + 8 * h) = packed;
    }
    rec[gen_scales_off(H, I, m, fmt) + gen_scale_index(r, kb, K / bl)] = (uint8_t)sb;
  }
}

__global__ void k_gen_x(uint64_t seed, int layer, int64_t draw0, int T, int H, float c,
                        uint16_t* out) {
  uint64_t n = (uint64_t)T * H;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x) {
    int t = (int)(i / H), h = (int)(i % H);
    uint64_t key = gen_key(seed, GEN_KIND_X, (uint64_t)layer, (uint64_t)(draw0 + t));
    float v = __fmul_rn((float)gen_ih(gen_draw(key, (uint64_t)h)), c);
    out[i] = gen_f32_to_bf16(v);
  }
}

__global__ void k_gen_router(uint64_t seed, int layer, int E, int H, float c, float* out) {
  uint64_t n = (uint64_t)E * H;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x) {
    int e = (int)(i / H), h = (int)(i % H);
    uint64_t key = gen_key(seed, GEN_KIND_ROUTER, (uint64_t)layer, (uint64_t)e);
    out[i] = __fmul_rn((float)gen_ih(gen_draw(key, (uint64_t)h)), c);
  }
}

__global__ void k_gen_shared(uint64_t seed, int layer, int m, uint64_t n, float c, uint16_t* out) {
  uint64_t key = gen_key(seed, GEN_KIND_SHARED, (uint64_t)layer, (uint64_t)m);
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = gen_f32_to_bf16(__fmul_rn((float)gen_ih(gen_draw(key, i)), c));
}

static int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 64) g = 152ull * 64;
  if (g < 1) g = 1;
  return (int)g;
}

GEN_API int gen_dev_expert_record(uint64_t seed, int layer, int expert, int H, int I, int fmt,
                                  uint8_t* dst, void* stream) {
  if (H % 128 || I % 128 || !dst || fmt < 0 || fmt > 1) return 1;
  uint64_t nb = 3ull * I * (H / gen_block_len(fmt));
  k_gen_expert<<<grid_for(nb), 256, 0, (cudaStream_t)stream>>>(seed, layer, expert, H, I, fmt,
                                                                dst);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

GEN_API int gen_dev_x_bf16(uint64_t seed, int layer, int64_t draw0, int T, int H, uint16_t* dst,
                           void* stream) {
  if (T <= 0) return 0;
  k_gen_x<<<grid_for((uint64_t)T * H), 256, 0, (cudaStream_t)stream>>>(
      seed, layer, draw0, T, H, (float)(1.0 / kSd), dst);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

GEN_API int gen_dev_router_f32(uint64_t seed, int layer, int E, int H, float* dst, void* stream) {
  k_gen_router<<<grid_for((uint64_t)E * H), 256, 0, (cudaStream_t)stream>>>(
      seed, layer, E, H, (float)(0.05 / kSd), dst);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

GEN_API int gen_dev_shared_bf16(uint64_t seed, int layer, int Is, int H, uint16_t* gate,
                                uint16_t* up, uint16_t* down, void* stream) {
  uint16_t* dst[3] = {gate, up, down};
  uint64_t n = (uint64_t)Is * H;
  for (int m = 0; m < 3; ++m) {
    if (!dst[m]) continue;
    k_gen_shared<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(seed, layer, m, n,
                                                              (float)(0.02 / kSd), dst[m]);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
