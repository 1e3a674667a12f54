/*
 * gen_core.h - seeded synthetic input generator: the definitions.
 *
 * This module only draws inputs.  It holds none of the MoE layer's
 * arithmetic (no routing, no dot products, no activation quantisation);
 * both the CPU oracle and the GPU path consume what it produces, and both
 * implementations of it (gen.c on the host, gen_cuda.cu on the device) use
 * these inline definitions so that they agree bit for bit.
 *
 * Counter-based generator
 *   mix64 is the splitmix64 output function (Steele, Lea, Flood,
 *   "Fast splittable pseudorandom number generators", OOPSLA 2014).
 *   A stream key is built from (seed, kind, a, b); draw i of a stream is
 *   mix64(key + (i + 1) * GOLDEN).
 *
 * Near-normal samples
 *   One 64-bit draw gives four 16-bit uniforms U1..U4; their sum S is an
 *   Irwin-Hall(4) variate scaled by 65535, mean 131070, standard deviation
 *   sqrt(4 * (65536^2 - 1) / 12) = 37837.228...  d = S - 131070 is an exact
 *   integer in [-131070, 131070]; a sample of N(0, sigma^2) is taken as
 *   d * sigma / 37837.228 (bounded support +-3.46 sigma, variance exact).
 *
 * Weight quantisation (input preparation, not the method)
 *   A block of 16 weights d_0..d_15 (integer domain) becomes one E4M3 block
 *   scale s (the smallest positive E4M3 value with 384 * s >= max|d|) and 16
 *   E2M1 codes (nearest magnitude of |d| / (64 s), ties to the even code).
 *   With the per-matrix global scale g, the represented weight is
 *   e2m1(code) * e4m3(s) * g and the weight "before quantisation" was
 *   d * g / 64.  Everything here is integer arithmetic.
 *   MXFP4 records (OCP Microscaling Formats v1.0, element E2M1, block 32,
 *   scale E8M0): a block of 32 weights w = d/64 shares the scale X =
 *   2^(floor(log2 max|w|) - 2) (byte 127 + floor(log2 max|d|) - 8; byte 0
 *   and codes 0 for an all-zero block) and each code is the nearest E2M1
 *   magnitude of |w| / X, ties to the even code, saturating at 6.
 */
#ifndef GEN_CORE_H
#define GEN_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define GEN_HD static __host__ __device__ __forceinline__
#else
#define GEN_HD static inline
#endif

#define GEN_GOLDEN 0x9E3779B97F4A7C15ULL
#define GEN_IH_MEAN 131070
#define GEN_IH_SD 37837.228

/* tensor kinds (stream separation) */
enum {
  GEN_KIND_X = 1,       /* activations, a = layer, b = draw index      */
  GEN_KIND_ROUTER = 2,  /* router weights, a = layer, b = expert        */
  GEN_KIND_SHARED = 3,  /* shared expert, a = layer, b = matrix (0,1,2) */
  GEN_KIND_EXPERT = 4,  /* routed expert, a = layer, b = expert*4+matrix*/
  GEN_KIND_GSCALE = 5,  /* per-matrix global scale factor               */
  GEN_KIND_PERM = 6     /* per-layer popularity permutation (Zipf bias)  */
};

GEN_HD uint64_t gen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

GEN_HD uint64_t gen_key(uint64_t seed, uint32_t kind, uint64_t a, uint64_t b) {
  uint64_t k = gen_mix64(seed * GEN_GOLDEN + (uint64_t)kind);
  k = gen_mix64(k + a);
  return gen_mix64(k + b);
}

GEN_HD uint64_t gen_draw(uint64_t key, uint64_t i) {
  return gen_mix64(key + (i + 1) * GEN_GOLDEN);
}

/* centred Irwin-Hall(4) integer, exact, in [-131070, 131070] */
GEN_HD int32_t gen_ih(uint64_t u) {
  int32_t s = (int32_t)(u & 0xFFFF) + (int32_t)((u >> 16) & 0xFFFF) +
              (int32_t)((u >> 32) & 0xFFFF) + (int32_t)(u >> 48);
  return s - GEN_IH_MEAN;
}

/* fp32 -> bf16 bit pattern, round to nearest even (inputs are finite) */
GEN_HD uint16_t gen_f32_to_bf16(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t lsb = (v.u >> 16) & 1u;
  return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

/* E4M3 (FN) positive value times 1024, as an exact integer, for byte b in
 * [0, 126]: subnormal (e = 0) m * 2^-9, normal (8 + m) * 2^(e - 10). */
GEN_HD int64_t gen_e4m3_v1024(int b) {
  int e = (b >> 3) & 15, m = b & 7;
  if (e == 0) return (int64_t)m * 2;
  return (int64_t)(8 + m) << e;
}

/* smallest E4M3 byte b in [1,126] with 384 * value(b) >= amax; 0 if amax == 0 */
GEN_HD int gen_block_scale_byte(int64_t amax) {
  if (amax <= 0) return 0;
  int lo = 1, hi = 126; /* value(126) = 448 >= 131070 / 384 */
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (gen_e4m3_v1024(mid) * 384 >= amax * 1024) hi = mid; else lo = mid + 1;
  }
  return lo;
}

/* E2M1 code of d for a block with scale byte sb: nearest magnitude of
 * |d| / (64 * value(sb)), ties to the even code, sign in bit 3 (zero -> 0). */
GEN_HD uint32_t gen_e2m1_code(int32_t d, int sb) {
  if (sb == 0) return 0;
  int64_t n = (int64_t)(d < 0 ? -d : d) * 64; /* compare n vs mid*V with mids x4 */
  int64_t V = gen_e4m3_v1024(sb);
  /* midpoints (x4) between consecutive E2M1 magnitudes 0,.5,1,1.5,2,3,4,6 */
  const int mid4[7] = {1, 3, 5, 7, 10, 14, 20};
  uint32_t c = 0;
  for (int j = 0; j < 7; ++j) {
    int64_t t = (int64_t)mid4[j] * V;
    if (n > t) c = (uint32_t)(j + 1);
    else if (n == t) { c = (uint32_t)(((j & 1) == 0) ? j : j + 1); break; }
    else break;
  }
  if (c > 7) c = 7;
  if (c != 0 && d < 0) c |= 8u;
  return c;
}

/* MXFP4 code of d in a block whose largest |d| has floor(log2) = E:
 * nearest E2M1 magnitude of q = |d| / 2^(E - 2), i.e. compare 16 |d| with
 * (4 x midpoint) x 2^E; ties to the even code; saturating at 6. */
GEN_HD uint32_t gen_e2m1_code_mx(int32_t d, int E) {
  int64_t n = (int64_t)(d < 0 ? -d : d) * 16;
  const int mid4[7] = {1, 3, 5, 7, 10, 14, 20};
  uint32_t c = 0;
  for (int j = 0; j < 7; ++j) {
    int64_t t = (int64_t)mid4[j] << E;
    if (n > t) c = (uint32_t)(j + 1);
    else if (n == t) { c = (uint32_t)(((j & 1) == 0) ? j : j + 1); break; }
    else break;
  }
  if (c != 0 && d < 0) c |= 8u;
  return c;
}

/* ---- expert record layout (the storage format) ----
 * Matrices: 0 = gate [I x H], 1 = up [I x H], 2 = down [H x I].
 * Codes: row-major, two E2M1 codes per byte, element 2j in the low nibble.
 * Scales: one E4M3 byte per 16 elements of a row, in 512-byte atoms:
 *   atom (row_tile = r / 128, k_group = kb / 4) at ((row_tile * KB/4) + k_group) * 512,
 *   byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4) inside the atom.
 */
/* fmt 0 = NVFP4 (E4M3 scale per 16 values), 1 = MXFP4 (E8M0 scale per 32,
 * in the same 512-byte atoms with kb counting blocks of 32) */
GEN_HD int gen_block_len(int fmt) { return fmt ? 32 : 16; }
GEN_HD uint64_t gen_codes_off(int H, int I, int m) {
  uint64_t gu = (uint64_t)I * (uint64_t)H / 2;
  return m == 0 ? 0 : (m == 1 ? gu : 2 * gu);
}
GEN_HD uint64_t gen_scales_off(int H, int I, int m, int fmt) {
  uint64_t codes = 3ull * (uint64_t)I * (uint64_t)H / 2;
  uint64_t gu = (uint64_t)I * (uint64_t)H / (uint64_t)gen_block_len(fmt);
  return codes + (m == 0 ? 0 : (m == 1 ? gu : 2 * gu));
}
GEN_HD uint64_t gen_record_bytes(int H, int I, int fmt) {
  return 3ull * (uint64_t)I * (uint64_t)H / 2 +
         3ull * (uint64_t)I * (uint64_t)H / (uint64_t)gen_block_len(fmt);
}
GEN_HD uint64_t gen_scale_index(int r, int kb, int KB) {
  return ((uint64_t)(r / 128) * (uint64_t)(KB / 4) + (uint64_t)(kb / 4)) * 512u +
         (uint64_t)(r % 32) * 16u + (uint64_t)((r % 128) / 32) * 4u + (uint64_t)(kb % 4);
}

/* One 16-element block (row r, block kb) of matrix m: writes 8 code bytes
 * and returns the scale byte.  K = row length of that matrix. */
GEN_HD int gen_expert_block(uint64_t key, int r, int kb, int K, uint8_t codes[8]) {
  int32_t d[16];
  int64_t amax = 0;
  uint64_t base = (uint64_t)r * (uint64_t)K + (uint64_t)kb * 16u;
  for (int j = 0; j < 16; ++j) {
    d[j] = gen_ih(gen_draw(key, base + (uint64_t)j));
    int64_t a = d[j] < 0 ? -(int64_t)d[j] : (int64_t)d[j];
    if (a > amax) amax = a;
  }
  int sb = gen_block_scale_byte(amax);
  for (int j = 0; j < 8; ++j) {
    uint32_t lo = gen_e2m1_code(d[2 * j], sb);
    uint32_t hi = gen_e2m1_code(d[2 * j + 1], sb);
    codes[j] = (uint8_t)(lo | (hi << 4));
  }
  return sb;
}

/* One 32-element MXFP4 block (row r, block kb of 32) of matrix m: writes 16
 * code bytes and returns the E8M0 scale byte. */
GEN_HD int gen_expert_block_mx(uint64_t key, int r, int kb, int K, uint8_t codes[16]) {
  int32_t d[32];
  int64_t amax = 0;
  uint64_t base = (uint64_t)r * (uint64_t)K + (uint64_t)kb * 32u;
  for (int j = 0; j < 32; ++j) {
    d[j] = gen_ih(gen_draw(key, base + (uint64_t)j));
    int64_t a = d[j] < 0 ? -(int64_t)d[j] : (int64_t)d[j];
    if (a > amax) amax = a;
  }
  if (amax == 0) {
    for (int j = 0; j < 16; ++j) codes[j] = 0;
    return 0;
  }
  int E = 0;
  while ((amax >> (E + 1)) != 0) ++E; /* floor(log2 amax) */
  for (int j = 0; j < 16; ++j) {
    uint32_t lo = gen_e2m1_code_mx(d[2 * j], E);
    uint32_t hi = gen_e2m1_code_mx(d[2 * j + 1], E);
    codes[j] = (uint8_t)(lo | (hi << 4));
  }
  return 127 + E - 8;
}

#endif
