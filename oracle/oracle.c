/*
 * oracle.c - plain, slow CPU oracle of the routed MoE layer (fp64).
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's CPU
 * baseline leg may call it; the library under routed_expert_layer_router_gb300/
 * never does, and the two share no code, header, table or constant.
 *
 * What it computes, step by step (sources: "Project Maya" page, sections
 * "Three tiers and the rules between them" and "A V100 has no BF16 and no FP8";
 * the dev.to page "A hot expert cache made a 181 GiB model faster", sections
 * "The wall: one PCIe transfer per token" and "A gather kernel that reads
 * wide"; the Strata-GLM blog "Day one" list):
 *   1. formats: E2M1 codes and E4M3 block scales decoded from their
 *      definitions; weight = e2m1(code) * e4m3(scale of its 16-block) * g.
 *   2. router: logits = W_r x + b in fp64; experts ordered by (logit desc,
 *      id asc) with a full sort; ids = first k; p_sel = full softmax of the
 *      selected; w = softmax over the selected logits (renormalised top-k).
 *   3. permute: stable counting sort of routes r = t*k + j by expert id.
 *   4. expert: g = Wg x, u = Wu x, h = silu(g) * u, o = Wd h (no biases).
 *   5. combine: y_t = sum_j w_tj * o(e_tj, x_t) + shared(x_t); no residual.
 *   6. prefill mode only: x (per token) and h (per route, after rounding to
 *      fp32) pass through NVFP4 activation quantisation first:
 *      G = amax/(6*448) (1 if amax == 0), s_b = e4m3_rne(amax_b / (6 G)),
 *      q = e2m1_rne_sat(v / (s_b G)), all in IEEE fp32 with correctly
 *      rounded division; the shared expert's h is rounded to bf16.
 *   7. cache residency is not an input: the output depends on (x, weights)
 *      (except under the optional renorm-skip of item 9).
 *   8. the adaptive cache's bookkeeping ("Project Maya" page, sections "How
 *      'most-used' is measured", "Promotion on every miss, eviction at the
 *      boundary" and "VRAM: one partition per layer"), an integer state
 *      machine simulated forward by forward (oracle_cache_policy_step).
 * Compiled with -ffp-contract=off so fp32 steps are single roundings.
 *   9. optional renorm-skip (Strata-GLM blog, section "Uncensoring without
 *      touching the weights"; oracle_renorm_skip): a token's cache-miss
 *      routes with weight below tau are dropped and its remaining weights
 *      renormalised.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ formats */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa; exponent 0
 * is subnormal (0 or 0.5). */
ORC_API double oracle_e2m1(unsigned c) {
  unsigned e = (c >> 1) & 3u, m = c & 1u;
  double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return (c & 8u) ? -mag : mag;
}

/* E4M3 (FN variant): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no inf. */
ORC_API double oracle_e4m3(unsigned b) {
  unsigned s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexp((double)m / 8.0, -6);
  else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

/* E8M0 (the MX scale, OCP Microscaling Formats v1.0): 8 exponent bits,
 * bias 127, no sign and no mantissa; 0xFF is NaN.  value = 2^(b - 127). */
ORC_API double oracle_e8m0(unsigned b) {
  b &= 0xFFu;
  return b == 0xFFu ? NAN : ldexp(1.0, (int)b - 127);
}

/* bf16 is the top half of an IEEE binary32 */
ORC_API double oracle_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Negative controls: a planted defect makes the oracle wrong on purpose, so a
 * test can show that the parity check fails by a wide margin when such a
 * mistake is present.  0 = none (always the default). */
enum { ORC_DEFECT_NONE = 0, ORC_DEFECT_NIBBLE_SWAP = 1, ORC_DEFECT_SCALE_UE8M0 = 2,
       ORC_DEFECT_BLOCK_OFF_BY_ONE = 3, ORC_DEFECT_TIE_HIGH_ID = 4, ORC_DEFECT_SCALING_2_5 = 5 };
static int g_defect = ORC_DEFECT_NONE;
ORC_API void oracle_set_defect(int d) { g_defect = d; }

static double g_e2m1[16];
static double g_e4m3[256];
static double g_e8m0[256];
static int g_tables_ready = 0;

static void tables_init(void) {
  if (g_tables_ready) return;
  for (unsigned c = 0; c < 16; ++c) g_e2m1[c] = oracle_e2m1(c);
  for (unsigned b = 0; b < 256; ++b) g_e4m3[b] = oracle_e4m3(b);
  for (unsigned b = 0; b < 256; ++b) g_e8m0[b] = oracle_e8m0(b);
  g_tables_ready = 1;
}

/* record formats: NVFP4 = E4M3 scale per 16 values; MXFP4 = E8M0 scale per
 * 32 values (windlass README: GLM-5.2 in MXFP4) */
enum { ORC_NVFP4 = 0, ORC_MXFP4 = 1 };
static int orc_block(int fmt) { return fmt == ORC_MXFP4 ? 32 : 16; }

/* ----------------------------------------------------------- record access */

/* Expert record: codes of gate [I][H], up [I][H], down [H][I] (row-major,
 * element 2j in the low nibble), then their scales, one per block of 16
 * (NVFP4, E4M3) or 32 (MXFP4, E8M0) elements, in 512-byte atoms: block kb of
 * row r in atom (r/128, kb/4) at ((r/128)*(KB/4) + kb/4)*512, byte
 * (r%32)*16 + ((r%128)/32)*4 + kb%4 inside it, KB = blocks per row. */
typedef struct {
  const uint8_t* codes;
  const uint8_t* scales;
  int R, K, fmt;
  double g;
} orc_mat;

static orc_mat orc_matrix(const uint8_t* rec, int H, int I, int fmt, int m, const float* g3) {
  orc_mat M;
  size_t gu_codes = (size_t)I * (size_t)H / 2;
  size_t all_codes = 3 * gu_codes;
  size_t gu_scales = (size_t)I * (size_t)H / (size_t)orc_block(fmt);
  M.R = (m == 2) ? H : I;
  M.K = (m == 2) ? I : H;
  M.fmt = fmt;
  M.codes = rec + (size_t)m * gu_codes;
  M.scales = rec + all_codes + (size_t)m * gu_scales;
  M.g = (double)g3[m];
  return M;
}

static size_t orc_scale_pos(int r, int kb, int KB) {
  size_t atom = (size_t)(r / 128) * (size_t)(KB / 4) + (size_t)(kb / 4);
  return atom * 512 + (size_t)(r % 32) * 16 + (size_t)((r % 128) / 32) * 4 + (size_t)(kb % 4);
}

/* W[r][c] as a double */
static double orc_w(const orc_mat* M, int r, int c) {
  uint8_t byte = M->codes[(size_t)r * (size_t)(M->K / 2) + (size_t)(c / 2)];
  int hi = (c & 1);
  if (g_defect == ORC_DEFECT_NIBBLE_SWAP) hi = !hi;
  unsigned code = hi ? (byte >> 4) : (byte & 15u);
  const int bl = orc_block(M->fmt), KB = M->K / bl;
  int kb = c / bl;
  if (g_defect == ORC_DEFECT_BLOCK_OFF_BY_ONE) kb = (kb + 1) % KB;
  uint8_t sb = M->scales[orc_scale_pos(r, kb, KB)];
  /* the scale-decoding defect reads each format's byte as the other's */
  int mx = M->fmt == ORC_MXFP4;
  if (g_defect == ORC_DEFECT_SCALE_UE8M0) mx = !mx;
  double s = mx ? g_e8m0[sb] : g_e4m3[sb];
  return g_e2m1[code] * s * M->g;
}

/* one dequantised weight, exported for the format pins */
ORC_API double oracle_weight(const uint8_t* rec, int H, int I, int fmt, int m, int r, int c,
                             const float* g3) {
  tables_init();
  orc_mat M = orc_matrix(rec, H, I, fmt, m, g3);
  return orc_w(&M, r, c);
}

/* y = W x for one matrix, fp64 */
static void orc_matvec(const orc_mat* M, const double* x, double* y) {
  #pragma omp parallel for schedule(static)
  for (int r = 0; r < M->R; ++r) {
    double acc = 0.0;
    for (int c = 0; c < M->K; ++c) acc += orc_w(M, r, c) * x[c];
    y[r] = acc;
  }
}

/* whole matrix dequantised, row-major [R][K], for brute-force pins */
ORC_API void oracle_dequant_matrix(const uint8_t* rec, int H, int I, int fmt, int m,
                                   const float* g3, double* out) {
  tables_init();
  orc_mat M = orc_matrix(rec, H, I, fmt, m, g3);
  for (int r = 0; r < M.R; ++r)
    for (int c = 0; c < M.K; ++c) out[(size_t)r * M.K + c] = orc_w(&M, r, c);
}

/* ------------------------------------------------------------------ router */

typedef struct { double l; int id; } orc_pair;

static int orc_pair_cmp(const void* a, const void* b) {
  const orc_pair* p = (const orc_pair*)a;
  const orc_pair* q = (const orc_pair*)b;
  if (p->l > q->l) return -1;
  if (p->l < q->l) return 1;
  if (g_defect == ORC_DEFECT_TIE_HIGH_ID) return (p->id > q->id) ? -1 : (p->id < q->id);
  return (p->id < q->id) ? -1 : (p->id > q->id);
}

/* Router for T tokens.  x [T][H] bf16, Wr [E][H] fp32, bias [E] (nullable).
 * Outputs ids [T][k], w [T][k], p_sel [T][k], logits [T][E] (nullable),
 * gap [T] (nullable) = smallest difference between consecutive logits among
 * the k+1 largest (E > k), used to reject near-ties when drawing inputs. */
ORC_API void oracle_route(const uint16_t* x, const float* Wr, const float* bias, int T, int H,
                          int E, int k, int32_t* ids, double* w, double* p_sel, double* logits,
                          double* gap) {
  #pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    orc_pair* ord = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)E);
    double* xd = (double*)malloc(sizeof(double) * (size_t)H);
    for (int h = 0; h < H; ++h) xd[h] = oracle_bf16(x[(size_t)t * H + h]);
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += (double)Wr[(size_t)e * H + h] * xd[h];
      if (bias) acc += (double)bias[e];
      ord[e].l = acc;
      ord[e].id = e;
      if (logits) logits[(size_t)t * E + e] = acc;
    }
    qsort(ord, (size_t)E, sizeof(orc_pair), orc_pair_cmp);
    double lmax = ord[0].l;
    double z_all = 0.0, z_sel = 0.0;
    for (int e = 0; e < E; ++e) z_all += exp(ord[e].l - lmax);
    for (int j = 0; j < k; ++j) z_sel += exp(ord[j].l - lmax);
    for (int j = 0; j < k; ++j) {
      double pj = exp(ord[j].l - lmax);
      ids[(size_t)t * k + j] = ord[j].id;
      if (p_sel) p_sel[(size_t)t * k + j] = pj / z_all;
      if (w) w[(size_t)t * k + j] = pj / z_sel;
    }
    if (gap) {
      double gmin = INFINITY;
      for (int j = 0; j < k && j + 1 < E; ++j) {
        double d = ord[j].l - ord[j + 1].l;
        if (d < gmin) gmin = d;
      }
      gap[t] = gmin;
    }
    free(xd);
    free(ord);
  }
}

/* ------------------------------------------------------------------ permute */

/* Stable counting sort of routes r = t*k + j by expert id: perm[p] = r for
 * the p-th route in (expert asc, r asc) order; inv[r] = p. */
ORC_API int oracle_permute(const int32_t* ids, int T, int k, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv) {
  int n = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int r = 0; r < n; ++r) {
    if (ids[r] < 0 || ids[r] >= E) return 1;
    counts[ids[r]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int r = 0; r < n; ++r) {
    int p = fill[ids[r]]++;
    perm[p] = r;
    inv[r] = p;
  }
  free(fill);
  return 0;
}

/* ------------------------------------------------- NVFP4 activation quant */

/* nearest E4M3 value to t >= 0 (brute force over the finite codes), ties to
 * the even code, values above 448 saturate to 448 (code 0x7E) */
ORC_API unsigned oracle_e4m3_rne(float t) {
  tables_init();
  if (!(t > 0.0f)) return 0;
  unsigned best = 0;
  double bd = INFINITY;
  for (unsigned b = 0; b <= 0x7E; ++b) {
    double d = fabs(g_e4m3[b] - (double)t);
    if (d < bd || (d == bd && (b & 1u) == 0)) { bd = d; best = b; }
  }
  return best;
}

/* nearest E2M1 magnitude to |q| (brute force), ties to the even code,
 * saturating at 6; the sign bit follows the sign bit of q */
ORC_API unsigned oracle_e2m1_rne_sat(float q) {
  tables_init();
  double a = fabs((double)q);
  unsigned best = 0;
  double bd = INFINITY;
  for (unsigned c = 0; c < 8; ++c) {
    double d = fabs(g_e2m1[c] - a);
    if (d < bd || (d == bd && (c & 1u) == 0)) { bd = d; best = c; }
  }
  if (a > 6.0) best = 7;
  return signbit(q) ? (best | 8u) : best;
}

/* NVFP4 quantisation of one row of n fp32 values (n % 16 == 0): codes [n/2]
 * (element 2j in the low nibble), scales [n/16] (row order, one per block),
 * G (per-row fp32 global).  Returns nothing; all steps in IEEE fp32. */
ORC_API void oracle_nvfp4_quant(const float* v, int n, uint8_t* codes, uint8_t* scales,
                                float* G_out) {
  tables_init();
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  volatile float six448 = 2688.0f;
  float G = (amax > 0.0f) ? amax / six448 : 1.0f;
  *G_out = G;
  for (int b = 0; b < n / 16; ++b) {
    float ab = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float a = fabsf(v[b * 16 + i]);
      if (a > ab) ab = a;
    }
    volatile float sixG = 6.0f * G;
    float t = ab / sixG;
    unsigned s = oracle_e4m3_rne(t);
    scales[b] = (uint8_t)s;
    volatile float sdq = (float)g_e4m3[s] * G;
    for (int i = 0; i < 16; i += 2) {
      unsigned lo = 0, hi = 0;
      if (s != 0) {
        float q0 = v[b * 16 + i] / sdq;
        float q1 = v[b * 16 + i + 1] / sdq;
        lo = oracle_e2m1_rne_sat(q0);
        hi = oracle_e2m1_rne_sat(q1);
      }
      codes[(b * 16 + i) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/* value of a quantised row, fp64 */
static void orc_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float G, int n,
                              double* out) {
  for (int i = 0; i < n; ++i) {
    unsigned c = (i & 1) ? (codes[i / 2] >> 4) : (codes[i / 2] & 15u);
    out[i] = g_e2m1[c] * g_e4m3[scales[i / 16]] * (double)G;
  }
}

/* nearest E2M1 magnitude to |q| for an exact double q (ties to the even
 * code, saturating at 6), sign bit from q */
static unsigned orc_e2m1_rne_sat_d(double q) {
  double a = fabs(q);
  unsigned best = 0;
  double bd = INFINITY;
  for (unsigned c = 0; c < 8; ++c) {
    double d = fabs(g_e2m1[c] - a);
    if (d < bd || (d == bd && (c & 1u) == 0)) { bd = d; best = c; }
  }
  if (a > 6.0) best = 7;
  return signbit(q) ? (best | 8u) : best;
}

/* MXFP4 quantisation of one row of n fp32 values (n % 32 == 0), after OCP
 * Microscaling Formats v1.0 (the conversion of a block of 32 values to an
 * MX block): the block's shared exponent is X = floor(log2(max |v|)) - 2 (2
 * = the exponent of E2M1's largest normal, 6 = 1.5 x 2^2), limited to the
 * E8M0 range [-127, 127]; scale byte X + 127; each element's code is the
 * E2M1 value nearest v / 2^X (exact), ties to even, saturating at 6.  An
 * all-zero block gets scale byte 0 and codes 0.  codes [n/2] (element 2j in
 * the low nibble), scales [n/32] in row order. */
ORC_API void oracle_mxfp4_quant(const float* v, int n, uint8_t* codes, uint8_t* scales) {
  tables_init();
  for (int b = 0; b < n / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      double a = fabs((double)v[b * 32 + i]);
      if (a > amax) amax = a;
    }
    int X = -127;
    if (amax > 0.0) {
      int e;
      frexp(amax, &e);  /* amax = f 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
      X = e - 1 - 2;
      if (X < -127) X = -127;
      if (X > 127) X = 127;
    }
    scales[b] = (uint8_t)(amax > 0.0 ? X + 127 : 0);
    for (int i = 0; i < 32; i += 2) {
      unsigned lo = 0, hi = 0;
      if (amax > 0.0) {
        lo = orc_e2m1_rne_sat_d(ldexp((double)v[b * 32 + i], -X));
        hi = orc_e2m1_rne_sat_d(ldexp((double)v[b * 32 + i + 1], -X));
      }
      codes[(b * 32 + i) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/* quantise-then-dequantise of a row given in fp32, in the prefill numerics
 * of the record format: NVFP4 (E4M3 per 16, fp32 global) or MXFP4 (E8M0 per
 * 32) - the tensor cores take both operands' block scales in one format */
static void orc_act_quant(const float* v, int n, int fmt, double* out) {
  uint8_t* codes = (uint8_t*)malloc((size_t)n / 2);
  uint8_t* scales = (uint8_t*)malloc((size_t)n / 16);
  if (fmt == ORC_MXFP4) {
    oracle_mxfp4_quant(v, n, codes, scales);
    for (int i = 0; i < n; ++i) {
      unsigned c = (i & 1) ? (codes[i / 2] >> 4) : (codes[i / 2] & 15u);
      out[i] = g_e2m1[c] * g_e8m0[scales[i / 32]];
    }
  } else {
    float G;
    oracle_nvfp4_quant(v, n, codes, scales, &G);
    orc_nvfp4_dequant(codes, scales, G, n, out);
  }
  free(codes);
  free(scales);
}

/* Rounding-boundary slack of an NVFP4 quantisation.  Two implementations
 * whose fp32 inputs differ in the last bits may round an element that sits
 * next to a rounding boundary to either neighbour; both results are correct.
 * The margins say how close counts as "next to":
 *   - an element whose scaled magnitude q = |v| / (s G) lies within
 *     g_flip_q code units of an E2M1 midpoint (0.25, 0.75, ..., 5) may take
 *     either neighbouring code: delta = the distance between the two codes'
 *     values, (hi - lo) s G;
 *   - a block whose scale argument t = amax_b / (6 G) lies within relative
 *     g_flip_t of an E4M3 midpoint may take either neighbouring scale s1 <
 *     s2.  Under s2 a value is within half a code step (at most 1, between
 *     codes 4 and 6) of v / (s2 G); under s1 the values above 6 s1 G
 *     saturate, by at most 6 G (t - s1) <= 3 s2 G (s1 = 0 included), the
 *     others are within s1 G.  So every element gets delta = 4 s2 G.
 * delta[i] receives the largest change of element i's quantised value that
 * such a flip can cause, 0 elsewhere.  Same fp32 steps as
 * oracle_nvfp4_quant.  The margins are set well above the difference
 * between an fp64 value rounded to fp32 and the same value summed in fp32
 * by another implementation (oracle_set_flip_margins). */
static double g_flip_q = 2e-5;
static double g_flip_t = 1e-5;
static double g_flip_bf16 = 2e-6;

ORC_API void oracle_set_flip_margins(double q_codes, double t_rel, double bf16_rel) {
  g_flip_q = q_codes;
  g_flip_t = t_rel;
  g_flip_bf16 = bf16_rel;
}

static const double g_mids[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
static const double g_lo_mag[7] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0};
static const double g_hi_mag[7] = {0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static void orc_nv_flip_delta(const float* v, int n, double* delta) {
  const double* mids = g_mids;
  const double* lo_mag = g_lo_mag;
  const double* hi_mag = g_hi_mag;
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  volatile float six448 = 2688.0f;
  float G = (amax > 0.0f) ? amax / six448 : 1.0f;
  for (int b = 0; b < n / 16; ++b) {
    float ab = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float a = fabsf(v[b * 16 + i]);
      if (a > ab) ab = a;
    }
    volatile float sixG = 6.0f * G;
    float t = ab / sixG;
    unsigned s = oracle_e4m3_rne(t);
    /* block scale next to an E4M3 rounding boundary (between codes c-1, c) */
    double s_hi = -1.0;
    for (unsigned c = 1; c <= 0x7E && s_hi < 0.0; ++c) {
      double mid = 0.5 * (g_e4m3[c - 1] + g_e4m3[c]);
      if (fabs((double)t - mid) <= g_flip_t * mid) s_hi = g_e4m3[c];
    }
    double sg = g_e4m3[s] * (double)G;
    for (int i = 0; i < 16; ++i) {
      double d = 0.0;
      if (s_hi >= 0.0) d = 4.0 * s_hi * (double)G;
      else if (s != 0) {
        double q = fabs((double)v[b * 16 + i]) / sg;
        for (int j = 0; j < 7; ++j)
          if (fabs(q - mids[j]) <= g_flip_q) d = (hi_mag[j] - lo_mag[j]) * sg;
      }
      delta[b * 16 + i] = d;
    }
  }
}

/* The same for MXFP4 blocks of 32: an element within g_flip_q code units of
 * an E2M1 midpoint of v / 2^X gets one code step x 2^X; a block whose max
 * |v| lies within relative g_flip_t of a power of two may take the shared
 * exponent X or X + 1: under 2^(X+1) a value is within one code unit
 * (2^(X+1)) of v, under 2^X within 2^X or, saturated at 6 x 2^X, within
 * 8 x 2^X - 6 x 2^X = 2^(X+1); every element gets delta = 2 x 2^(X+1). */
static void orc_mx_flip_delta(const float* v, int n, double* delta) {
  for (int b = 0; b < n / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      double a = fabs((double)v[b * 32 + i]);
      if (a > amax) amax = a;
    }
    int X = -127, near_pow2 = 0;
    if (amax > 0.0) {
      int e;
      double f = frexp(amax, &e);  /* amax = f 2^e, f in [0.5, 1) */
      X = e - 3;
      if (X < -127) X = -127;
      if (X > 127) X = 127;
      /* distance to 2^(e-1) (just above it) or 2^e (just below it) */
      near_pow2 = (f - 0.5) <= g_flip_t * 0.5 || (1.0 - f) <= g_flip_t;
      if (near_pow2 && (1.0 - f) <= g_flip_t) X = X + 1 > 127 ? 127 : X + 1;
    }
    const double sx = ldexp(1.0, X);
    for (int i = 0; i < 32; ++i) {
      double d = 0.0;
      if (near_pow2) d = 2.0 * sx;
      else if (amax > 0.0) {
        double q = fabs((double)v[b * 32 + i]) / sx;
        for (int j = 0; j < 7; ++j)
          if (fabs(q - g_mids[j]) <= g_flip_q) d = (g_hi_mag[j] - g_lo_mag[j]) * sx;
      }
      delta[b * 32 + i] = d;
    }
  }
}

static void orc_quant_flip_delta(const float* v, int n, int fmt, double* delta) {
  if (fmt == ORC_MXFP4) orc_mx_flip_delta(v, n, delta);
  else orc_nv_flip_delta(v, n, delta);
}

ORC_API void oracle_quant_flip_delta(const float* v, int n, int fmt, double* delta) {
  tables_init();
  orc_quant_flip_delta(v, n, fmt, delta);
}

/* bf16 rounding slack: one bf16 step when the value lies within relative
 * g_flip_bf16 of a bf16 rounding midpoint */
static double orc_bf16_flip_delta(double hv) {
  float f = (float)hv;
  uint32_t b;
  memcpy(&b, &f, 4);
  uint32_t lo = b & 0xFFFF0000u, hi = lo + 0x10000u;
  float flo, fhi;
  memcpy(&flo, &lo, 4);
  memcpy(&fhi, &hi, 4);
  double mid = 0.5 * ((double)flo + (double)fhi);
  return (fabs(hv - mid) <= g_flip_bf16 * fabs(mid)) ? fabs((double)fhi - (double)flo) : 0.0;
}

ORC_API void oracle_bf16_flip_delta(const double* v, int n, double* delta) {
  for (int i = 0; i < n; ++i) delta[i] = orc_bf16_flip_delta(v[i]);
}

/* ------------------------------------------------------------------ experts */

static double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* h = silu(Wg x) * (Wu x), fp64, for one activation vector x [H] -> h [I] */
static void orc_expert_h(const orc_mat* Mg, const orc_mat* Mu, int I, const double* x,
                         double* h) {
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  orc_matvec(Mg, x, g);
  orc_matvec(Mu, x, u);
  for (int i = 0; i < I; ++i) h[i] = orc_silu(g[i]) * u[i];
  free(g);
  free(u);
}

/* One routed expert on one activation vector x [H] -> o [H].
 * act_quant != 0: prefill numerics (h rounded to fp32 and NVFP4-quantised
 * before the down projection; x must already be the quantised value).
 * bound (nullable, act_quant only): bound[r] += wabs * sum_i |Wd[r][i]| *
 * delta_i, the most that rounding-boundary flips of h can move o[r] * wabs. */
static void orc_expert_impl(const uint8_t* rec, int H, int I, int fmt, const float* g3,
                            const double* x,
                            int act_quant, double* o, double wabs, double* bound) {
  tables_init();
  orc_mat Mg = orc_matrix(rec, H, I, fmt, 0, g3);
  orc_mat Mu = orc_matrix(rec, H, I, fmt, 1, g3);
  orc_mat Md = orc_matrix(rec, H, I, fmt, 2, g3);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  orc_expert_h(&Mg, &Mu, I, x, h);
  if (act_quant) {
    float* hf = (float*)malloc(sizeof(float) * (size_t)I);
    for (int i = 0; i < I; ++i) hf[i] = (float)h[i];
    if (bound) {
      double* delta = (double*)malloc(sizeof(double) * (size_t)I);
      orc_quant_flip_delta(hf, I, fmt, delta);
      for (int i = 0; i < I; ++i) {
        if (delta[i] == 0.0) continue;
        for (int r = 0; r < H; ++r) bound[r] += wabs * fabs(orc_w(&Md, r, i)) * delta[i];
      }
      free(delta);
    }
    orc_act_quant(hf, I, fmt, h);
    free(hf);
  }
  orc_matvec(&Md, h, o);
  free(h);
}

ORC_API void oracle_expert(const uint8_t* rec, int H, int I, int fmt, const float* g3,
                           const double* x,
                           int act_quant, double* o) {
  orc_expert_impl(rec, H, I, fmt, g3, x, act_quant, o, 0.0, NULL);
}

/* h [I] (fp64, before any quantisation) of one routed expert on x [H]
 * (already the quantised value in prefill numerics) */
ORC_API void oracle_expert_h(const uint8_t* rec, int H, int I, int fmt, const float* g3,
                             const double* x,
                             double* h) {
  tables_init();
  orc_mat Mg = orc_matrix(rec, H, I, fmt, 0, g3);
  orc_mat Mu = orc_matrix(rec, H, I, fmt, 1, g3);
  orc_expert_h(&Mg, &Mu, I, x, h);
}

/* Prefill numerics: for each token t of x [T][H] (bf16) with routes ids
 * [T][k], the number of elements of its routes' h (rounded to fp32) that
 * lie within the margins of an NVFP4 rounding boundary (nonzero slack of
 * orc_quant_flip_delta), where another implementation's fp32 sums may round
 * them to the neighbouring code.  rec[e] as in oracle_layer_forward. */
ORC_API void oracle_prefill_near_boundary(const uint16_t* x, int T, int H, int I, int fmt, int k,
                                          const int32_t* ids, const uint8_t* const* rec,
                                          const float* g, int32_t* count) {
  tables_init();
  #pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    double* xq = (double*)malloc(sizeof(double) * (size_t)H);
    float* xf = (float*)malloc(sizeof(float) * (size_t)H);
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    float* hf = (float*)malloc(sizeof(float) * (size_t)I);
    double* delta = (double*)malloc(sizeof(double) * (size_t)I);
    for (int c = 0; c < H; ++c) xf[c] = (float)oracle_bf16(x[(size_t)t * H + c]);
    orc_act_quant(xf, H, fmt, xq);
    int n = 0;
    for (int j = 0; j < k; ++j) {
      const int e = ids[(size_t)t * k + j];
      orc_mat Mg = orc_matrix(rec[e], H, I, fmt, 0, g + 3 * e);
      orc_mat Mu = orc_matrix(rec[e], H, I, fmt, 1, g + 3 * e);
      orc_expert_h(&Mg, &Mu, I, xq, h);
      for (int i = 0; i < I; ++i) hf[i] = (float)h[i];
      orc_quant_flip_delta(hf, I, fmt, delta);
      for (int i = 0; i < I; ++i) n += delta[i] != 0.0;
    }
    count[t] = n;
    free(xq); free(xf); free(h); free(hf); free(delta);
  }
}

/* Shared expert with bf16 weights gate/up [Is][H], down [H][Is].
 * round_h_bf16 != 0: h is rounded to bf16 (RNE) before the down projection. */
static void orc_shared_impl(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, int H,
                            int Is, const double* x, int round_h_bf16, double* o, double* bound) {
  double* h = (double*)malloc(sizeof(double) * (size_t)Is);
  double* hd = bound ? (double*)calloc((size_t)Is, sizeof(double)) : NULL;
  #pragma omp parallel for schedule(static)
  for (int i = 0; i < Is; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += oracle_bf16(wg[(size_t)i * H + c]) * x[c];
      u += oracle_bf16(wu[(size_t)i * H + c]) * x[c];
    }
    double hv = orc_silu(g) * u;
    if (hd) hd[i] = orc_bf16_flip_delta(hv);
    if (round_h_bf16) {
      float f = (float)hv;
      uint32_t b;
      memcpy(&b, &f, 4);
      b = (b + 0x7FFFu + ((b >> 16) & 1u)) & 0xFFFF0000u;
      memcpy(&f, &b, 4);
      hv = (double)f;
    }
    h[i] = hv;
  }
  #pragma omp parallel for schedule(static)
  for (int r = 0; r < H; ++r) {
    double acc = 0.0, bd = 0.0;
    for (int i = 0; i < Is; ++i) {
      acc += oracle_bf16(wd[(size_t)r * Is + i]) * h[i];
      if (hd && hd[i] != 0.0) bd += fabs(oracle_bf16(wd[(size_t)r * Is + i])) * hd[i];
    }
    o[r] = acc;
    if (bound) bound[r] += bd;
  }
  free(h);
  free(hd);
}

ORC_API void oracle_shared(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, int H,
                           int Is, const double* x, int round_h_bf16, double* o) {
  orc_shared_impl(wg, wu, wd, H, Is, x, round_h_bf16, o, NULL);
}

/* -------------------------------------------------------------------- layer */

/* Full layer on T tokens.  rec[e] points to expert e's record (may be NULL
 * for experts no token selects; selecting one returns 2).  g [E][3].
 * Shared weights may be NULL (Is == 0).  mode 0 = decode numerics, 1 =
 * prefill numerics (activation quantisation).  Outputs y [T][H] (fp64) and,
 * when non-NULL, ids/w/p_sel [T][k] and, in mode 1, ybound [T][H]: the most
 * that rounding-boundary flips of the intermediate quantisations (h to NVFP4,
 * shared h to bf16) can move each output, for comparisons with another
 * implementation of the same rounding steps. */
/* --renorm-skip (Strata-GLM blog, "Uncensoring without touching the weights"):
 * a route of token t whose expert is a cache miss (resident[e] == 0) and
 * whose combine weight is below tau is dropped - never gathered or computed -
 * and the token's remaining weights are renormalised to sum to 1.  keep[r] = 1 for kept routes; w_eff
 * the renormalised weights (0 for dropped routes).  tau = 0 keeps every route
 * and w_eff = w. */
ORC_API void oracle_renorm_skip(const int32_t* ids, const double* w, int T, int k,
                                const uint8_t* resident, double tau, double* w_eff,
                                uint8_t* keep) {
  for (int t = 0; t < T; ++t) {
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      const int r = t * k + j;
      keep[r] = !(resident && !resident[ids[r]] && w[r] < tau);
      if (keep[r]) sum += w[r];
    }
    for (int j = 0; j < k; ++j) {
      const int r = t * k + j;
      w_eff[r] = keep[r] ? w[r] / sum : 0.0;
    }
  }
}

/* The layer.  resident/tau: the renorm-skip above (resident == NULL: exact). */
ORC_API int oracle_layer_forward(const uint16_t* x, int T, int H, int I, int fmt, int E, int k,
                                 int Is,
                                 const float* Wr, const float* bias, const uint8_t* const* rec,
                                 const float* g, const uint16_t* sg, const uint16_t* su,
                                 const uint16_t* sd, int mode, const uint8_t* resident,
                                 double tau, double* y, int32_t* ids_out, double* w_out,
                                 double* p_out, double* ybound) {
  tables_init();
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  double* p = (double*)malloc(sizeof(double) * (size_t)T * k);
  double* weff = (double*)malloc(sizeof(double) * (size_t)T * k);
  uint8_t* keep = (uint8_t*)malloc((size_t)T * k);
  oracle_route(x, Wr, bias, T, H, E, k, ids, w, p, NULL, NULL);
  oracle_renorm_skip(ids, w, T, k, resident, resident ? tau : 0.0, weff, keep);
  for (int r = 0; r < T * k; ++r)
    if (keep[r] && !rec[ids[r]]) {
      free(ids); free(w); free(p); free(weff); free(keep);
      return 2;
    }
  /* tokens are independent: one per thread (each token's own steps in order);
   * a single token keeps the threads for its row loops instead */
  #pragma omp parallel for schedule(dynamic, 1) if (T > 1)
  for (int t = 0; t < T; ++t) {
    double* xd = (double*)malloc(sizeof(double) * (size_t)H);
    double* xq = (double*)malloc(sizeof(double) * (size_t)H);
    float* xf = (float*)malloc(sizeof(float) * (size_t)H);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    for (int c = 0; c < H; ++c) {
      xd[c] = oracle_bf16(x[(size_t)t * H + c]);
      xf[c] = (float)xd[c];
    }
    if (mode == 1) orc_act_quant(xf, H, fmt, xq);
    else memcpy(xq, xd, sizeof(double) * (size_t)H);
    double* yt = y + (size_t)t * H;
    double* bt = (ybound && mode == 1) ? ybound + (size_t)t * H : NULL;
    if (ybound) for (int c = 0; c < H; ++c) ybound[(size_t)t * H + c] = 0.0;
    for (int c = 0; c < H; ++c) yt[c] = 0.0;
    for (int j = 0; j < k; ++j) {
      if (!keep[(size_t)t * k + j]) continue;
      int e = ids[(size_t)t * k + j];
      double wj = weff[(size_t)t * k + j];
      orc_expert_impl(rec[e], H, I, fmt, g + 3 * e, xq, mode == 1, o, fabs(wj), bt);
      if (g_defect == ORC_DEFECT_SCALING_2_5) wj *= 2.5;
      for (int c = 0; c < H; ++c) yt[c] += wj * o[c];
    }
    if (Is > 0 && sg && su && sd) {
      orc_shared_impl(sg, su, sd, H, Is, xd, mode == 1, o, bt);
      for (int c = 0; c < H; ++c) yt[c] += o[c];
    }
    free(xd); free(xq); free(xf); free(o);
  }
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * k);
  if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)T * k);
  if (p_out) memcpy(p_out, p, sizeof(double) * (size_t)T * k);
  free(ids); free(w); free(p); free(weff); free(keep);
  return 0;
}

/* ------------------------------------------------------- adaptive cache policy */

/* One layer forward of the adaptive expert cache ("Project Maya" page).
 * State (caller-owned, all layers): table[L*E] slot or -1; cnt[L*E] decayed
 * route counts; last[L*E] the layer-forward number of the expert's latest
 * route (0 = never); stamp[L] forwards of each layer so far; *events route
 * events since the last halving; freeslot[n_cache] 1 = a free (spare) slot.
 * Layer `layer` owns cache slots [slot_lo, slot_hi).  counts[E] = this
 * forward's routes per expert.  In this order:
 *   1. lookup: the active experts (counts > 0) not in the table are the
 *      misses, in ascending id;
 *   2. promotion on the miss: miss i takes the i-th lowest free slot of the
 *      layer, while there is one, and is resident from then on
 *      (promoted[i] = that slot, else -1: it goes through a staging slot);
 *   3. counts: each route adds 1, capped at 2^24; the expert's last = this
 *      forward's number; every 32,768 route events (counted over all layers,
 *      checked after a forward) every count of every layer is halved;
 *   4. boundary: while the layer has fewer than K free slots, its resident
 *      with the smallest (count, last, id) is evicted and its slot is free.
 * Returns the number of misses. */
ORC_API int oracle_cache_policy_step(int L, int E, int layer, int slot_lo, int slot_hi, int K,
                                     int32_t* table, uint32_t* cnt, uint32_t* last,
                                     uint32_t* stamp, uint32_t* events, uint8_t* freeslot,
                                     const int32_t* counts, int32_t* promoted) {
  int32_t* tab = table + (size_t)layer * E;
  uint32_t* c = cnt + (size_t)layer * E;
  uint32_t* ls = last + (size_t)layer * E;
  int n_miss = 0;
  for (int e = 0; e < E; ++e) {
    if (counts[e] <= 0 || tab[e] >= 0) continue;
    int slot = -1;
    for (int s = slot_lo; s < slot_hi; ++s)
      if (freeslot[s]) { slot = s; break; }
    if (slot >= 0) {
      freeslot[slot] = 0;
      tab[e] = slot;
    }
    promoted[n_miss++] = slot;
  }
  const uint32_t now = ++stamp[layer];
  uint64_t routes = 0;
  for (int e = 0; e < E; ++e) {
    if (counts[e] <= 0) continue;
    routes += (uint64_t)counts[e];
    uint64_t v = (uint64_t)c[e] + (uint64_t)counts[e];
    c[e] = v > (1u << 24) ? (1u << 24) : (uint32_t)v;
    ls[e] = now;
  }
  *events += (uint32_t)routes;
  if (*events >= 32768u) {
    for (size_t i = 0; i < (size_t)L * E; ++i) cnt[i] >>= 1;
    *events = 0;
  }
  for (;;) {
    int n_free = 0;
    for (int s = slot_lo; s < slot_hi; ++s) n_free += freeslot[s] != 0;
    if (n_free >= K) break;
    int victim = -1;
    for (int e = 0; e < E; ++e) {
      if (tab[e] < 0) continue;
      if (victim < 0 || c[e] < c[victim] || (c[e] == c[victim] && ls[e] < ls[victim]))
        victim = e;  /* ascending e: the lowest id wins the remaining ties */
    }
    if (victim < 0) break;
    freeslot[tab[victim]] = 1;
    tab[victim] = -1;
  }
  return n_miss;
}

/* ----------------------------------------------- per-layer slot budgets */

/* Greedy per-layer slot budget ("Project Maya" page, section "VRAM: one
 * partition per layer, sized by what the layer routes"): with counts[l][e]
 * the routes of expert e in layer l (per-layer sums below 2^32):
 *   1. order each layer's experts by count, descending, ties to the lower id
 *      (order[l][0..E));
 *   2. every layer gets `floor` slots (its `floor` most-routed experts);
 *   3. each further slot, one at a time, goes to the layer whose next
 *      expert in that order serves the largest share of the layer's lookups,
 *      counts[l][next] / sum_e counts[l][e] (0 for a layer without routes),
 *      ties to the lower layer; a layer whose E experts all have slots takes
 *      no more.
 * Slots left once every layer is full stay unassigned.  layer_slots[L+1] =
 * the partition's prefix sums (layer l owns [layer_slots[l],
 * layer_slots[l+1])); layer l's residents are order[l][0 .. n_l).  Returns
 * 0, or 1 when floor > E or total < L * floor. */
ORC_API int oracle_slot_budget(int L, int E, const uint32_t* counts, int total, int floor,
                               int32_t* layer_slots, int32_t* order) {
  if (floor < 0 || floor > E || total < L * floor) return 1;
  uint64_t* sum = (uint64_t*)calloc((size_t)L, sizeof(uint64_t));
  int* n = (int*)malloc(sizeof(int) * (size_t)L);
  for (int l = 0; l < L; ++l) {
    const uint32_t* c = counts + (size_t)l * E;
    int32_t* o = order + (size_t)l * E;
    for (int e = 0; e < E; ++e) {
      o[e] = e;
      sum[l] += c[e];
    }
    /* insertion sort: count descending, then id ascending */
    for (int i = 1; i < E; ++i) {
      int32_t v = o[i];
      int j = i - 1;
      while (j >= 0 && (c[o[j]] < c[v] || (c[o[j]] == c[v] && o[j] > v))) {
        o[j + 1] = o[j];
        --j;
      }
      o[j + 1] = v;
    }
    n[l] = floor;
  }
  for (int given = L * floor; given < total; ++given) {
    int best = -1;
    for (int l = 0; l < L; ++l) {
      if (n[l] >= E) continue;
      if (best < 0) { best = l; continue; }
      /* share of l's next expert > share of best's next expert, exactly:
       * c_l / S_l > c_b / S_b  <=>  c_l * S_b > c_b * S_l (a layer without
       * routes has share 0) */
      uint64_t cl = sum[l] ? counts[(size_t)l * E + order[(size_t)l * E + n[l]]] : 0;
      uint64_t cb = sum[best] ? counts[(size_t)best * E + order[(size_t)best * E + n[best]]] : 0;
      uint64_t Sl = sum[l] ? sum[l] : 1, Sb = sum[best] ? sum[best] : 1;
      if (cl * Sb > cb * Sl) best = l;
    }
    if (best < 0) break;
    ++n[best];
  }
  layer_slots[0] = 0;
  for (int l = 0; l < L; ++l) layer_slots[l + 1] = layer_slots[l] + n[l];
  free(sum);
  free(n);
  return 0;
}
