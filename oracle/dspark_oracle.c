/*
 * dspark_oracle.c -- plain, slow, CPU reference of the DSpark sequential
 * Markov draft-sampling loop and its verify side.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA sources.
 *
 * Every function follows the definition on the pages it cites, written out
 * element by element with no blocking, fusion or reordering:
 *
 *   [P1] "Dspark Kernels" (TensorRT Edge-LLM C++ API, dsparkKernels.html):
 *        dsparkBuildVerifyTokens, dsparkGreedyAccept.
 *   [P2] vllm.models.kimi_k3.nvidia.specialized_decode.drafter.markov:
 *        module docstring (exactness paragraph), _gumbel_key, _loop_rest.
 *   [P3] vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.markov:
 *        module docstring, _StepKernel.kernel, _logit, _gumbel,
 *        _murmur_prefix, _combine, _w1_row, _nonzero_f32, anchor_embed.
 *   [P4] vllm.models.deepseek_v41.amd.ops.fused_markov: module docstring.
 *
 * Floating point: compile with -O2 -ffp-contract=off and no fast-math, so
 * that every float expression below is one IEEE binary32 operation rounded
 * to nearest even, and fmaf() is the fused multiply-add.
 *
 * Readings of points the pages leave open:
 *   - the MurmurHash3 block step (_MURMUR_MIX, not printed) is the published
 *     MurmurHash3_x86_32 block mix; the printed tail fixes the finaliser;
 *   - logf/tanhf are the library's own functions (below), because the pages'
 *     logf and tanhf are a vendor math library's; division is IEEE;
 *   - the bias is the exactly rounded dot product (any FP32 order is allowed
 *     by [P2]/[P4]; the exact value is the one order-free definition);
 *   - a request index outside [0, num_req) marks the row invalid, like a
 *     negative one ([P3] _StepKernel.kernel: valid = req >= 0).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "dspark_oracle.h"

/* ------------------------------------------------------------------------ */
/* BF16 <-> FP32                                                            */
/* ------------------------------------------------------------------------ */

float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round-to-nearest-even FP32 -> BF16; every NaN becomes the canonical
 * 0x7FFF (the value a cvt.rn.bf16.f32 of [P3] _logit produces). */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return 0x7FFF;
  uint32_t upper = u >> 16, lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* ------------------------------------------------------------------------ */
/* Own natural logarithm (replaces the pages' vendor logf).                */
/* For positive normal finite x:                                            */
/*   x = 2^e * m with m in [sqrt(1/2), sqrt(2)),  f = m - 1 (exact),        */
/*   log(1 + f) = 2 atanh(s),  s = f / (2 + f),                             */
/*   2 atanh(s) = 2s + s*R,  R = sum_{n>=1} 2 z^n / (2n+1),  z = s^2,       */
/*   and since 2s = f - s*f = f - (hfsq - s*hfsq) with hfsq = f^2 / 2:      */
/*   log(1 + f) = f - (hfsq - s * (hfsq + R)),                              */
/*   log x = e * ln2 + log m, ln2 split as LN2_HI + LN2_LO (Cody-Waite), so */
/*   that e * LN2_HI is exact.                                              */
/* Coefficients 2/(2n+1) are the Taylor coefficients of 2 atanh, each       */
/* rounded once to binary32 (the compiler rounds the double quotient; none  */
/* of these quotients lies on a binary32 rounding boundary).                */
/* ------------------------------------------------------------------------ */

static const float LOG_C3 = (float)(2.0 / 3.0);
static const float LOG_C5 = (float)(2.0 / 5.0);
static const float LOG_C7 = (float)(2.0 / 7.0);
static const float LOG_C9 = (float)(2.0 / 9.0);
static const float LOG_C11 = (float)(2.0 / 11.0);
/* ln 2 with its last 8 significand bits cleared: e * LN2_HI is exact for
 * |e| < 2^8.  LN2_LO is the rest, rounded once. */
static const float LN2_HI = 0.693145751953125f;
#define ORACLE_LN2_DOUBLE 0.69314718055994530941723212145818
static const float LN2_LO = (float)(ORACLE_LN2_DOUBLE - 0.693145751953125);

float oracle_logf(float x) {
  uint32_t bits;
  memcpy(&bits, &x, 4);
  int e = (int)(bits >> 23) - 127;
  uint32_t mbits = (bits & 0x007FFFFFu) | 0x3F800000u; /* m in [1, 2) */
  if (mbits > 0x3FB504F3u) {                           /* m > RN(sqrt 2) */
    mbits -= 0x00800000u;                              /* m / 2 */
    e += 1;
  }
  float m;
  memcpy(&m, &mbits, 4);
  float f = m - 1.0f;
  float s = f / (2.0f + f);
  float z = s * s;
  float p = fmaf(z, LOG_C11, LOG_C9);
  p = fmaf(z, p, LOG_C7);
  p = fmaf(z, p, LOG_C5);
  p = fmaf(z, p, LOG_C3);
  float R = z * p;
  float hfsq = (0.5f * f) * f;
  float t = hfsq + R;
  float corr = fmaf(-s, t, hfsq);
  float logm = f - corr;
  float fe = (float)e;
  return fmaf(fe, LN2_HI, fmaf(fe, LN2_LO, logm));
}

/* ------------------------------------------------------------------------ */
/* Own hyperbolic tangent (replaces the pages' vendor tanhf, [P3] _logit). */
/*   tanh|z| = E / (E + 2),  E = expm1(2|z|),  sign restored at the end;    */
/*   |z| > 9.1: tanh rounds to 1 in binary32;  NaN propagates.              */
/*   expm1(x), x >= 0:  k = nearest integer to x / ln2,                     */
/*   r = x - k ln2 (Cody-Waite, |r| <= ln2/2 + tiny),                       */
/*   expm1(r) = r + r^2 (1/2! + r/3! + ... + r^7/9!)  (Taylor),             */
/*   expm1(x) = 2^k expm1(r) + (2^k - 1).                                   */
/* ------------------------------------------------------------------------ */

static const float INV_LN2 = (float)(1.0 / ORACLE_LN2_DOUBLE);
static const float EXP_C2 = (float)(1.0 / 2.0);
static const float EXP_C3 = (float)(1.0 / 6.0);
static const float EXP_C4 = (float)(1.0 / 24.0);
static const float EXP_C5 = (float)(1.0 / 120.0);
static const float EXP_C6 = (float)(1.0 / 720.0);
static const float EXP_C7 = (float)(1.0 / 5040.0);
static const float EXP_C8 = (float)(1.0 / 40320.0);
static const float EXP_C9 = (float)(1.0 / 362880.0);

static float own_expm1f_nonneg(float x) {
  float kf = rintf(x * INV_LN2);
  float r = fmaf(-kf, LN2_HI, x);
  r = fmaf(-kf, LN2_LO, r);
  float p = fmaf(r, EXP_C9, EXP_C8);
  p = fmaf(r, p, EXP_C7);
  p = fmaf(r, p, EXP_C6);
  p = fmaf(r, p, EXP_C5);
  p = fmaf(r, p, EXP_C4);
  p = fmaf(r, p, EXP_C3);
  p = fmaf(r, p, EXP_C2);
  float em1 = fmaf(r * r, p, r);
  int k = (int)kf;
  if (k == 0) return em1;
  float two_k = ldexpf(1.0f, k);
  return fmaf(two_k, em1, two_k - 1.0f);
}

float oracle_tanhf(float z) {
  if (isnan(z)) return z;
  float a = fabsf(z);
  float t;
  if (a > 9.1f) {
    t = 1.0f;
  } else {
    float E = own_expm1f_nonneg(2.0f * a);
    t = E / (E + 2.0f);
  }
  return copysignf(t, z);
}

/* ------------------------------------------------------------------------ */
/* Output transform ([P3] _logit; [P2] module docstring "the add is one    */
/* FP32 add rounded to the logits dtype"):                                  */
/*   hx = RN_bf16(f32(base) + f32(bias))          (add.bf16)                */
/*   y  = RN(mult * f32(hx))                                                */
/*   w  = has_cap ? RN(cap * tanh(RN(inv_cap * y))) : y                     */
/*   c  = RN_bf16(w), the cached (pre-temperature) logit; l = f32(c).       */
/* ------------------------------------------------------------------------ */

uint16_t oracle_logit(uint16_t base, uint16_t bias, float mult, int has_cap,
                      float inv_cap, float cap, float *l_out) {
  float sum = oracle_bf16_to_f32(base) + oracle_bf16_to_f32(bias);
  float x = oracle_bf16_to_f32(oracle_f32_to_bf16(sum));
  float y = mult * x;
  float w = y;
  if (has_cap) {
    float z = inv_cap * y;
    w = cap * oracle_tanhf(z);
  }
  uint16_t c = oracle_f32_to_bf16(w);
  if (l_out) *l_out = oracle_bf16_to_f32(c);
  return c;
}

/* ------------------------------------------------------------------------ */
/* Noise hash ([P3] _StepKernel.kernel, _murmur_prefix, _gumbel):          */
/* MurmurHash3_x86_32 with seed 0 over the four little-endian words         */
/*   lo32(step_seed), hi32(step_seed), lo32(pos - 1 + salt), vocab id,      */
/* step_seed = seed XOR (step << 32).                                       */
/* ------------------------------------------------------------------------ */

static uint32_t rotl32(uint32_t x, int r) { return (x << r) | (x >> (32 - r)); }

uint32_t oracle_murmur_block(uint32_t h, uint32_t k) {
  k *= 0xcc9e2d51u;
  k = rotl32(k, 15);
  k *= 0x1b873593u;
  h ^= k;
  h = rotl32(h, 13);
  h = h * 5u + 0xe6546b64u;
  return h;
}

uint32_t oracle_murmur_fmix(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

uint32_t oracle_noise_hash(int64_t seed, int32_t step, int64_t sample_pos,
                           uint32_t salt, uint32_t vocab_id) {
  uint64_t step_seed = (uint64_t)seed ^ ((uint64_t)(uint32_t)step << 32);
  uint64_t salted = (uint64_t)sample_pos - 1u + (uint64_t)salt;
  uint32_t h = 0;
  h = oracle_murmur_block(h, (uint32_t)(step_seed & 0xFFFFFFFFu));
  h = oracle_murmur_block(h, (uint32_t)(step_seed >> 32));
  h = oracle_murmur_block(h, (uint32_t)(salted & 0xFFFFFFFFu));
  h = oracle_murmur_block(h, vocab_id);
  h ^= 16u; /* key length in bytes */
  return oracle_murmur_fmix(h);
}

/* u = RN_f32((h + 0.5) / 2^32): [P3] _gumbel builds it as
 * fma(f32(h >> 16), 2^-16, (f32(h & 0xffff) + 0.5) * 2^-32), a single
 * rounding of the same exact value. */
float oracle_uniform(uint32_t h) {
  return (float)(((double)h + 0.5) * 0x1p-32);
}

/* log(1 - u) as [P3] _gumbel (and [P2] _log1p_neg_stable) computes it:
 * below 0.25 the Taylor series -u * (1 + u/2 + ... + u^7/8) in Horner form
 * with coefficients RN_f32(1/n); else log(max(RN(1 - u), 2^-24)). */
float oracle_log1m(float u) {
  if (u < 0.25f) {
    float poly = fmaf(u, (float)(1.0 / 8.0), (float)(1.0 / 7.0));
    poly = fmaf(u, poly, (float)(1.0 / 6.0));
    poly = fmaf(u, poly, (float)(1.0 / 5.0));
    poly = fmaf(u, poly, (float)(1.0 / 4.0));
    poly = fmaf(u, poly, (float)(1.0 / 3.0));
    poly = fmaf(u, poly, (float)(1.0 / 2.0));
    poly = fmaf(u, poly, 1.0f);
    return poly * (-u);
  }
  float om = 1.0f - u;
  float xa = om > 0x1p-24f ? om : 0x1p-24f;
  return oracle_logf(xa);
}

/* L(h) = log(-log(1 - u(h))); the Gumbel noise is -L ([P2] _gumbel_key,
 * _gumbel_log_arg32: the kernel takes the outer log itself). */
float oracle_noise_L(uint32_t h) {
  float u = oracle_uniform(h);
  float sel = oracle_log1m(u);
  return oracle_logf(-sel);
}

/* [P3] _nonzero_f32: temp != 0.0 as an ordered compare (NaN counts as
 * nonzero).  [P2] _gumbel_key: key = l / temp + g, g = -L, else l. */
float oracle_key(float l, float temp, uint32_t h) {
  if (temp == 0.0f) return l;
  float q = l / temp;
  return q - oracle_noise_L(h);
}

/* ------------------------------------------------------------------------ */
/* Total-order argmax ([P3] module docstring, _combine): the first NaN,    */
/* else the lowest index of the maximum (+0 == -0).                         */
/* ------------------------------------------------------------------------ */

int64_t oracle_argmax(const float *keys, int64_t n) {
  if (n <= 0) return -1;
  int64_t bi = 0;
  float best = keys[0];
  for (int64_t v = 1; v < n; v++) {
    if (isnan(best)) break;
    if (isnan(keys[v]) || keys[v] > best) {
      best = keys[v];
      bi = v;
    }
  }
  return bi;
}

/* [P3] _combine, written from its description: the first pair if v1 > v2,
 * or v1 == v2 and i1 < i2, or v1 is NaN and (v2 is not NaN or i1 < i2). */
int oracle_combine_first_wins(float v1, int64_t i1, float v2, int64_t i2) {
  if (isnan(v1)) return !isnan(v2) || i1 < i2;
  if (isnan(v2)) return 0;
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

/* ------------------------------------------------------------------------ */
/* Exactly rounded BF16 dot product ([P2] module docstring: "the FP32 dot  */
/* product of the embedding and the markov_w2 row rounded once"; any FP32   */
/* summation order is allowed, the exact sum is the order-free value).      */
/* Each BF16 value is sig * 2^exp with an integer sig < 256.  Products are  */
/* integers < 2^16 scaled by 2^(exp1+exp2), exp1 + exp2 >= -266; the sum   */
/* is kept exactly in two unsigned 640-bit integers (positive and negative  */
/* parts, bit 0 = 2^-266) and rounded once, to nearest even, to BF16.       */
/* ------------------------------------------------------------------------ */

#define ACC_LIMBS 10
#define ACC_OFFSET 266

typedef struct {
  uint64_t w[ACC_LIMBS];
} wide_t;

static void wide_add_shifted(wide_t *a, uint64_t mag, int pos) {
  int limb = pos / 64, sh = pos % 64;
  uint64_t lo = mag << sh;
  uint64_t hi = sh ? (mag >> (64 - sh)) : 0;
  uint64_t carry = 0;
  for (int i = limb; i < ACC_LIMBS; i++) {
    uint64_t add = (i == limb) ? lo : (i == limb + 1 ? hi : 0);
    uint64_t s = a->w[i] + add;
    uint64_t c1 = s < add;
    uint64_t s2 = s + carry;
    uint64_t c2 = s2 < carry;
    a->w[i] = s2;
    carry = c1 + c2;
    if (i > limb + 1 && carry == 0) break;
  }
}

static int wide_cmp(const wide_t *a, const wide_t *b) {
  for (int i = ACC_LIMBS - 1; i >= 0; i--) {
    if (a->w[i] != b->w[i]) return a->w[i] > b->w[i] ? 1 : -1;
  }
  return 0;
}

static void wide_sub(wide_t *r, const wide_t *a, const wide_t *b) { /* a >= b */
  uint64_t borrow = 0;
  for (int i = 0; i < ACC_LIMBS; i++) {
    uint64_t d = a->w[i] - b->w[i];
    uint64_t b1 = a->w[i] < b->w[i];
    uint64_t d2 = d - borrow;
    uint64_t b2 = d < borrow;
    r->w[i] = d2;
    borrow = b1 + b2;
  }
}

static int wide_bit(const wide_t *a, int pos) {
  if (pos < 0) return 0;
  return (int)((a->w[pos / 64] >> (pos % 64)) & 1u);
}

static int wide_any_below(const wide_t *a, int pos) { /* bits [0, pos) */
  for (int i = 0; i < pos; i++)
    if (wide_bit(a, i)) return 1;
  return 0;
}

static int wide_top(const wide_t *a) {
  for (int i = ACC_LIMBS - 1; i >= 0; i--) {
    if (a->w[i]) {
      for (int b = 63; b >= 0; b--)
        if ((a->w[i] >> b) & 1u) return i * 64 + b;
    }
  }
  return -1;
}

/* BF16 fields -> (sig, exp) with value = sig * 2^exp; 0 for zero. */
static void bf16_parts(uint16_t b, uint32_t *sig, int *exp) {
  int E = (b >> 7) & 0xFF;
  uint32_t M = b & 0x7F;
  if (E == 0) {
    *sig = M;
    *exp = 1 - 134;
  } else {
    *sig = 128u + M;
    *exp = E - 134;
  }
}

/* Round sign * mag * 2^-ACC_OFFSET to BF16, nearest even. */
static uint16_t wide_to_bf16(const wide_t *mag, int negative) {
  uint16_t sign = negative ? 0x8000 : 0;
  int t = wide_top(mag);
  if (t < 0) return sign;
  /* lowest kept bit: 8 significant bits, but never below the BF16
   * subnormal quantum 2^-133 (accumulator bit 133). */
  int q = t - 7;
  if (q < 133) q = 133;
  uint32_t kept = 0;
  for (int b = t; b >= q; b--) kept = (kept << 1) | (uint32_t)wide_bit(mag, b);
  int rbit = wide_bit(mag, q - 1);
  int sticky = wide_any_below(mag, q - 1);
  if (rbit && (sticky || (kept & 1u))) kept += 1u;
  if (kept == 0) return sign;
  if (q == 133 && kept < 128u) return (uint16_t)(sign | kept); /* subnormal */
  if (kept >= 256u) {
    kept >>= 1;
    q += 1;
  }
  int E = q - 132;
  if (E >= 255) return (uint16_t)(sign | 0x7F80);
  return (uint16_t)(sign | ((uint32_t)E << 7) | (kept - 128u));
}

uint16_t oracle_dot_bf16(const uint16_t *a, const uint16_t *b, int n) {
  int has_nan = 0, has_pinf = 0, has_ninf = 0, all_negzero = 1;
  wide_t pos, neg;
  memset(&pos, 0, sizeof(pos));
  memset(&neg, 0, sizeof(neg));
  for (int j = 0; j < n; j++) {
    uint16_t x = a[j], y = b[j];
    int x_nan = ((x & 0x7F80) == 0x7F80) && (x & 0x7F);
    int y_nan = ((y & 0x7F80) == 0x7F80) && (y & 0x7F);
    int x_inf = (x & 0x7FFF) == 0x7F80, y_inf = (y & 0x7FFF) == 0x7F80;
    int x_zero = (x & 0x7FFF) == 0, y_zero = (y & 0x7FFF) == 0;
    int negative = ((x ^ y) & 0x8000) != 0;
    if (x_nan || y_nan) {
      has_nan = 1;
      continue;
    }
    if (x_inf || y_inf) {
      if (x_zero || y_zero) has_nan = 1; /* inf * 0 */
      else if (negative) has_ninf = 1;
      else has_pinf = 1;
      continue;
    }
    if (x_zero || y_zero) {
      if (!negative) all_negzero = 0;
      continue;
    }
    all_negzero = 0;
    uint32_t sx, sy;
    int ex, ey;
    bf16_parts(x, &sx, &ex);
    bf16_parts(y, &sy, &ey);
    uint64_t mag = (uint64_t)sx * (uint64_t)sy;
    int at = ex + ey + ACC_OFFSET;
    wide_add_shifted(negative ? &neg : &pos, mag, at);
  }
  if (has_nan || (has_pinf && has_ninf)) return 0x7FFF;
  if (has_pinf) return 0x7F80;
  if (has_ninf) return 0xFF80;
  int c = wide_cmp(&pos, &neg);
  if (c == 0) return (n > 0 && all_negzero) ? 0x8000 : 0x0000;
  wide_t mag;
  if (c > 0) wide_sub(&mag, &pos, &neg);
  else wide_sub(&mag, &neg, &pos);
  return wide_to_bf16(&mag, c < 0);
}

/* ------------------------------------------------------------------------ */
/* [P1] dsparkQuantizeMarkovW2Fp8 / dsparkMarkovGreedyFusedStepFp8: w2 as   */
/* E4M3 bytes (bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN,   */
/* largest 448) with one FP16 scale per row, rowScale = rowAbsMax / 448.   */
/* Readings (the pages give the format and the scale rule only):           */
/*   - rowAbsMax = max |w| over the row's non-NaN BF16 values; the scale is */
/*     RN(rowAbsMax / 448) in FP32, then to FP16 (nearest even; beyond      */
/*     65504 it saturates to 65504);                                        */
/*   - q = E4M3(RN(w / s)) in FP32, nearest even, saturating to +-448 (the  */
/*     hardware conversion's satfinite mode); NaN gives 0x7F; a row whose  */
/*     scale is 0 stores zeros;                                             */
/*   - the step's bias is s * (sum_j e_j * decode(q_j)), the scale applied  */
/*     to the exact sum, rounded once to BF16, as the BF16 path's dot       */
/*     ([P2] module docstring).                                             */
/* ------------------------------------------------------------------------ */

float oracle_e4m3_value(uint8_t q) {
  const int E = (q >> 3) & 15, M = q & 7;
  const double sg = (q & 0x80) ? -1.0 : 1.0;
  if (E == 15 && M == 7) return NAN;
  if (E == 0) return (float)(sg * ldexp((double)M, -9));
  return (float)(sg * ldexp((double)(8 + M), E - 10));
}

uint8_t oracle_e4m3_from_f32(float x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) { /* subnormals: multiples of 2^-9; 8 is the smallest normal */
    const double m = nearbyint(ldexp(a, 9));
    return (uint8_t)(sign | (uint8_t)m);
  }
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int E = e - 1 + 7;
  double m = nearbyint(ldexp(a, 3 - (e - 1))); /* [8, 16] */
  if (m == 16.0) {
    m = 8.0;
    E += 1;
  }
  return (uint8_t)(sign | (uint8_t)((E << 3) | ((int)m - 8)));
}

float oracle_f16_value(uint16_t h) {
  const int E = (h >> 10) & 31, M = h & 1023;
  const double sg = (h & 0x8000) ? -1.0 : 1.0;
  if (E == 31) return M ? NAN : (float)(sg * INFINITY);
  if (E == 0) return (float)(sg * ldexp((double)M, -24));
  return (float)(sg * ldexp((double)(1024 + M), E - 25));
}

uint16_t oracle_f16_from_f32(float x) {
  if (isnan(x)) return 0x7E00;
  const uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
  const double a = fabs((double)x);
  if (a >= 65504.0) return (uint16_t)(sign | 0x7BFF);
  if (a < ldexp(1.0, -14)) { /* subnormals: multiples of 2^-24; 1024 is the smallest normal */
    const double m = nearbyint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)m);
  }
  int e;
  frexp(a, &e);
  int E = e - 1 + 15;
  double m = nearbyint(ldexp(a, 10 - (e - 1))); /* [1024, 2048] */
  if (m == 2048.0) {
    m = 1024.0;
    E += 1;
  }
  return (uint16_t)(sign | (uint16_t)((E << 10) | ((int)m - 1024)));
}

void oracle_quantize_w2_fp8(const uint16_t *w2, uint8_t *q, uint16_t *scale, int64_t vocab, int rank) {
  for (int64_t v = 0; v < vocab; v++) {
    const uint16_t *row = w2 + v * rank;
    float amax = 0.0f;
    for (int j = 0; j < rank; j++) {
      const float w = oracle_bf16_to_f32(row[j]);
      if (!isnan(w) && fabsf(w) > amax) amax = fabsf(w);
    }
    const uint16_t s16 = oracle_f16_from_f32(amax / 448.0f);
    const float s = oracle_f16_value(s16);
    scale[v] = s16;
    for (int j = 0; j < rank; j++)
      q[v * rank + j] = s == 0.0f ? 0x00 : oracle_e4m3_from_f32(oracle_bf16_to_f32(row[j]) / s);
  }
}

static void f16_parts(uint16_t h, uint32_t *sig, int *exp) {
  const int E = (h >> 10) & 31;
  const uint32_t M = h & 1023u;
  if (E == 0) {
    *sig = M;
    *exp = -24;
  } else {
    *sig = 1024u + M;
    *exp = E - 25;
  }
}

static void e4m3_parts(uint8_t q, uint32_t *sig, int *exp) {
  const int E = (q >> 3) & 15;
  const uint32_t M = q & 7u;
  if (E == 0) {
    *sig = M;
    *exp = -9;
  } else {
    *sig = 8u + M;
    *exp = E - 10;
  }
}

/* RN_bf16(s * sum_j e_j * decode(q_j)) exactly, the scale applied to the
 * exact sum.  For a finite nonzero scale each product of the three factors
 * is an integer below 2^23 times 2^(sum of exponents) >= 2^-166, kept in the
 * same 640-bit accumulators as the BF16 dot; a zero, infinite or NaN scale
 * meets the exact sum's class (zero with its sign, infinite, NaN) by the
 * IEEE rules of one multiplication. */
uint16_t oracle_dot_fp8(const uint16_t *e, const uint8_t *q, uint16_t scale, int n) {
  const int s_nan = ((scale & 0x7C00) == 0x7C00) && (scale & 0x3FF);
  const int s_inf = (scale & 0x7FFF) == 0x7C00;
  const int s_zero = (scale & 0x7FFF) == 0;
  const int s_neg = (scale & 0x8000) != 0;
  const int s_finite = !s_nan && !s_inf && !s_zero;
  int has_nan = 0, has_pinf = 0, has_ninf = 0, all_negzero = 1;
  wide_t pos, neg;
  memset(&pos, 0, sizeof(pos));
  memset(&neg, 0, sizeof(neg));
  uint32_t ss = 1;
  int es = 0;
  if (s_finite) f16_parts(scale, &ss, &es);
  for (int j = 0; j < n; j++) {
    const uint16_t x = e[j];
    const uint8_t y = q[j];
    const int x_nan = ((x & 0x7F80) == 0x7F80) && (x & 0x7F);
    const int y_nan = (y & 0x7F) == 0x7F;
    const int x_inf = (x & 0x7FFF) == 0x7F80;
    const int x_zero = (x & 0x7FFF) == 0, y_zero = (y & 0x7F) == 0;
    const int negative = (((x & 0x8000) != 0) ^ ((y & 0x80) != 0)) != 0; /* sign of e_j * d_j */
    if (x_nan || y_nan) {
      has_nan = 1;
      continue;
    }
    if (x_inf) {
      if (y_zero) has_nan = 1; /* inf * 0 */
      else if (negative) has_ninf = 1;
      else has_pinf = 1;
      continue;
    }
    if (x_zero || y_zero) {
      if (!negative) all_negzero = 0;
      continue;
    }
    all_negzero = 0;
    uint32_t sx, sy;
    int ex, ey;
    bf16_parts(x, &sx, &ex);
    e4m3_parts(y, &sy, &ey);
    wide_add_shifted(negative ? &neg : &pos, (uint64_t)sx * sy * ss, ex + ey + es + ACC_OFFSET);
  }
  const int sum_nan = has_nan || (has_pinf && has_ninf);
  const int sum_inf = has_pinf || has_ninf;
  const int c = wide_cmp(&pos, &neg);
  /* sign of the exact sum: an infinity's, else the accumulators', else -0 when every product was -0 */
  const int sum_neg = sum_inf ? has_ninf : (c != 0 ? c < 0 : (n > 0 && all_negzero));
  const uint16_t sign = (uint16_t)((sum_neg ^ s_neg) ? 0x8000 : 0x0000);
  if (s_nan || sum_nan) return 0x7FFF;
  if (sum_inf) return s_zero ? 0x7FFF : (uint16_t)(sign | 0x7F80);
  if (s_inf) return c == 0 ? 0x7FFF : (uint16_t)(sign | 0x7F80); /* inf * 0 */
  if (s_zero || c == 0) return sign;
  wide_t mag;
  if (c > 0) wide_sub(&mag, &pos, &neg);
  else wide_sub(&mag, &neg, &pos);
  return (uint16_t)(wide_to_bf16(&mag, 0) | sign);
}

void oracle_dot_fp8_rows(const uint16_t *e, const uint8_t *q, const uint16_t *scale, uint16_t *out, int64_t rows,
                         int n) {
  for (int64_t r = 0; r < rows; r++) out[r] = oracle_dot_fp8(e + r * n, q + r * n, scale[r], n);
}
void oracle_e4m3_value_array(const uint8_t *q, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_value(q[i]);
}
void oracle_e4m3_from_f32_array(const float *x, uint8_t *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_from_f32(x[i]);
}
void oracle_f16_value_array(const uint16_t *h, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_f16_value(h[i]);
}
void oracle_f16_from_f32_array(const float *x, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_f16_from_f32(x[i]);
}

/* ------------------------------------------------------------------------ */
/* The loop ([P2] _loop_rest; [P3] module docstring, _StepKernel.kernel,   */
/* anchor_embed, _w1_row).  For each step s and row r:                     */
/*   prev(0)   = sext32(input_ids[anchor_idx[r]])                           */
/*   e         = w1[min(u64(prev), w1_rows - 1)]                            */
/*   bias[v]   = RN_bf16(exact dot(e, w2[v]))   (or the fed bias)           */
/*   (c, l)    = transform(base[r, s, v], bias[v])                          */
/*   cache[req, s, v] = c when the row is valid                             */
/*   key[v]    = temp != 0 ? RN(RN(l / temp) - L(h(r, s, v))) : l           */
/*   token     = total-order argmax of key; tokens[r, s] = token; prev = it */
/* ------------------------------------------------------------------------ */

typedef struct {
  const oracle_loop_args *a;
  int32_t r, s;
  const uint16_t *e;
  int64_t req;
  int valid;
  float temp;
  int64_t seed;
  int64_t pos;
  int has_cap;
  float inv_cap;
  float *keys;
  int64_t v0, v1;
} row_step_job;

static void *row_step_range(void *arg) {
  row_step_job *j = (row_step_job *)arg;
  const oracle_loop_args *a = j->a;
  const int64_t V = a->vocab;
  const uint16_t *base_row = a->base + (int64_t)j->r * a->base_s0 + (int64_t)j->s * a->base_s1;
  for (int64_t v = j->v0; v < j->v1; v++) {
    uint16_t b;
    if (a->fed_bias)
      b = a->fed_bias[((int64_t)j->r * a->steps + j->s) * V + v];
    else if (a->w2_fp8)
      b = oracle_dot_fp8(j->e, a->w2_fp8 + v * a->rank, a->w2_scale[v], a->rank);
    else
      b = oracle_dot_bf16(j->e, a->w2 + v * a->rank, a->rank);
    if (a->bias_out) a->bias_out[((int64_t)j->r * a->steps + j->s) * V + v] = b;
    float l;
    uint16_t c = oracle_logit(base_row[v], b, a->mult, j->has_cap, j->inv_cap, a->cap, &l);
    if (j->valid && a->cache) a->cache[j->req * a->cache_s0 + (int64_t)j->s * a->cache_s1 + v] = c;
    if (a->logits_out) a->logits_out[((int64_t)j->r * a->steps + j->s) * V + v] = c;
    uint32_t h = oracle_noise_hash(j->seed, j->s, j->pos, a->salt, (uint32_t)v);
    j->keys[v] = oracle_key(l, j->temp, h);
  }
  return NULL;
}

int oracle_markov_loop(const oracle_loop_args *a) {
  if (!a || a->vocab <= 0 || a->rank <= 0 || a->w1_rows <= 0 || a->rows < 0 || a->steps < 0)
    return -1;
  const int64_t V = a->vocab;
  int nthreads = a->nthreads > 0 ? a->nthreads : 1;
  if (nthreads > 256) nthreads = 256;
  float *keys = (float *)malloc(sizeof(float) * (size_t)V);
  if (!keys) return -2;
  int has_cap = a->cap != 0.0f;
  float inv_cap = has_cap ? 1.0f / a->cap : 0.0f;
  pthread_t th[256];
  row_step_job jobs[256];
  for (int32_t r = 0; r < a->rows; r++) {
    int64_t prev = (int64_t)a->input_ids[a->anchor_idx[r]]; /* int32, sign-extended */
    for (int32_t s = 0; s < a->steps; s++) {
      uint64_t last = (uint64_t)(a->w1_rows - 1);
      uint64_t row = (uint64_t)prev < last ? (uint64_t)prev : last;
      const uint16_t *e = a->w1 + (int64_t)row * a->rank;
      int64_t req = a->req_idx ? a->req_idx[(int64_t)r * a->req_s0 + s] : r;
      int valid = req >= 0 && req < a->num_req;
      float temp = valid ? a->temperature[req] : 0.0f;
      int64_t seed = valid ? a->seeds[req] : 0;
      int64_t pos = a->sample_pos[(int64_t)r * a->pos_s0 + s];
      int64_t chunk = (V + nthreads - 1) / nthreads;
      int launched[256];
      int njobs = 0;
      for (int t = 0; t < nthreads; t++) {
        int64_t v0 = (int64_t)t * chunk, v1 = v0 + chunk;
        if (v0 >= V) break;
        if (v1 > V) v1 = V;
        row_step_job jb = {a, r, s, e, req, valid, temp, seed, pos, has_cap, inv_cap, keys, v0, v1};
        jobs[t] = jb;
        launched[t] = nthreads > 1 && pthread_create(&th[t], NULL, row_step_range, &jobs[t]) == 0;
        if (!launched[t]) row_step_range(&jobs[t]);
        njobs++;
      }
      for (int t = 0; t < njobs; t++)
        if (launched[t]) pthread_join(th[t], NULL);
      int64_t tok = oracle_argmax(keys, V);
      a->tokens[(int64_t)r * a->tokens_s0 + s] = tok;
      if (a->keys_out) memcpy(a->keys_out + ((int64_t)r * a->steps + s) * V, keys, sizeof(float) * (size_t)V);
      prev = tok;
    }
  }
  free(keys);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* [P1] dsparkBuildVerifyTokens:                                            */
/*   verify[b, 0] = last[b];  verify[b, j + 1] = draft[b, j], j < P.        */
/* ------------------------------------------------------------------------ */

void oracle_build_verify_tokens(const int64_t *last, const int64_t *draft, int64_t *verify,
                                int32_t batch, int32_t draft_stride, int32_t P) {
  for (int32_t b = 0; b < batch; b++) {
    verify[(int64_t)b * (P + 1)] = last[b];
    for (int32_t j = 0; j < P; j++)
      verify[(int64_t)b * (P + 1) + j + 1] = draft[(int64_t)b * draft_stride + j];
  }
}

/* ------------------------------------------------------------------------ */
/* [P1] dsparkGreedyAccept: a_j = argmax(logits[b, j, :]) (total order);    */
/* accept draft[b, j] while it equals a_j, j < min(proposal_len[b], P);    */
/* then append the bonus a_n.  accepted[b] = a_0 .. a_n, then -1;           */
/* accept_len[b] = n + 1 (the accepted drafts plus the bonus token).        */
/* ------------------------------------------------------------------------ */

static int64_t argmax_bf16_row(const uint16_t *row, int64_t n, float *scratch) {
  for (int64_t v = 0; v < n; v++) scratch[v] = oracle_bf16_to_f32(row[v]);
  return oracle_argmax(scratch, n);
}

int oracle_greedy_accept(const uint16_t *logits, const int64_t *draft, const int32_t *proposal_len,
                         int64_t *accepted, int32_t *accept_len, int32_t batch, int32_t draft_stride,
                         int32_t P, int64_t vocab) {
  float *scratch = (float *)malloc(sizeof(float) * (size_t)(vocab > 0 ? vocab : 1));
  if (!scratch) return -2;
  for (int32_t b = 0; b < batch; b++) {
    int32_t pl = proposal_len[b];
    if (pl < 0) pl = 0;
    if (pl > P) pl = P;
    const uint16_t *rows = logits + (int64_t)b * (P + 1) * vocab;
    int32_t n = 0;
    int64_t a = argmax_bf16_row(rows, vocab, scratch);
    while (n < pl && draft[(int64_t)b * draft_stride + n] == a) {
      accepted[(int64_t)b * (P + 1) + n] = a;
      n++;
      a = argmax_bf16_row(rows + (int64_t)n * vocab, vocab, scratch);
    }
    accepted[(int64_t)b * (P + 1) + n] = a;
    for (int32_t j = n + 1; j <= P; j++) accepted[(int64_t)b * (P + 1) + j] = -1;
    accept_len[b] = n + 1;
  }
  free(scratch);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Probabilistic verify side ([P1] dsparkFillUniforms,                       */
/* dsparkProbabilisticAccept).                                               */
/* ------------------------------------------------------------------------ */

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011): ten rounds of
 *   (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
 * with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key bumped by the Weyl
 * constants (0x9E3779B9, 0xBB67AE85) between rounds. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; round++) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
    const uint32_t n1 = (uint32_t)p1;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
    const uint32_t n3 = (uint32_t)p0;
    c[0] = n0;
    c[1] = n1;
    c[2] = n2;
    c[3] = n3;
  }
  for (int i = 0; i < 4; i++) out[i] = c[i];
}

/* [P1] dsparkFillUniforms: deterministic uniforms in [0, 1).  Reading:
 * element i takes word i % 4 of Philox4x32-10 at counter (offset + i / 4) as
 * a 64-bit number in the low two words (the high two zero) and key (lo, hi)
 * of the seed; the word's top 24 bits scaled by 2^-24 are the uniform. */
void oracle_fill_uniforms(float *u, int64_t n, uint64_t seed, uint64_t offset) {
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  for (int64_t i = 0; i < n; i++) {
    const uint64_t block = offset + (uint64_t)i / 4u;
    const uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), 0u, 0u};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    u[i] = (float)(out[i % 4] >> 8) * (1.0f / 16777216.0f);
  }
}

/* A probability as a fixed-point weight in units of 2^-40: clamp to [0, 1]
 * (NaN and negatives weigh 0) and truncate.  Sums of weights are exact, so
 * the sampled index does not depend on the order of the additions. */
uint64_t oracle_weight(float p) {
  if (!(p > 0.0f)) return 0u;
  if (p >= 1.0f) return (uint64_t)1 << 40;
  return (uint64_t)ldexp((double)p, 40);
}

/* Inverse-CDF sample of n weights with uniform u: U = floor(u 2^24),
 * T = floor(U S / 2^24) for the total S, the smallest index whose inclusive
 * prefix sum exceeds T; -1 when S = 0. */
int64_t oracle_sample_weights(const uint64_t *w, int64_t n, float u) {
  uint64_t total = 0;
  for (int64_t v = 0; v < n; v++) total += w[v];
  if (total == 0) return -1;
  float uu = u;
  if (!(uu > 0.0f)) uu = 0.0f;
  uint64_t U = (uint64_t)ldexp((double)uu, 24);
  if (U > 0xFFFFFFu) U = 0xFFFFFFu;
  const uint64_t T = (uint64_t)(((unsigned __int128)U * total) >> 24);
  uint64_t prefix = 0;
  for (int64_t v = 0; v < n; v++) {
    prefix += w[v];
    if (prefix > T) return v;
  }
  return n - 1; /* unreachable: T < S */
}

/* [P1] dsparkProbabilisticAccept, speculative sampling with residual
 * sampling.  target [B, P+1, V], draft [B, P, V] (FP32 probabilities),
 * uniforms [B, 2P+1]: u[j] decides draft position j, u[P + j] drives the
 * residual sample after a rejection at j, u[2P] the bonus sample after a full
 * accept.  Readings: position j accepts its draft token d when
 * RN(u[j] * q) < t, t = target[b, j, d], q = draft[b, j, d] (the multiplied
 * form of u < t / q; an id outside [0, V) is rejected); the residual is
 * max(0, RN(target - draft)) per id, sampled by oracle_sample_weights; a
 * residual of weight 0 samples the target row instead, and a target row of
 * weight 0 gives id 0; accepted[b] holds the accepted drafts then the sample,
 * then -1; accept_len = accepted drafts + 1 (as for greedy accept). */
int oracle_probabilistic_accept(const float *target, const float *draft_probs, const int64_t *draft,
                                const int32_t *proposal_len, const float *uniforms, int64_t *accepted,
                                int32_t *accept_len, int32_t batch, int32_t draft_stride, int32_t P,
                                int64_t vocab) {
  uint64_t *w = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(vocab > 0 ? vocab : 1));
  if (!w) return -2;
  for (int32_t b = 0; b < batch; b++) {
    int32_t pl = proposal_len[b];
    if (pl < 0) pl = 0;
    if (pl > P) pl = P;
    const float *tb = target + (int64_t)b * (P + 1) * vocab;
    const float *qb = draft_probs + (int64_t)b * P * vocab;
    const float *ub = uniforms + (int64_t)b * (2 * P + 1);
    int64_t *acc = accepted + (int64_t)b * (P + 1);
    int32_t j = 0;
    while (j < pl) {
      const int64_t d = draft[(int64_t)b * draft_stride + j];
      if (d < 0 || d >= vocab) break;
      const float t = tb[(int64_t)j * vocab + d];
      const float q = qb[(int64_t)j * vocab + d];
      if (!(ub[j] * q < t)) break;
      acc[j] = d;
      j++;
    }
    int64_t pick = -1;
    if (j < pl) {
      for (int64_t v = 0; v < vocab; v++) {
        float r = tb[(int64_t)j * vocab + v] - qb[(int64_t)j * vocab + v];
        w[v] = oracle_weight(r);
      }
      pick = oracle_sample_weights(w, vocab, ub[P + j]);
    }
    if (pick < 0) {
      const float ut = j < pl ? ub[P + j] : ub[2 * P];
      for (int64_t v = 0; v < vocab; v++) w[v] = oracle_weight(tb[(int64_t)j * vocab + v]);
      pick = oracle_sample_weights(w, vocab, ut);
      if (pick < 0) pick = 0;
    }
    acc[j] = pick;
    for (int32_t i = j + 1; i <= P; i++) acc[i] = -1;
    accept_len[b] = j + 1;
  }
  free(w);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* [P1] dsparkLogitsToProbabilities: a dense probability row after         */
/* temperature, top-k and top-p.  The pages name the three filters only;   */
/* the arithmetic below is this build's reading, chosen so that every      */
/* decision is an exact comparison:                                        */
/*   - temperature <= 0 or NaN is greedy: probability 1 at the lowest id   */
/*     of the largest non-NaN logit.                                        */
/*   - z = RN(l / T); -0 counts as +0; an id whose z is NaN (a NaN logit,  */
/*     or an infinite one over an infinite T) is dropped (probability 0).  */
/*   - top-k (0 < K < number of non-NaN logits): the K first ids in the    */
/*     order (z descending, id ascending).                                  */
/*   - e = own exp(x), x = z - m for the kept maximum m (x = 0 where        */
/*     z == m, so infinite logits share their mass); w = floor(e 2^40).    */
/*   - top-p (p < 1): the shortest prefix of the kept ids in the order     */
/*     (w descending, id ascending) whose weight sum reaches               */
/*     max(1, ceil(p W)), W the kept total (p <= 0: one id).               */
/*   - probability = RN(e / S) over the final set, S = RN(sum of its w)    */
/*     2^-40; 0 elsewhere.                                                  */
/* ------------------------------------------------------------------------ */

/* Own exp for x <= 0 (Cody-Waite with the ln 2 split above, Taylor degree
 * 7 on |r| <= ln2/2, scaling by 2^k in one rounding): NaN propagates, below
 * -104 (exp rounds to 0 in binary32) gives 0. */
float oracle_expf_nonpos(float x) {
  if (isnan(x)) return x;
  if (x < -104.0f) return 0.0f;
  float kf = rintf(x * INV_LN2);
  float r = fmaf(-kf, LN2_HI, x);
  r = fmaf(-kf, LN2_LO, r);
  float p = fmaf(r, EXP_C7, EXP_C6);
  p = fmaf(r, p, EXP_C5);
  p = fmaf(r, p, EXP_C4);
  p = fmaf(r, p, EXP_C3);
  p = fmaf(r, p, EXP_C2);
  p = fmaf(r, p, 1.0f);
  p = fmaf(r, p, 1.0f);
  int k = (int)kf;
  if (k >= -125) return p * ldexpf(1.0f, k);          /* exact */
  return (p * ldexpf(1.0f, k + 64)) * ldexpf(1.0f, -64); /* one rounding */
}

typedef struct {
  float key;
  uint64_t w;
  int64_t id;
} l2p_item;

static int cmp_key_desc(const void *a, const void *b) {
  const l2p_item *x = (const l2p_item *)a, *y = (const l2p_item *)b;
  if (x->key > y->key) return -1;
  if (x->key < y->key) return 1;
  return x->id < y->id ? -1 : (x->id > y->id);
}

static int cmp_w_desc(const void *a, const void *b) {
  const l2p_item *x = (const l2p_item *)a, *y = (const l2p_item *)b;
  if (x->w > y->w) return -1;
  if (x->w < y->w) return 1;
  return x->id < y->id ? -1 : (x->id > y->id);
}

/* max(1, ceil(p W)) for 0 < p < 1, exactly: p = M 2^E with M a 24-bit
 * integer. */
static uint64_t top_p_threshold(float p, uint64_t W) {
  if (!(p > 0.0f)) return 1;
  int e;
  float f = frexpf(p, &e); /* p = f 2^e, f in [0.5, 1) */
  uint64_t M = (uint64_t)ldexpf(f, 24);
  int shift = 24 - e;      /* p W = M W / 2^shift */
  if (shift >= 100) return 1;
  unsigned __int128 prod = (unsigned __int128)M * W;
  unsigned __int128 c = (prod + (((unsigned __int128)1 << shift) - 1)) >> shift;
  return c < 1 ? 1 : (uint64_t)c;
}

int oracle_logits_to_probs(const float *logits, float *probs, int32_t rows, int64_t vocab, float temperature,
                           int32_t top_k, float top_p) {
  l2p_item *it = (l2p_item *)malloc(sizeof(l2p_item) * (size_t)(vocab > 0 ? vocab : 1));
  float *e = (float *)malloc(sizeof(float) * (size_t)(vocab > 0 ? vocab : 1));
  if (!it || !e) {
    free(it);
    free(e);
    return -2;
  }
  for (int32_t r = 0; r < rows; r++) {
    const float *l = logits + (int64_t)r * vocab;
    float *out = probs + (int64_t)r * vocab;
    for (int64_t v = 0; v < vocab; v++) out[v] = 0.0f;
    if (!(temperature > 0.0f)) { /* greedy */
      int64_t best = -1;
      for (int64_t v = 0; v < vocab; v++)
        if (!isnan(l[v]) && (best < 0 || l[v] > l[best])) best = v;
      if (best >= 0) out[best] = 1.0f;
      continue;
    }
    int64_t n = 0;
    for (int64_t v = 0; v < vocab; v++) {
      float z = l[v] / temperature;
      if (isnan(z)) continue;
      if (z == 0.0f) z = 0.0f;
      it[n].key = z;
      it[n].id = v;
      n++;
    }
    if (n == 0) continue;
    qsort(it, (size_t)n, sizeof(l2p_item), cmp_key_desc);
    int64_t kept = (top_k > 0 && top_k < n) ? top_k : n;
    const float m = it[0].key;
    uint64_t W = 0;
    for (int64_t i = 0; i < kept; i++) {
      float x = it[i].key == m ? 0.0f : it[i].key - m;
      e[it[i].id] = oracle_expf_nonpos(x);
      it[i].w = oracle_weight(e[it[i].id]);
      W += it[i].w;
    }
    int64_t fin = kept;
    uint64_t S = W;
    if (top_p < 1.0f) {
      qsort(it, (size_t)kept, sizeof(l2p_item), cmp_w_desc);
      const uint64_t thr = top_p_threshold(top_p, W);
      uint64_t cum = 0;
      fin = 0;
      while (fin < kept && cum < thr) cum += it[fin++].w;
      S = cum;
    }
    const float Sf = ldexpf((float)S, -40);
    for (int64_t i = 0; i < fin; i++) out[it[i].id] = e[it[i].id] / Sf;
  }
  free(it);
  free(e);
  return 0;
}

void oracle_expf_nonpos_array(const float *x, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_expf_nonpos(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Array helpers for the tests (plain loops over the scalar functions).    */
/* ------------------------------------------------------------------------ */

void oracle_noise_L_array(const uint32_t *h, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_noise_L(h[i]);
}
void oracle_uniform_array(const uint32_t *h, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_uniform(h[i]);
}
void oracle_log1m_array(const float *u, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_log1m(u[i]);
}
void oracle_logf_array(const float *x, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_logf(x[i]);
}
void oracle_tanhf_array(const float *x, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_tanhf(x[i]);
}
void oracle_logit_array(const uint16_t *base, const uint16_t *bias, uint16_t *c, float *l,
                        int64_t n, float mult, float cap) {
  int has_cap = cap != 0.0f;
  float inv_cap = has_cap ? 1.0f / cap : 0.0f;
  for (int64_t i = 0; i < n; i++) c[i] = oracle_logit(base[i], bias[i], mult, has_cap, inv_cap, cap, &l[i]);
}
void oracle_noise_hash_array(int64_t seed, int32_t step, int64_t sample_pos, uint32_t salt,
                             const uint32_t *vocab_ids, uint32_t *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_noise_hash(seed, step, sample_pos, salt, vocab_ids[i]);
}
void oracle_dot_bf16_rows(const uint16_t *a, const uint16_t *b, uint16_t *out, int64_t rows, int n) {
  for (int64_t r = 0; r < rows; r++) out[r] = oracle_dot_bf16(a + r * n, b + r * n, n);
}
void oracle_f32_to_bf16_array(const float *x, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_bf16(x[i]);
}
void oracle_key_array(const float *l, float temp, const uint32_t *h, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_key(l[i], temp, h[i]);
}

/* ------------------------------------------------------------------------ */
/* Vocabulary-sharded loop ([P3] module docstring: with a vocab-parallel w2  */
/* each rank works on its vocab range, its last block writes a packet       */
/* instead of the token, markov_pick picks the winner from the gathered     */
/* per-rank packets, cache_fill scatters the gathered draft-logits shards). */
/* ------------------------------------------------------------------------ */

/* [P3] _finish, sharded: the packet of one rank's winner over its slice,
 * keys[0 .. width) being the keys of global ids vocab_offset + local:
 * [bits of the key, global id, 0, 0], the winner by the total order. */
void oracle_shard_packet(const float *keys, int64_t width, int64_t vocab_offset, uint32_t packet[4]) {
  int64_t local = oracle_argmax(keys, width);
  float v = keys[local];
  uint32_t bits;
  memcpy(&bits, &v, 4);
  packet[0] = bits;
  packet[1] = (uint32_t)(int32_t)(vocab_offset + local);
  packet[2] = 0;
  packet[3] = 0;
}

/* [P3] markov_pick: per row, the winner over the ranks' packets
 * packets[(k * rows + r) * 4 + ...], k = 0 .. tp - 1, by the total order on
 * (value, global id): the first NaN, else the largest value, ties to the
 * lower id (which, with rank k holding the ids above rank k - 1's, is the
 * unsharded argmax).  Written as a left-to-right pass with _combine. */
void oracle_pick(const uint32_t *packets, int32_t tp, int32_t rows, int64_t *tokens) {
  for (int32_t r = 0; r < rows; r++) {
    float best = 0.0f;
    int64_t best_id = -1;
    for (int32_t k = 0; k < tp; k++) {
      const uint32_t *pk = packets + ((int64_t)k * rows + r) * 4;
      float v;
      memcpy(&v, &pk[0], 4);
      int64_t id = (int64_t)(int32_t)pk[1];
      if (best_id < 0 || oracle_combine_first_wins(v, id, best, best_id)) {
        best = v;
        best_id = id;
      }
    }
    tokens[r] = best_id;
  }
}

/* [P3] cache_fill: the gathered rank-local caches src[k * src_s0 + (r *
 * steps + i) * shard + local] (rank k, row r, step i, local id) go to
 * cache[req * cache_s0 + i * cache_s1 + v] for v = k * shard + local < vocab,
 * for every (r, i) whose request req = req_idx[r * req_s0 + i] (r without
 * req_idx) is valid: 0 <= req < num_req.  Other rows are left as they are. */
void oracle_cache_fill(const uint16_t *src, int64_t src_s0, uint16_t *cache, int64_t cache_s0, int64_t cache_s1,
                       const int64_t *req_idx, int64_t req_s0, int64_t num_req, int32_t rows, int32_t steps,
                       int32_t shard, int32_t tp, int64_t vocab) {
  for (int32_t r = 0; r < rows; r++)
    for (int32_t i = 0; i < steps; i++) {
      int64_t req = req_idx ? req_idx[(int64_t)r * req_s0 + i] : r;
      if (req < 0 || req >= num_req) continue;
      for (int64_t v = 0; v < vocab; v++) {
        int64_t k = v / shard, local = v - k * shard;
        if (k >= tp) break;
        cache[req * cache_s0 + (int64_t)i * cache_s1 + v] =
            src[k * src_s0 + ((int64_t)r * steps + i) * shard + local];
      }
    }
}

/* ------------------------------------------------------------------------ */
/* Confidence-scored proposal lengths ([P1] "Dspark Kernels":               */
/* dsparkComputeConfidenceScores, dsparkComputeConfidenceAndProposalLengths, */
/* dsparkComputeConfidenceAndSPSProposalLengths).  The page gives the       */
/* inputs and one-line contracts; the readings taken:                       */
/*   - the confidence that draft position j is accepted is a logistic head: */
/*     z = RN_f32(exact dot(weight, feature)) + bias (one FP32 add), with   */
/*     feature = the draft hidden state of (b, j), followed (with the       */
/*     Markov term) by the Markov embedding w1[prev] of the token before    */
/*     position j (firstPrevTokens[b] for j = 0, draft[b, j - 1] after;     */
/*     clamped to the last w1 row as in the loop); score = sigmoid(z) by    */
/*     the library's own exp: E = exp(-|z|), RN(1 / RN(1 + E)) for z >= 0,  */
/*     RN(E / RN(1 + E)) below;                                             */
/*   - threshold scheduling proposes while the running product of scores   */
/*     (the chance that every draft so far is accepted) stays >= threshold, */
/*     clamped to [minProposalLen, maxProposalLen];                         */
/*   - SPS scheduling takes the length L in [min, max] whose expected       */
/*     output, 1 + the sum of the first L running products, per verify cost */
/*     cost[L] is largest (ties to the shorter), considering L > min only   */
/*     while the running product at L - 1 is >= the survival floor; the     */
/*     verify-bucket costs are the caller's (the page names a B100 cost     */
/*     model without giving it).                                            */
/* ------------------------------------------------------------------------ */

/* Round sign * mag * 2^-ACC_OFFSET to FP32, nearest even. */
static float wide_to_f32(const wide_t *mag, int negative) {
  int t = wide_top(mag);
  if (t < 0) return negative ? -0.0f : 0.0f;
  int q = t - 23; /* 24 significant bits, never below the quantum 2^-149 */
  if (q < ACC_OFFSET - 149) q = ACC_OFFSET - 149;
  uint32_t kept = 0;
  for (int b = t; b >= q; b--) kept = (kept << 1) | (uint32_t)wide_bit(mag, b);
  int rbit = wide_bit(mag, q - 1);
  int sticky = wide_any_below(mag, q - 1);
  if (rbit && (sticky || (kept & 1u))) kept += 1u;
  float v = ldexpf((float)kept, q - ACC_OFFSET); /* exact: kept <= 2^24 */
  return negative ? -v : v;
}

float oracle_dot_bf16_f32(const uint16_t *a, const uint16_t *b, int n) {
  int has_nan = 0, has_pinf = 0, has_ninf = 0, all_negzero = 1;
  wide_t pos, neg;
  memset(&pos, 0, sizeof(pos));
  memset(&neg, 0, sizeof(neg));
  for (int j = 0; j < n; j++) {
    uint16_t x = a[j], y = b[j];
    int x_nan = ((x & 0x7F80) == 0x7F80) && (x & 0x7F);
    int y_nan = ((y & 0x7F80) == 0x7F80) && (y & 0x7F);
    int x_inf = (x & 0x7FFF) == 0x7F80, y_inf = (y & 0x7FFF) == 0x7F80;
    int x_zero = (x & 0x7FFF) == 0, y_zero = (y & 0x7FFF) == 0;
    int negative = ((x ^ y) & 0x8000) != 0;
    if (x_nan || y_nan) {
      has_nan = 1;
      continue;
    }
    if (x_inf || y_inf) {
      if (x_zero || y_zero) has_nan = 1;
      else if (negative) has_ninf = 1;
      else has_pinf = 1;
      continue;
    }
    if (x_zero || y_zero) {
      if (!negative) all_negzero = 0;
      continue;
    }
    all_negzero = 0;
    uint32_t sx, sy;
    int ex, ey;
    bf16_parts(x, &sx, &ex);
    bf16_parts(y, &sy, &ey);
    wide_add_shifted(negative ? &neg : &pos, (uint64_t)sx * (uint64_t)sy, ex + ey + ACC_OFFSET);
  }
  if (has_nan || (has_pinf && has_ninf)) return NAN;
  if (has_pinf) return INFINITY;
  if (has_ninf) return -INFINITY;
  int c = wide_cmp(&pos, &neg);
  if (c == 0) return (n > 0 && all_negzero) ? -0.0f : 0.0f;
  wide_t mag;
  if (c > 0) wide_sub(&mag, &pos, &neg);
  else wide_sub(&mag, &neg, &pos);
  return wide_to_f32(&mag, c < 0);
}

float oracle_sigmoid(float z) {
  if (isnan(z)) return z;
  float a = z < 0.0f ? -z : z;
  float E = oracle_expf_nonpos(-a);
  float d = 1.0f + E;
  return z >= 0.0f ? 1.0f / d : E / d;
}

void oracle_confidence(const uint16_t *hidden, int64_t hidden_stride, int64_t hidden_offset, const uint16_t *w1,
                       int64_t w1_rows, int32_t rank, const uint16_t *weight, float bias, const int64_t *first_prev,
                       const int64_t *draft, int64_t draft_stride, int32_t batch, int32_t P, int32_t hidden_size,
                       int32_t with_markov, const float *fed_logits, float *logits_out, float *scores) {
  uint16_t *feat = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(hidden_size + rank));
  int64_t hs = hidden_stride > 0 ? hidden_stride : hidden_size;
  for (int32_t b = 0; b < batch; b++)
    for (int32_t j = 0; j < P; j++) {
      float z;
      if (fed_logits) {
        z = fed_logits[(int64_t)b * P + j];
      } else {
        const uint16_t *h = hidden + hidden_offset + ((int64_t)b * P + j) * hs;
        int n = hidden_size;
        memcpy(feat, h, sizeof(uint16_t) * (size_t)hidden_size);
        if (with_markov) {
          int64_t prev = j == 0 ? first_prev[b] : draft[(int64_t)b * draft_stride + j - 1];
          uint64_t last = (uint64_t)(w1_rows - 1);
          uint64_t row = (uint64_t)prev < last ? (uint64_t)prev : last;
          memcpy(feat + hidden_size, w1 + row * (uint64_t)rank, sizeof(uint16_t) * (size_t)rank);
          n += rank;
        }
        z = oracle_dot_bf16_f32(weight, feat, n) + bias;
      }
      if (logits_out) logits_out[(int64_t)b * P + j] = z;
      scores[(int64_t)b * P + j] = oracle_sigmoid(z);
    }
  free(feat);
}

static int32_t clamp_len(int32_t L, int32_t min_len, int32_t max_len, int32_t P) {
  if (max_len > P) max_len = P;
  if (max_len < 0) max_len = 0;
  if (min_len < 0) min_len = 0;
  if (min_len > max_len) min_len = max_len;
  return L < min_len ? min_len : (L > max_len ? max_len : L);
}

int32_t oracle_threshold_length(const float *scores, int32_t P, float threshold, int32_t min_len, int32_t max_len) {
  float S = 1.0f;
  int32_t L = 0;
  for (int32_t j = 0; j < P; j++) {
    S = S * scores[j];
    if (!(S >= threshold)) break;
    L = j + 1;
  }
  return clamp_len(L, min_len, max_len, P);
}

int32_t oracle_sps_length(const float *scores, int32_t P, float survival_floor, int32_t min_len, int32_t max_len,
                          const float *cost) {
  int32_t lo = clamp_len(min_len, min_len, max_len, P), hi = clamp_len(max_len, min_len, max_len, P);
  float S = 1.0f, T = 1.0f; /* running product before position L; expected output of length L */
  int32_t best = lo;
  float best_ratio = 0.0f;
  int have = 0;
  for (int32_t L = 0; L <= hi; L++) {
    if (L > 0) {
      S = S * scores[L - 1];
      T = T + S;
      if (L > lo && !(S >= survival_floor)) break;
    }
    if (L < lo) continue;
    if (!(cost[L] > 0.0f)) continue;
    float ratio = T / cost[L];
    if (!have || ratio > best_ratio) {
      best = L;
      best_ratio = ratio;
      have = 1;
    }
  }
  return best;
}
