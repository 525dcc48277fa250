// markov_math.cuh -- per-element arithmetic of the DSpark Markov step on the
// GPU: the output transform, the MurmurHash3 noise, the library's own log,
// tanh and exp, and the packed total-order key.
//
// Every floating-point operation is an explicit round-to-nearest intrinsic
// (__fadd_rn, __fmul_rn, __fmaf_rn, __fdiv_rn), which nvcc never contracts or
// reassociates, so the results are fixed bit for bit by the operation order
// written here.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace dspark {

// ---------------------------------------------------------------------------
// Own natural logarithm of a positive normal finite float (the pages' logf
// is a vendor library's and is not used).  With x = 2^e m, m in [1/sqrt2,
// sqrt2), f = m - 1 and s = f / (2 + f):
//   log(1 + f) = 2 atanh(s) = f - (f^2/2 - s (f^2/2 + R)),
//   R = 2z/3 + 2z^2/5 + 2z^3/7 + 2z^4/9 + 2z^5/11,  z = s^2,
// and log x = e ln2 + log(1 + f) with ln2 = LN2_HI + LN2_LO, LN2_HI having
// 16 significant bits so that e * LN2_HI is exact.
// Constants: 2/(2n+1) and ln 2 rounded to binary32 (hex below).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float own_logf(float x) {
  constexpr float kC3 = 0x1.555556p-1f;   // 2/3
  constexpr float kC5 = 0x1.99999ap-2f;   // 2/5
  constexpr float kC7 = 0x1.24924ap-2f;   // 2/7
  constexpr float kC9 = 0x1.c71c72p-3f;   // 2/9
  constexpr float kC11 = 0x1.745d18p-3f;  // 2/11
  constexpr float kLn2Hi = 0x1.62e400p-1f;  // 0.693145751953125
  constexpr float kLn2Lo = 0x1.7f7d1cp-20f; // ln2 - kLn2Hi
  const uint32_t bits = __float_as_uint(x);
  int e = static_cast<int>(bits >> 23) - 127;
  uint32_t mbits = (bits & 0x007FFFFFu) | 0x3F800000u;
  if (mbits > 0x3FB504F3u) {  // m above RN(sqrt 2): halve it
    mbits -= 0x00800000u;
    e += 1;
  }
  const float f = __fsub_rn(__uint_as_float(mbits), 1.0f);
  const float s = __fdiv_rn(f, __fadd_rn(2.0f, f));
  const float z = __fmul_rn(s, s);
  float p = __fmaf_rn(z, kC11, kC9);
  p = __fmaf_rn(z, p, kC7);
  p = __fmaf_rn(z, p, kC5);
  p = __fmaf_rn(z, p, kC3);
  const float R = __fmul_rn(z, p);
  const float hfsq = __fmul_rn(__fmul_rn(0.5f, f), f);
  const float corr = __fmaf_rn(-s, __fadd_rn(hfsq, R), hfsq);
  const float logm = __fsub_rn(f, corr);
  const float fe = __int2float_rn(e);
  return __fmaf_rn(fe, kLn2Hi, __fmaf_rn(fe, kLn2Lo, logm));
}

// ---------------------------------------------------------------------------
// Own tanh (the pages' tanhf is a vendor library's).
//   tanh|z| = E / (E + 2),  E = expm1(2|z|);  |z| > 9.1 rounds to 1.
//   expm1(x), 0 <= x <= 18.2: k = rint(x / ln2), r = x - k ln2 (two fmas),
//   expm1(r) = r + r^2 (1/2! + r (1/3! + ... + r/9!)),
//   expm1(x) = 2^k expm1(r) + (2^k - 1).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float own_expm1f_nonneg(float x) {
  constexpr float kInvLn2 = 0x1.715476p+0f;
  constexpr float kLn2Hi = 0x1.62e400p-1f;
  constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
  constexpr float k2 = 0x1.000000p-1f;   // 1/2!
  constexpr float k3 = 0x1.555556p-3f;   // 1/3!
  constexpr float k4 = 0x1.555556p-5f;   // 1/4!
  constexpr float k5 = 0x1.111112p-7f;   // 1/5!
  constexpr float k6 = 0x1.6c16c2p-10f;  // 1/6!
  constexpr float k7 = 0x1.a01a02p-13f;  // 1/7!
  constexpr float k8 = 0x1.a01a02p-16f;  // 1/8!
  constexpr float k9 = 0x1.71de3ap-19f;  // 1/9!
  const float kf = rintf(__fmul_rn(x, kInvLn2));
  float r = __fmaf_rn(-kf, kLn2Hi, x);
  r = __fmaf_rn(-kf, kLn2Lo, r);
  float p = __fmaf_rn(r, k9, k8);
  p = __fmaf_rn(r, p, k7);
  p = __fmaf_rn(r, p, k6);
  p = __fmaf_rn(r, p, k5);
  p = __fmaf_rn(r, p, k4);
  p = __fmaf_rn(r, p, k3);
  p = __fmaf_rn(r, p, k2);
  const float em1 = __fmaf_rn(__fmul_rn(r, r), p, r);
  const int k = __float2int_rn(kf);
  if (k == 0) return em1;
  const float two_k = __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
  return __fmaf_rn(two_k, em1, __fsub_rn(two_k, 1.0f));
}

__device__ __forceinline__ float own_tanhf(float z) {
  if (z != z) return z;
  const float a = fabsf(z);
  float t = 1.0f;
  if (!(a > 9.1f)) {
    const float E = own_expm1f_nonneg(__fmul_rn(2.0f, a));
    t = __fdiv_rn(E, __fadd_rn(E, 2.0f));
  }
  return copysignf(t, z);
}

// ---------------------------------------------------------------------------
// Own exp(x) for x <= 0 (the pages' expf is a vendor library's): Cody-Waite
// reduction by ln 2 (its high part with the last 8 significand bits cleared,
// so k * hi is exact for |k| < 2^8) and the Taylor series of exp to degree 7
// on |r| <= ln2/2.  NaN propagates, below -104 gives 0, and 2^k scales the
// polynomial exactly (k >= -125) or with one rounding into the subnormals.
// k = rint(RN(x / ln2)) comes from adding and removing 1.5 2^23, which
// rounds to an integer with ties to even as rint does (|x / ln2| < 2^22),
// and leaves k in the low bits of the sum.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float own_exp_nonpos(float x) {
  constexpr double kLn2 = 0.69314718055994530941723212145818;
  constexpr float kInvLn2 = static_cast<float>(1.0 / kLn2);
  constexpr float kLn2Hi = 0.693145751953125f;
  constexpr float kLn2Lo = static_cast<float>(kLn2 - 0.693145751953125);
  constexpr float kC2 = static_cast<float>(1.0 / 2.0);
  constexpr float kC3 = static_cast<float>(1.0 / 6.0);
  constexpr float kC4 = static_cast<float>(1.0 / 24.0);
  constexpr float kC5 = static_cast<float>(1.0 / 120.0);
  constexpr float kC6 = static_cast<float>(1.0 / 720.0);
  constexpr float kC7 = static_cast<float>(1.0 / 5040.0);
  constexpr float kRound = 0x1.8p23f;
  if (isnan(x)) return x;
  if (x < -104.0f) return 0.0f;
  const float t = __fadd_rn(__fmul_rn(x, kInvLn2), kRound);
  const float kf = __fsub_rn(t, kRound);
  float r = __fmaf_rn(-kf, kLn2Hi, x);
  r = __fmaf_rn(-kf, kLn2Lo, r);
  float p = __fmaf_rn(r, kC7, kC6);
  p = __fmaf_rn(r, p, kC5);
  p = __fmaf_rn(r, p, kC4);
  p = __fmaf_rn(r, p, kC3);
  p = __fmaf_rn(r, p, kC2);
  p = __fmaf_rn(r, p, 1.0f);
  p = __fmaf_rn(r, p, 1.0f);
  const int k = static_cast<int>(__float_as_uint(t) - 0x4B400000u);  // in [-150, 0]
  if (k >= -125) return __fmul_rn(p, __int_as_float((k + 127) << 23));
  return __fmul_rn(__fmul_rn(p, __int_as_float((k + 64 + 127) << 23)), 0x1p-64f);
}

// ---------------------------------------------------------------------------
// Correctly rounded division by one divisor d, many dividends: with
// y = RN(1/d), q = RN(x y) is a faithful quotient, the remainder x - q d is
// exact (one fma) and RN(q + (x - q d) y) is RN(x / d) -- P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990 -- provided nothing overflows or
// underflows.  `fast` holds for 2^-20 <= |d| < 2^40; the quotient is taken
// that way for 2^-60 <= |x| < 2^60 (remainders stay multiples of 2^-146,
// quotients normal), by the IEEE division otherwise.
// ---------------------------------------------------------------------------
struct Divider {
  float d, y;
  bool fast;
};

__device__ __forceinline__ Divider make_divider(float d) {
  const uint32_t a = __float_as_uint(d) & 0x7FFFFFFFu;
  // 2^-20 has exponent field 107, 2^40 has 167
  return Divider{d, __frcp_rn(d), a >= (107u << 23) && a < (167u << 23)};
}

__device__ __forceinline__ float div_rn(float x, const Divider& D) {
  const uint32_t a = __float_as_uint(x) & 0x7FFFFFFFu;
  // 2^-60 has exponent field 67, 2^60 has 187
  if (D.fast && a - (67u << 23) < (120u << 23)) {
    const float q = __fmul_rn(x, D.y);
    const float r = __fmaf_rn(-q, D.d, x);
    return __fmaf_rn(r, D.y, q);
  }
  return __fdiv_rn(x, D.d);
}

// ---------------------------------------------------------------------------
// Output transform ([P3] _logit): BF16 add (one FP32 add rounded to BF16),
// multiplier, optional soft cap cap * tanh(inv_cap * y), round to BF16.
// Returns the cached BF16 bits; *l is their FP32 value.  transform_sum is
// the part after the BF16 add, a function of the rounded sum x alone.
// ---------------------------------------------------------------------------
template <bool kHasCap>
__device__ __forceinline__ uint16_t transform_sum(float x, float mult, float inv_cap, float cap, float* l) {
  const float y = __fmul_rn(mult, x);
  float w = y;
  if (kHasCap) w = __fmul_rn(cap, own_tanhf(__fmul_rn(inv_cap, y)));
  const __nv_bfloat16 c = __float2bfloat16_rn(w);
  *l = __bfloat162float(c);
  return __bfloat16_as_ushort(c);
}

template <bool kHasCap>
__device__ __forceinline__ uint16_t transform_logit(float base, float bias, float mult, float inv_cap,
                                                    float cap, float* l) {
  const float x = __bfloat162float(__float2bfloat16_rn(__fadd_rn(base, bias)));
  return transform_sum<kHasCap>(x, mult, inv_cap, cap, l);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// ---------------------------------------------------------------------------
// MurmurHash3_x86_32 (seed 0) of the four words [lo(step_seed),
// hi(step_seed), lo(pos - 1 + salt), vocab id] ([P3] _murmur_prefix,
// _gumbel).  The prefix covers the first three words (per row and step).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t murmur_round(uint32_t h, uint32_t k) {
  k *= 0xcc9e2d51u;
  k = __funnelshift_l(k, k, 15);
  k *= 0x1b873593u;
  h ^= k;
  h = __funnelshift_l(h, h, 13);
  return h * 5u + 0xe6546b64u;
}

__device__ __forceinline__ uint32_t murmur_prefix(uint64_t seed, int32_t step, int64_t pos, uint32_t salt) {
  const uint64_t step_seed = seed ^ (static_cast<uint64_t>(static_cast<uint32_t>(step)) << 32);
  const uint32_t salted = static_cast<uint32_t>(static_cast<uint64_t>(pos) - 1u + salt);
  uint32_t h = murmur_round(0u, static_cast<uint32_t>(step_seed));
  h = murmur_round(h, static_cast<uint32_t>(step_seed >> 32));
  return murmur_round(h, salted);
}

// The block step split in its key half (which depends only on the vocab id,
// so it is shared by every row) and its state half.
__device__ __forceinline__ uint32_t murmur_kmix(uint32_t k) {
  k *= 0xcc9e2d51u;
  k = __funnelshift_l(k, k, 15);
  return k * 0x1b873593u;
}

__device__ __forceinline__ uint32_t murmur_finish_mixed(uint32_t prefix, uint32_t kmixed) {
  uint32_t h = prefix ^ kmixed;
  h = __funnelshift_l(h, h, 13);
  h = (h * 5u + 0xe6546b64u) ^ 16u;
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

__device__ __forceinline__ uint32_t murmur_finish(uint32_t prefix, uint32_t vocab_id) {
  return murmur_finish_mixed(prefix, murmur_kmix(vocab_id));
}

// ---------------------------------------------------------------------------
// Noise L(h) = log(-log(1 - u)), u = RN((h + 0.5) 2^-32) ([P3] _gumbel):
// u is built as the page builds it, one fma of the two 16-bit halves;
// log(1 - u) is the 8-term series below 0.25, else log(max(1 - u, 2^-24)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float noise_uniform(uint32_t h) {
  const float lo = __fmul_rn(__fadd_rn(__uint2float_rn(h & 0xFFFFu), 0.5f), 0x1p-32f);
  return __fmaf_rn(__uint2float_rn(h >> 16), 0x1p-16f, lo);
}

__device__ __forceinline__ float noise_L(uint32_t h) {
  const float u = noise_uniform(h);
  float sel;
  if (u < 0.25f) {
    float poly = __fmaf_rn(u, 0x1p-3f, 0x1.24924ap-3f);  // 1/8, 1/7
    poly = __fmaf_rn(u, poly, 0x1.555556p-3f);            // 1/6
    poly = __fmaf_rn(u, poly, 0x1.99999ap-3f);            // 1/5
    poly = __fmaf_rn(u, poly, 0x1p-2f);                   // 1/4
    poly = __fmaf_rn(u, poly, 0x1.555556p-2f);            // 1/3
    poly = __fmaf_rn(u, poly, 0x1p-1f);                   // 1/2
    poly = __fmaf_rn(u, poly, 1.0f);
    sel = __fmul_rn(poly, -u);
  } else {
    const float om = __fsub_rn(1.0f, u);
    sel = own_logf(om > 0x1p-24f ? om : 0x1p-24f);
  }
  return own_logf(-sel);
}

// key = RN(RN(l / t) - L) at a nonzero temperature ([P2] _gumbel_key).
__device__ __forceinline__ float noised_key(float l, float temp, uint32_t h) {
  return __fsub_rn(__fdiv_rn(l, temp), noise_L(h));
}

// ---------------------------------------------------------------------------
// Packed total-order key: (orderable value << 32) | ~id.  The 64-bit maximum
// is the first NaN, else the lowest id of the largest value, with +0 == -0
// ([P3] module docstring, _combine) -- in any reduction order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t orderable(float v) {
  const uint32_t b = __float_as_uint(v);
  if (v != v) return 0xFFFFFFFFu;
  if ((b & 0x7FFFFFFFu) == 0) return 0x80000000u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned long long pack_key(float v, uint32_t id) {
  return (static_cast<unsigned long long>(orderable(v)) << 32) | static_cast<uint32_t>(~id);
}

// The float bits of an orderable key (NaN comes back as the canonical NaN).
__device__ __forceinline__ uint32_t key_bits(uint32_t o) {
  if (o == 0xFFFFFFFFu) return 0x7FFFFFFFu;
  return (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
}

__device__ __forceinline__ int64_t slot_token(unsigned long long slot) {
  return static_cast<int64_t>(static_cast<int32_t>(~static_cast<uint32_t>(slot)));
}

}  // namespace dspark
