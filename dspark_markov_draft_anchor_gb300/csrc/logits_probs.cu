// logits_probs.cu -- [P1] dsparkLogitsToProbabilities: a dense probability
// row after temperature, top-k and top-p, behind the C ABI of
// include/dspark_markov.h.
//
// Every decision is an exact comparison, so the result does not depend on
// how threads split a row:
//   - temperature <= 0 (or NaN) is greedy: 1 at the lowest id of the
//     largest non-NaN logit;
//   - z = RN(l / T), -0 as +0; an id whose z is NaN (a NaN logit, or an
//     infinite one over an infinite temperature) weighs nothing; top-k
//     (0 < K < count of the others) keeps the first K ids in the order
//     (z descending, id ascending);
//   - e = exp(x) by the library's own exp, x = z - m (m the largest z; x = 0
//     where z == m), w = floor(e 2^40);
//   - top-p (p < 1) keeps the shortest prefix in the order (w descending, id
//     ascending) whose weight reaches max(1, ceil(p W)), W the kept total;
//   - probability = RN(e / S), S = RN(sum of the final w) 2^-40; 0 elsewhere.
//
// The plain setting (no top-k, no top-p, T > 0) on aligned rows runs on
// clusters that hold each row in shared memory (probs_plain_cluster_kernel).
// Otherwise one CTA of 1024 threads per row: top-k with K <= 1024 is cut
// from the few ids at or above the K-th largest per-thread maximum
// (prefilter_tau), else the k-th largest key is a radix select over the row
// (8 bits a pass: four passes of counts over the 32-bit logit keys) with an
// ordered scan for ties; with K <= 2048 the rest happens on the kept ids in
// shared memory (compact_finish), else the top-p cut is a radix select of
// weight sums over the 48-bit weights (six passes), and a last pass writes
// the row.  The output row holds z, then e, between passes (see
// logits_probs_row).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "dspark_markov.h"
#include "kernels.h"
#include "markov_math.cuh"
#include "ptx.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// floor(e 2^40) for e in [0, 1], in two halves and FP32/INT32 instructions
// only (a float-to-64-bit conversion runs on this part's small FP64 pipe):
// with y = e 2^20 (exact, subnormal e included) the weight is
// floor(y) 2^20 + floor(frac(y) 2^20).  Each floor is the low mantissa bits of
// a round-toward-zero add of 2^23 (exact for values below 2^23; both are at
// most 2^20), and frac(y) = y - floor(y) is exact.
struct WeightHalves {
  uint32_t hi, lo;
};
__device__ __forceinline__ WeightHalves weight_halves(float e) {
  const float y = __fmul_rn(e, 0x1p20f);
  const float hm = __fadd_rz(y, 0x1p23f);
  const float lm = __fmaf_rz(__fsub_rn(y, __fsub_rn(hm, 0x1p23f)), 0x1p20f, 0x1p23f);
  return {__float_as_uint(hm) - 0x4B000000u, __float_as_uint(lm) - 0x4B000000u};
}
__device__ __forceinline__ uint64_t weight(float e) {
  const WeightHalves h = weight_halves(e);
  return (static_cast<uint64_t>(h.hi) << 20) | h.lo;
}
// A thread's total of up to 4095 weights: each half is at most 2^20, so
// their 32-bit sums are exact.
struct WeightSum {
  uint32_t hi = 0, lo = 0;
  __device__ __forceinline__ void add(float e) {
    const WeightHalves h = weight_halves(e);
    hi += h.hi;
    lo += h.lo;
  }
  __device__ __forceinline__ uint64_t total() const { return (static_cast<uint64_t>(hi) << 20) + lo; }
};

// An order-preserving 32-bit key of a non-NaN float (+0 and -0 equal).
__device__ __forceinline__ uint32_t order_key(float z) {
  const uint32_t b = __float_as_uint(z == 0.0f ? 0.0f : z);
  return b ^ ((b >> 31) ? 0xFFFFFFFFu : 0x80000000u);
}

// max(1, ceil(p W)) for p < 1, exactly: p = M 2^(E - 150) with M the 24-bit
// significand and E the biased exponent field, so p W = M W / 2^(150 - E).
__device__ uint64_t top_p_threshold(float p, uint64_t W) {
  if (!(p > 0.0f)) return 1ull;
  const uint32_t b = __float_as_uint(p);
  const int E = static_cast<int>(b >> 23);
  const int shift = 150 - E;  // >= 24 since p < 1; subnormals give 150
  if (shift >= 100) return 1ull;
  const uint64_t M = (b & 0x7FFFFFu) | 0x800000u;
  uint64_t lo = M * W, hi = __umul64hi(M, W);
  // + 2^shift - 1, then >> shift
  const uint64_t add_lo = shift >= 64 ? ~0ull : (1ull << shift) - 1;
  const uint64_t add_hi = shift >= 64 ? (1ull << (shift - 64)) - 1 : 0ull;
  const uint64_t lo2 = lo + add_lo;
  hi += add_hi + (lo2 < lo ? 1ull : 0ull);
  lo = lo2;
  const uint64_t c = shift >= 64 ? hi >> (shift - 64) : (lo >> shift) | (hi << (64 - shift));
  return c < 1 ? 1ull : c;
}

struct RowSmem {
  unsigned int hist[256];
  unsigned long long whist[256];
  unsigned long long red_u64[kWarps];
  float red_f[kWarps];
  int red_i[kWarps];
  int64_t red_id[kWarps];
  int64_t found;
  // decisions, written by thread 0
  uint32_t k_prefix, k_mask;
  int64_t k_rem;
  uint64_t p_prefix, p_mask, p_above, p_thr;
  uint32_t tkey[kThreads];  // per thread: the order key of its largest z (0 if it has none)
  int cand_n;
};

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  return x;
}

__device__ uint64_t block_sum_u64(uint64_t x, RowSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  x = warp_sum_u64(x);
  if (lane == 0) sm.red_u64[warp] = x;
  __syncthreads();
  uint64_t t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += sm.red_u64[w];
  __syncthreads();
  return t;
}

// The id of the r-th id (1-based, id order) that satisfies pred, by one
// ordered scan of the row kThreads ids at a time; vocab if there are fewer.
template <class Pred>
__device__ int64_t nth_in_order(int64_t vocab, int64_t r, Pred pred, RowSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t seen = 0;
  for (int64_t c0 = 0; c0 < vocab; c0 += kThreads) {
    const int64_t v = c0 + threadIdx.x;
    const bool f = v < vocab && pred(v);
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, f);
    if (lane == 0) sm.red_i[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = sm.red_i[w];
      if (w < warp) before += c;
      total += c;
    }
    if (seen + total >= r) {  // the same in every thread
      const int64_t rank = seen + before + __popc(bal & ((1u << lane) - 1u)) + 1;
      if (f && rank == r) sm.found = v;
      __syncthreads();
      const int64_t id = sm.found;
      __syncthreads();
      return id;
    }
    seen += total;
    __syncthreads();
  }
  return vocab;
}

// Row iteration: every id of a row, four at a time (float4) where the row
// allows it.  Each thread issues the loads of kBatch groups (or ids) before
// it uses any: the passes that stream from or to HBM batch 4 so that one CTA
// per SM keeps enough requests in flight, as does the top-k prefilter's
// light pass over L2; the other passes over L2 take 1 (more would spill
// their inlined per-id work).
// row_map writes f's value back in place of what it read (the same thread
// reads and then writes each id, so src may equal dst).
template <int kBatch = 1, class F>
__device__ __forceinline__ void row_each(const float* src, int64_t vocab, bool vec, F&& f) {
  const int n = static_cast<int>(vocab);  // < 2^31 (the C ABI's vocab is an int32)
  const int t = static_cast<int>(threadIdx.x);
  if (vec) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    const int n4 = n >> 2;
    for (int g0 = t; g0 < n4; g0 += kBatch * kThreads) {
      float4 x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (g0 + k * kThreads < n4) x[k] = s4[g0 + k * kThreads];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int g = g0 + k * kThreads;
        if (g < n4) {
          f(4 * g, x[k].x);
          f(4 * g + 1, x[k].y);
          f(4 * g + 2, x[k].z);
          f(4 * g + 3, x[k].w);
        }
      }
    }
  } else {
    for (int v0 = t; v0 < n; v0 += kBatch * kThreads) {
      float x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (v0 + k * kThreads < n) x[k] = src[v0 + k * kThreads];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (v0 + k * kThreads < n) f(v0 + k * kThreads, x[k]);
    }
  }
}

template <bool kStreamIn, bool kStreamOut, int kBatch = 1, class F>
__device__ __forceinline__ void row_map(const float* src, float* dst, int64_t vocab, bool vec, F&& f) {
  const int n = static_cast<int>(vocab);
  const int t = static_cast<int>(threadIdx.x);
  if (vec) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* d4 = reinterpret_cast<float4*>(dst);
    const int n4 = n >> 2;
    for (int g0 = t; g0 < n4; g0 += kBatch * kThreads) {
      float4 x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int g = g0 + k * kThreads;
        if (g < n4) x[k] = kStreamIn ? __ldcs(s4 + g) : s4[g];
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int g = g0 + k * kThreads;
        if (g < n4) {
          const float4 y =
              make_float4(f(4 * g, x[k].x), f(4 * g + 1, x[k].y), f(4 * g + 2, x[k].z), f(4 * g + 3, x[k].w));
          if (kStreamOut)
            __stcs(d4 + g, y);
          else
            d4[g] = y;
        }
      }
    }
  } else {
    for (int v0 = t; v0 < n; v0 += kBatch * kThreads) {
      float x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int v = v0 + k * kThreads;
        if (v < n) x[k] = kStreamIn ? __ldcs(src + v) : src[v];
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int v = v0 + k * kThreads;
        if (v < n) {
          const float y = f(v, x[k]);
          if (kStreamOut)
            __stcs(dst + v, y);
          else
            dst[v] = y;
        }
      }
    }
  }
}

// Small top-k: the kept ids in shared memory (at most kCompactMax).
constexpr int kCompactMax = 2048;

struct CompactSmem {
  int32_t id[kCompactMax];
  float e[kCompactMax];  // z, then e
  unsigned long long w[kCompactMax];
  int n;
};

// Sort a[0, n) descending, n a power of two: a bitonic network, one
// compare-exchange per pair and stage, kThreads threads.
template <class T>
__device__ void bitonic_desc(T* a, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const T x = a[i], y = a[ixj];
          if ((i & k) == 0 ? x < y : x > y) {
            a[i] = y;
            a[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

// The top-k cut (k_key, k_id) without radix passes over the row, for K <=
// kThreads.  Each thread's largest z (from pass 1, sm.tkey) is an element of
// the row, so the K-th largest of the kThreads thread maxima, tau, is at most
// the K-th largest key: every id the cut keeps has a key >= tau (a thread
// without a number counts as key 0, and if one of those is among the K
// largest, tau is 0 and every number passes).  The ids passing tau -- about
// K for a row of independent logits -- are gathered into shared memory and
// sorted by (key descending, id ascending); the K-th entry is the cut, as
// the radix passes and the ordered tie scan would find it, and the first K
// entries are the ids it keeps: they go to cs.id / cs.e (z from its key) as
// compact_finish's gather would leave them; the row's zeros are written
// here (nothing reads the row after the gather).  False, nothing decided and
// nothing written, when more than kCompactMax ids pass.
__device__ __noinline__ bool prefilter_cut(float* out, int64_t vocab, bool vec, int K, uint32_t& k_key,
                                           int64_t& k_id, RowSmem& sm, CompactSmem& cs) {
  bitonic_desc(sm.tkey, kThreads);
  const uint32_t tau = sm.tkey[K - 1];
  if (threadIdx.x == 0) sm.cand_n = 0;
  __syncthreads();
  row_each<4>(out, vocab, vec, [&](int64_t v, float z) {  // four loads in flight a thread: an L2 pass
    if (isnan(z)) return;
    const uint32_t key = order_key(z);
    if (key >= tau) {
      const int slot = atomicAdd(&sm.cand_n, 1);
      if (slot < kCompactMax)  // (key, ~id): larger first is key descending, id ascending
        cs.w[slot] = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(v));
    }
  });
  __syncthreads();
  const int n = sm.cand_n;
  if (n > kCompactMax) return false;  // the same in every thread
  // The row is not read again: its zeros go out now, under the sorts below
  // and compact_finish's work on the kept ids (which then only scatters).
  if (vec) {
    float4* d4 = reinterpret_cast<float4*>(out);
    for (int64_t g = threadIdx.x; g < (vocab >> 2); g += kThreads) __stcs(d4 + g, make_float4(0.f, 0.f, 0.f, 0.f));
  } else {
    for (int64_t v = threadIdx.x; v < vocab; v += kThreads) __stcs(out + v, 0.0f);
  }
  int P2 = 1;
  while (P2 < n) P2 <<= 1;
  for (int i = n + static_cast<int>(threadIdx.x); i < P2; i += kThreads) cs.w[i] = 0ull;  // below every key
  __syncthreads();
  bitonic_desc(cs.w, P2);
  const unsigned long long c = cs.w[K - 1];
  k_key = static_cast<uint32_t>(c >> 32);
  k_id = static_cast<int64_t>(0xFFFFFFFFu - static_cast<uint32_t>(c));
  for (int i = threadIdx.x; i < K; i += kThreads) {
    const unsigned long long ci = cs.w[i];
    const uint32_t key = static_cast<uint32_t>(ci >> 32);  // order_key inverted (no NaN here)
    cs.id[i] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(ci));
    cs.e[i] = __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
  }
  if (threadIdx.x == 0) cs.n = K;
  __syncthreads();
  return true;
}

// After a top-k cut of K <= kCompactMax ids: gather them (and their z) into
// shared memory, take e and w there, cut top-p on the K entries sorted by
// (w descending, id ascending) (a bitonic sort, then a block scan for the
// shortest prefix reaching the threshold), then zero the row and scatter
// the probabilities.  Equal to the full-row passes: the same sets, sums and
// roundings.
__device__ __noinline__ void compact_finish(float* out, int64_t vocab, bool vec, int K, uint32_t k_key, int64_t k_id,
                                            float m, float top_p, bool gathered, RowSmem& sm, CompactSmem& cs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!gathered) {  // (else prefilter_cut left the kept ids there)
    if (threadIdx.x == 0) cs.n = 0;
    __syncthreads();
    row_each(out, vocab, vec, [&](int64_t v, float z) {
      if (isnan(z)) return;
      const uint32_t key = order_key(z);
      if (key > k_key || (key == k_key && v <= k_id)) {
        const int slot = atomicAdd(&cs.n, 1);
        if (slot < kCompactMax) {  // exactly K ids pass the cut
          cs.id[slot] = static_cast<int32_t>(v);
          cs.e[slot] = z;
        }
      }
    });
    __syncthreads();
  }
  K = cs.n < K ? cs.n : K;  // equal in correct operation; never past what was gathered
  const bool topp = top_p < 1.0f;
  int P2 = 1;
  while (P2 < K) P2 <<= 1;
  uint64_t part = 0;
  for (int i = threadIdx.x; i < (topp ? P2 : K); i += kThreads) {
    if (i < K) {
      const float z = cs.e[i];
      const float e = own_exp_nonpos(z == m ? 0.0f : __fsub_rn(z, m));
      const uint64_t w = weight(e);
      cs.e[i] = e;
      cs.w[i] = w;
      part += w;
    } else {  // padding that sorts after every real entry
      cs.e[i] = 0.0f;
      cs.w[i] = 0ull;
      cs.id[i] = 0x7FFFFFFF;
    }
  }
  const uint64_t W = block_sum_u64(part, sm);
  int n_final = K;
  uint64_t S = W;
  if (topp) {
    for (int k = 2; k <= P2; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = threadIdx.x; i < P2; i += kThreads) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const uint64_t wa = cs.w[i], wb = cs.w[ixj];
            const int32_t ia = cs.id[i], ib = cs.id[ixj];
            const bool a_first = wa > wb || (wa == wb && ia < ib);
            if (((i & k) == 0) != a_first) {
              cs.w[i] = wb;
              cs.w[ixj] = wa;
              cs.id[i] = ib;
              cs.id[ixj] = ia;
              const float ea = cs.e[i];
              cs.e[i] = cs.e[ixj];
              cs.e[ixj] = ea;
            }
          }
        }
        __syncthreads();
      }
    }
    // shortest prefix whose weight reaches the threshold: two entries a thread
    if (threadIdx.x == 0) {
      sm.p_thr = top_p_threshold(top_p, W);
      sm.found = K;  // replaced by the crossing thread
      sm.p_above = W;
    }
    const int i0 = 2 * threadIdx.x;
    const uint64_t w0 = i0 < P2 ? cs.w[i0] : 0ull, w1 = i0 + 1 < P2 ? cs.w[i0 + 1] : 0ull;
    const uint64_t mine = w0 + w1;
    uint64_t incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) sm.red_u64[warp] = incl;
    __syncthreads();
    uint64_t before = 0;
    for (int w = 0; w < warp; ++w) before += sm.red_u64[w];
    const uint64_t thr = sm.p_thr;
    const uint64_t excl = before + incl - mine;
    if (excl < thr && thr <= excl + mine) {  // one thread: the prefix crosses here
      const bool first = excl + w0 >= thr;
      sm.found = first ? i0 + 1 : i0 + 2;
      sm.p_above = first ? excl + w0 : excl + mine;
    }
    __syncthreads();
    n_final = static_cast<int>(sm.found);
    S = sm.p_above;
    __syncthreads();
  }
  const float Sf = __fmul_rn(__ull2float_rn(S), 0x1p-40f);
  if (!gathered) {  // (else prefilter_cut wrote the zeros)
    if (vec) {
      float4* d4 = reinterpret_cast<float4*>(out);
      for (int64_t g = threadIdx.x; g < (vocab >> 2); g += kThreads) __stcs(d4 + g, make_float4(0.f, 0.f, 0.f, 0.f));
    } else {
      for (int64_t v = threadIdx.x; v < vocab; v += kThreads) __stcs(out + v, 0.0f);
    }
  }
  __syncthreads();  // the zeros are ordered before the scattered values
  for (int i = threadIdx.x; i < n_final; i += kThreads) out[cs.id[i]] = __fdiv_rn(cs.e[i], Sf);
}

// ---------------------------------------------------------------------------
// The plain setting -- T > 0, no top-k, no top-p -- on a 16-byte-aligned
// row, four ids at a time.  Each group of four takes one range check that
// keeps the reciprocal division (div_rn's fast form) and the exp's fast form
// exact, with the general forms behind it, so the common path is a few
// instructions an id.  Same passes and values as logits_probs_row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float min_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// z = RN(x / T), -0 as +0
__device__ __forceinline__ float4 scaled4(float4 x, const Divider& D) {
  const float lo = fminf(fminf(fabsf(x.x), fabsf(x.y)), fminf(fabsf(x.z), fabsf(x.w)));
  const float hi = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
  float4 z;
  if (D.fast && lo >= 0x1p-60f && hi < 0x1p60f) {  // a NaN id is NaN either way
    const auto q = [&](float v) { const float a = __fmul_rn(v, D.y); return __fmaf_rn(__fmaf_rn(-a, D.d, v), D.y, a); };
    z = make_float4(q(x.x), q(x.y), q(x.z), q(x.w));
  } else {
    z = make_float4(__fdiv_rn(x.x, D.d), __fdiv_rn(x.y, D.d), __fdiv_rn(x.z, D.d), __fdiv_rn(x.w, D.d));
  }
  return make_float4(__fadd_rn(z.x, 0.0f), __fadd_rn(z.y, 0.0f), __fadd_rn(z.z, 0.0f), __fadd_rn(z.w, 0.0f));
}

// exp(x) for -86.5 <= x <= 0: own_exp_nonpos with k >= -125 (one scaling),
// no zero clamp and no NaN
__device__ __forceinline__ float exp_mid(float x) {
  constexpr double kLn2 = 0.69314718055994530941723212145818;
  constexpr float kInvLn2 = static_cast<float>(1.0 / kLn2);
  constexpr float kLn2Hi = 0.693145751953125f;
  constexpr float kLn2Lo = static_cast<float>(kLn2 - 0.693145751953125);
  constexpr float kRound = 0x1.8p23f;
  const float t = __fadd_rn(__fmul_rn(x, kInvLn2), kRound);
  const float kf = __fsub_rn(t, kRound);
  float r = __fmaf_rn(-kf, kLn2Hi, x);
  r = __fmaf_rn(-kf, kLn2Lo, r);
  float p = __fmaf_rn(r, static_cast<float>(1.0 / 5040.0), static_cast<float>(1.0 / 720.0));
  p = __fmaf_rn(r, p, static_cast<float>(1.0 / 120.0));
  p = __fmaf_rn(r, p, static_cast<float>(1.0 / 24.0));
  p = __fmaf_rn(r, p, static_cast<float>(1.0 / 6.0));
  p = __fmaf_rn(r, p, 0.5f);
  p = __fmaf_rn(r, p, 1.0f);
  p = __fmaf_rn(r, p, 1.0f);
  // 2^k: k + 127 in the exponent field, k the low bits of t
  return __fmul_rn(p, __uint_as_float((__float_as_uint(t) - (0x4B400000u - 127u)) << 23));
}

// e = exp(z - m) (1 where z == m), -1 for a NaN z
__device__ __forceinline__ float weight_e(float z, float m) {
  if (z != z) return -1.0f;
  return own_exp_nonpos(z == m ? 0.0f : __fsub_rn(z, m));
}

// ---------------------------------------------------------------------------
// The plain setting on clusters: a row's ids are split over the C CTAs of a
// cluster, CTA c keeping ids [c S, c S + S) (S = slice) in its shared memory,
// so the row is read from HBM once, written once, and its three passes run
// over shared memory -- the passes of the one-CTA-per-row kernels go through
// L2, whose traffic, not HBM, bounds them.  The row's largest z and its
// weight total are combined across the cluster through distributed shared
// memory.  CTAs are small (256 threads, one slice buffer) so that two or
// three of them, from different clusters, share an SM and one's copies and
// barriers overlap another's arithmetic.  The slice travels in two halves,
// each on its own mbarrier: pass 1 starts on the first half while the second
// lands, and the next row's first half is copied while pass 3 finishes the
// second.  Each cluster takes rows cid, cid + clusters, ...; its CTAs take
// the same rows and the same branches, so every cluster barrier is reached
// by all of them.
// ---------------------------------------------------------------------------
// Cluster pushes: a store into a peer CTA's shared memory (a shared::cluster
// address from mapa) that completes its bytes on the peer's mbarrier (in the
// same CTA as the destination), so the peer waits on its own barrier.
__device__ __forceinline__ void push_f32x2(uint32_t dst, float a, float b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(dst),
               "f"(a), "f"(b), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void push_u64(uint32_t dst, unsigned long long v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(dst), "l"(v),
               "r"(bar)
               : "memory");
}

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr int kCSliceBytesMax = 100 * 1024;
constexpr int kCMaxCluster = 8;
static_assert(kCSliceBytesMax / 4 / kCThreads <= 4095, "a thread's weights must sum exactly in WeightSum");
constexpr uint32_t kCopyWaitLimit = 1u << 24;  // polls of a slice copy's mbarrier

__global__ void __launch_bounds__(kCThreads, 3)
    probs_plain_cluster_kernel(const float* __restrict__ logits, float* __restrict__ probs, int rows, int vocab,
                               float temperature, int slice) {
  extern __shared__ __align__(128) float sbuf[];  // [slice]: halves [0, h) and [h, cnt)
  __shared__ uint64_t bar[2];                     // one per half
  // The row's exchanges, pushed by every CTA into every CTA's slots: per row
  // parity, each CTA's (largest z, smallest z or NaN if any z is NaN), its
  // "some z is -inf" flag (rows of only NaN and -inf), its weight total;
  // xbar[exchange][parity] completes when all of the cluster's have landed.
  __shared__ float2 x_mm[2][kCMaxCluster];
  __shared__ unsigned long long x_any[2][kCMaxCluster];
  __shared__ unsigned long long x_sum[2][kCMaxCluster];
  __shared__ uint64_t xbar[3][2];
  __shared__ float2 red_f[kCWarps];
  __shared__ unsigned long long red_u[kCWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t csize = ptx::cluster_nctarank();
  const uint32_t rank = ptx::cluster_ctarank();
  const int cid = static_cast<int>(ptx::clusterid_x()), ncl = static_cast<int>(ptx::nclusterid_x());
  const int v0 = static_cast<int>(ptx::cluster_ctarank()) * slice;
  const int cnt = vocab - v0 < slice ? (vocab - v0 > 0 ? vocab - v0 : 0) : slice;  // a multiple of 4
  const int n4 = cnt >> 2;
  const int h4 = n4 >> 1;  // float4 groups of the first half
  float4* b4 = reinterpret_cast<float4*>(sbuf);
  if (tid == 0) {
    ptx::mbar_init(&bar[0], 1);
    ptx::mbar_init(&bar[1], 1);
    for (int e = 0; e < 3; ++e) {
      ptx::mbar_init(&xbar[e][0], 1);
      ptx::mbar_init(&xbar[e][1], 1);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::cluster_sync();  // every CTA's exchange barriers exist before any push
  // warp 0: push this CTA's value of exchange e (parity p) to every CTA of
  // the cluster (lane q to CTA q); lane 0 arms the local barrier for the
  // cluster's values (a push may land before it: the transaction count may
  // go below zero until then)
  auto push2 = [&](int e, int p, float2* slots, float a, float c) {
    if (lane == 0) ptx::mbar_arrive_expect_tx(&xbar[e][p], csize * 8u);
    if (static_cast<uint32_t>(lane) < csize)
      push_f32x2(ptx::dsmem_addr(&slots[rank], lane), a, c, ptx::dsmem_addr(&xbar[e][p], lane));
  };
  auto push8 = [&](int e, int p, unsigned long long* slots, unsigned long long v) {
    if (lane == 0) ptx::mbar_arrive_expect_tx(&xbar[e][p], csize * 8u);
    if (static_cast<uint32_t>(lane) < csize)
      push_u64(ptx::dsmem_addr(&slots[rank], lane), v, ptx::dsmem_addr(&xbar[e][p], lane));
  };
  // every thread: the k-th phase of exchange e's barrier p landed (bounded;
  // the answer is made the same in the whole CTA)
  auto landed = [&](int e, int p, int k) {
    return __syncthreads_and(ptx::mbar_wait(&xbar[e][p], static_cast<uint32_t>(k) & 1u, kCopyWaitLimit));
  };
  // thread 0: half hf of row r's slice into the buffer (the half's last
  // generic reads, ordered before this thread by a CTA barrier, before the
  // async write)
  auto issue = [&](int r, int hf) {
    ptx::fence_proxy_async_smem();
    const int g0 = hf ? h4 : 0, g1 = hf ? n4 : h4;
    if (g1 > g0) {
      const uint32_t bytes = static_cast<uint32_t>(g1 - g0) * 16u;
      ptx::mbar_arrive_expect_tx(&bar[hf], bytes);
      ptx::bulk_load(b4 + g0, logits + static_cast<int64_t>(r) * vocab + v0 + 4 * g0, bytes, &bar[hf]);
    } else {
      ptx::mbar_arrive(&bar[hf]);
    }
  };
  if (tid == 0 && cid < rows) {
    issue(cid, 0);
    issue(cid, 1);
  }
  // wait for half hf of the i-th row (every half completes one phase a row);
  // a wait that gives up (never in correct operation) lets the copy land
  // (bounded) and marks the half by NaN results, keeping to the protocol
  auto land = [&](int i, int hf) {
    const bool ok = ptx::mbar_wait(&bar[hf], i & 1, kCopyWaitLimit);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) ptx::mbar_wait(&bar[hf], i & 1, kCopyWaitLimit);
      for (int g = (hf ? h4 : 0) + tid; g < (hf ? n4 : h4); g += kCThreads) b4[g] = make_float4(NAN, NAN, NAN, NAN);
      __syncthreads();
    }
  };
  const Divider by_t = make_divider(temperature);
  int i = 0, n_any = 0, n_sum = 0;  // exchanges of each kind so far (a row of zeros takes no sum)
  for (int r = cid; r < rows; r += ncl, ++i) {
    const int b = i & 1;  // the (largest, smallest) exchange's slots and barrier alternate between rows
    const bool next = r + ncl < rows;
    float4* o4 = reinterpret_cast<float4*>(probs + static_cast<int64_t>(r) * vocab + v0);

    // pass 1: z in place; the cluster's largest z, and its smallest (NaN if
    // any z is NaN), which decides whether the later passes need the range
    // checks of their fast forms
    float m = -INFINITY, lo = INFINITY;
    for (int hf = 0; hf < 2; ++hf) {
      land(i, hf);
      for (int g = (hf ? h4 : 0) + tid; g < (hf ? n4 : h4); g += kCThreads) {
        const float4 z = scaled4(b4[g], by_t);
        m = fmaxf(m, fmaxf(fmaxf(z.x, z.y), fmaxf(z.z, z.w)));
        lo = min_nan(lo, min_nan(min_nan(z.x, z.y), min_nan(z.z, z.w)));
        b4[g] = z;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
      lo = min_nan(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
    }
    if (lane == 0) red_f[warp] = make_float2(m, lo);
    __syncthreads();
    if (warp == 0) {
      float2 t = make_float2(-INFINITY, INFINITY);
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) t = make_float2(fmaxf(t.x, red_f[w].x), min_nan(t.y, red_f[w].y));
      push2(0, b, x_mm[b], t.x, t.y);
    }
    // lane q takes CTA q's values (NaN, never in correct operation, if the
    // cluster's did not all land)
    const bool ok_mm = landed(0, b, i >> 1);
    m = -INFINITY;
    lo = INFINITY;
    if (static_cast<uint32_t>(lane) < csize) {
      const float2 v = x_mm[b][lane];
      m = v.x;
      lo = v.y;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
      lo = min_nan(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
    }
    if (!ok_mm) m = NAN;
    if (m == -INFINITY) {  // every z of the row is NaN or -inf: is any -inf?
      int any = 0;
      for (int g = tid; g < n4; g += kCThreads) {
        const float4 z = b4[g];
        any |= (z.x == z.x) | (z.y == z.y) | (z.z == z.z) | (z.w == z.w);
      }
      any = __syncthreads_or(any);
      const int xa = n_any & 1;
      if (warp == 0) push8(1, xa, x_any[xa], static_cast<unsigned long long>(any));
      const bool ok_any = landed(1, xa, n_any >> 1);
      ++n_any;
      any = ok_any && static_cast<uint32_t>(lane) < csize ? static_cast<int>(x_any[xa][lane]) : 0;
      if (!__any_sync(0xFFFFFFFFu, any)) {  // all NaN: a row of zeros
        for (int g = tid; g < n4; g += kCThreads) __stcs(o4 + g, make_float4(0.f, 0.f, 0.f, 0.f));
        __syncthreads();
        if (tid == 0 && next) {
          issue(r + ncl, 0);
          issue(r + ncl, 1);
        }
        continue;
      }
    }

    // pass 2: e in place (-1 for a NaN z); the cluster's weight total.  When
    // every z is a number within 86.5 of m (and m is finite), every id takes
    // exp's fast form with no check: RN(z - m) >= RN(lo - m) >= -86.5.
    WeightSum ws;  // at most kCSliceBytesMax / (16 kCThreads) groups of four a thread
    const bool m_finite = fabsf(m) <= 3.4028235e38f;
    const float spread = __fsub_rn(lo, m);  // NaN if any z is NaN
    if (m_finite && spread >= -86.5f) {
      for (int g = tid; g < n4; g += kCThreads) {
        const float4 z = b4[g];
        const float4 e = make_float4(exp_mid(__fsub_rn(z.x, m)), exp_mid(__fsub_rn(z.y, m)),
                                     exp_mid(__fsub_rn(z.z, m)), exp_mid(__fsub_rn(z.w, m)));
        ws.add(e.x);
        ws.add(e.y);
        ws.add(e.z);
        ws.add(e.w);
        b4[g] = e;
      }
    } else {
      for (int g = tid; g < n4; g += kCThreads) {
        const float4 z = b4[g];
        float4 e;
        const float4 x = make_float4(__fsub_rn(z.x, m), __fsub_rn(z.y, m), __fsub_rn(z.z, m), __fsub_rn(z.w, m));
        if (m_finite && min_nan(min_nan(x.x, x.y), min_nan(x.z, x.w)) >= -86.5f)
          e = make_float4(exp_mid(x.x), exp_mid(x.y), exp_mid(x.z), exp_mid(x.w));
        else
          e = make_float4(weight_e(z.x, m), weight_e(z.y, m), weight_e(z.z, m), weight_e(z.w, m));
        ws.add(fmaxf(e.x, 0.0f));  // -1 (a NaN z) weighs nothing
        ws.add(fmaxf(e.y, 0.0f));
        ws.add(fmaxf(e.z, 0.0f));
        ws.add(fmaxf(e.w, 0.0f));
        b4[g] = e;
      }
    }
    uint64_t part = warp_sum_u64(ws.total());
    if (lane == 0) red_u[warp] = part;
    __syncthreads();
    if (warp == 0) {
      unsigned long long t = 0;
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) t += red_u[w];
      push8(2, n_sum & 1, x_sum[n_sum & 1], t);
    }
    const bool ok_sum = landed(2, n_sum & 1, n_sum >> 1);
    uint64_t S = ok_sum && static_cast<uint32_t>(lane) < csize ? x_sum[n_sum & 1][lane] : 0ull;
    ++n_sum;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);

    // pass 3: the probabilities of this slice, a half at a time, each half
    // then taking the next row's
    // (every e >= exp(-41) > 2^-60 when the spread is within 41: no checks)
    const Divider by_s = make_divider(__fmul_rn(__ull2float_rn(S), 0x1p-40f));
    const bool all_fast = by_s.fast && m_finite && spread >= -41.0f;
    for (int hf = 0; hf < 2; ++hf) {
      for (int g = (hf ? h4 : 0) + tid; g < (hf ? n4 : h4); g += kCThreads) {
        const float4 e = b4[g];
        float4 p;
        if (all_fast || (by_s.fast && fminf(fminf(e.x, e.y), fminf(e.z, e.w)) >= 0x1p-60f)) {
          const auto q = [&](float v) {
            const float a = __fmul_rn(v, by_s.y);
            return __fmaf_rn(__fmaf_rn(-a, by_s.d, v), by_s.y, a);
          };
          p = make_float4(q(e.x), q(e.y), q(e.z), q(e.w));
        } else {
          const auto q = [&](float v) { return v >= 0.0f ? div_rn(v, by_s) : 0.0f; };
          p = make_float4(q(e.x), q(e.y), q(e.z), q(e.w));
        }
        __stcs(o4 + g, p);
      }
      __syncthreads();  // the half is free
      if (tid == 0 && next) issue(r + ncl, hf);
    }
  }
  ptx::cluster_sync();  // no CTA leaves while another may still read its slots
}

// One row.  The output row doubles as scratch: pass 1 stores z there, the
// weight pass replaces it by e (or -1 for an id that top-k or a NaN z
// dropped), and the last pass by the probability, so later passes read a
// value instead of recomputing a division and an exp, from L2 (one row per
// SM is in flight).
__device__ void logits_probs_row(const float* l, float* out, int64_t vocab, float temperature, int32_t top_k,
                                 float top_p, RowSmem& sm, CompactSmem& cs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool vec = (((reinterpret_cast<uintptr_t>(l) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0) &&
                   (vocab & 3) == 0;

  if (!(temperature > 0.0f)) {  // greedy: lowest id of the largest non-NaN logit
    float best = 0.0f;
    int64_t best_id = -1;
    row_each(l, vocab, vec, [&](int64_t v, float x) {
      if (!isnan(x) && (best_id < 0 || x > best || (x == best && v < best_id))) {
        best = x;
        best_id = v;
      }
    });
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, off);
      const int64_t oi = __shfl_xor_sync(0xFFFFFFFFu, best_id, off);
      if (oi >= 0 && (best_id < 0 || ob > best || (ob == best && oi < best_id))) {
        best = ob;
        best_id = oi;
      }
    }
    if (lane == 0) {
      sm.red_f[warp] = best;
      sm.red_id[warp] = best_id;
    }
    __syncthreads();
    best = 0.0f;
    best_id = -1;
    for (int w = 0; w < kWarps; ++w) {
      const float ob = sm.red_f[w];
      const int64_t oi = sm.red_id[w];
      if (oi >= 0 && (best_id < 0 || ob > best || (ob == best && oi < best_id))) {
        best = ob;
        best_id = oi;
      }
    }
    __syncthreads();
    row_map<false, true>(out, out, vocab, vec, [&](int64_t v, float) { return v == best_id ? 1.0f : 0.0f; });
    return;
  }

  // pass 1: z into the output row; non-NaN count and the largest z
  int n_local = 0;
  float m = -INFINITY;
  const Divider by_t = make_divider(temperature);
  row_map<true, false, 4>(l, out, vocab, vec, [&](int64_t, float x) {
    const float z = __fadd_rn(div_rn(x, by_t), 0.0f);  // -0 becomes +0
    n_local += z == z;
    m = fmaxf(m, z);  // a NaN z leaves m as it is
    return z;
  });
  sm.tkey[threadIdx.x] = n_local > 0 ? order_key(m) : 0u;  // read after the barriers below
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    n_local += __shfl_xor_sync(0xFFFFFFFFu, n_local, off);
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  }
  if (lane == 0) {
    sm.red_i[warp] = n_local;
    sm.red_f[warp] = m;
  }
  __syncthreads();
  int64_t n_valid = 0;
  m = -INFINITY;
  for (int w = 0; w < kWarps; ++w) {
    n_valid += sm.red_i[w];
    m = fmaxf(m, sm.red_f[w]);
  }
  __syncthreads();
  if (n_valid == 0) {
    row_map<false, true>(out, out, vocab, vec, [](int64_t, float) { return 0.0f; });
    return;
  }

  // top-k: the k-th largest key by four 8-bit passes over z, then the tie cut
  const bool topk = top_k > 0 && top_k < n_valid;
  uint32_t k_key = 0;
  int64_t k_id = vocab;
  const bool gathered = topk && top_k <= kThreads && prefilter_cut(out, vocab, vec, top_k, k_key, k_id, sm, cs);
  if (topk && !gathered) {
    if (threadIdx.x == 0) {
      sm.k_prefix = 0;
      sm.k_mask = 0;
      sm.k_rem = top_k;
    }
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kThreads) sm.hist[i] = 0;
      __syncthreads();
      const uint32_t prefix = sm.k_prefix, mask = sm.k_mask;
      row_each(out, vocab, vec, [&](int64_t, float z) {
        if (isnan(z)) return;
        const uint32_t key = order_key(z);
        if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
      });
      __syncthreads();
      if (threadIdx.x == 0) {
        int64_t rem = sm.k_rem;
        int b = 255;
        for (; b > 0; --b) {
          const int64_t c = sm.hist[b];
          if (c >= rem) break;
          rem -= c;
        }
        sm.k_prefix = prefix | (static_cast<uint32_t>(b) << shift);
        sm.k_mask = mask | (255u << shift);
        sm.k_rem = rem;
        if (shift == 0) sm.found = sm.hist[b];  // ids with exactly this key
      }
      __syncthreads();
    }
    k_key = sm.k_prefix;
    const int64_t rem = sm.k_rem, ties = sm.found;
    __syncthreads();
    if (rem < ties)
      k_id = nth_in_order(
          vocab, rem,
          [&](int64_t v) {
            const float z = out[v];
            return !isnan(z) && order_key(z) == k_key;
          },
          sm);
  }
  if (topk && top_k <= kCompactMax) {
    compact_finish(out, vocab, vec, top_k, k_key, k_id, m, top_p, gathered, sm, cs);
    return;
  }

  // weight pass: e (or -1 for a dropped id) into the output row; the kept total
  uint64_t part = 0;
  row_map<false, false>(out, out, vocab, vec, [&](int64_t v, float z) {
    if (isnan(z)) return -1.0f;
    if (topk) {
      const uint32_t key = order_key(z);
      if (!(key > k_key || (key == k_key && v <= k_id))) return -1.0f;
    }
    const float e = own_exp_nonpos(z == m ? 0.0f : __fsub_rn(z, m));
    part += weight(e);
    return e;
  });
  const uint64_t W = block_sum_u64(part, sm);

  // top-p: the cut weight by six 8-bit passes of weight sums, then the tie cut
  const bool topp = top_p < 1.0f;
  uint64_t S = W, p_w = 0;
  int64_t p_id = vocab;
  if (topp) {
    if (threadIdx.x == 0) {
      sm.p_thr = top_p_threshold(top_p, W);
      sm.p_prefix = 0;
      sm.p_mask = 0;
      sm.p_above = 0;
    }
    for (int shift = 40; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kThreads) sm.whist[i] = 0;
      __syncthreads();
      const uint64_t prefix = sm.p_prefix, mask = sm.p_mask;
      row_each(out, vocab, vec, [&](int64_t, float e) {
        if (e < 0.0f) return;
        const uint64_t w = weight(e);
        if ((w & mask) == prefix) atomicAdd(&sm.whist[(w >> shift) & 255u], static_cast<unsigned long long>(w));
      });
      __syncthreads();
      if (threadIdx.x == 0) {
        uint64_t above = sm.p_above;
        const uint64_t thr = sm.p_thr;
        int b = 255;
        for (; b > 0; --b) {
          if (above + sm.whist[b] >= thr) break;
          above += sm.whist[b];
        }
        sm.p_prefix = prefix | (static_cast<uint64_t>(b) << shift);
        sm.p_mask = mask | (255ull << shift);
        sm.p_above = above;
        if (shift == 0) sm.found = static_cast<int64_t>(sm.whist[b]);  // mass at exactly this weight
      }
      __syncthreads();
    }
    p_w = sm.p_prefix;
    const uint64_t above = sm.p_above, thr = sm.p_thr, at_cut = static_cast<uint64_t>(sm.found);
    __syncthreads();
    const uint64_t tau = p_w > 0 ? p_w : 1ull;
    const uint64_t need = (thr - above + tau - 1) / tau;  // ids of weight p_w to take
    const uint64_t ties = at_cut / tau;
    S = above + need * p_w;
    if (need < ties)
      p_id = nth_in_order(
          vocab, static_cast<int64_t>(need),
          [&](int64_t v) {
            const float e = out[v];
            return e >= 0.0f && weight(e) == p_w;
          },
          sm);
  }

  const float Sf = __fmul_rn(__ull2float_rn(S), 0x1p-40f);
  const Divider by_s = make_divider(Sf);
  row_map<false, true>(out, out, vocab, vec, [&](int64_t v, float e) {
    bool keep = e >= 0.0f;
    if (keep && topp) {
      const uint64_t w = weight(e);
      keep = w > p_w || (w == p_w && v <= p_id);
    }
    return keep ? div_rn(e, by_s) : 0.0f;
  });
}

// A persistent grid of one CTA per SM takes rows in turn, so that the rows in
// flight (one output row each) stay in L2 across their passes.
__global__ void __launch_bounds__(kThreads)
    logits_probs_kernel(const float* logits, float* probs, int32_t rows, int64_t vocab, float temperature,
                        int32_t top_k, float top_p) {
  __shared__ RowSmem sm;
  __shared__ CompactSmem cs;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    logits_probs_row(logits + r * vocab, probs + r * vocab, vocab, temperature, top_k, top_p, sm, cs);
    __syncthreads();  // shared state is reused by the next row
  }
}

constexpr int kAttrMaxDevices = 64;
std::atomic<unsigned long long> g_cluster_attr_ctx[kAttrMaxDevices];

// The cluster kernel's shared-memory limit, set once per device context.
bool cluster_attr_ready(int device) {
  if (device < 0 || device >= kAttrMaxDevices) return false;
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && g_cluster_attr_ctx[device].load(std::memory_order_acquire) == ctx) return true;
  if (cudaFuncSetAttribute(probs_plain_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kCSliceBytesMax) != cudaSuccess)
    return false;
  g_cluster_attr_ctx[device].store(ctx, std::memory_order_release);
  return true;
}

// The plain setting on clusters; false when that does not apply (a
// vocabulary of more than 8 slices, or no cluster fits), and the caller
// takes the one-CTA-per-row kernel.
bool launch_plain_cluster(const float* logits, float* probs, int rows, int vocab, float temperature, int device,
                          cudaStream_t stream, int* rc) {
  int C = 1, slice = 0;
  for (; C <= kCMaxCluster; C *= 2) {
    slice = ((vocab + C - 1) / C + 3) & ~3;
    if (slice * 4 <= kCSliceBytesMax) break;
  }
  if (C > kCMaxCluster || !cluster_attr_ready(device)) return false;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(slice) * 4;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(C);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, probs_plain_cluster_kernel, &cfg) != cudaSuccess || clusters < 1) {
    (void)cudaGetLastError();
    return false;
  }
  cfg.gridDim = dim3((rows < clusters ? rows : clusters) * C);
  *rc = cudaLaunchKernelEx(&cfg, probs_plain_cluster_kernel, logits, probs, rows, vocab, temperature, slice) ==
                cudaSuccess
            ? DSPARK_OK
            : DSPARK_ERR_CUDA;
  return true;
}

}  // namespace
}  // namespace dspark

extern "C" int dspark_logits_to_probs(const float* logits, float* probs, int32_t rows, int32_t vocab,
                                      float temperature, int32_t top_k, float top_p, cudaStream_t stream) {
  if (rows < 0 || vocab < 1) return DSPARK_ERR_INVALID_ARG;
  if (rows == 0) return DSPARK_OK;
  if (!logits || !probs) return DSPARK_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const int grid = rows < sms ? rows : sms;
  const bool vec = (vocab & 3) == 0 && ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(probs)) & 15u) == 0;
  if (vec && temperature > 0.0f && !(top_k > 0 && top_k < vocab) && !(top_p < 1.0f)) {
    int rc = DSPARK_OK;
    if (dspark::launch_plain_cluster(logits, probs, rows, vocab, temperature, dev, stream, &rc)) return rc;
  }
  dspark::logits_probs_kernel<<<grid, dspark::kThreads, 0, stream>>>(logits, probs, rows, vocab, temperature, top_k,
                                                                     top_p);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
