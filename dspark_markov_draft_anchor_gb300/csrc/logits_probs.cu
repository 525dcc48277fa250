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
// One CTA of 1024 threads per row.  The k-th largest key and the top-p cut
// are radix selects over the row (8 bits a pass: four passes of counts over
// the 32-bit logit keys, six passes of weight sums over the 48-bit weights),
// ties at a cut are resolved by one ordered scan, and a last pass writes the
// row.  The output row holds z, then e, between passes (see
// logits_probs_row).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dspark_markov.h"
#include "markov_math.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// floor(e 2^40) for e in [0, 1], in integer instructions (significand
// shifted by the exponent).
__device__ __forceinline__ uint64_t weight(float e) {
  if (!(e > 0.0f)) return 0ull;
  if (e >= 1.0f) return 1ull << 40;
  const uint32_t b = __float_as_uint(e);
  const uint32_t ex = b >> 23;
  const uint32_t m = (b & 0x7FFFFFu) | (ex ? 0x800000u : 0u);
  const int sh = static_cast<int>(ex ? ex : 1u) - 110;
  return sh >= 0 ? static_cast<uint64_t>(m) << sh : static_cast<uint64_t>(m >> (-sh < 31 ? -sh : 31));
}

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
// per SM keeps enough requests in flight; the passes over L2 take 1 (more
// would spill the inlined per-id work).
// row_map writes f's value back in place of what it read (the same thread
// reads and then writes each id, so src may equal dst).
template <int kBatch = 1, class F>
__device__ __forceinline__ void row_each(const float* src, int64_t vocab, bool vec, F&& f) {
  if (vec) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    const int64_t n4 = vocab >> 2;
    for (int64_t g0 = threadIdx.x; g0 < n4; g0 += kBatch * kThreads) {
      float4 x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (g0 + k * kThreads < n4) x[k] = s4[g0 + k * kThreads];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t g = g0 + k * kThreads;
        if (g < n4) {
          f(4 * g, x[k].x);
          f(4 * g + 1, x[k].y);
          f(4 * g + 2, x[k].z);
          f(4 * g + 3, x[k].w);
        }
      }
    }
  } else {
    for (int64_t v0 = threadIdx.x; v0 < vocab; v0 += kBatch * kThreads) {
      float x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (v0 + k * kThreads < vocab) x[k] = src[v0 + k * kThreads];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (v0 + k * kThreads < vocab) f(v0 + k * kThreads, x[k]);
    }
  }
}

template <bool kStreamIn, bool kStreamOut, int kBatch = 1, class F>
__device__ __forceinline__ void row_map(const float* src, float* dst, int64_t vocab, bool vec, F&& f) {
  if (vec) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* d4 = reinterpret_cast<float4*>(dst);
    const int64_t n4 = vocab >> 2;
    for (int64_t g0 = threadIdx.x; g0 < n4; g0 += kBatch * kThreads) {
      float4 x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t g = g0 + k * kThreads;
        if (g < n4) x[k] = kStreamIn ? __ldcs(s4 + g) : s4[g];
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t g = g0 + k * kThreads;
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
    for (int64_t v0 = threadIdx.x; v0 < vocab; v0 += kBatch * kThreads) {
      float x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t v = v0 + k * kThreads;
        if (v < vocab) x[k] = kStreamIn ? __ldcs(src + v) : src[v];
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int64_t v = v0 + k * kThreads;
        if (v < vocab) {
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

// After a top-k cut of K <= kCompactMax ids: gather them (and their z) into
// shared memory, take e and w there, cut top-p on the K entries sorted by
// (w descending, id ascending) (a bitonic sort, then a block scan for the
// shortest prefix reaching the threshold), then zero the row and scatter
// the probabilities.  Equal to the full-row passes: the same sets, sums and
// roundings.
__device__ __noinline__ void compact_finish(float* out, int64_t vocab, bool vec, int K, uint32_t k_key, int64_t k_id,
                                            float m, float top_p, RowSmem& sm, CompactSmem& cs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  if (vec) {
    float4* d4 = reinterpret_cast<float4*>(out);
    for (int64_t g = threadIdx.x; g < (vocab >> 2); g += kThreads) __stcs(d4 + g, make_float4(0.f, 0.f, 0.f, 0.f));
  } else {
    for (int64_t v = threadIdx.x; v < vocab; v += kThreads) __stcs(out + v, 0.0f);
  }
  __syncthreads();  // the zeros are ordered before the scattered values
  for (int i = threadIdx.x; i < n_final; i += kThreads) out[cs.id[i]] = __fdiv_rn(cs.e[i], Sf);
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
  row_map<true, false, 4>(l, out, vocab, vec, [&](int64_t, float x) {
    float z = __fdiv_rn(x, temperature);
    if (!isnan(z)) {
      ++n_local;
      if (z == 0.0f) z = 0.0f;
      m = fmaxf(m, z);
    }
    return z;
  });
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
  if (topk) {
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
    if (top_k <= kCompactMax) {
      compact_finish(out, vocab, vec, top_k, k_key, k_id, m, top_p, sm, cs);
      return;
    }
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
  row_map<false, true>(out, out, vocab, vec, [&](int64_t v, float e) {
    bool keep = e >= 0.0f;
    if (keep && topp) {
      const uint64_t w = weight(e);
      keep = w > p_w || (w == p_w && v <= p_id);
    }
    return keep ? __fdiv_rn(e, Sf) : 0.0f;
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
  dspark::logits_probs_kernel<<<grid, dspark::kThreads, 0, stream>>>(logits, probs, rows, vocab, temperature, top_k,
                                                                     top_p);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
