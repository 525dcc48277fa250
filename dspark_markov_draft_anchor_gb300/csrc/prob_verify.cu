// prob_verify.cu -- the probabilistic verify side: deterministic uniforms
// ([P1] dsparkFillUniforms) and speculative acceptance with residual
// sampling ([P1] dsparkProbabilisticAccept), behind the C ABI of
// include/dspark_markov.h.
//
// Sampling from a probability row is an inverse CDF over fixed-point weights
// (each probability clamped to [0, 1] and truncated to units of 2^-40), so
// every sum is exact and the sampled id does not depend on the order in which
// threads add: U = floor(u 2^24), T = floor(U S / 2^24) for the row's total
// S, and the sample is the smallest id whose inclusive prefix exceeds T.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "dspark_markov.h"
#include "kernels.h"
#include "ptx.cuh"

namespace dspark {
namespace {

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011): ten rounds of the
// 4x32 bijection, multipliers 0xD2511F53 and 0xCD9E8D57, key bumped by
// 0x9E3779B9 / 0xBB67AE85 between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// Element i is word i % 4 of the block at counter offset + i / 4 (a 64-bit
// number in the low two words), key (lo, hi) of the seed; its top 24 bits
// times 2^-24.  One thread per counter block.
__global__ void fill_uniforms_kernel(float* __restrict__ u, int64_t n, uint64_t seed, uint64_t offset) {
  const int64_t blocks = (n + 3) / 4;
  const uint2 key = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  for (int64_t blk = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; blk < blocks;
       blk += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint64_t ctr = offset + static_cast<uint64_t>(blk);
    const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32), 0u, 0u), key);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    const int64_t i0 = blk * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i0 + j < n) u[i0 + j] = static_cast<float>(w[j] >> 8) * (1.0f / 16777216.0f);
  }
}

// A probability as a weight in units of 2^-40: [0, 1] clamped (NaN and
// negatives weigh 0), truncated.  For 0 < p < 1 the value is the 24-bit
// significand m (implicit bit included; subnormals use exponent field 1)
// shifted by e - 110 (e the biased exponent field), i.e. floor(p 2^40), in
// integer instructions only: a float-to-64-bit conversion would run on the
// FP64 pipe, which this part has little of.
__device__ __forceinline__ uint64_t weight(float p) {
  if (!(p > 0.0f)) return 0ull;
  if (p >= 1.0f) return 1ull << 40;
  const uint32_t b = __float_as_uint(p);
  const uint32_t e = b >> 23;
  const uint32_t m = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  const int sh = static_cast<int>(e ? e : 1u) - 110;  // <= 16
  return sh >= 0 ? static_cast<uint64_t>(m) << sh : static_cast<uint64_t>(m >> (-sh < 31 ? -sh : 31));
}

// T = floor(U S / 2^24), U = floor(u 2^24) clamped to [0, 2^24 - 1].
__device__ __forceinline__ uint64_t threshold(float u, uint64_t total) {
  const float uu = u > 0.0f ? u : 0.0f;
  uint64_t U = __float2ull_rz(uu * 0x1p24f);
  if (U > 0xFFFFFFull) U = 0xFFFFFFull;
  const uint64_t lo = U * total, hi = __umul64hi(U, total);
  return (hi << 40) | (lo >> 24);
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  return x;
}

__device__ __forceinline__ uint64_t warp_incl_scan_u64(uint64_t x, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  return x;
}

constexpr int kAcceptThreads = 512;
constexpr int kAcceptWarps = kAcceptThreads / 32;
constexpr int kScanSpan = 4 * kAcceptThreads;  // ids one block-wide scan covers
constexpr int kMaxChunks = 1024;               // chunk totals kept in shared memory
constexpr int kPiece = 512;                    // ids one warp streams per bulk copy
static_assert(kPiece / 32 <= 16, "wacc adds at most 16 halves exactly");
constexpr uint32_t kCopyWaitLimit = 1u << 24;  // polls of a copy's mbarrier
constexpr size_t kStageBytes = size_t{kAcceptWarps} * 2 * kPiece * sizeof(float);

// One row being sampled: the target row t and, for a residual, the draft
// row q (null for the target row itself).  vec: both rows start on a
// 16-byte boundary, so groups of four ids load as float4; bulk: also a
// vocabulary of a multiple of four ids, so that every piece of the row is a
// whole number of 16-byte units and streams by bulk copies.
struct Row {
  const float* t;
  const float* q;
  int64_t vocab;
  bool vec;
  bool bulk;
};

// Warp w's staging area: one piece of t and one of q, refilled by the warp
// itself once it has read them, completing on mbarrier full[w].  `used`
// counts the pieces the warp has taken from it (the next one's phase parity
// is used & 1); `failed` is set when a wait gave up.
struct Stage {
  float* buf;
  uint64_t* full;
  uint32_t used;
  bool failed;
};

// The weights of ids v .. v+3 (ids past the end weigh 0): max(0, RN(t - q))
// for a residual, else t, each through weight().
__device__ __forceinline__ void weights4(const Row& r, int64_t v, uint64_t w[4]) {
  if (r.vec && v + 4 <= r.vocab) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(r.t + v));
    if (r.q) {
      const float4 b = __ldg(reinterpret_cast<const float4*>(r.q + v));
      w[0] = weight(__fsub_rn(a.x, b.x));
      w[1] = weight(__fsub_rn(a.y, b.y));
      w[2] = weight(__fsub_rn(a.z, b.z));
      w[3] = weight(__fsub_rn(a.w, b.w));
    } else {
      w[0] = weight(a.x);
      w[1] = weight(a.y);
      w[2] = weight(a.z);
      w[3] = weight(a.w);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t x = v + k;
    w[k] = x < r.vocab ? (r.q ? weight(__fsub_rn(r.t[x], r.q[x])) : weight(r.t[x])) : 0ull;
  }
}

template <bool kRes>
__device__ __forceinline__ uint64_t weight_at(const Row& r, int64_t x) {
  return kRes ? weight(__fsub_rn(r.t[x], r.q[x])) : weight(r.t[x]);
}

// The same weight on the FP32 pipe, split in two exact halves and added to
// two float accumulators: with y = c 2^20 (c the probability clamped to
// [0, 1], NaN to 0 by fmaxf), floor(c 2^40) = floor(y) 2^20 +
// floor(frac(y) 2^20); each floor is a round-toward-zero add of 2^23 (exact
// for values below 2^23), frac(y) = y - floor(y) is exact, and each half is an
// integer of at most 2^20, so up to 16 of them add exactly in FP32.  Sixteen
// ids cost ten FP32 operations each and one conversion pair (wflush) instead
// of about twenty integer ones each.
__device__ __forceinline__ void wacc(float p, float& hi, float& lo) {
  const float c = fminf(fmaxf(p, 0.0f), 1.0f);
  const float y = c * 0x1p20f;
  const float fl = __fsub_rn(__fadd_rz(y, 0x1p23f), 0x1p23f);
  hi += fl;
  lo += __fsub_rn(__fmaf_rz(__fsub_rn(y, fl), 0x1p20f, 0x1p23f), 0x1p23f);
}

__device__ __forceinline__ uint64_t wflush(float hi, float lo) {
  return (static_cast<uint64_t>(__float2uint_rz(hi)) << 20) + __float2uint_rz(lo);
}

template <bool kRes>
__device__ __forceinline__ void wacc4(float4 a, float4 b, float& hi, float& lo) {
  wacc(kRes ? __fsub_rn(a.x, b.x) : a.x, hi, lo);
  wacc(kRes ? __fsub_rn(a.y, b.y) : a.y, hi, lo);
  wacc(kRes ? __fsub_rn(a.z, b.z) : a.z, hi, lo);
  wacc(kRes ? __fsub_rn(a.w, b.w) : a.w, hi, lo);
}

template <bool kRes>
__device__ __forceinline__ uint64_t weight_sum4(float4 a, float4 b) {
  float hi = 0.0f, lo = 0.0f;
  wacc4<kRes>(a, b, hi, lo);
  return wflush(hi, lo);
}

// The weight of ids [c0, c1) summed by one warp (all lanes get the total).
// The main loops issue four loads per row before using any, with no branch
// between them, so that each lane keeps several requests in flight.
template <bool kRes>
__device__ __forceinline__ uint64_t chunk_sum(const Row& r, int64_t c0, int64_t c1, int lane) {
  uint64_t part = 0;
  if (r.vec) {
    const int64_t groups = (c1 - c0) >> 2;  // whole float4 groups
    const float4* t4 = reinterpret_cast<const float4*>(r.t + c0);
    const float4* q4 = reinterpret_cast<const float4*>(kRes ? r.q + c0 : r.t + c0);
    int64_t g = lane;
    for (; g + 96 < groups; g += 128) {
      const float4 a0 = __ldg(t4 + g), a1 = __ldg(t4 + g + 32), a2 = __ldg(t4 + g + 64), a3 = __ldg(t4 + g + 96);
      float4 b0 = a0, b1 = a1, b2 = a2, b3 = a3;
      if (kRes) {
        b0 = __ldg(q4 + g);
        b1 = __ldg(q4 + g + 32);
        b2 = __ldg(q4 + g + 64);
        b3 = __ldg(q4 + g + 96);
      }
      float hi = 0.0f, lo = 0.0f;  // 16 ids: exact (see wacc)
      wacc4<kRes>(a0, b0, hi, lo);
      wacc4<kRes>(a1, b1, hi, lo);
      wacc4<kRes>(a2, b2, hi, lo);
      wacc4<kRes>(a3, b3, hi, lo);
      part += wflush(hi, lo);
    }
    for (; g < groups; g += 32) part += weight_sum4<kRes>(__ldg(t4 + g), kRes ? __ldg(q4 + g) : float4{});
    const int64_t x = c0 + 4 * groups + lane;  // at most three ids left
    if (x < c1) part += weight_at<kRes>(r, x);
  } else {
    int64_t x = c0 + lane;
    for (; x + 96 < c1; x += 128) {
      const float a0 = r.t[x], a1 = r.t[x + 32], a2 = r.t[x + 64], a3 = r.t[x + 96];
      if (kRes) {
        const float b0 = r.q[x], b1 = r.q[x + 32], b2 = r.q[x + 64], b3 = r.q[x + 96];
        part += (weight(__fsub_rn(a0, b0)) + weight(__fsub_rn(a1, b1))) +
                (weight(__fsub_rn(a2, b2)) + weight(__fsub_rn(a3, b3)));
      } else {
        part += (weight(a0) + weight(a1)) + (weight(a2) + weight(a3));
      }
    }
    for (; x < c1; x += 32) part += weight_at<kRes>(r, x);
  }
  return warp_sum_u64(part);
}

// Stage 1 over bulk copies: warp w streams pieces w, w + kAcceptWarps, ...
// of the row (kPiece ids of t, and of q for a residual) into its own stage,
// sums each piece's weights (16 ids a lane, float4 reads of shared memory),
// hands the stage back to the copy engine for its next piece as soon as the
// values are in registers, and adds the piece's total to its chunk's.
template <bool kRes>
__device__ __forceinline__ void stream_sums(const Row& r, int64_t chunk_len, uint64_t* chunk, Stage& st, int warp,
                                            int lane) {
  const int64_t n_pieces = (r.vocab + kPiece - 1) / kPiece;
  float* st_t = st.buf;
  float* st_q = st.buf + kPiece;
  auto issue = [&](int64_t piece) {
    const int64_t v0 = piece * kPiece;
    const uint32_t bytes = static_cast<uint32_t>((r.vocab - v0 < kPiece ? r.vocab - v0 : kPiece) * sizeof(float));
    ptx::mbar_arrive_expect_tx(st.full, kRes ? 2 * bytes : bytes);
    ptx::bulk_load(st_t, r.t + v0, bytes, st.full);
    if (kRes) ptx::bulk_load(st_q, r.q + v0, bytes, st.full);
  };
  int64_t piece = warp;
  if (lane == 0 && piece < n_pieces) issue(piece);
  for (; piece < n_pieces; piece += kAcceptWarps) {
    if (!ptx::mbar_wait(st.full, st.used & 1, kCopyWaitLimit)) {
      st.failed = true;  // leave the copy to land (bounded) before the kernel exits
      ptx::mbar_wait(st.full, st.used & 1, kCopyWaitLimit);
      return;
    }
    ++st.used;
    const int64_t v0 = piece * kPiece;
    const int64_t cnt = r.vocab - v0 < kPiece ? r.vocab - v0 : kPiece;  // a multiple of 4
    float hi = 0.0f, lo = 0.0f;  // kPiece / 32 = 16 ids a lane: exact (see wacc)
#pragma unroll
    for (int k = 0; k < kPiece / 128; ++k) {
      const int e = 4 * (lane + 32 * k);
      if (e < cnt) {
        const float4 a = *reinterpret_cast<const float4*>(st_t + e);
        const float4 b = kRes ? *reinterpret_cast<const float4*>(st_q + e) : a;
        wacc4<kRes>(a, b, hi, lo);
      }
    }
    uint64_t part = wflush(hi, lo);
    __syncwarp();
    // the stage's next fill is an async-proxy write: the proxy fence orders
    // it after the warp's generic reads of the stage (synchronised by the
    // warp barrier above)
    if (lane == 0 && piece + kAcceptWarps < n_pieces) {
      ptx::fence_proxy_async_smem();
      issue(piece + kAcceptWarps);
    }
    part = warp_sum_u64(part);
    if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long*>(&chunk[v0 / chunk_len]), part);
  }
}

struct SampleSmem {
  uint64_t chunk[kMaxChunks];  // weight of each chunk of the row
  uint64_t wsum[kAcceptWarps];  // block scan: each warp's total
  uint64_t rest;                // threshold left inside the chosen chunk
  int64_t chunk_id;             // chosen chunk, -1 when the row weighs 0
  int64_t pick;
};

// Inverse-CDF sample of one row by the whole CTA, in three steps:
//  1. the row is cut into chunks of chunk_len ids (kScanSpan, or a multiple
//     of it for rows of more than kMaxChunks spans) and each chunk's total
//     weight is kept: streamed through shared memory by bulk copies where
//     the row allows (stream_sums), else warp w sums chunks w,
//     w + kAcceptWarps, ... with float4 or scalar loads;
//  2. warp 0 adds the totals, takes T from u, and finds the chunk whose
//     running total first exceeds T (a warp scan over 32 chunks at a time);
//  3. the CTA scans that chunk kScanSpan ids at a time (four ids a thread,
//     a block-wide exclusive scan of the thread sums) and the one thread
//     whose range holds the threshold picks the id.
// Returns -1 (in every thread) when the row weighs 0.
__device__ int64_t sample_row(const Row& r, float u, SampleSmem& sm, Stage& st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t spans = (r.vocab + kScanSpan - 1) / kScanSpan;
  const int64_t chunk_len = kScanSpan * ((spans + kMaxChunks - 1) / kMaxChunks);
  const int64_t n_chunks = (r.vocab + chunk_len - 1) / chunk_len;

  if (r.bulk) {
    for (int64_t c = threadIdx.x; c < n_chunks; c += kAcceptThreads) sm.chunk[c] = 0;
    __syncthreads();
    if (r.q)
      stream_sums<true>(r, chunk_len, sm.chunk, st, warp, lane);
    else
      stream_sums<false>(r, chunk_len, sm.chunk, st, warp, lane);
  } else {
    for (int64_t c = warp; c < n_chunks; c += kAcceptWarps) {
      const int64_t c0 = c * chunk_len;
      const int64_t c1 = c0 + chunk_len < r.vocab ? c0 + chunk_len : r.vocab;
      const uint64_t part = r.q ? chunk_sum<true>(r, c0, c1, lane) : chunk_sum<false>(r, c0, c1, lane);
      if (lane == 0) sm.chunk[c] = part;
    }
  }
  __syncthreads();

  if (warp == 0) {
    uint64_t total = 0;
    for (int64_t c = lane; c < n_chunks; c += 32) total += sm.chunk[c];
    total = warp_sum_u64(total);
    int64_t chosen = -1;
    uint64_t rest = 0;
    if (total > 0) {
      const uint64_t T = threshold(u, total);  // T < total: some chunk holds it
      uint64_t run = 0;
      for (int64_t base = 0; base < n_chunks; base += 32) {
        const int64_t c = base + lane;
        const uint64_t x = c < n_chunks ? sm.chunk[c] : 0ull;
        const uint64_t incl = warp_incl_scan_u64(x, lane);
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, run + incl > T);
        if (hit) {
          const int src = __ffs(hit) - 1;
          const uint64_t before = run + __shfl_sync(0xFFFFFFFFu, incl - x, src);
          chosen = base + src;
          rest = T - before;
          break;
        }
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
    if (lane == 0) {
      sm.chunk_id = chosen;
      sm.rest = rest;
      sm.pick = -1;
    }
  }
  __syncthreads();
  const int64_t chosen = sm.chunk_id;
  if (chosen < 0) {
    __syncthreads();  // sm is reused by the next call
    return -1;
  }

  uint64_t rest = sm.rest;
  const int64_t c_end = (chosen + 1) * chunk_len < r.vocab ? (chosen + 1) * chunk_len : r.vocab;
  for (int64_t s0 = chosen * chunk_len; s0 < c_end; s0 += kScanSpan) {
    const int64_t v = s0 + 4 * threadIdx.x;
    uint64_t w[4];
    weights4(r, v, w);
    const uint64_t mine = (w[0] + w[1]) + (w[2] + w[3]);
    const uint64_t incl = warp_incl_scan_u64(mine, lane);
    if (lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    uint64_t offset = 0, span_total = 0;
#pragma unroll
    for (int k = 0; k < kAcceptWarps; ++k) {
      const uint64_t x = sm.wsum[k];
      if (k < warp) offset += x;
      span_total += x;
    }
    const uint64_t excl = offset + incl - mine;
    if (rest >= excl && rest - excl < mine) {  // exactly one thread, when rest < span_total
      uint64_t left = rest - excl;  // < mine, so one of the four ids holds it
      int k = 3;
      if (left < w[0]) {
        k = 0;
      } else if ((left -= w[0]) < w[1]) {
        k = 1;
      } else if (left - w[1] < w[2]) {
        k = 2;
      }
      sm.pick = v + k;
    }
    __syncthreads();
    if (sm.pick >= 0) break;
    rest -= span_total;
  }
  const int64_t pick = sm.pick;
  __syncthreads();  // sm is reused by the next call
  return pick;
}

// One CTA per batch row.  Warp 0 evaluates up to 32 positions of the accept
// chain at once (draft id, then the two probabilities at it) and the first
// rejection ends it; then the CTA draws one inverse-CDF sample: the residual
// after a rejection (the target row when that weighs 0), else the bonus.
__global__ void __launch_bounds__(kAcceptThreads, 2)
    prob_accept_kernel(const float* __restrict__ target, const float* __restrict__ draft_probs,
                       const int64_t* __restrict__ draft, const int32_t* __restrict__ proposal_len,
                       const float* __restrict__ uniforms, int64_t* __restrict__ accepted,
                       int32_t* __restrict__ accept_len, int32_t draft_stride, int32_t P, int64_t vocab) {
  extern __shared__ __align__(128) float s_stage[];  // kStageBytes: one stage per warp
  __shared__ SampleSmem sm;
  __shared__ __align__(8) uint64_t s_full[kAcceptWarps];
  __shared__ int s_j, s_pl, s_failed;
  if (threadIdx.x < kAcceptWarps) ptx::mbar_init(&s_full[threadIdx.x], 1);
  if (threadIdx.x == 0) s_failed = 0;
  ptx::fence_mbar_init();
  const int b = blockIdx.x;
  const float* tb = target + static_cast<int64_t>(b) * (P + 1) * vocab;
  const float* qb = draft_probs + static_cast<int64_t>(b) * P * vocab;
  const float* ub = uniforms + static_cast<int64_t>(b) * (2 * P + 1);
  int64_t* acc = accepted + static_cast<int64_t>(b) * (P + 1);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int pl = proposal_len[b];
    pl = pl < 0 ? 0 : (pl > P ? P : pl);
    int j = pl;
    for (int base = 0; base < pl; base += 32) {
      const int i = base + lane;
      bool ok = false;
      int64_t d = 0;
      if (i < pl) {
        d = draft[static_cast<int64_t>(b) * draft_stride + i];
        if (d >= 0 && d < vocab) {
          const float t = tb[static_cast<int64_t>(i) * vocab + d];
          const float q = qb[static_cast<int64_t>(i) * vocab + d];
          ok = __fmul_rn(ub[i], q) < t;
        }
      }
      const unsigned fail = __ballot_sync(0xFFFFFFFFu, i < pl && !ok);
      const int first = fail ? base + __ffs(fail) - 1 : pl;
      if (i < first) acc[i] = d;
      if (fail) {
        j = first;
        break;
      }
    }
    if (lane == 0) {
      s_j = j;
      s_pl = pl;
    }
  }
  __syncthreads();
  const int j = s_j, pl = s_pl;
  const int warp = threadIdx.x >> 5;
  Stage st{s_stage + warp * 2 * kPiece, &s_full[warp], 0u, false};
  const float* trow = tb + static_cast<int64_t>(j) * vocab;
  const bool t_vec = (reinterpret_cast<uintptr_t>(trow) & 15u) == 0;
  const bool four = (vocab & 3) == 0;
  int64_t pick = -1;
  if (j < pl) {
    const float* qrow = qb + static_cast<int64_t>(j) * vocab;
    const bool vec = t_vec && (reinterpret_cast<uintptr_t>(qrow) & 15u) == 0;
    pick = sample_row(Row{trow, qrow, vocab, vec, vec && four}, ub[P + j], sm, st);
  }
  if (st.failed) s_failed = 1;
  __syncthreads();
  if (pick < 0 && !s_failed)
    pick = sample_row(Row{trow, nullptr, vocab, t_vec, t_vec && four}, j < pl ? ub[P + j] : ub[2 * P], sm, st);
  if (st.failed) s_failed = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (s_failed) {  // a copy wait gave up: the row is marked, not sampled
      accept_len[b] = 0;
      return;
    }
    acc[j] = pick < 0 ? 0 : pick;
    for (int i = j + 1; i <= P; ++i) acc[i] = -1;
    accept_len[b] = j + 1;
  }
}

int done() { return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

// The accept kernel's dynamic shared-memory limit, raised once per context
// of each device (a kernel attribute lives in the context: a device reset or
// another context needs it set again).  The context the attribute was set in
// is kept per device ordinal; setting it twice is harmless, so two threads
// racing here only repeat the call.
constexpr int kAttrMaxDevices = 64;
std::atomic<unsigned long long> g_accept_attr_ctx[kAttrMaxDevices];

bool accept_attr_ready() {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kAttrMaxDevices) {
    (void)cudaGetLastError();
    return false;
  }
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && g_accept_attr_ctx[device].load(std::memory_order_acquire) == ctx) return true;
  if (cudaFuncSetAttribute(prob_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kStageBytes)) != cudaSuccess)
    return false;
  g_accept_attr_ctx[device].store(current_context_id(), std::memory_order_release);
  return true;
}

}  // namespace
}  // namespace dspark

extern "C" {

int dspark_fill_uniforms(float* uniforms, int64_t n, uint64_t seed, uint64_t offset, cudaStream_t stream) {
  if (n < 0 || (n > 0 && !uniforms)) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  const int64_t blocks = (n + 3) / 4;
  const int64_t grid = (blocks + 255) / 256;
  dspark::fill_uniforms_kernel<<<static_cast<int>(grid < 152 * 32 ? grid : 152 * 32), 256, 0, stream>>>(
      uniforms, n, seed, offset);
  return dspark::done();
}

int dspark_probabilistic_accept(const float* target_probs, const float* draft_probs, const int64_t* draft,
                                const int32_t* proposal_len, const float* uniforms, int64_t* accepted,
                                int32_t* accept_len, int32_t batch, int32_t draft_stride, int32_t P, int32_t vocab,
                                cudaStream_t stream) {
  if (batch < 0 || P < 0 || vocab < 1 || (P > 0 && draft_stride < P)) return DSPARK_ERR_INVALID_ARG;
  if (batch == 0) return DSPARK_OK;
  if (!target_probs || !uniforms || !accepted || !accept_len || !proposal_len ||
      (P > 0 && (!draft_probs || !draft)))
    return DSPARK_ERR_INVALID_ARG;
  if (!dspark::accept_attr_ready()) return DSPARK_ERR_CUDA;
  dspark::prob_accept_kernel<<<batch, dspark::kAcceptThreads, dspark::kStageBytes, stream>>>(
      target_probs, draft_probs, draft, proposal_len, uniforms, accepted, accept_len, draft_stride, P, vocab);
  return dspark::done();
}

}  // extern "C"
