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

#include "dspark_markov.h"

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
// negatives weigh 0), truncated.  p * 2^40 is exact in FP32.
__device__ __forceinline__ uint64_t weight(float p) {
  if (!(p > 0.0f)) return 0ull;
  if (p >= 1.0f) return 1ull << 40;
  return __float2ull_rz(p * 0x1p40f);
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

constexpr int kAcceptThreads = 256;
constexpr int kAcceptWarps = kAcceptThreads / 32;

// The weight of id v of the row being sampled: the residual max(0, RN(t - q))
// when q is given, else the target probability.
__device__ __forceinline__ uint64_t row_weight(const float* t, const float* q, int64_t v) {
  return q ? weight(__fsub_rn(t[v], q[v])) : weight(t[v]);
}

// Inverse-CDF sample of one row by the whole CTA: warp w sums the weights of
// its contiguous segment (lanes strided, loads coalesced), thread 0 finds the
// segment holding the threshold, and that warp rescans it 32 ids at a time
// with a warp prefix sum.  Returns -1 (in every thread) when the row weighs 0.
__device__ int64_t sample_row(const float* t, const float* q, int64_t vocab, float u, uint64_t* s_seg,
                              int64_t* s_pick) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t seg = (vocab + kAcceptWarps - 1) / kAcceptWarps;
  const int64_t b0 = warp * seg, b1 = b0 + seg < vocab ? b0 + seg : vocab;
  uint64_t part = 0;
  for (int64_t v = b0 + lane; v < b1; v += 32) part += row_weight(t, q, v);
  part = warp_sum_u64(part);
  if (lane == 0) s_seg[warp] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t total = 0;
    for (int w = 0; w < kAcceptWarps; ++w) total += s_seg[w];
    int64_t pick = -1;
    if (total > 0) {
      const uint64_t T = threshold(u, total);
      uint64_t before = 0;
      int w = 0;
      while (before + s_seg[w] <= T) before += s_seg[w++];  // T < total: stops at a segment
      s_seg[kAcceptWarps] = T - before;                   // threshold within segment w
      pick = -2 - w;                                      // segment to rescan
    }
    *s_pick = pick;
  }
  __syncthreads();
  const int64_t code = *s_pick;
  if (code == -1) return -1;
  const int target_warp = static_cast<int>(-2 - code);
  if (warp == target_warp) {
    const uint64_t Tw = s_seg[kAcceptWarps];
    uint64_t run = 0;
    for (int64_t base = b0; base < b1; base += 32) {
      const int64_t v = base + lane;
      const uint64_t x = v < b1 ? row_weight(t, q, v) : 0ull;
      uint64_t incl = x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, run + incl > Tw);
      if (hit) {
        if (lane == 0) *s_pick = base + __ffs(hit) - 1;
        break;
      }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  __syncthreads();
  const int64_t pick = *s_pick;
  __syncthreads();  // s_pick and s_seg are reused by the next call
  return pick;
}

// One CTA per batch row: the accept chain on thread 0, then one inverse-CDF
// sample (the residual after a rejection, else the bonus) by the whole CTA.
__global__ void __launch_bounds__(kAcceptThreads)
    prob_accept_kernel(const float* __restrict__ target, const float* __restrict__ draft_probs,
                       const int64_t* __restrict__ draft, const int32_t* __restrict__ proposal_len,
                       const float* __restrict__ uniforms, int64_t* __restrict__ accepted,
                       int32_t* __restrict__ accept_len, int32_t draft_stride, int32_t P, int64_t vocab) {
  __shared__ uint64_t s_seg[kAcceptWarps + 1];
  __shared__ int64_t s_pick;
  __shared__ int s_j, s_pl;
  const int b = blockIdx.x;
  const float* tb = target + static_cast<int64_t>(b) * (P + 1) * vocab;
  const float* qb = draft_probs + static_cast<int64_t>(b) * P * vocab;
  const float* ub = uniforms + static_cast<int64_t>(b) * (2 * P + 1);
  int64_t* acc = accepted + static_cast<int64_t>(b) * (P + 1);
  if (threadIdx.x == 0) {
    int pl = proposal_len[b];
    pl = pl < 0 ? 0 : (pl > P ? P : pl);
    int j = 0;
    while (j < pl) {
      const int64_t d = draft[static_cast<int64_t>(b) * draft_stride + j];
      if (d < 0 || d >= vocab) break;
      const float t = tb[static_cast<int64_t>(j) * vocab + d];
      const float q = qb[static_cast<int64_t>(j) * vocab + d];
      if (!(__fmul_rn(ub[j], q) < t)) break;
      acc[j] = d;
      ++j;
    }
    s_j = j;
    s_pl = pl;
  }
  __syncthreads();
  const int j = s_j, pl = s_pl;
  const float* trow = tb + static_cast<int64_t>(j) * vocab;
  int64_t pick = -1;
  if (j < pl) pick = sample_row(trow, qb + static_cast<int64_t>(j) * vocab, vocab, ub[P + j], s_seg, &s_pick);
  if (pick < 0) pick = sample_row(trow, nullptr, vocab, j < pl ? ub[P + j] : ub[2 * P], s_seg, &s_pick);
  if (threadIdx.x == 0) {
    acc[j] = pick < 0 ? 0 : pick;
    for (int i = j + 1; i <= P; ++i) acc[i] = -1;
    accept_len[b] = j + 1;
  }
}

int done() { return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

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
  dspark::prob_accept_kernel<<<batch, dspark::kAcceptThreads, 0, stream>>>(
      target_probs, draft_probs, draft, proposal_len, uniforms, accepted, accept_len, draft_stride, P, vocab);
  return dspark::done();
}

}  // extern "C"
