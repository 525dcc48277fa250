// sharded.cu -- the vocabulary-sharded form of the Markov loop ([P3]
// "muse_spark cutedsl draft markov": module docstring, _finish, markov_pick,
// cache_fill).  Each rank runs the step over its vocabulary shard (the
// tensor-core step with a vocabulary offset, dspark_markov_shard_step in
// api.cu) and writes one 16-byte packet per row; the caller all-gathers the
// packets into [tp, rows, 4] on every rank; the pick kernel reduces them
// under the loop's total order and feeds the next step; after the loop the
// gathered rank-local caches are placed into the request cache.
#include <cuda_runtime.h>

#include "dspark_markov.h"
#include "kernels.h"

namespace dspark {
namespace {

// One warp per row: lane k < tp takes rank k's packet (value bits, global
// id); a butterfly maximum of the packed (orderable value, ~id) words is the
// total-order winner (first NaN, else the largest value, ties to the lower
// id) -- the unsharded argmax, the ranks holding consecutive id ranges.
// Writes tokens[r * tokens_s0 + step] and the packed winner into the slot
// the next step reads its previous token from.
__global__ void pick_kernel(const int32_t* __restrict__ packets, int tp, int rows, int64_t* __restrict__ tokens,
                            int64_t tokens_s0, int step, unsigned long long* __restrict__ slot_next) {
  const int r = blockIdx.x;
  const int lane = threadIdx.x;
  unsigned long long key = 0ull;
  if (lane < tp) {
    const int4 pk = *reinterpret_cast<const int4*>(packets + (static_cast<int64_t>(lane) * rows + r) * 4);
    key = pack_key(__int_as_float(pk.x), static_cast<uint32_t>(pk.y));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, key, off);
    key = o > key ? o : key;
  }
  if (lane == 0) {
    tokens[static_cast<int64_t>(r) * tokens_s0 + step] = slot_token(key);
    slot_next[r] = key;
  }
}

// Grid (rows * steps, vocabulary blocks of 1024): the entries of (row r,
// step i) whose request is valid go from the gathered rank-local caches
// src[k * src_s0 + (r * steps + i) * shard + local] to cache[req, i, v],
// v = k * shard + local < vocab; 16-byte copies where everything is aligned.
constexpr int kFillBlock = 1024;
constexpr int kFillThreads = 128;

template <bool kVec>
__global__ void cache_fill_kernel(const uint16_t* __restrict__ src, int64_t src_s0, uint16_t* __restrict__ cache,
                                  int64_t cache_s0, int64_t cache_s1, const int64_t* __restrict__ req_idx,
                                  int64_t req_s0, int64_t num_req, int steps, int64_t shard, int tp, int64_t vocab) {
  const int rs = blockIdx.x;
  const int r = rs / steps, i = rs - (rs / steps) * steps;
  const int64_t req = req_idx ? req_idx[static_cast<int64_t>(r) * req_s0 + i] : r;
  if (req < 0 || req >= num_req) return;
  uint16_t* dst = cache + req * cache_s0 + static_cast<int64_t>(i) * cache_s1;
  const int64_t row = static_cast<int64_t>(rs) * shard;
  const int64_t v0 = static_cast<int64_t>(blockIdx.y) * kFillBlock;
  if constexpr (kVec) {  // 8 entries a thread, all in one rank's shard (shard % 8 == 0)
    const int64_t v = v0 + threadIdx.x * 8;
    if (v >= vocab) return;
    const int64_t k = v / shard, local = v - k * shard;
    *reinterpret_cast<uint4*>(dst + v) = *reinterpret_cast<const uint4*>(src + k * src_s0 + row + local);
  } else {
    for (int64_t v = v0 + threadIdx.x; v < v0 + kFillBlock && v < vocab; v += kFillThreads) {
      const int64_t k = v / shard, local = v - k * shard;
      if (k < tp) dst[v] = src[k * src_s0 + row + local];
    }
  }
}

}  // namespace

cudaError_t launch_pick(const int32_t* packets, int tp, int rows, int64_t* tokens, int64_t tokens_s0, int step,
                        unsigned long long* slot_next, cudaStream_t stream) {
  pick_kernel<<<rows, 32, 0, stream>>>(packets, tp, rows, tokens, tokens_s0, step, slot_next);
  return cudaGetLastError();
}

}  // namespace dspark

extern "C" {

int dspark_cache_fill(const void* src, int64_t src_s0, void* cache, int64_t cache_s0, int64_t cache_s1,
                      const int64_t* req_idx, int64_t req_s0, int64_t num_req, int32_t rows, int32_t steps,
                      int32_t shard, int32_t tp, int32_t vocab, cudaStream_t stream) {
  if (rows < 0 || steps < 0 || shard < 1 || tp < 1 || vocab < 0 || num_req < 0) return DSPARK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(shard) * tp < vocab) return DSPARK_ERR_INVALID_ARG;  // the shards must cover the vocabulary
  if (rows == 0 || steps == 0 || vocab == 0) return DSPARK_OK;
  if (!src || !cache || src_s0 < static_cast<int64_t>(rows) * steps * shard || cache_s0 < 0 || cache_s1 < 0 ||
      (req_idx && req_s0 < steps))
    return DSPARK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(cache)) & 1u) return DSPARK_ERR_MISALIGNED;
  const int64_t rs = static_cast<int64_t>(rows) * steps;
  const int64_t blocks = (vocab + dspark::kFillBlock - 1) / dspark::kFillBlock;
  if (rs > 0x7FFFFFFF || blocks > 65535) return DSPARK_ERR_INVALID_ARG;
  const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(cache)) & 15u) == 0 &&
                   shard % 8 == 0 && vocab % 8 == 0 && src_s0 % 8 == 0 && cache_s0 % 8 == 0 && cache_s1 % 8 == 0;
  const dim3 grid(static_cast<unsigned>(rs), static_cast<unsigned>(blocks));
  if (vec)
    dspark::cache_fill_kernel<true><<<grid, dspark::kFillBlock / 8, 0, stream>>>(
        static_cast<const uint16_t*>(src), src_s0, static_cast<uint16_t*>(cache), cache_s0, cache_s1, req_idx,
        req_s0, num_req, steps, shard, tp, vocab);
  else
    dspark::cache_fill_kernel<false><<<grid, dspark::kFillThreads, 0, stream>>>(
        static_cast<const uint16_t*>(src), src_s0, static_cast<uint16_t*>(cache), cache_s0, cache_s1, req_idx,
        req_s0, num_req, steps, shard, tp, vocab);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // extern "C"
