// confidence.cu -- DSpark confidence-scored proposal lengths ([P1] "Dspark
// Kernels": dsparkComputeConfidenceScores, dsparkComputeConfidenceAnd-
// ProposalLengths, dsparkComputeConfidenceAndSPSProposalLengths) behind the C
// ABI of include/dspark_markov.h.
//
// The confidence that draft position j of request b is accepted is a logistic
// head over the feature that produced the draft: the draft hidden state of
// (b, j), followed (with the Markov term) by the Markov embedding w1[prev] of
// the token before position j (the request's first previous token for j = 0,
// draft j - 1 after it; the id clamped to the last w1 row as in the loop):
//   z = (weight . feature) + bias   (FP32 accumulation, one FP32 bias add),
//   score = sigmoid(z) = 1 / (1 + E) for z >= 0, E / (1 + E) below,
//           E = exp(-|z|) by the library's own exp.
// Threshold scheduling proposes while the running product of scores stays at
// or above the threshold; SPS scheduling picks the length whose expected
// output (1 + the sum of the running products) per verify cost is largest,
// stopping where the running product falls below the survival floor.  Both
// clamp to [min, max] and to P.
//
// One CTA per request.  The work is a read of batch * P * (H + rank) BF16
// values, HBM-bound, so the CTA's whole input goes out in one round trip:
// the staged kernel bulk-copies the weight, the request's P hidden rows and
// (one thread per position, after loading its previous-token id) the P
// gathered w1 rows into shared memory on one mbarrier, and the dots run from
// shared memory.  Where the rows are not 16-byte aligned or do not fit, the
// register kernel loads them into registers directly.  In both, W warps
// share each position's dot in a fixed order (a fixed butterfly inside each
// warp, then a fixed sum over the W partials), so the logit does not depend
// on scheduling; thread 0 then runs the scheduler over the request's P
// scores in shared memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "dspark_markov.h"
#include "kernels.h"
#include "markov_math.cuh"
#include "ptx.cuh"

namespace dspark {
namespace {

constexpr int kConfMaxP = DSPARK_CONFIDENCE_MAX_P;
constexpr int kConfMaxWarps = 32;
constexpr int kStagedMaxBytes = 200 * 1024;     // shared memory of the staged kernel
constexpr uint32_t kCopyWaitLimit = 1u << 24;   // polls of the copies' mbarrier

struct ConfParams {
  const uint16_t* hidden;
  int64_t hidden_stride;
  int64_t hidden_offset;
  const uint16_t* w1;
  int64_t w1_rows;
  const uint16_t* weight;
  const float* bias;
  const int64_t* first_prev;
  const int64_t* draft;
  int64_t draft_s0;
  float* scores;
  float* logits;
  int32_t* lengths;
  const float* cost;
  float level;  // threshold or survival floor
  int H, rank, with_markov, P;
  int mode;     // 0 scores only, 1 threshold, 2 SPS
  int lo, hi;   // clamped length bounds
  int W;        // warps per position
  int slots;    // positions in flight per CTA pass
};

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// acc + x . w over eight BF16 pairs, in element order (each product is exact
// in FP32; each fma rounds once).
__device__ __forceinline__ float dot8(uint4 x, uint4 w, float acc) {
  acc = __fmaf_rn(bf_lo(x.x), bf_lo(w.x), acc);
  acc = __fmaf_rn(bf_hi(x.x), bf_hi(w.x), acc);
  acc = __fmaf_rn(bf_lo(x.y), bf_lo(w.y), acc);
  acc = __fmaf_rn(bf_hi(x.y), bf_hi(w.y), acc);
  acc = __fmaf_rn(bf_lo(x.z), bf_lo(w.z), acc);
  acc = __fmaf_rn(bf_hi(x.z), bf_hi(w.z), acc);
  acc = __fmaf_rn(bf_lo(x.w), bf_lo(w.w), acc);
  acc = __fmaf_rn(bf_hi(x.w), bf_hi(w.w), acc);
  return acc;
}

// This lane's share of weight . feature for one position: hidden row h
// (H values), then the Markov row of id `prev` (rank values; p.rank is 0
// without the Markov term).  The row's address is formed where a chunk
// first needs it, so the hidden loads before it do not wait for the id.
// Vector form: 8-value chunks c = part * 32 + lane + t * 32 W.
template <bool kVec>
__device__ __forceinline__ float dot_part(const ConfParams& p, const uint16_t* h, int64_t prev, int part,
                                          int lane) {
  const int n = p.H + p.rank;
  const uint64_t last = static_cast<uint64_t>(p.w1_rows - 1);
  const uint64_t row = static_cast<uint64_t>(prev) < last ? static_cast<uint64_t>(prev) : last;
  const uint16_t* m = p.w1 + row * static_cast<uint64_t>(p.rank);
  const int stride = 32 * p.W;
  float acc = 0.0f;
  if (kVec) {
    const int nh = p.H >> 3, nc = n >> 3;
    for (int c0 = part * 32 + lane; c0 < nc; c0 += 4 * stride) {
      uint4 x[4], w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * stride;
        if (c < nc) {
          x[u] = c < nh ? ld_stream_v4(h + static_cast<int64_t>(c) * 8)
                        : __ldg(reinterpret_cast<const uint4*>(m + static_cast<int64_t>(c - nh) * 8));
          w[u] = __ldg(reinterpret_cast<const uint4*>(p.weight + static_cast<int64_t>(c) * 8));
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + u * stride < nc) acc = dot8(x[u], w[u], acc);
    }
  } else {
    for (int e = part * 32 + lane; e < n; e += stride) {
      const uint32_t x = e < p.H ? h[e] : m[e - p.H];
      acc = __fmaf_rn(__uint_as_float(x << 16), __uint_as_float(static_cast<uint32_t>(p.weight[e]) << 16), acc);
    }
  }
  return acc;
}

__device__ __forceinline__ float own_sigmoid(float z) {
  if (z != z) return z;
  const float E = own_exp_nonpos(-fabsf(z));
  const float d = __fadd_rn(1.0f, E);
  return z >= 0.0f ? __fdiv_rn(1.0f, d) : __fdiv_rn(E, d);
}

__device__ int threshold_length(const float* sc, int P, float thr, int lo, int hi) {
  float S = 1.0f;
  int L = 0;
  for (int j = 0; j < P; ++j) {
    S = __fmul_rn(S, sc[j]);
    if (!(S >= thr)) break;
    L = j + 1;
  }
  return L < lo ? lo : (L > hi ? hi : L);
}

__device__ int sps_length(const float* sc, float floor_, int lo, int hi, const float* cost) {
  float S = 1.0f, T = 1.0f, best_ratio = 0.0f;
  int best = lo;
  bool have = false;
  for (int L = 0; L <= hi; ++L) {
    if (L > 0) {
      S = __fmul_rn(S, sc[L - 1]);
      T = __fadd_rn(T, S);
      if (L > lo && !(S >= floor_)) break;
    }
    if (L < lo) continue;
    const float c = cost[L];
    if (!(c > 0.0f)) continue;
    const float ratio = __fdiv_rn(T, c);
    if (!have || ratio > best_ratio) {
      best = L;
      best_ratio = ratio;
      have = true;
    }
  }
  return best;
}

// The logit and score of position j from the CTA's W partial sums; records
// the score for the scheduler.
__device__ __forceinline__ void finish_position(const ConfParams& p, int b, int j, const float* partial, float bias,
                                                float* sc) {
  float s = partial[0];
  for (int q = 1; q < p.W; ++q) s = __fadd_rn(s, partial[q]);
  const float z = __fadd_rn(s, bias);
  const float score = own_sigmoid(z);
  const int64_t o = static_cast<int64_t>(b) * p.P + j;
  if (p.logits) p.logits[o] = z;
  p.scores[o] = score;
  sc[j] = score;
}

__device__ __forceinline__ void schedule(const ConfParams& p, int b, const float* sc) {
  if (p.mode != 0)
    p.lengths[b] = p.mode == 1 ? threshold_length(sc, p.P, p.level, p.lo, p.hi)
                               : sps_length(sc, p.level, p.lo, p.hi, p.cost);
}

__device__ __forceinline__ float warp_sum_lane0(float acc) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, off));
  return acc;  // lane 0's value is the one kept: its order is fixed
}

__device__ __forceinline__ uint64_t markov_row(const ConfParams& p, int b, int j) {
  const int64_t prev = j == 0 ? p.first_prev[b] : p.draft[static_cast<int64_t>(b) * p.draft_s0 + j - 1];
  const uint64_t last = static_cast<uint64_t>(p.w1_rows - 1);
  return static_cast<uint64_t>(prev) < last ? static_cast<uint64_t>(prev) : last;
}

// Staged: shared memory holds the weight [n], the hidden rows [P][H] and the
// Markov rows [P][rank] (n = H + rank; every piece a multiple of 16 bytes).
__global__ void __launch_bounds__(1024) confidence_staged_kernel(ConfParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bar;
  __shared__ float partial[kConfMaxWarps];
  __shared__ float sc[kConfMaxP];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, rank = p.rank, n = H + rank, P = p.P;
  uint16_t* s_w = reinterpret_cast<uint16_t*>(smem);
  uint16_t* s_h = s_w + n;
  uint16_t* s_m = s_h + static_cast<int64_t>(P) * H;
  // The ids the Markov copies depend on, and the bias, go out first, ahead
  // of the bulk of the request's bytes.
  const uint64_t row0 = rank > 0 && tid < P ? markov_row(p, b, tid) : 0;
  const float bias = *p.bias;
  if (tid == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar, static_cast<uint32_t>((P + 1) * n * 2));
  }
  __syncthreads();
  if (tid == 0) ptx::bulk_load(s_w, p.weight, n * 2, &bar);
  for (int j = tid; j < P; j += blockDim.x)
    if (H > 0)
      ptx::bulk_load(s_h + static_cast<int64_t>(j) * H,
                     p.hidden + p.hidden_offset + (static_cast<int64_t>(b) * P + j) * p.hidden_stride, H * 2, &bar);
  for (int j = tid; j < P; j += blockDim.x)
    if (rank > 0)
      ptx::bulk_load(s_m + static_cast<int64_t>(j) * rank, p.w1 + (j == tid ? row0 : markov_row(p, b, j)) * rank,
                     rank * 2, &bar);
  bool ok = ptx::mbar_wait(&bar, 0, kCopyWaitLimit);
  if (!__syncthreads_and(ok)) {
    // Never in correct operation: let the copies land (bounded) before the
    // CTA exits, then mark the request (NaN scores, length -1).
    if (tid == 0) ptx::mbar_wait(&bar, 0, kCopyWaitLimit);
    for (int j = tid; j < P; j += blockDim.x) p.scores[static_cast<int64_t>(b) * P + j] = __uint_as_float(0x7FC00000u);
    if (tid == 0 && p.mode != 0) p.lengths[b] = -1;
    return;
  }
  const int slot = warp / p.W, part = warp - slot * p.W;
  const int nh = H >> 3, nc = n >> 3, stride = 32 * p.W;
  for (int j0 = 0; j0 < P; j0 += p.slots) {
    const int j = j0 + slot;
    float acc = 0.0f;
    if (j < P) {
      const uint32_t h = ptx::smem_addr(s_h + static_cast<int64_t>(j) * H);
      const uint32_t m = ptx::smem_addr(s_m + static_cast<int64_t>(j) * rank);
      const uint32_t w = ptx::smem_addr(s_w);
      for (int c = part * 32 + lane; c < nc; c += stride) {
        const uint4 x = c < nh ? ptx::lds_v4(h + c * 16) : ptx::lds_v4(m + (c - nh) * 16);
        acc = dot8(x, ptx::lds_v4(w + c * 16), acc);
      }
    }
    acc = warp_sum_lane0(acc);
    if (lane == 0) partial[warp] = acc;
    __syncthreads();
    if (tid < p.slots && j0 + tid < P) finish_position(p, b, j0 + tid, partial + tid * p.W, bias, sc);
    __syncthreads();
  }
  if (tid == 0) schedule(p, b, sc);
}

// Registers: each lane loads its chunks of the position's feature itself.
template <bool kVec>
__global__ void __launch_bounds__(1024) confidence_kernel(ConfParams p) {
  __shared__ float partial[kConfMaxWarps];
  __shared__ float sc[kConfMaxP];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = warp / p.W, part = warp - slot * p.W;
  const float bias = p.P > 0 ? *p.bias : 0.0f;
  for (int j0 = 0; j0 < p.P; j0 += p.slots) {
    const int j = j0 + slot;
    float acc = 0.0f;
    if (j < p.P) {
      const uint16_t* h = p.hidden + p.hidden_offset + (static_cast<int64_t>(b) * p.P + j) * p.hidden_stride;
      const int64_t prev = !p.with_markov ? 0
                           : j == 0      ? p.first_prev[b]
                                         : p.draft[static_cast<int64_t>(b) * p.draft_s0 + j - 1];
      acc = dot_part<kVec>(p, h, prev, part, lane);
    }
    acc = warp_sum_lane0(acc);
    if (lane == 0) partial[warp] = acc;
    __syncthreads();
    const int t = threadIdx.x;
    if (t < p.slots && j0 + t < p.P) finish_position(p, b, j0 + t, partial + t * p.W, bias, sc);
    __syncthreads();
  }
  if (threadIdx.x == 0) schedule(p, b, sc);
}

constexpr int kAttrMaxDevices = 64;
std::atomic<unsigned long long> g_staged_attr_ctx[kAttrMaxDevices];

// The staged kernel's shared-memory limit, set once per device context.
bool staged_attr_ready() {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kAttrMaxDevices) {
    (void)cudaGetLastError();
    return false;
  }
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && g_staged_attr_ctx[device].load(std::memory_order_acquire) == ctx) return true;
  if (cudaFuncSetAttribute(confidence_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kStagedMaxBytes) != cudaSuccess)
    return false;
  g_staged_attr_ctx[device].store(ctx, std::memory_order_release);
  return true;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int launch_confidence(const dspark_confidence_args* a, int mode, float level, int32_t min_len, int32_t max_len,
                      const float* cost, int32_t* lengths, cudaStream_t stream) {
  if (!a) return DSPARK_ERR_INVALID_ARG;
  const int32_t B = a->batch, P = a->proposal_len, H = a->hidden_size;
  const int32_t rank = a->with_markov ? a->rank : 0;
  if (B < 0 || P < 0 || P > kConfMaxP || H < 0 || a->hidden_offset < 0) return DSPARK_ERR_INVALID_ARG;
  const int64_t hs = a->hidden_stride == 0 ? H : a->hidden_stride;
  if (hs < H) return DSPARK_ERR_INVALID_ARG;
  if (a->with_markov && (a->rank < 1 || a->w1_rows < 1 || (P > 1 && a->draft_s0 < P)))
    return DSPARK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(H) + rank > 0x7FFFFFF0) return DSPARK_ERR_INVALID_ARG;
  if (B == 0) return DSPARK_OK;
  if (mode != 0 && (!lengths || (mode == 2 && !cost))) return DSPARK_ERR_INVALID_ARG;
  if (a->with_markov && ((P > 0 && (!a->w1 || !a->first_prev)) || (P > 1 && !a->draft)))
    return DSPARK_ERR_INVALID_ARG;
  if (P > 0 && (!a->bias || !a->scores || (H > 0 && !a->hidden) || (H + rank > 0 && !a->weight)))
    return DSPARK_ERR_INVALID_ARG;
  if (mode == 0 && P == 0) return DSPARK_OK;

  ConfParams p{};
  p.hidden = static_cast<const uint16_t*>(a->hidden);
  p.hidden_stride = hs;
  p.hidden_offset = a->hidden_offset;
  p.w1 = static_cast<const uint16_t*>(a->w1);
  p.w1_rows = a->w1_rows;
  p.weight = static_cast<const uint16_t*>(a->weight);
  p.bias = a->bias;
  p.first_prev = a->first_prev;
  p.draft = a->draft;
  p.draft_s0 = a->draft_s0;
  p.scores = a->scores;
  p.logits = a->logits;
  p.lengths = lengths;
  p.cost = cost;
  p.level = level;
  p.H = H;
  p.rank = rank;
  p.with_markov = a->with_markov ? 1 : 0;
  p.P = P;
  p.mode = mode;
  int32_t hi = max_len < P ? max_len : P;
  if (hi < 0) hi = 0;
  int32_t lo = min_len < 0 ? 0 : min_len;
  if (lo > hi) lo = hi;
  p.lo = lo;
  p.hi = hi;

  // 16-byte loads where every feature row and the weight start on 16 bytes.
  const bool vec = (H % 8 == 0) && (rank % 8 == 0) && (hs % 8 == 0) && (a->hidden_offset % 8 == 0) &&
                   (H == 0 || aligned16(a->hidden)) && (rank == 0 || aligned16(a->w1)) &&
                   (H + rank == 0 || aligned16(a->weight));
  const int chunks = (H + rank + 7) / 8;
  const int Pe = P > 0 ? P : 1;
  const int64_t staged_bytes = static_cast<int64_t>(Pe + 1) * (H + rank) * 2;
  const bool staged = vec && P > 0 && H + rank > 0 && staged_bytes <= kStagedMaxBytes;
  // W warps per position: about four 16-byte chunks a lane for the register
  // kernel (all of them in flight at once); at most four warps for the staged
  // kernel, whose dots read shared memory; at most 32 warps per CTA.
  int W = staged ? (chunks + 255) / 256 : (chunks + 127) / 128;
  if (staged && W > 4) W = 4;
  const int wmax = kConfMaxWarps / (Pe < kConfMaxWarps ? Pe : kConfMaxWarps);
  if (W > wmax) W = wmax;
  if (W < 1) W = 1;
  p.W = W;
  p.slots = (Pe < kConfMaxWarps / W ? Pe : kConfMaxWarps / W);
  const int threads = 32 * W * p.slots;
  if (staged) {
    if (!staged_attr_ready()) return DSPARK_ERR_CUDA;
    confidence_staged_kernel<<<B, threads, static_cast<size_t>(staged_bytes), stream>>>(p);
  } else if (vec) {
    confidence_kernel<true><<<B, threads, 0, stream>>>(p);
  } else {
    confidence_kernel<false><<<B, threads, 0, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace
}  // namespace dspark

extern "C" {

int dspark_confidence_scores(const dspark_confidence_args* args, cudaStream_t stream) {
  return dspark::launch_confidence(args, 0, 0.0f, 0, 0, nullptr, nullptr, stream);
}

int dspark_confidence_and_proposal_lengths(const dspark_confidence_args* args, float threshold,
                                           int32_t min_proposal_len, int32_t max_proposal_len,
                                           int32_t* proposal_lengths, cudaStream_t stream) {
  return dspark::launch_confidence(args, 1, threshold, min_proposal_len, max_proposal_len, nullptr,
                                   proposal_lengths, stream);
}

int dspark_confidence_and_sps_proposal_lengths(const dspark_confidence_args* args, float survival_floor,
                                               int32_t min_proposal_len, int32_t max_proposal_len,
                                               const float* verify_cost, int32_t* proposal_lengths,
                                               cudaStream_t stream) {
  return dspark::launch_confidence(args, 2, survival_floor, min_proposal_len, max_proposal_len, verify_cost,
                                   proposal_lengths, stream);
}

}  // extern "C"
