// verify.cu -- the verify side of a DSpark round ([P1] dsparkBuildVerifyTokens,
// dsparkGreedyAccept).
//
// Greedy accept is an HBM scan: every (b, j) row of the verify logits that
// the acceptance can reach (j <= min(proposal_len[b], P)) is split into
// 8192-entry chunks; a 256-thread CTA reduces its chunk with 16-byte loads to
// one packed (orderable value, ~id) key and folds it into the row's slot with
// a 64-bit atomicMax.  The last CTA to arrive walks the slots and writes the
// accepted tokens and lengths.  A first small kernel clears the slots, so the
// caller's scratch needs no initialisation.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "dspark_markov.h"
#include "markov_math.cuh"
#include "step_common.cuh"

// Scratch of dspark_greedy_accept_noalloc: one argmax slot per verify row
// plus the arrival counter, in a fixed array of the module, so that the entry
// point needs no allocation.  Every device that loads the library keeps it
// (64 KB + 16 bytes) until the process exits.  Host code must not pass
// `g_accept_noalloc_scratch` itself to a kernel: on the host the name denotes
// a stand-in, not the device address; that comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned long long g_accept_noalloc_scratch[DSPARK_NOALLOC_MAX_VERIFY_ROWS + 2];

namespace dspark {
namespace {

constexpr int kAcceptThreads = 256;
constexpr int kAcceptChunk = 8192;  // BF16 entries per CTA (16 KB)

__global__ void build_verify_kernel(const int64_t* __restrict__ last, const int64_t* __restrict__ draft,
                                    int64_t* __restrict__ verify, int batch, int draft_stride, int P) {
  const int64_t n = static_cast<int64_t>(batch) * (P + 1);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = i / (P + 1);
    const int j = static_cast<int>(i - b * (P + 1));
    verify[i] = j == 0 ? last[b] : draft[b * draft_stride + j - 1];
  }
}

__global__ void accept_clear_kernel(unsigned long long* slots, unsigned int* counter, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    slots[i] = 0ull;
  if (blockIdx.x == 0 && threadIdx.x == 0) *counter = 0u;
}

__device__ __forceinline__ int clamp_plen(int pl, int P) { return pl < 0 ? 0 : (pl > P ? P : pl); }

__global__ void __launch_bounds__(kAcceptThreads)
accept_scan_kernel(const uint16_t* __restrict__ logits, const int64_t* __restrict__ draft,
                   const int32_t* __restrict__ proposal_len, int64_t* __restrict__ accepted,
                   int32_t* __restrict__ accept_len, unsigned long long* __restrict__ slots,
                   unsigned int* __restrict__ counter, int batch, int draft_stride, int P, int vocab) {
  __shared__ unsigned long long warp_best[kAcceptThreads / 32];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;  // b * (P + 1) + j
  const int b = static_cast<int>(row / (P + 1));
  const int j = static_cast<int>(row - static_cast<int64_t>(b) * (P + 1));
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kAcceptChunk;
  const bool needed = j <= clamp_plen(proposal_len[b], P) && c0 < vocab;
  if (needed) {
    const uint16_t* src = logits + row * vocab;
    float best = -INFINITY;
    uint32_t best_id = 0xFFFFFFFFu;
#pragma unroll
    for (int it = 0; it < kAcceptChunk / (8 * kAcceptThreads); ++it) {
      const int64_t e0 = c0 + (static_cast<int64_t>(it) * kAcceptThreads + tid) * 8;
      if (e0 < vocab) {
        const uint4 w = ldg_nc_v4(src + e0);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float x = __uint_as_float(q & 1 ? (words[q >> 1] & 0xFFFF0000u) : (words[q >> 1] << 16));
          const uint32_t id = static_cast<uint32_t>(e0 + q);
          // in-order combine: the later id wins only if strictly larger, or
          // if it is the first NaN
          const bool take = (x != x) ? (best == best) : (x > best);
          if (take || best_id == 0xFFFFFFFFu) {
            best = x;
            best_id = id;
          }
        }
      }
    }
    unsigned long long cand = best_id == 0xFFFFFFFFu ? 0ull : pack_key(best, best_id);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, cand, off);
      cand = o > cand ? o : cand;
    }
    if ((tid & 31) == 0) warp_best[tid >> 5] = cand;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kAcceptThreads / 32; ++w) m = warp_best[w] > m ? warp_best[w] : m;
      atomicMax(slots + row, m);
    }
  }
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(counter, 1u) == gridDim.x * gridDim.y - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int bb = tid; bb < batch; bb += kAcceptThreads) {
    const int pl = clamp_plen(proposal_len[bb], P);
    const int64_t r0 = static_cast<int64_t>(bb) * (P + 1);
    int n = 0;
    int64_t a = slot_token(atomicAdd(slots + r0, 0ull));
    while (n < pl && draft[static_cast<int64_t>(bb) * draft_stride + n] == a) {
      accepted[r0 + n] = a;
      ++n;
      a = slot_token(atomicAdd(slots + r0 + n, 0ull));
    }
    accepted[r0 + n] = a;
    for (int q = n + 1; q <= P; ++q) accepted[r0 + q] = -1;
    accept_len[bb] = n + 1;
  }
}

constexpr int kNoAllocMaxDevices = 64;

std::atomic<void*> g_noalloc_addr[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// The device address of the array on the current device, looked up once per
// device; nullptr if the lookup failed.
void* noalloc_scratch_address(int device) {
  void* p = g_noalloc_addr[device].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  p = g_noalloc_addr[device].load(std::memory_order_relaxed);
  if (p) return p;
  if (cudaGetSymbolAddress(&p, ::g_accept_noalloc_scratch) != cudaSuccess || !p) {
    (void)cudaGetLastError();
    return nullptr;
  }
  g_noalloc_addr[device].store(p, std::memory_order_release);
  return p;
}

}  // namespace
}  // namespace dspark

extern "C" {

int dspark_build_verify_tokens(const int64_t* last, const int64_t* draft, int64_t* verify, int32_t batch,
                               int32_t draft_stride, int32_t P, cudaStream_t stream) {
  if (batch < 0 || P < 0 || draft_stride < P) return DSPARK_ERR_INVALID_ARG;
  if (batch == 0) return DSPARK_OK;
  if (!last || !verify || (P > 0 && !draft)) return DSPARK_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(batch) * (P + 1);
  const int grid = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  dspark::build_verify_kernel<<<grid, 256, 0, stream>>>(last, draft, verify, batch, draft_stride, P);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

size_t dspark_greedy_accept_scratch_bytes(int32_t batch, int32_t P, int32_t vocab) {
  (void)vocab;
  if (batch < 0 || P < 0) return 0;
  return static_cast<size_t>(batch) * (P + 1) * sizeof(unsigned long long) + 16;
}

int dspark_greedy_accept(const void* logits, const int64_t* draft, const int32_t* proposal_len, int64_t* accepted,
                         int32_t* accept_len, void* scratch, size_t scratch_bytes, int32_t batch,
                         int32_t draft_stride, int32_t P, int32_t vocab, cudaStream_t stream) {
  if (batch < 0 || P < 0 || vocab < 1 || draft_stride < P) return DSPARK_ERR_INVALID_ARG;
  if (batch == 0) return DSPARK_OK;
  if (!logits || !proposal_len || !accepted || !accept_len || !scratch || (P > 0 && !draft))
    return DSPARK_ERR_INVALID_ARG;
  if (scratch_bytes < dspark_greedy_accept_scratch_bytes(batch, P, vocab)) return DSPARK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) || (reinterpret_cast<uintptr_t>(scratch) & 15u) || (vocab % 8))
    return DSPARK_ERR_MISALIGNED;
  const int64_t rows = static_cast<int64_t>(batch) * (P + 1);
  if (rows > 0x7FFFFFFF) return DSPARK_ERR_INVALID_ARG;
  const int chunks = (vocab + dspark::kAcceptChunk - 1) / dspark::kAcceptChunk;
  if (chunks > 65535) return DSPARK_ERR_INVALID_ARG;
  unsigned long long* slots = static_cast<unsigned long long*>(scratch);
  unsigned int* counter = reinterpret_cast<unsigned int*>(slots + rows);
  const int cgrid = static_cast<int>((rows + 255) / 256 < 1024 ? (rows + 255) / 256 : 1024);
  dspark::accept_clear_kernel<<<cgrid, 256, 0, stream>>>(slots, counter, rows);
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>(chunks));
  dspark::accept_scan_kernel<<<grid, dspark::kAcceptThreads, 0, stream>>>(
      static_cast<const uint16_t*>(logits), draft, proposal_len, accepted, accept_len, slots, counter, batch,
      draft_stride, P, vocab);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

int dspark_greedy_accept_noalloc(const void* logits, const int64_t* draft, const int32_t* proposal_len,
                                 int64_t* accepted, int32_t* accept_len, int32_t batch, int32_t draft_stride,
                                 int32_t P, int32_t vocab, cudaStream_t stream) {
  if (batch < 0 || P < 0 || vocab < 1 || draft_stride < P) return DSPARK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * (P + 1) > DSPARK_NOALLOC_MAX_VERIFY_ROWS) return DSPARK_ERR_TOO_MANY_ROWS;
  if (batch == 0) return DSPARK_OK;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= dspark::kNoAllocMaxDevices) {
    (void)cudaGetLastError();
    return DSPARK_ERR_CUDA;
  }
  void* scratch = dspark::noalloc_scratch_address(device);
  if (!scratch) return DSPARK_ERR_CUDA;
  // The slots and the counter are cleared by the first kernel of every call
  // (dspark_greedy_accept's own sequence), so whatever the previous call left
  // in the array does not matter.
  return dspark_greedy_accept(logits, draft, proposal_len, accepted, accept_len, scratch,
                              static_cast<size_t>(DSPARK_NOALLOC_MAX_VERIFY_ROWS + 2) * sizeof(unsigned long long),
                              batch, draft_stride, P, vocab, stream);
}

}  // extern "C"
