// verify.cu -- the verify side of a DSpark round ([P1] dsparkBuildVerifyTokens,
// dsparkGreedyAccept).
//
// Greedy accept is an HBM scan: every (b, j) row of the verify logits that
// the acceptance can reach (j <= min(proposal_len[b], P)) is split into
// 16384-entry chunks, one 256-thread CTA each.  A thread takes 64 entries
// (eight 16-byte loads, all issued before any is used) and reduces them with
// the packed NaN-propagating BF16 maximum; the CTA reduces the threads'
// maxima as orderable keys, and only the threads holding the maximum look
// for its first id, so the total order (first NaN, else the lowest id of the
// maximum) costs about half an instruction per entry.  The CTA folds its
// packed (orderable value, ~id) key into the row's slot with one 64-bit
// atomicMax and is done: no fence, no arrival.  A third kernel, one thread
// per batch row, walks the slots and writes the accepted tokens and lengths.
// A first small kernel clears the slots, so the caller's scratch needs no
// initialisation.  The three launches are chained with programmatic
// dependent launch: each starts while the previous one runs and waits for it
// only before it touches the slots.
#include <cuda_runtime.h>

#include <mutex>

#include "dspark_markov.h"
#include "kernels.h"
#include "markov_math.cuh"
#include "step_common.cuh"

// Scratch of dspark_greedy_accept_noalloc: one argmax slot per verify row
// and the alignment pad, in a fixed array of the module, so that the entry
// point needs no allocation.  Every device that loads the library keeps it
// (64 KB + 16 bytes) until the process exits.  Host code must not pass
// `g_accept_noalloc_scratch` itself to a kernel: on the host the name denotes
// a stand-in, not the device address; that comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned long long
    g_accept_noalloc_scratch[DSPARK_NOALLOC_MAX_VERIFY_ROWS + 2];

namespace dspark {
namespace {

constexpr int kAcceptThreads = 256;
constexpr int kAcceptLoads = 8;                                  // 16-byte loads per thread
constexpr int kAcceptChunk = kAcceptThreads * kAcceptLoads * 8;  // BF16 entries per CTA (32 KB)

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

__global__ void accept_clear_kernel(unsigned long long* slots, int64_t n) {
  pdl_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    slots[i] = 0ull;
}

__device__ __forceinline__ int clamp_plen(int pl, int P) { return pl < 0 ? 0 : (pl > P ? P : pl); }

// The NaN-propagating maximum of two BF16 pairs (a NaN in either lane gives
// NaN in that lane).
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Orderable key of a BF16 value (NaN highest, +0 == -0): the FP32 key of the
// value it widens to.
__device__ __forceinline__ uint32_t bf16_key(uint32_t bits16) { return orderable(__uint_as_float(bits16 << 16)); }

// grid (batch * (P + 1), chunks): blockIdx.y is the chunk of verify row
// blockIdx.x = b * (P + 1) + j.
__global__ void __launch_bounds__(kAcceptThreads)
accept_scan_kernel(const uint16_t* __restrict__ logits, const int32_t* __restrict__ proposal_len,
                   unsigned long long* __restrict__ slots, int P, int vocab) {
  __shared__ uint32_t warp_key[kAcceptThreads / 32];
  __shared__ uint32_t warp_id[kAcceptThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int b = static_cast<int>(row / (P + 1));
  const int j = static_cast<int>(row - static_cast<int64_t>(b) * (P + 1));
  pdl_launch_dependents();
  if (j > clamp_plen(proposal_len[b], P)) return;  // not reachable: not scanned
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kAcceptChunk;
  const uint16_t* src = logits + row * vocab;

  // (1) this thread's 64 entries: ids c0 + (it * 256 + tid) * 8 + q
  uint4 w[kAcceptLoads];
#pragma unroll
  for (int it = 0; it < kAcceptLoads; ++it) {
    const int64_t e0 = c0 + (static_cast<int64_t>(it) * kAcceptThreads + tid) * 8;
    w[it] = e0 < vocab ? ldg_nc_v4(src + e0) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  }
  uint32_t m2 = 0xFF80FF80u;  // -inf, -inf (past the row's end too: never above a real entry)
#pragma unroll
  for (int it = 0; it < kAcceptLoads; ++it)
    m2 = max_nan_bf16x2(max_nan_bf16x2(m2, w[it].x), max_nan_bf16x2(w[it].y, max_nan_bf16x2(w[it].z, w[it].w)));
  const uint32_t mine = max(bf16_key(m2 & 0xFFFFu), bf16_key(m2 >> 16));

  // (2) the CTA's largest key
  uint32_t k = __reduce_max_sync(0xFFFFFFFFu, mine);
  if (lane == 0) warp_key[warp] = k;
  __syncthreads();
  k = warp_key[0];
#pragma unroll
  for (int i = 1; i < kAcceptThreads / 32; ++i) k = max(k, warp_key[i]);

  // (3) its first id: only threads holding the maximum look (in id order)
  uint32_t id = 0xFFFFFFFFu;
  if (mine == k) {
    for (int it = 0; it < kAcceptLoads && id == 0xFFFFFFFFu; ++it) {
      const uint32_t words[4] = {w[it].x, w[it].y, w[it].z, w[it].w};
      const uint32_t e0 = static_cast<uint32_t>(c0 + (static_cast<int64_t>(it) * kAcceptThreads + tid) * 8);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t bits = q & 1 ? words[q >> 1] >> 16 : words[q >> 1] & 0xFFFFu;
        if (id == 0xFFFFFFFFu && bf16_key(bits) == k && e0 + q < static_cast<uint32_t>(vocab)) id = e0 + q;
      }
    }
  }
  id = __reduce_min_sync(0xFFFFFFFFu, id);
  if (lane == 0) warp_id[warp] = id;
  __syncthreads();
  if (tid == 0) {
    uint32_t first = warp_id[0];
    for (int i = 1; i < kAcceptThreads / 32; ++i) first = min(first, warp_id[i]);
    pdl_wait();  // the slots were cleared by the previous launch
    atomicMax(slots + row, (static_cast<unsigned long long>(k) << 32) | static_cast<uint32_t>(~first));
  }
}

// One thread per batch row: accept while the draft equals the argmax, then
// the bonus token.
__global__ void accept_walk_kernel(const int64_t* __restrict__ draft, const int32_t* __restrict__ proposal_len,
                                   int64_t* __restrict__ accepted, int32_t* __restrict__ accept_len,
                                   const unsigned long long* __restrict__ slots, int batch, int draft_stride, int P) {
  pdl_wait();  // every scan CTA has folded its key
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int pl = clamp_plen(proposal_len[b], P);
  const int64_t r0 = static_cast<int64_t>(b) * (P + 1);
  int n = 0;
  int64_t a = slot_token(slots[r0]);
  while (n < pl && draft[static_cast<int64_t>(b) * draft_stride + n] == a) {
    accepted[r0 + n] = a;
    ++n;
    a = slot_token(slots[r0 + n]);
  }
  accepted[r0 + n] = a;
  for (int q = n + 1; q <= P; ++q) accepted[r0 + q] = -1;
  accept_len[b] = n + 1;
}

// A launch with programmatic stream serialisation: it may start while the
// previous kernel on the stream runs (its own griddepcontrol.wait orders it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kNoAllocMaxDevices = 64;

// Per device: the array's address and the context it was looked up in.  A
// device reset (or another context made current) gives a new context id, and
// the next call looks the address up again.
struct NoAllocEntry {
  void* addr = nullptr;
  unsigned long long ctx = 0;
};
NoAllocEntry g_noalloc[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// The device address of the array in the current context of `device`,
// looked up once per context; nullptr if the lookup failed.
void* noalloc_scratch_address(int device) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocEntry& e = g_noalloc[device];
  const unsigned long long ctx = current_context_id();
  if (e.addr && ctx != 0 && e.ctx == ctx) return e.addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, ::g_accept_noalloc_scratch) != cudaSuccess || !p) {
    (void)cudaGetLastError();
    e.addr = nullptr;
    return nullptr;
  }
  e.addr = p;
  e.ctx = current_context_id();  // the lookup makes the primary context current if none was
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
  const int chunks = (vocab + dspark::kAcceptChunk - 1) / dspark::kAcceptChunk;  // <= 65535: vocab < 2^31
  unsigned long long* slots = static_cast<unsigned long long*>(scratch);
  const int cgrid = static_cast<int>((rows + 255) / 256 < 1024 ? (rows + 255) / 256 : 1024);
  dspark::accept_clear_kernel<<<cgrid, 256, 0, stream>>>(slots, rows);
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  if (dspark::launch_pdl(dspark::accept_scan_kernel, dim3(static_cast<unsigned>(rows), static_cast<unsigned>(chunks)),
                         dim3(dspark::kAcceptThreads), stream, static_cast<const uint16_t*>(logits), proposal_len,
                         slots, P, vocab) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (dspark::launch_pdl(dspark::accept_walk_kernel, dim3((batch + 127) / 128), dim3(128), stream, draft,
                         proposal_len, accepted, accept_len, static_cast<const unsigned long long*>(slots), batch,
                         draft_stride, P) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return DSPARK_OK;
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
  // The slots are cleared by the first kernel of every call
  // (dspark_greedy_accept's own sequence), so whatever the previous call left
  // in the array does not matter.
  return dspark_greedy_accept(logits, draft, proposal_len, accepted, accept_len, scratch,
                              sizeof(::g_accept_noalloc_scratch), batch, draft_stride, P, vocab, stream);
}

}  // extern "C"
