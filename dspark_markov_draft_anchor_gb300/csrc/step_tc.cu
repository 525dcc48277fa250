// step_tc.cu -- the fused Markov step on Blackwell tensor cores (sm_103a).
//
// One persistent CTA per SM owns a contiguous vocabulary range (whole
// 32-entry units, the ranges differing by at most one unit) and every request
// row.  Per 128-entry vocabulary tile:
//   * warps 0 and 2 (even and odd tiles) stream the tile's w2 rows with TMA
//     into rings of 16 KB stages (128 rows x 64 K, 128-byte swizzle), 4
//     stages per tile, and then its base logits, 16 rows x 128 entries per
//     4 KB chunk, into rings of their own;
//   * warps 1 and 3 issue tcgen05.mma (M = 128 vocab rows, N = rows padded
//     to 16, K = 256 in 16 steps of 16) for the even and the odd tiles into
//     TMEM accumulators;
//   * warps 4..19 (four quartets: tile parity x half of each 16-row chunk,
//     each warp reading its TMEM lane quarter) load the FP32 dots with
//     tcgen05.ld and run the per-element epilogue of [P3]
//     _StepKernel.kernel: bias rounded once to BF16, BF16 add, multiplier,
//     soft cap, cache store, Gumbel key ([P3] _logit, _gumbel).
// The row maxima live in shared memory as packed (orderable key, ~id) words,
// so any update order gives the total-order winner ([P3] module docstring);
// one global atomicMax per row and CTA publishes them ([P3] _finish).
//
// One launch runs one step or, as a cooperative launch whose CTAs are all
// resident, every step of the loop: after a step each CTA publishes its
// maxima and adds one to the step's arrival counter; once the counter
// reaches the grid size every CTA reads the step's tokens, gathers their w1
// rows and goes on.  The producers do not wait at that boundary: w2 (the same
// range every step) and the next step's base logits keep streaming into the
// rings.  CTA 0 writes each step's tokens during the next step's gather; the
// last step's are written by the CTA that arrives last.
//
// The Gumbel key of an element is only evaluated when it can win: the noise
// -L(h) falls as the hash h grows, so h's top byte bounds it above and below
// (tables computed on the host in double precision, with margins far above
// the FP32 rounding).  An element whose upper bound l/t + noise bound is below
// its row's threshold cannot be the argmax and is skipped; a threshold is
// never above the row's maximum key, so skipping never changes the result.
//
// The bias is the previous step's token's w1 row (clamped to the last row)
// times w2 in FP32, the summation order being the tensor core's; the pages
// allow any order ([P2] module docstring, [P4] module docstring).
//
// Programmatic dependent launch: the TMA producers read only inputs written
// before the loop (w2, base) and start before griddepcontrol.wait, and the
// epilogue warps read the per-row sampling constants (also inputs) before it;
// only the previous tokens wait.  All waits are bounded; a wait that gives up
// records DSPARK_ERR_DEVICE_TIMEOUT in the status word and raises the loop's
// abort word (which ends the other CTAs' waits), and the CTA leaves its
// loops, waits (bounded) for its copies in flight and frees its TMEM.
#include <atomic>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 640;
constexpr int kTileV = 128;
constexpr int kUnit = 32;              // vocabulary rows per partition unit / TMA box
constexpr int kKBlock = 64;            // K per w2 stage (one 128-byte swizzle row)
constexpr int kKBlocks = kRank / kKBlock;
constexpr int kW2StageBytes = kTileV * kKBlock * 2;  // 16 KB
constexpr int kChunkRows = 16;         // base rows per chunk (one epilogue pass)
constexpr int kChunkBytes = kChunkRows * kTileV * 2;  // 4 KB
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 16;          // four quartets: tile parity x half of each chunk's rows
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kHalfRows = kChunkRows / 2;  // rows of a chunk one epilogue warp handles
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint64_t kWaitNs = 10000000000ull;  // a role's wait gives up after 10 s
constexpr uint32_t kSuspendNs = 20000;        // suspend-time hint of one poll
// Polls of a step's arrival counter before the grid wait gives up (each an L2
// round trip: a few seconds at most, shorter than the roles' own waits).
constexpr uint32_t kGridWaitLimit = 1u << 22;
// Entries of a warp's key-evaluation queue: a push adds at most 32 to fewer
// than 32 left after a flush, so 64 never overflows.
constexpr int kQCap = 64;
constexpr int kNoiseT = kNoiseBuckets;

struct TcLayout {
  int n;         // MMA N: rows padded to 16
  int nacc;      // TMEM accumulators (tiles the MMA may run ahead)
  int stages;    // w2 ring stages (E4M3 w2: stages of 128 rows x 128 K bytes)
  int stages16;  // E4M3 w2 only: FP16 operand stages (128 rows x 64 K), two rings, one per MMA warp
  int nbase;     // base ring slots (two rings, one per tile parity)
  int tmem_cols;
  int res_tiles; // w2 tiles kept in tensor memory as the MMA's A operand after the first step
  int res_col;   // their first column (128 columns a tile)
  int smem;      // dynamic shared memory bytes (0: the layout does not fit)
  int emb_off, w2_off, f16_off, base_off, bar_off, row_off, queue_off, scale_off;
};

__host__ __device__ inline int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

// Per-row arrays in shared memory (structure of arrays, kMaxRows entries
// each) and their byte offsets inside the row region.
constexpr int kRowBest = 0;                            // u64 packed maxima
constexpr int kRowCoff = kRowBest + 8 * kMaxRows;      // i64 cache row addresses
constexpr int kRowPrefix = kRowCoff + 8 * kMaxRows;    // u32 Murmur3 prefixes
constexpr int kRowRinv = kRowPrefix + 4 * kMaxRows;    // f32 RN(1/t) (1 for greedy rows)
constexpr int kRowNs = kRowRinv + 4 * kMaxRows;        // f32 noise scale (0 greedy, 1 else)
constexpr int kRowTemp = kRowNs + 4 * kMaxRows;        // f32 temperature
constexpr int kRowThr = kRowTemp + 4 * kMaxRows;       // f32 pruning threshold
constexpr int kRowGmask = kRowThr + 4 * kMaxRows;      // u32 per 16-row chunk: store bits 0..15, live bits 16..31
constexpr int kRowGtab = kRowGmask + 4 * (kMaxRows / kChunkRows);  // f32 noise upper bound by clz
constexpr int kRowLtab = kRowGtab + 4 * kNoiseT;                   // f32 noise lower bound by bucket
constexpr int kRowKs = kRowLtab + 4 * kNoiseT;                      // f32 E4M3 w2: 2^-k of the row's B scaling
constexpr int kRowBytes = kRowKs + 4 * kMaxRows;

constexpr int kSmemBudget = 232448 - 64;  // 227 KB less the static shared variables
// E4M3 w2: the FP16 row scales of a CTA's vocabulary range are kept in shared
// memory when the range has at most this many rows (every step reads them)
constexpr int kScaleRowsMax = 2048;

// Shared memory of one CTA.  BF16 w2: the rest of the budget goes to the w2
// ring (at most 12 stages).  E4M3 w2: four FP16 operand stages (two per MMA
// warp) and the rest to the E4M3 ring (at most 8 stages); smem = 0 when the
// ring would have fewer than two stages (E4M3 w2 above 128 rows).
TcLayout tc_layout(int rows, bool fp8 = false) {
  TcLayout L;
  L.n = ((rows + 15) / 16) * 16;
  // even: each accumulator belongs to one tile parity
  L.nacc = 8 * L.n <= 512 ? 8 : (4 * L.n <= 512 ? 4 : 2);
  L.tmem_cols = pow2_at_least(L.nacc * L.n);
  // the columns the accumulators leave hold whole w2 tiles (128 rows x 256 K
  // of 16-bit values: 128 columns): the whole tensor memory is then allocated
  L.res_col = (L.nacc * L.n + 127) / 128 * 128;
  L.res_tiles = (512 - L.res_col) / 128;
  if (L.res_tiles > 0) L.tmem_cols = 512;
  // 4 KB chunks, half per parity's ring; more slots where a tile has several
  // chunks, or three per parity at 16 rows, where the w2 ring can spare them
  L.nbase = (L.n > kChunkRows && L.n < 128) ? 8 : (L.n == kChunkRows ? 6 : 4);
  const int bars_max = 8 * (2 * 12 + 4 + 2 * L.nbase + 2 * 8 + 3);
  const int fixed = L.n * kRank * 2 + L.nbase * kChunkBytes + bars_max + 16 + kRowBytes + kEpiWarps * kQCap * 8 +
                    (fp8 ? kScaleRowsMax * 2 : 0) + 1024 + 64;
  const int avail = (kSmemBudget - fixed) / kW2StageBytes;  // 16 KB stages that fit
  L.smem = 0;
  if (!fp8) {
    L.stages16 = 0;
    L.stages = avail > 12 ? 12 : avail;
    L.stages &= ~1;  // two w2 rings of stages / 2, one per MMA warp
    if (L.stages < 2) return L;
  } else {
    L.stages16 = 4;  // two per MMA warp: one is filled while the other's MMAs run
    L.stages = avail - L.stages16 > 8 ? 8 : avail - L.stages16;
    L.stages &= ~1;  // two E4M3 rings, one per tile parity
    if (L.stages < 2) return L;
  }
  int off = 0;
  L.emb_off = off;
  off += L.n * kRank * 2;
  L.w2_off = off;
  off += L.stages * kW2StageBytes;
  L.f16_off = off;
  off += L.stages16 * kW2StageBytes;
  L.base_off = off;
  off += L.nbase * kChunkBytes;
  L.bar_off = off;
  off += 8 * (2 * L.stages + L.stages16 + 2 * L.nbase + 2 * L.nacc + 3);
  off = (off + 15) & ~15;
  L.row_off = off;
  off += kRowBytes;
  off = (off + 15) & ~15;
  L.queue_off = off;
  off += kEpiWarps * kQCap * 8;
  L.scale_off = off;
  if (fp8) off += kScaleRowsMax * 2;
  L.smem = off + 1024;  // room to align the base to 1024 bytes
  return L;
}

struct TcParams {
  StepParams p;
  int32_t n;
  int32_t nacc;
  int32_t stages;
  int32_t stages16;
  int32_t nbase;
  int32_t tmem_cols;
  int32_t res_tiles;  // the CTA's last res_tiles tiles stay in tensor memory from the second step on
  int32_t res_col;
  int32_t emb_off, w2_off, f16_off, base_off, bar_off, row_off, queue_off, scale_off;
  int32_t num_units;  // ceil(V / 32)
  int32_t base_steps_mid;  // base tensor map dims are (vocab, step, row), else (vocab, row, step)
};

// A warp's queue of elements whose Gumbel key must be evaluated (their exact
// bound reaches the row's current maximum).  Evaluating them 32 at a time,
// one per lane, keeps rare survivors from costing the warp a full pass each.
// An entry is 8 bytes (the hash is formed again at evaluation), so vocabulary
// ids must stay below 2^24 (the host sends larger vocabularies to the other
// step kernel).
struct Cand {
  float l;
  uint32_t vr;  // row << 24 | vocabulary id
};
struct Shared;

struct WarpQueue {
  Cand* q;
  uint32_t head = 0, count = 0;  // warp-uniform

  __device__ __forceinline__ void push(bool take, int lane, uint32_t v, float l, int r) {
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, take);
    if (take) {
      const uint32_t pos = (head + count + __popc(m & ((1u << lane) - 1u))) & (kQCap - 1);
      q[pos] = Cand{l, (static_cast<uint32_t>(r) << 24) | v};
    }
    count += __popc(m);
  }
  __device__ __forceinline__ void flush(uint32_t min_count, const Shared& sh);
};

struct Shared {
  unsigned char* emb;
  unsigned char* w2;
  unsigned char* base;
  uint64_t* full_w2;
  uint64_t* empty_w2;
  uint64_t* full_base;
  uint64_t* empty_base;
  uint64_t* tmem_full;   // [nacc]
  uint64_t* tmem_empty;  // [nacc]
  uint64_t* emb_ready;
  uint64_t* spare;       // [2], one per MMA warp
  uint64_t* empty_f16;   // E4M3 w2: [stages16], FP16 operand stage free (its MMAs completed)
  unsigned char* f16;    // E4M3 w2: FP16 operand stages
  unsigned long long* best;
  int64_t* cache_off;  // per row: the address of its cache row (an int64)
  uint32_t* prefix;
  float* rinv;
  float* ns;
  float* temp;
  float* thr;       // per-row pruning threshold: never above the row's maximum key
  uint32_t* gmask;  // per 16-row chunk: rows that store (bits 0..15), rows that exist (16..31)
  float* gtab;      // the computed noise never exceeds gtab[noise_index(h)]
  float* ltab;      // the computed noise is never below ltab[noise_index(h)]
  float* kscale;    // E4M3 w2: per row, 2^-k undoing the FP16 embedding's power-of-two scaling
  Cand* queues;
  uint16_t* w2s;       // E4M3 w2: the FP16 scales of the CTA's rows (range of at most kScaleRowsMax rows)
  uint32_t id_offset;  // the global id of local vocabulary id 0 (a vocabulary shard's offset; else 0)
};

// Bounds of the noise -L(h) by bucket of the hash h: with g = h | 1, the
// position k of g's leading one and the 4 bits m after it, bucket 16 k + m
// (the exponent and top mantissa bits of g converted to float rounding toward
// zero).  -L falls as u = RN((h + 0.5) 2^-32) grows, so a bucket's bounds are
// the noise at the float u of its smallest and of its largest h, computed on
// the host in double with a margin (1e-3) far above the FP32 evaluation's
// error.  Where u < 1/16 (the large noise values that can win) a bucket spans
// a factor of at most 17/16 in u, so its noise range is about ln(17/16) = 0.06
// wide.
__constant__ float c_noise_ub[kNoiseT];
__constant__ float c_noise_lb[kNoiseT];

__device__ __forceinline__ uint32_t noise_index(uint32_t h) {
  return (__float_as_uint(__uint2float_rz(h | 1u)) >> 19) - (127u << 4);
}

// The Gumbel key of one element, out of line: it is evaluated for few
// elements, and one copy keeps the kernel's code small.
__device__ __noinline__ float eval_key(float l, float temp, uint32_t h) { return noised_key(l, temp, h); }

// Two-launch select: this CTA's row maxima into partials[r * grid + block]
// (out of line: it stays out of the register allocation of the hot loop).
__device__ __noinline__ void store_partials(unsigned long long* partials, const unsigned long long* best, int rows,
                                            int et) {
  for (int r = et; r < rows; r += kEpiThreads)
    partials[static_cast<int64_t>(r) * gridDim.x + blockIdx.x] = best[r];
}

// Explicit shared-space loads of per-row data, by the runtime shared address
// (the compiler need not order them against the epilogue's global stores).
__device__ __forceinline__ uint4 lds_u4(const void* ptr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(ptx::smem_addr(ptr)));
  return r;
}
__device__ __forceinline__ longlong2 lds_ll2(const void* ptr) {
  longlong2 r;
  asm volatile("ld.shared.v2.s64 {%0, %1}, [%2];" : "=l"(r.x), "=l"(r.y) : "r"(ptx::smem_addr(ptr)));
  return r;
}
__device__ __forceinline__ uint32_t lds_u32(const void* ptr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(ptx::smem_addr(ptr)));
  return r;
}

__device__ __forceinline__ long long lds_i64(const void* ptr) {
  long long r;
  asm volatile("ld.shared.s64 %0, [%1];" : "=l"(r) : "r"(ptx::smem_addr(ptr)));
  return r;
}
__device__ __forceinline__ float ld_shared_f32(const float* ptr) {
  float r;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(ptx::smem_addr(ptr)));
  return r;
}
__device__ __forceinline__ float ld_volatile_f32(const float* ptr) {
  float r;
  asm volatile("ld.volatile.shared.f32 %0, [%1];" : "=f"(r) : "r"(ptx::smem_addr(ptr)));
  return r;
}

// Four floats of shared memory that other warps update (never cached).
__device__ __forceinline__ float4 ld_volatile_f4(const float* ptr) {
  float4 r;
  asm volatile("ld.volatile.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(ptx::smem_addr(ptr)));
  return r;
}

__device__ __forceinline__ void WarpQueue::flush(uint32_t min_count, const Shared& sh) {
  const int lane = threadIdx.x & 31;
  while (count >= min_count && count > 0) {
    __syncwarp();
    const uint32_t n = count < 32u ? count : 32u;
    if (static_cast<uint32_t>(lane) < n) {
      const Cand e = q[(head + lane) & (kQCap - 1)];
      const uint32_t r = e.vr >> 24, v = e.vr & 0xFFFFFFu;
      const float t = sh.temp[r];
      const float key =
          t != 0.0f ? eval_key(e.l, t, murmur_finish_mixed(sh.prefix[r], murmur_kmix(v + sh.id_offset))) : e.l;
      const unsigned long long cand = pack_key(key, v);
      const unsigned long long old = atomicMax(sh.best + r, cand);
      if (cand > old) sh.thr[r] = key != key ? INFINITY : key;
    }
    head = (head + n) & (kQCap - 1);
    count -= n;
  }
  __syncwarp();
}

// Four E4M3 values (bytes of w, lowest first) as two FP16 pairs: lo holds
// values 0 and 1, hi values 2 and 3 (the hardware conversion, exact).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  // each cvt takes an E4M3 pair (lower byte = lower half of the result)
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// E4M3 w2: one embedding row (eight BF16 values a lane, the warp holding
// the whole row) as FP16 values of e * 2^k, the power of two k chosen per row
// so that the largest finite |e| lands in [2^14, 2^15): then every entry
// within 2^32 of the row's largest converts exactly (smaller ones, whose
// products are below 2^-32 of the row's largest, round to the FP16 grid), and
// infinities and NaN stay what they are.  Lane 0 stores 2^-k for the
// epilogue.  k is clamped to [-112, 126] so that 2^k and 2^-k are normal floats.
__device__ __forceinline__ uint4 embedding_to_f16(uint4 v, float* kscale, int lane) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t emax = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t e0 = (w[i] >> 7) & 0xFFu, e1 = (w[i] >> 23) & 0xFFu;
    emax = max(emax, max(e0 == 0xFFu ? 0u : e0, e1 == 0xFFu ? 0u : e1));
  }
  emax = __reduce_max_sync(0xFFFFFFFFu, emax);
  int k = 14 - (static_cast<int>(emax < 1u ? 1u : emax) - 127);
  k = k < -112 ? -112 : (k > 126 ? 126 : k);
  const float up = __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
  if (lane == 0) *kscale = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half lo = __float2half_rn(__fmul_rn(__uint_as_float(w[i] << 16), up));
    const __half hi = __float2half_rn(__fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), up));
    o[i] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The kernel's bounded mbarrier wait as a value that out-of-line helpers can
// take (the same polls, limits and give-up record as the kernel's own).
struct BoundedWait {
  volatile int* abort_flag;
  unsigned int* abort_word;
  int* status;
  __device__ __forceinline__ bool operator()(uint64_t* bar, uint32_t parity, int site, int detail) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
      if (ptx::mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
      if ((it & 15) == 15 && (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitNs)) break;
    }
    if (*abort_flag) return false;
    *abort_flag = 1;
    atomicExch(abort_word, 1u);
    if (atomicCAS(status, 0, kStatusTimeout) == 0) {
      status[1] = site;
      status[2] = static_cast<int>(blockIdx.x);
      status[3] = detail;
    }
    return false;
  }
};

// A resident tile in the first step of a launch: each w2 stage is taken from
// the ring as usual, copied into tensor memory (from column `at`, 32 columns
// a stage) and multiplied from shared memory; the stage's commit covers the
// copy too.  Returns false if a wait gave up.
__device__ __noinline__ bool resident_first_step(uint64_t* full_w2, uint64_t* empty_w2, int g, int SG, uint32_t d,
                                                 uint32_t at, uint64_t a0, uint64_t b0, uint64_t b_kstep,
                                                 uint32_t idesc, int k, BoundedWait wait, int detail) {
  for (int kb = 0; kb < kKBlocks; ++kb, ++k) {
    const int s = g * SG + k % SG;
    if (!wait(&full_w2[s], (k / SG) & 1, 5, detail | (k & 0xFFF))) return false;
    ptx::tc_fence_after();
    const uint64_t a = a0 + static_cast<uint64_t>(s * (kW2StageBytes >> 4));
    const uint64_t bd = b0 + static_cast<uint64_t>(kb) * b_kstep;
    const uint32_t ak = at + static_cast<uint32_t>(kb * 32);
    ptx::tmem_cp_128x256b(ak, a);
    ptx::tmem_cp_128x256b(ak + 8, a + 2);
    ptx::tmem_cp_128x256b(ak + 16, a + 4);
    ptx::tmem_cp_128x256b(ak + 24, a + 6);
    if (kb == 0)
      ptx::mma_bf16_c<false>(d, a, bd, idesc);
    else
      ptx::mma_bf16_c<true>(d, a, bd, idesc);
    ptx::mma_bf16_c<true>(d, a + 2, bd + 2, idesc);
    ptx::mma_bf16_c<true>(d, a + 4, bd + 4, idesc);
    ptx::mma_bf16_c<true>(d, a + 6, bd + 6, idesc);
    ptx::mma_commit(&empty_w2[s]);
  }
  return true;
}

// The MMAs of one tile whose A operand (w2, 128 rows x 256 K of 16-bit
// values) sits in tensor memory from column `at` (8 columns a K step).
__device__ __noinline__ void resident_step(uint32_t d, uint32_t at, uint64_t b0, uint64_t b_kstep, uint32_t idesc) {
  for (int kb = 0; kb < kKBlocks; ++kb) {
    const uint64_t bd = b0 + static_cast<uint64_t>(kb) * b_kstep;
    const uint32_t ak = at + static_cast<uint32_t>(kb * 32);
    if (kb == 0)
      ptx::mma_tmem_a_c<false>(d, ak, bd, idesc);
    else
      ptx::mma_tmem_a_c<true>(d, ak, bd, idesc);
    ptx::mma_tmem_a_c<true>(d, ak + 8, bd + 2, idesc);
    ptx::mma_tmem_a_c<true>(d, ak + 16, bd + 4, idesc);
    ptx::mma_tmem_a_c<true>(d, ak + 24, bd + 6, idesc);
  }
}

// kRW: rows of a chunk each epilogue warp takes -- kHalfRows, or 1 or 4 for
// loops of at most that many rows (the second half's warps then only keep
// the barriers).
// kFp8: w2 as E4M3 bytes with FP16 row scales (the w2 tensor maps then
// describe the E4M3 table: boxes of 128 K bytes).
template <bool kHasCap, bool kMultOne, bool kTestStall = false, int kRW = kHalfRows, bool kFp8 = false>
__global__ void __launch_bounds__(kThreads, 1)
step_tc_kernel(const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_w2_tile,
               const __grid_constant__ CUtensorMap tmap_base, const TcParams tp) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // The 1024-byte alignment is taken from the runtime address of the array.
  // (A build that instead offset the array by a pad computed from its shared
  // address faulted on the GPU; shared-space loads below convert runtime
  // addresses explicitly.)
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_last;

  const StepParams& p = tp.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = tp.n;
  const int S = tp.stages;
  const int NB = tp.nbase;
  const int NBG = NB / 2;  // slots of each tile parity's base ring
  const int NACC = tp.nacc;
  const int NA = NACC / 2;  // accumulators of each tile parity (MMA warp and its two quartets)
  const int n_steps = p.step_end - p.step;

  Shared sh;
  sh.emb = smem + tp.emb_off;
  sh.w2 = smem + tp.w2_off;
  sh.base = smem + tp.base_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + tp.bar_off);
  sh.full_w2 = bars;
  sh.empty_w2 = bars + S;
  sh.full_base = bars + 2 * S;
  sh.empty_base = bars + 2 * S + NB;
  sh.tmem_full = bars + 2 * S + 2 * NB;
  sh.tmem_empty = sh.tmem_full + NACC;
  sh.emb_ready = sh.tmem_full + 2 * NACC;
  sh.spare = sh.emb_ready + 1;
  sh.empty_f16 = sh.spare + 2;
  sh.f16 = smem + tp.f16_off;
  unsigned char* rowreg = smem + tp.row_off;
  sh.best = reinterpret_cast<unsigned long long*>(rowreg + kRowBest);
  sh.cache_off = reinterpret_cast<int64_t*>(rowreg + kRowCoff);
  sh.prefix = reinterpret_cast<uint32_t*>(rowreg + kRowPrefix);
  sh.rinv = reinterpret_cast<float*>(rowreg + kRowRinv);
  sh.ns = reinterpret_cast<float*>(rowreg + kRowNs);
  sh.temp = reinterpret_cast<float*>(rowreg + kRowTemp);
  sh.thr = reinterpret_cast<float*>(rowreg + kRowThr);
  sh.gmask = reinterpret_cast<uint32_t*>(rowreg + kRowGmask);
  sh.gtab = reinterpret_cast<float*>(rowreg + kRowGtab);
  sh.ltab = reinterpret_cast<float*>(rowreg + kRowLtab);
  sh.kscale = reinterpret_cast<float*>(rowreg + kRowKs);
  sh.queues = reinterpret_cast<Cand*>(smem + tp.queue_off);
  sh.w2s = reinterpret_cast<uint16_t*>(smem + tp.scale_off);
  sh.id_offset = static_cast<uint32_t>(p.vocab_offset);

  // This CTA's vocabulary range.
  const int G = gridDim.x;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * tp.num_units / G;
  const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * tp.num_units / G;
  const int64_t v_begin = u0 * kUnit;
  const int64_t v_end = min(u1 * kUnit, p.vocab);
  const int n_tiles = static_cast<int>((v_end - v_begin + kTileV - 1) / kTileV);
  const int chunks = (p.rows + kChunkRows - 1) / kChunkRows;
  // tiles res0 .. n_tiles - 1 are copied into tensor memory in the first step
  // and read from there afterwards (their w2 is streamed once per launch)
  const int res0 = n_tiles - tp.res_tiles > 0 ? n_tiles - tp.res_tiles : 0;

  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(&sh.full_w2[i], 1);
      ptx::mbar_init(&sh.empty_w2[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      ptx::mbar_init(&sh.full_base[i], 1);
      ptx::mbar_init(&sh.empty_base[i], 8);  // the eight warps of the consuming quartets
    }
    for (int i = 0; i < NACC; ++i) {
      ptx::mbar_init(&sh.tmem_full[i], 1);
      ptx::mbar_init(&sh.tmem_empty[i], 8);  // the eight warps of the consuming quartets
    }
    ptx::mbar_init(sh.emb_ready, 1);
    ptx::mbar_init(sh.spare, 1);
    ptx::mbar_init(sh.spare + 1, 1);
    for (int i = 0; i < tp.stages16; ++i) ptx::mbar_init(&sh.empty_f16[i], 1);
    s_abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&s_tmem_base, static_cast<uint32_t>(tp.tmem_cols));
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort_flag = &s_abort;

  // A wait that gives up records where: status[1] = wait site,
  // status[2] = block, status[3] = detail (step, tile, sequence number); it
  // also raises the loop's abort word, which ends the other CTAs' waits for
  // this one.
  auto give_up = [&](int site, int detail) {
    *abort_flag = 1;
    atomicExch(p.abort_word, 1u);
    if (atomicCAS(p.status, 0, kStatusTimeout) == 0) {
      p.status[1] = site;
      p.status[2] = static_cast<int>(blockIdx.x);
      p.status[3] = detail;
    }
  };
  // A bounded wait: polls that may suspend the thread until the phase
  // completes, up to kWaitNs of the global timer (and at most kWaitLimit
  // polls); it leaves early once the CTA is aborting.
  auto wait = [&](uint64_t* bar, uint32_t parity, int site, int detail) -> bool {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
      if (ptx::mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
      if ((it & 15) == 15 && (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitNs)) break;
    }
    if (*abort_flag) return false;
    give_up(site, detail);
    return false;
  };

  if (warp == 0 || warp == 2) {
    // ---------------- producers ----------------
    // Warp 0 fills the rings of the even tiles, warp 2 those of the odd ones:
    // per tile its four w2 stages (ring g of SG = S / 2 slots, consumed by MMA
    // warp g) and then its base chunks (ring g of NBG slots, consumed by
    // quartets of parity g).  Every ring has one producer and one consumer
    // taking its slots in order, across steps (an mbarrier's parity only
    // tells adjacent phases apart), and neither parity waits for the other.
    // Every step streams the same w2 range; the tensor map of the base logits
    // spans the launch's steps.
    const int g = warp == 0 ? 0 : 1;
    if (lane == 0 && n_tiles > g) {
      ptx::prefetch_tmap(&tmap_w2);
      ptx::prefetch_tmap(&tmap_w2_tile);
      ptx::prefetch_tmap(&tmap_base);
      // every step reads the same w2: ask L2 to keep it; each base logit is
      // read once: let it leave L2 first
      const uint64_t keep = ptx::make_policy_evict_last();
      const uint64_t stream = ptx::make_policy_evict_first();
      const int SG = S / 2;
      int issued = 0, issued_b = 0;
      bool stop = false;
      for (int st = 0; st < n_steps && !stop; ++st) {
        for (int i = g; i < n_tiles && !stop && !*abort_flag; i += 2) {
          const int64_t t0 = v_begin + static_cast<int64_t>(i) * kTileV;
          const int rows_i = static_cast<int>(v_end - t0 < kTileV ? v_end - t0 : kTileV);
          const int boxes = (rows_i + kUnit - 1) / kUnit;
          // a stage holds 128 bytes of each of the tile's rows: 64 K of BF16
          // (four stages a tile) or 128 K of E4M3 (two)
          constexpr int kStagesPerTile = kFp8 ? 2 : kKBlocks;
          constexpr int kStageK = kFp8 ? 128 : kKBlock;
          const bool w2_resident = st > 0 && i >= res0;  // in tensor memory since the first step
          for (int kb = 0; kb < kStagesPerTile && !w2_resident; ++kb) {
            const int k = issued;
            const int s = g * SG + k % SG;
            if (!wait(&sh.empty_w2[s], ((k / SG) & 1) ^ 1, 1, (st << 24) | (i << 12) | (k & 0xFFF))) {
              stop = true;
              break;
            }
            ptx::mbar_arrive_expect_tx(&sh.full_w2[s], static_cast<uint32_t>(boxes * kUnit * 128));
            if (boxes == kTileV / kUnit) {  // a whole tile: one 128-row copy
              ptx::tma_load_2d_hint(sh.w2 + s * kW2StageBytes, &tmap_w2_tile, &sh.full_w2[s], kb * kStageK,
                                    static_cast<int32_t>(t0), keep);
            } else {
              for (int bx = 0; bx < boxes; ++bx)
                ptx::tma_load_2d_hint(sh.w2 + s * kW2StageBytes + bx * kUnit * 128, &tmap_w2, &sh.full_w2[s],
                                      kb * kStageK, static_cast<int32_t>(t0 + bx * kUnit), keep);
            }
            issued = k + 1;
          }
          for (int c = 0; c < chunks && !stop; ++c) {
            const int k = issued_b;
            const int s = g * NBG + k % NBG;
            if (!wait(&sh.empty_base[s], ((k / NBG) & 1) ^ 1, 2, (st << 24) | (i << 12) | (k & 0xFFF))) {
              stop = true;
              break;
            }
            // the epilogue read this slot with generic loads (released to
            // this thread through the barrier); the refill is an async-proxy
            // write, which the proxy fence orders after them
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive_expect_tx(&sh.full_base[s], kChunkBytes);
            if (tp.base_steps_mid)  // dims (vocab, step, row)
              ptx::tma_load_3d_hint(sh.base + s * kChunkBytes, &tmap_base, &sh.full_base[s],
                                    static_cast<int32_t>(t0), st, c * kChunkRows, stream);
            else  // dims (vocab, row, step)
              ptx::tma_load_3d_hint(sh.base + s * kChunkBytes, &tmap_base, &sh.full_base[s],
                                    static_cast<int32_t>(t0), c * kChunkRows, st, stream);
            issued_b = k + 1;
          }
        }
        if (*abort_flag) stop = true;
      }
      if (*abort_flag) {  // let copies in flight land before the CTA exits
        for (int k = max(0, issued - SG); k < issued; ++k)
          ptx::mbar_wait(&sh.full_w2[g * SG + k % SG], (k / SG) & 1, kWaitLimit);
        for (int k = max(0, issued_b - NBG); k < issued_b; ++k)
          ptx::mbar_wait(&sh.full_base[g * NBG + k % NBG], (k / NBG) & 1, kWaitLimit);
      } else {
        // Producer tail: observe the MMA's release of every w2 stage in
        // flight, so that no tensor-core arrival on this CTA's barriers is
        // still pending when the CTA exits.
        for (int k = issued; k < issued + SG; ++k)
          if (!wait(&sh.empty_w2[g * SG + k % SG], ((k / SG) & 1) ^ 1, 8, k)) break;
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ---------------- MMA issuers ----------------
    // Two warps issue (one instruction stream alone cannot keep up with the
    // w2 stream at N = 16): in every step warp 1 takes the even tiles, warp 3
    // the odd ones, each with its own w2 ring and accumulators g, g + 2, ...
    // (its j-th tile uses accumulator g + 2 (j % NA)).  A step's MMAs start
    // once the epilogue has written that step's embeddings.
    const int g = warp == 1 ? 0 : 1;
    if constexpr (kFp8) {
      // E4M3 w2: the whole warp turns each E4M3 stage (128 rows x 128 K) into
      // two FP16 operand stages (128 rows x 64 K each, the MMA's 128-byte
      // swizzle layout) of this warp's ring, one hardware conversion per pair
      // (exact: every E4M3 value is an FP16 value), releases the E4M3 stage,
      // and lane 0 issues the two K-blocks' MMAs (FP16 x FP16 into FP32) with
      // one commit per FP16 stage.
      if (n_tiles > g) {
        const int SG = S / 2;                 // E4M3 slots of this parity's ring
        const int SG16 = tp.stages16 / 2;     // FP16 slots of this warp's ring
        const uint32_t idesc = ptx::idesc_f16_f32(kTileV, static_cast<uint32_t>(N));
        const uint64_t a0 = ptx::sw128_desc(ptx::smem_addr(sh.f16), 1024);
        const uint64_t b0 = ptx::sw128_desc(ptx::smem_addr(sh.emb), 1024);
        const uint64_t b_kstep = static_cast<uint64_t>((N * 128) >> 4);
        // a lane converts rows 8 q + (lane & 7) of 16-byte chunk (lane >> 3) +
        // 4 h of each E4M3 row: the eight lanes of a shared-memory phase take
        // eight rows of one chunk, so neither the reads nor the writes of a
        // phase share a bank
        const int rl = lane & 7, cq = lane >> 3;
        bool ok = true;
        int k = 0;   // E4M3 stages taken from this parity's ring
        int k16 = 0; // FP16 stages used
        int j = 0;   // tiles issued
        for (int st = 0; st < n_steps && ok; ++st) {
          if (!(ok = __all_sync(0xFFFFFFFFu, wait(sh.emb_ready, st & 1, 3, st << 24)))) break;
          ptx::tc_fence_after();
          for (int i = g; i < n_tiles && ok; i += 2, ++j) {
            const int b = g + 2 * (j % NA);
            if (!(ok = __all_sync(0xFFFFFFFFu, wait(&sh.tmem_empty[b], ((j / NA) & 1) ^ 1, 4, (st << 24) | (i << 12)))))
              break;
            ptx::tc_fence_after();
            const uint32_t d = tmem_base + static_cast<uint32_t>(b * N);
            const bool res = i >= res0;
            const uint32_t at = tmem_base + static_cast<uint32_t>(tp.res_col + (i - res0) * 128);
            if (res && st > 0) {  // converted in the first step and kept in tensor memory
              if (lane == 0) {
                for (int kb = 0; kb < kKBlocks; ++kb) {
                  const uint64_t bd = b0 + static_cast<uint64_t>(kb) * b_kstep;
                  const uint32_t ak = at + static_cast<uint32_t>(kb * 32);
                  if (kb == 0)
                    ptx::mma_tmem_a_c<false>(d, ak, bd, idesc);
                  else
                    ptx::mma_tmem_a_c<true>(d, ak, bd, idesc);
                  ptx::mma_tmem_a_c<true>(d, ak + 8, bd + 2, idesc);
                  ptx::mma_tmem_a_c<true>(d, ak + 16, bd + 4, idesc);
                  ptx::mma_tmem_a_c<true>(d, ak + 24, bd + 6, idesc);
                }
                ptx::mma_commit(&sh.tmem_full[b]);
              }
              __syncwarp();
              continue;
            }
            for (int h = 0; h < 2 && ok; ++h, ++k, k16 += 2) {
              const int s8 = g * SG + k % SG;
              const int sa = g * SG16 + k16 % SG16, sb = g * SG16 + (k16 + 1) % SG16;
              ok = __all_sync(0xFFFFFFFFu,
                              wait(&sh.full_w2[s8], (k / SG) & 1, 5, (st << 24) | (i << 12) | (k & 0xFFF)) &&
                                  wait(&sh.empty_f16[sa], ((k16 / SG16) & 1) ^ 1, 10, (st << 24) | (i << 12)) &&
                                  wait(&sh.empty_f16[sb], (((k16 + 1) / SG16) & 1) ^ 1, 10, (st << 24) | (i << 12)));
              if (!ok) break;
              const uint32_t src = ptx::smem_addr(sh.w2 + s8 * kW2StageBytes) + rl * 128;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int c = cq + 4 * hh;  // logical 16-byte chunk: K 16 c .. 16 c + 15 of this stage
                const uint32_t dst =
                    ptx::smem_addr(sh.f16 + (hh ? sb : sa) * kW2StageBytes) + rl * 128;
                const uint32_t rd = src + ((c ^ rl) << 4);
                const uint32_t w0 = dst + (((2 * cq) ^ rl) << 4), w1 = dst + (((2 * cq + 1) ^ rl) << 4);
                // eight 16-byte loads in flight, then their conversions
#pragma unroll
                for (int q0 = 0; q0 < kTileV / 8; q0 += 8) {
                  uint4 v8[8];
#pragma unroll
                  for (int q = 0; q < 8; ++q) v8[q] = ptx::lds_v4(rd + (q0 + q) * 1024);
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    uint4 lo, hi;
                    e4m3x4_to_f16(v8[q].x, lo.x, lo.y);
                    e4m3x4_to_f16(v8[q].y, lo.z, lo.w);
                    e4m3x4_to_f16(v8[q].z, hi.x, hi.y);
                    e4m3x4_to_f16(v8[q].w, hi.z, hi.w);
                    ptx::sts_v4(w0 + (q0 + q) * 1024, lo);
                    ptx::sts_v4(w1 + (q0 + q) * 1024, hi);
                  }
                }
              }
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::mbar_arrive(&sh.empty_w2[s8]);
                ptx::tc_fence_after();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const int s16 = hh ? sb : sa;
                  const uint64_t a = a0 + static_cast<uint64_t>(s16 * (kW2StageBytes >> 4));
                  const uint64_t bd = b0 + static_cast<uint64_t>(2 * h + hh) * b_kstep;
                  if (res) {  // first step: keep the FP16 stage in tensor memory for the later steps
                    const uint32_t ak = at + static_cast<uint32_t>((2 * h + hh) * 32);
                    ptx::tmem_cp_128x256b(ak, a);
                    ptx::tmem_cp_128x256b(ak + 8, a + 2);
                    ptx::tmem_cp_128x256b(ak + 16, a + 4);
                    ptx::tmem_cp_128x256b(ak + 24, a + 6);
                  }
                  if (h == 0 && hh == 0)
                    ptx::mma_f16_c<false>(d, a, bd, idesc);
                  else
                    ptx::mma_f16_c<true>(d, a, bd, idesc);
                  ptx::mma_f16_c<true>(d, a + 2, bd + 2, idesc);
                  ptx::mma_f16_c<true>(d, a + 4, bd + 4, idesc);
                  ptx::mma_f16_c<true>(d, a + 6, bd + 6, idesc);
                  ptx::mma_commit(&sh.empty_f16[s16]);
                }
              }
              __syncwarp();
            }
            if (ok && lane == 0) ptx::mma_commit(&sh.tmem_full[b]);
          }
        }
        // every MMA lane 0 issued has completed before TMEM is freed
        if (lane == 0) {
          ptx::mma_commit(sh.spare + g);
          ptx::mbar_wait(sh.spare + g, 0, kWaitLimit);
        }
        __syncwarp();
      }
    } else if (lane == 0 && n_tiles > g) {
      const int SG = S / 2;
      const uint32_t idesc = ptx::idesc_bf16_f32(kTileV, static_cast<uint32_t>(N));
      // descriptors of stage 0 / K-block 0; a stage is 16 KB (1024 in the
      // descriptor's 16-byte units), a K step of 16 is 32 bytes (2 units)
      const uint64_t a0 = ptx::sw128_desc(ptx::smem_addr(sh.w2), 1024);
      const uint64_t b0 = ptx::sw128_desc(ptx::smem_addr(sh.emb), 1024);
      const uint64_t b_kstep = static_cast<uint64_t>((N * 128) >> 4);
      bool ok = true;
      int k = 0;  // stages this warp has taken from its ring
      int j = 0;  // tiles this warp has issued
      for (int st = 0; st < n_steps && ok; ++st) {
        // every step's embeddings, in order (each phase of emb_ready is seen)
        if (!(ok = wait(sh.emb_ready, st & 1, 3, st << 24))) break;
        ptx::tc_fence_after();
        for (int i = g; i < n_tiles && ok; i += 2, ++j) {
          const int b = g + 2 * (j % NA);
          if (!(ok = wait(&sh.tmem_empty[b], ((j / NA) & 1) ^ 1, 4, (st << 24) | (i << 12)))) break;
          ptx::tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(b * N);
          if (i < res0) {  // w2 streamed through the ring
            for (int kb = 0; kb < kKBlocks && ok; ++kb, ++k) {
              const int s = g * SG + k % SG;
              if (!(ok = wait(&sh.full_w2[s], (k / SG) & 1, 5, (st << 24) | (i << 12) | (k & 0xFFF)))) break;
              ptx::tc_fence_after();
              const uint64_t a = a0 + static_cast<uint64_t>(s * (kW2StageBytes >> 4));
              const uint64_t bd = b0 + static_cast<uint64_t>(kb) * b_kstep;
              if (kb == 0)
                ptx::mma_bf16_c<false>(d, a, bd, idesc);
              else
                ptx::mma_bf16_c<true>(d, a, bd, idesc);
              ptx::mma_bf16_c<true>(d, a + 2, bd + 2, idesc);
              ptx::mma_bf16_c<true>(d, a + 4, bd + 4, idesc);
              ptx::mma_bf16_c<true>(d, a + 6, bd + 6, idesc);
              ptx::mma_commit(&sh.empty_w2[s]);
            }
          } else if (st == 0) {  // a resident tile's first step: streamed, and copied into tensor memory
            ok = resident_first_step(sh.full_w2, sh.empty_w2, g, SG, d,
                                     tmem_base + static_cast<uint32_t>(tp.res_col + (i - res0) * 128), a0, b0, b_kstep,
                                     idesc, k, BoundedWait{abort_flag, p.abort_word, p.status}, (st << 24) | (i << 12));
            k += kKBlocks;
          } else {  // a resident tile: A read from tensor memory
            resident_step(d, tmem_base + static_cast<uint32_t>(tp.res_col + (i - res0) * 128), b0, b_kstep, idesc);
          }
          if (ok) ptx::mma_commit(&sh.tmem_full[b]);
        }
      }
      // every MMA this thread issued has completed before TMEM is freed
      ptx::mma_commit(sh.spare + g);
      ptx::mbar_wait(sh.spare + g, 0, kWaitLimit);
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------- epilogue ----------------
    const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..511
    const int quartet = (warp - kEpiWarp0) >> 2;
    const int wg = quartet & 1;                   // takes tiles i = wg, wg + 2, ... of every step
    const int half = quartet >> 1;                // takes rows 8 half .. 8 half + 7 of every chunk
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp

    // Per-row sampling constants of relative step st, one thread per row
    // slot (the first kMaxRows epilogue threads); slots beyond the rows are
    // never taken.  They are inputs of the loop (no grid dependency).
    auto row_init = [&](int st) {
      if (et >= kMaxRows) return;  // whole warps
      const int r = et;
      float thr = INFINITY, rinv = 1.0f, ns = 0.0f, temp = 0.0f;
      uint32_t prefix = 0;
      int64_t coff = 0;
      bool store = false;
      if (r < p.rows) {
        const RowInfo ri = row_info(p, r, p.step + st);
        temp = ri.temp;
        const bool noisy = ri.temp != 0.0f;
        rinv = noisy ? __frcp_rn(ri.temp) : 1.0f;
        ns = noisy ? 1.0f : 0.0f;
        prefix = ri.prefix;
        coff = ri.cache_off + static_cast<int64_t>(st) * p.cache_s1;
        store = ri.valid != 0;
        thr = -INFINITY;
      }
      sh.best[r] = 0ull;
      // the row's cache row as an address (read only where the row stores)
      sh.cache_off[r] = store ? reinterpret_cast<int64_t>(p.cache + coff) : 0;
      sh.prefix[r] = prefix;
      sh.rinv[r] = rinv;
      sh.ns[r] = ns;
      sh.temp[r] = temp;
      sh.thr[r] = thr;
      const uint32_t sb = __ballot_sync(0xFFFFFFFFu, store), lb = __ballot_sync(0xFFFFFFFFu, r < p.rows);
      if ((lane & 15) == 0) sh.gmask[r >> 4] = ((sb >> lane) & 0xFFFFu) | (((lb >> lane) & 0xFFFFu) << 16);
    };

    // Markov embeddings of relative step st's previous tokens, in the MMA's
    // B layout: 4 K-blocks of [N rows x 128 bytes], 128-byte swizzle.  CTA 0
    // writes those tokens as the previous step's output.  Every MMA of the
    // step before has completed (the epilogue consumed all its tiles).
    const uint64_t last_row = static_cast<uint64_t>(p.w1_rows - 1);
    auto gather = [&](int st) {
      const unsigned long long* prev = p.slots_prev + static_cast<int64_t>(st) * p.slots_s;
      const bool write_prev = blockIdx.x == 0 && (st > 0 || p.write_prev);
      const int64_t prev_step = static_cast<int64_t>(p.step) + st - 1;
      for (int idx = et; idx < N * 32; idx += kEpiThreads) {
        const int r = idx >> 5, ch = idx & 31;  // a warp takes one row
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.rows) {
          const int64_t tok = st == 0 && p.self_reset ? static_cast<int64_t>(__ldg(p.input_ids + __ldg(p.anchor_idx + r)))
                                                      : slot_token(__ldcg(prev + r));
          const uint64_t row = static_cast<uint64_t>(tok) < last_row ? static_cast<uint64_t>(tok) : last_row;
          val = ldg_nc_v4(p.w1 + row * kRank + ch * 8);
          if (write_prev && ch == 0) p.tokens[static_cast<int64_t>(r) * p.tokens_s0 + prev_step] = tok;
        }
        if constexpr (kFp8) val = embedding_to_f16(val, sh.kscale + r, ch);
        const int kb = ch >> 3, c = ch & 7;
        *reinterpret_cast<uint4*>(sh.emb + kb * N * 128 + r * 128 + ((c ^ (r & 7)) << 4)) = val;
      }
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(1, kEpiThreads);
      if (et == 0) ptx::mbar_arrive(sh.emb_ready);
    };

    // All CTAs have published relative step st's row maxima (its arrival
    // counter reached the grid size).  Every CTA of the cooperative launch is
    // resident, so the wait ends unless a CTA gave up; the loop's abort word
    // then ends it early.
    auto wait_grid = [&](int st) -> bool {
      const unsigned int* ctr = p.counter + st;
      // (the checking aid waits for one arrival too many at the first boundary)
      const uint32_t target = static_cast<uint32_t>(G) + (kTestStall && st == 0 ? 1u : 0u);
      for (uint32_t it = 0; it < kGridWaitLimit; ++it) {
        if (ptx::ld_acquire_gpu(ctr) >= target) return true;
        if ((it & 15) == 15 && (*abort_flag || ptx::ld_volatile_global(p.abort_word) != 0u)) {
          *abort_flag = 1;
          return false;
        }
      }
      give_up(9, st << 24);
      return false;
    };

    row_init(0);
    for (int t = et; t < kNoiseT; t += kEpiThreads) {
      sh.gtab[t] = c_noise_ub[t];
      sh.ltab[t] = c_noise_lb[t];
    }
    // E4M3 w2: the range's row scales, read by every step (a weight table:
    // no wait on the previous launch); published by gather's barrier
    const bool w2s_local = kFp8 && v_end - v_begin <= kScaleRowsMax;
    if (w2s_local)
      for (int t = et; t < v_end - v_begin; t += kEpiThreads) sh.w2s[t] = __ldg(p.w2_scale + v_begin + t);
    pdl_wait();
    gather(0);

    WarpQueue q;
    q.q = sh.queues + (warp - kEpiWarp0) * kQCap;
    int taken = 0;  // chunks this warp's quartet has taken from its base ring
    int j = 0;      // tiles this warp's quartet has taken
    const int vr = quarter * 32 + lane;  // this thread's vocabulary row of a tile
    for (int st = 0; st < n_steps; ++st) {
      const int step = p.step + st;
      bool ok = true;
      for (int i = wg; i < n_tiles && ok; i += 2, ++j) {
        const int b = wg + 2 * (j % NA);
        const int64_t v = v_begin + static_cast<int64_t>(i) * kTileV + vr;
        const bool in = v < v_end;
        const uint32_t kv = murmur_kmix(static_cast<uint32_t>(v) + sh.id_offset);  // the global id
        float w2s = 0.0f;  // E4M3 w2: this vocabulary row's FP16 scale (read while the tile's MMAs run)
        if constexpr (kFp8)
          w2s = in ? __half2float(__ushort_as_half(w2s_local ? sh.w2s[v - v_begin] : __ldg(p.w2_scale + v))) : 0.0f;
        ok = __all_sync(0xFFFFFFFFu, wait(&sh.tmem_full[b], (j / NA) & 1, 6, (st << 24) | (i << 12)));
        if (!ok) break;
        ptx::tc_fence_after();
        const bool first = i == wg;
        for (int c = 0; c < chunks && ok; ++c) {
          const int k = taken++;
          const int s = wg * NBG + k % NBG;
          ok = __all_sync(0xFFFFFFFFu, wait(&sh.full_base[s], (k / NBG) & 1, 7, (st << 24) | (i << 12) | (k & 0xFFF)));
          if (!ok) break;
          constexpr int R = kRW;
          const int r0 = c * kChunkRows + half * kHalfRows;  // this warp's first row of the chunk
          if (kRW < kHalfRows && half == 1) {
            // few-row build: no row for this warp; the slot's data has
            // landed, so release it (and the accumulator) in step
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive(&sh.empty_base[s]);
              if (c == chunks - 1) ptx::mbar_arrive(&sh.tmem_empty[b]);
            }
            continue;
          }
          const uint16_t* bs =
              reinterpret_cast<const uint16_t*>(sh.base + s * kChunkBytes) + half * kHalfRows * kTileV;
          uint32_t bb[R];
#pragma unroll
          for (int rr = 0; rr < R; ++rr) bb[rr] = bs[rr * kTileV + vr];
          uint32_t acc[R];
          const uint32_t taddr =
              tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(b * N + r0);
          if constexpr (R == 1)
            ptx::tmem_ld1_sync(taddr, acc);
          else if constexpr (R == 4)
            ptx::tmem_ld4_sync(taddr, acc);
          else
            ptx::tmem_ld8_sync(taddr, acc);
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(&sh.empty_base[s]);
            // the tile's last chunk is in registers: the accumulator is free
            if (c == chunks - 1) ptx::mbar_arrive(&sh.tmem_empty[b]);
          }

          // (a) bias rounded to BF16 and the BF16 add on packed pairs (the
          // BF16 add is the FP32 add rounded once), then the transform of the
          // sum x: none with multiplier 1 and no cap (x * 1 rounds to x), the
          // call's lookup table with a soft cap, else the multiplier
          uint32_t cb[R], biasb[R];
          float lv[R];
          if constexpr (kFp8) {
            // E4M3 w2: the dot of e 2^k with decode(q), back to e's scale
            // (exact) and times the FP16 row scale, rounded once to FP32
            // ([P1] dsparkMarkovGreedyFusedStepFp8: the scale meets the FP32
            // sum); then the BF16 rounding below
#pragma unroll
            for (int rr = 0; rr < R; ++rr)
              acc[rr] = __float_as_uint(
                  __fmul_rn(__fmul_rn(__uint_as_float(acc[rr]), ld_shared_f32(sh.kscale + r0 + rr)), w2s));
          }
          if constexpr (R == 1) {
            const uint32_t bias1 = ptx::cvt_bf16x2(__uint_as_float(acc[0]), 0.0f);
            biasb[0] = bias1 & 0xFFFFu;
            cb[0] = ptx::add_bf16x2(bb[0], bias1) & 0xFFFFu;
          } else {
#pragma unroll
            for (int pr = 0; pr < R / 2; ++pr) {
              const uint32_t bias2 =
                  ptx::cvt_bf16x2(__uint_as_float(acc[2 * pr]), __uint_as_float(acc[2 * pr + 1]));
              const uint32_t x2 = ptx::add_bf16x2(bb[2 * pr] | (bb[2 * pr + 1] << 16), bias2);
              biasb[2 * pr] = bias2 & 0xFFFFu;
              biasb[2 * pr + 1] = bias2 >> 16;
              cb[2 * pr] = x2 & 0xFFFFu;
              cb[2 * pr + 1] = x2 >> 16;
            }
          }
          if (kHasCap) {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) cb[rr] = __ldg(p.xform_lut + cb[rr]);
          } else if (!kMultOne) {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) cb[rr] = transform_sum<false>(bf16_bits_to_float(cb[rr]), p.mult, 0.0f, 0.0f, &lv[rr]);
          }
#pragma unroll
          for (int rr = 0; rr < R; ++rr) lv[rr] = bf16_bits_to_float(cb[rr]);

          // the rows' constants, all loaded before any global store
          uint32_t pf[R], ri[R], nsb[R];
          if constexpr (R == 1) {
            pf[0] = lds_u32(sh.prefix + r0);
            ri[0] = lds_u32(sh.rinv + r0);
            nsb[0] = lds_u32(sh.ns + r0);
          }
#pragma unroll
          for (int q4 = 0; q4 < R / 4; ++q4) {
            const uint4 a = lds_u4(sh.prefix + r0 + 4 * q4);
            const uint4 bq = lds_u4(sh.rinv + r0 + 4 * q4);
            const uint4 cq = lds_u4(sh.ns + r0 + 4 * q4);
            pf[4 * q4] = a.x; pf[4 * q4 + 1] = a.y; pf[4 * q4 + 2] = a.z; pf[4 * q4 + 3] = a.w;
            ri[4 * q4] = bq.x; ri[4 * q4 + 1] = bq.y; ri[4 * q4 + 2] = bq.z; ri[4 * q4 + 3] = bq.w;
            nsb[4 * q4] = cq.x; nsb[4 * q4 + 1] = cq.y; nsb[4 * q4 + 2] = cq.z; nsb[4 * q4 + 3] = cq.w;
          }
          const uint32_t gm16 = lds_u32(sh.gmask + c) >> (half * kHalfRows);
          const uint32_t gm = (gm16 & 0xFFu) | (gm16 >> 16 & 0xFFu) << 16;  // store bits 0..7, live bits 16..23
          const uint32_t live = in ? gm >> 16 : 0u;  // this warp's rows that exist, this lane in range

          // hash and the exact upper bound of each key: key <= l/t + (the
          // noise bound of h's bucket) with rounding margins; a greedy row's
          // bound is l (plus a margin), its key l itself
          float bnd[R], qa[R];
          uint32_t hv[R];
#pragma unroll
          for (int rr = 0; rr < R; ++rr) {
            hv[rr] = murmur_finish_mixed(pf[rr], kv);
            qa[rr] = __fmul_rn(lv[rr], __uint_as_float(ri[rr]));
            const float g = __uint_as_float(lds_u32(sh.gtab + noise_index(hv[rr])));
            bnd[rr] = __fmaf_rn(__uint_as_float(nsb[rr]), g, __fmaf_rn(fabsf(qa[rr]), 0x1p-20f, qa[rr]));
          }

          // (b) the quartet's first tile of the step: raise each row's
          // threshold to the warp's largest exact lower bound of a key, l/t +
          // (least noise of h's bucket) with rounding margins; a threshold
          // at or below some key of this CTA's range never prunes its argmax
          if (first) {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
              if (gm & (0x10000u << rr)) {
                const float lb =
                    __fmaf_rn(__uint_as_float(nsb[rr]), __uint_as_float(lds_u32(sh.ltab + noise_index(hv[rr]))),
                              __fmaf_rn(-fabsf(qa[rr]), 0x1p-20f, qa[rr]));
                const uint32_t o = ((live >> rr) & 1u) && lb == lb ? orderable(lb) : 0u;
                const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, o);
                if (lane == 0 && top != 0u) {
                  const float m = __uint_as_float((top & 0x80000000u) ? (top & 0x7FFFFFFFu) : ~top);
                  float* t = sh.thr + r0 + rr;
                  if (m > *reinterpret_cast<volatile float*>(t)) *t = m;
                }
              }
            }
            __syncwarp();
          }

          // (c) an element whose bound is below its row's threshold cannot be
          // the argmax; the rest are queued and evaluated 32 at a time
          uint32_t take = 0;
          if constexpr (R == 1) take = bnd[0] < ld_volatile_f32(sh.thr + r0) ? 0u : 1u;
#pragma unroll
          for (int q4 = 0; q4 < R / 4; ++q4) {
            const float4 th = ld_volatile_f4(sh.thr + r0 + 4 * q4);
            take |= (bnd[4 * q4] < th.x ? 0u : 1u) << (4 * q4);
            take |= (bnd[4 * q4 + 1] < th.y ? 0u : 1u) << (4 * q4 + 1);
            take |= (bnd[4 * q4 + 2] < th.z ? 0u : 1u) << (4 * q4 + 2);
            take |= (bnd[4 * q4 + 3] < th.w ? 0u : 1u) << (4 * q4 + 3);
          }
          take &= live;
          if (__any_sync(0xFFFFFFFFu, take != 0u)) {
            // one warp scan places every survivor in the queue when they fit
            const uint32_t nt = __popc(take);
            uint32_t incl = nt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
              if (lane >= off) incl += y;
            }
            const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
            if (q.count + total <= static_cast<uint32_t>(kQCap)) {
              uint32_t pos = q.head + q.count + incl - nt;
#pragma unroll
              for (int rr = 0; rr < R; ++rr)
                if ((take >> rr) & 1u) {
                  q.q[pos & (kQCap - 1)] =
                      Cand{lv[rr], (static_cast<uint32_t>(r0 + rr) << 24) | static_cast<uint32_t>(v)};
                  ++pos;
                }
              q.count += total;
              q.flush(32, sh);
            } else {
#pragma unroll
              for (int rr = 0; rr < R; ++rr) {
                const bool t = (take >> rr) & 1u;
                if (__any_sync(0xFFFFFFFFu, t)) {
                  q.push(t, lane, static_cast<uint32_t>(v), lv[rr], r0 + rr);
                  q.flush(32, sh);
                }
              }
            }
          }

          // (d) cache and bias stores of the chunk
          if (in) {
            if constexpr (R == 1) {
              if (gm & 1u)
                __stcs(reinterpret_cast<unsigned short*>(lds_i64(sh.cache_off + r0)) + v,
                       static_cast<unsigned short>(cb[0]));
            }
#pragma unroll
            for (int q2 = 0; q2 < R / 2; ++q2) {
              const longlong2 co = lds_ll2(sh.cache_off + r0 + 2 * q2);
              // streaming stores: the cache is not read back by the loop
              if (gm & (1u << (2 * q2)))
                __stcs(reinterpret_cast<unsigned short*>(co.x) + v, static_cast<unsigned short>(cb[2 * q2]));
              if (gm & (2u << (2 * q2)))
                __stcs(reinterpret_cast<unsigned short*>(co.y) + v, static_cast<unsigned short>(cb[2 * q2 + 1]));
            }
            if (p.bias_out) {
#pragma unroll
              for (int rr = 0; rr < R; ++rr)
                if (gm & (0x10000u << rr))
                  p.bias_out[(static_cast<int64_t>(r0 + rr) * p.steps + step) * p.vocab + v] =
                      static_cast<uint16_t>(biasb[rr]);
            }
          }
        }
      }
      q.flush(1, sh);

      // Every quartet is done with the step (a wait that gave up anywhere
      // in the CTA ends the loop here, the same way in every thread).
      if (ptx::named_bar_or(1, kEpiThreads, *abort_flag != 0)) break;
      // Publish this CTA's row maxima.  Within a launch the next step waits
      // until every CTA has published; a launch's last step either leaves its
      // tokens to the next launch's CTA 0 or (finish) lets the CTA that
      // arrives last write them.
      if (p.partials) {  // the select launch reduces the CTAs' maxima (one step per launch)
        store_partials(p.partials, sh.best, p.rows, et);
        break;
      }
      unsigned long long* out = p.slots_out + static_cast<int64_t>(st) * p.slots_s;
      for (int r = et; r < p.rows; r += kEpiThreads) atomicMax(out + r, sh.best[r]);
      const bool last = st == n_steps - 1;
      if (last && !p.finish) break;
      // the arrival is released after every thread's maxima (the barrier
      // orders them before the one fence, which is cumulative)
      ptx::named_bar_sync(1, kEpiThreads);
      if (et == 0) {
        __threadfence();
        s_last = atomicAdd(p.counter + st, 1u) == static_cast<unsigned int>(G - 1);
        if (p.self_reset && s_last && st > 0) {
          // every CTA is past step st - 1's grid wait and has read the slots
          // of step st's previous tokens: clear both for the next call
          p.counter[st - 1] = 0u;
          unsigned long long* used = p.slots_out + static_cast<int64_t>(st - 1) * p.slots_s;
          for (int r = 0; r < p.rows; ++r) used[r] = 0ull;
        }
      }
      if (last) {
        ptx::named_bar_sync(1, kEpiThreads);
        if (s_last) {
          __threadfence();
          if (p.self_reset && et == 0) p.counter[st] = 0u;
          for (int r = et; r < p.rows; r += kEpiThreads) {
            const unsigned long long sv = atomicAdd(out + r, 0ull);
            if (p.self_reset) out[r] = 0ull;
            if (p.packets) {  // a rank of a sharded loop: its winner's packet ([P3] _finish)
              const int4 pk = make_int4(static_cast<int>(key_bits(static_cast<uint32_t>(sv >> 32))),
                                        static_cast<int>(static_cast<int64_t>(p.vocab_offset) + slot_token(sv)), 0, 0);
              *reinterpret_cast<int4*>(p.packets + 4 * r) = pk;
            } else {
              p.tokens[static_cast<int64_t>(r) * p.tokens_s0 + step] = slot_token(sv);
            }
          }
        }
        break;
      }
      // The next step's row constants (the rows' shared state is free: all
      // quartets are past the barrier) while the other CTAs arrive.
      row_init(st + 1);
      const bool arrived = et != 0 || wait_grid(st);
      if (ptx::named_bar_or(1, kEpiThreads, !arrived || *abort_flag != 0)) break;
      gather(st + 1);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, static_cast<uint32_t>(tp.tmem_cols));
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

int max_tc_smem() {
  int m = 0;
  for (int r = 1; r <= kMaxRows; ++r) {
    m = tc_layout(r).smem > m ? tc_layout(r).smem : m;
    m = tc_layout(r, true).smem > m ? tc_layout(r, true).smem : m;
  }
  return m;
}

template <bool C, bool M, bool T = false, int RW = kHalfRows, bool F = false>
cudaError_t set_attrs() {
  return cudaFuncSetAttribute(step_tc_kernel<C, M, T, RW, F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_tc_smem());
}

// u of hash h as the kernels form it (two FP32 roundings, one of them an fma).
float noise_u(uint32_t h) {
  const float lo = (static_cast<float>(h & 0xFFFFu) + 0.5f) * 0x1p-32f;
  return fmaf(static_cast<float>(h >> 16), 0x1p-16f, lo);
}

// -L(u) = -log(-log(1 - u)) in double, with the kernels' clamp of 1 - u at 2^-24.
double neg_noise_L(float u) {
  const double om = 1.0 - static_cast<double>(u);
  const double l1m = om < 0x1p-24 ? log(0x1p-24) : log1p(-static_cast<double>(u));
  return -log(-l1m);
}

}  // namespace

void noise_bound_tables(float* ub, float* lb) {
  const double margin = 1e-3;
  // The bucket's smallest and largest hash: enumerated below 2^16, a range
  // above (there h | 1 leaves the 4 bits after the leading one alone).
  int64_t lo[kNoiseT], hi[kNoiseT];
  for (int b = 0; b < kNoiseT; ++b) lo[b] = hi[b] = -1;
  for (int64_t h = 0; h < (int64_t{1} << 16); ++h) {
    const int64_t g = h | 1;
    int k = 0;
    while ((g >> (k + 1)) != 0) ++k;
    const int m = static_cast<int>(k >= 4 ? (g >> (k - 4)) & 15 : (g << (4 - k)) & 15);
    const int b = 16 * k + m;
    if (lo[b] < 0) lo[b] = h;
    hi[b] = h;
  }
  for (int k = 16; k < 32; ++k)
    for (int m = 0; m < 16; ++m) {
      const int b = 16 * k + m;
      lo[b] = (int64_t{1} << k) + (static_cast<int64_t>(m) << (k - 4));
      hi[b] = lo[b] + (int64_t{1} << (k - 4)) - 1;
    }
  for (int b = 0; b < kNoiseT; ++b) {
    if (lo[b] < 0) {
      ub[b] = lb[b] = 0.0f;  // never looked up
      continue;
    }
    ub[b] = static_cast<float>(neg_noise_L(noise_u(static_cast<uint32_t>(lo[b]))) + margin);
    lb[b] = static_cast<float>(neg_noise_L(noise_u(static_cast<uint32_t>(hi[b]))) - margin);
  }
}

namespace {

// Fill the kernel's noise-bound tables (see c_noise_ub / c_noise_lb).
cudaError_t upload_noise_tables() {
  float ub[kNoiseT], lb[kNoiseT];
  noise_bound_tables(ub, lb);
  cudaError_t e = cudaMemcpyToSymbol(c_noise_ub, ub, sizeof(ub));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(c_noise_lb, lb, sizeof(lb));
}

}  // namespace

cudaError_t setup_step_tc() {
  if (!encode_fn()) return cudaErrorNotSupported;
  cudaError_t e = upload_noise_tables();
  if (e != cudaSuccess) return e;
  if ((e = set_attrs<false, false>()) != cudaSuccess) return e;
  if ((e = set_attrs<false, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<true, false>()) != cudaSuccess) return e;
  if ((e = set_attrs<false, true, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<false, true, false, 1>()) != cudaSuccess) return e;
  if ((e = set_attrs<false, true, false, 4>()) != cudaSuccess) return e;
  if ((e = set_attrs<true, true>()) != cudaSuccess) return e;
  // E4M3 w2
  if ((e = set_attrs<false, false, false, kHalfRows, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<false, true, false, kHalfRows, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<true, false, false, kHalfRows, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<true, true, false, kHalfRows, true>()) != cudaSuccess) return e;
  if ((e = set_attrs<false, true, false, 1, true>()) != cudaSuccess) return e;
  return set_attrs<false, true, false, 4, true>();
}

int tc_fp8_max_rows() {
  int m = 0;
  for (int r = 1; r <= kMaxRows; ++r)
    if (tc_layout(r, true).smem > 0) m = r;
  return m;
}

int tc_smem_bytes(int rows) { return tc_layout(rows).smem; }

bool encode_w2_fp8_map(CUtensorMap* map, const void* w2_fp8, int64_t vocab, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRank), static_cast<cuuint64_t>(vocab)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRank)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};  // 128 K bytes: one swizzle row
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w2_fp8), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_w2_map(CUtensorMap* map, const void* w2, int64_t vocab, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRank), static_cast<cuuint64_t>(vocab)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRank * 2)};
  const cuuint32_t box[2] = {kKBlock, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w2), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Base logits of steps p.step .. p.step_end - 1 as one 3-D tensor: the
// (vocab, row, step) or (vocab, step, row) order, whichever has increasing
// strides; boxes of 128 vocabulary entries x 16 rows x 1 step.  A dimension of
// extent 1 takes the placeholder stride (previous stride x previous extent).
bool encode_base_map(CUtensorMap* map, const StepParams& p, bool* steps_mid) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int64_t nsteps = p.step_end - p.step;
  const bool mid = nsteps > 1 && p.base_s1 < p.base_s0;
  const int64_t ext1 = mid ? nsteps : p.rows, ext2 = mid ? p.rows : nsteps;
  const int64_t row0 = (p.vocab * 2 + 15) / 16 * 16;
  const int64_t str1 = ext1 > 1 ? 2 * (mid ? p.base_s1 : p.base_s0) : row0;
  const int64_t str2 = ext2 > 1 ? 2 * (mid ? p.base_s0 : p.base_s1) : str1 * ext1;
  if (str1 <= 0 || str2 <= 0 || (str1 & 15) || (str2 & 15) || str2 >= (int64_t{1} << 40)) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.vocab), static_cast<cuuint64_t>(ext1),
                              static_cast<cuuint64_t>(ext2)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(str1), static_cast<cuuint64_t>(str2)};
  const cuuint32_t box[3] = {kTileV, mid ? 1u : static_cast<cuuint32_t>(kChunkRows),
                             mid ? static_cast<cuuint32_t>(kChunkRows) : 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  *steps_mid = mid;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(p.base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_step_grid(int64_t vocab, int sm_count) {
  const int64_t units = (vocab + kUnit - 1) / kUnit;
  return static_cast<int>(units < sm_count ? units : sm_count);
}

namespace {

// Resident CTAs per SM of one build of the kernel at its launch shape.
template <bool C, bool M, bool T = false, int RW = kHalfRows, bool F = false>
int tc_blocks_per_sm() {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_tc_kernel<C, M, T, RW, F>, kThreads, max_tc_smem()) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return per_sm;
}

}  // namespace

bool tc_cooperative_ok(int grid) {
  int dev = 0, coop = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  // every build a loop may launch (their register counts may differ)
  const int counts[] = {tc_blocks_per_sm<false, false>(),
                        tc_blocks_per_sm<false, true>(),
                        tc_blocks_per_sm<true, false>(),
                        tc_blocks_per_sm<true, true>(),
                        tc_blocks_per_sm<false, true, true>(),
                        tc_blocks_per_sm<false, true, false, 1>(),
                        tc_blocks_per_sm<false, true, false, 4>(),
                        tc_blocks_per_sm<false, false, false, kHalfRows, true>(),
                        tc_blocks_per_sm<false, true, false, kHalfRows, true>(),
                        tc_blocks_per_sm<true, false, false, kHalfRows, true>(),
                        tc_blocks_per_sm<true, true, false, kHalfRows, true>(),
                        tc_blocks_per_sm<false, true, false, 1, true>(),
                        tc_blocks_per_sm<false, true, false, 4, true>()};
  int per_sm = counts[0];
  for (int c : counts) per_sm = c < per_sm ? c : per_sm;
  return coop != 0 && per_sm >= 1 && grid <= per_sm * sms;
}

namespace {
// Whether a cooperative launch may also carry programmatic stream
// serialisation, per device: unknown until the first such launch on it (1
// yes, 0 no, -1 unknown).
constexpr int kCoopMaxDevices = 64;
std::atomic<int> g_coop_pdl[kCoopMaxDevices];
struct CoopPdlInit {
  CoopPdlInit() {
    for (auto& v : g_coop_pdl) v.store(-1, std::memory_order_relaxed);
  }
} g_coop_pdl_init;
}  // namespace

cudaError_t launch_step_tc(const StepParams& p, const CUtensorMap& w2_map, const CUtensorMap& w2_tile_map, int grid,
                           bool pdl, bool cooperative, cudaStream_t stream, bool fp8) {
  CUtensorMap base_map;
  bool steps_mid = false;
  if (!encode_base_map(&base_map, p, &steps_mid)) return cudaErrorInvalidValue;
  const TcLayout L = tc_layout(p.rows, fp8);
  if (L.smem == 0 || (fp8 && !p.w2_scale)) return cudaErrorInvalidValue;
  TcParams tp;
  tp.p = p;
  tp.n = L.n;
  tp.nacc = L.nacc;
  tp.stages = L.stages;
  tp.stages16 = L.stages16;
  tp.nbase = L.nbase;
  tp.tmem_cols = L.tmem_cols;
  tp.res_tiles = L.res_tiles;
  tp.res_col = L.res_col;
  tp.emb_off = L.emb_off;
  tp.w2_off = L.w2_off;
  tp.f16_off = L.f16_off;
  tp.base_off = L.base_off;
  tp.bar_off = L.bar_off;
  tp.row_off = L.row_off;
  tp.queue_off = L.queue_off;
  tp.scale_off = L.scale_off;
  tp.num_units = static_cast<int32_t>((p.vocab + kUnit - 1) / kUnit);
  tp.base_steps_mid = steps_mid ? 1 : 0;

  const bool cap = p.cap != 0.0f;
  const bool one = p.mult == 1.0f;
  auto kernel = cap ? (one ? step_tc_kernel<true, true> : step_tc_kernel<true, false>)
                    : (one ? step_tc_kernel<false, true> : step_tc_kernel<false, false>);
  if (fp8) {
    if (p.test_stall) return cudaErrorNotSupported;
    kernel = cap ? (one ? step_tc_kernel<true, true, false, kHalfRows, true>
                        : step_tc_kernel<true, false, false, kHalfRows, true>)
                 : (one ? step_tc_kernel<false, true, false, kHalfRows, true>
                        : step_tc_kernel<false, false, false, kHalfRows, true>);
    if (p.rows <= 4 && !cap && one)
      kernel = p.rows == 1 ? step_tc_kernel<false, true, false, 1, true> : step_tc_kernel<false, true, false, 4, true>;
  } else if (p.test_stall) {  // the checking aid is built for multiplier 1 without a cap only
    if (cap || !one) return cudaErrorNotSupported;
    kernel = step_tc_kernel<false, true, true>;
  } else if (p.rows <= 4 && !cap && one) {  // few rows: the few-row epilogue
    kernel = p.rows == 1 ? step_tc_kernel<false, true, false, 1> : step_tc_kernel<false, true, false, 4>;
  }
  auto launch = [&](bool with_pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (with_pdl) {
      attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[n].val.programmaticStreamSerializationAllowed = 1;
      ++n;
    }
    if (cooperative) {
      attr[n].id = cudaLaunchAttributeCooperative;
      attr[n].val.cooperative = 1;
      ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, w2_map, w2_tile_map, base_map, tp);
  };
  if (!cooperative || !pdl) return launch(pdl);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kCoopMaxDevices) {
    (void)cudaGetLastError();
    return launch(false);
  }
  std::atomic<int>& known = g_coop_pdl[dev];
  if (known.load(std::memory_order_relaxed) != 0) {
    const cudaError_t e = launch(true);
    if (e == cudaSuccess) {
      known.store(1, std::memory_order_relaxed);
      return e;
    }
    if (known.load(std::memory_order_relaxed) == 1) return e;
    (void)cudaGetLastError();
    known.store(0, std::memory_order_relaxed);
  }
  return launch(false);
}

}  // namespace dspark
