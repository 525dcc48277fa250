// step_simple.cu -- the anchor kernel and a straightforward fused Markov step.
//
// The step kernel gives one CTA of 128 threads a 128-entry vocabulary tile and
// every request row.  It stages the tile's w2 rows in shared memory, gathers
// the rows' w1 embeddings (their previous tokens clamped to the last w1 row),
// forms the bias with FP32 FMAs (one vocab entry per thread), and runs the
// per-element epilogue: BF16 add, multiplier, soft cap, cache store, Gumbel
// key ([P3] _StepKernel.kernel, _logit, _gumbel).  The row's argmax is a
// 64-bit packed-key maximum: per warp by shuffles, per CTA in shared memory,
// over the grid by one atomicMax per row; the last CTA to arrive writes the
// step's tokens ([P3] _finish; [P1] dsparkMarkovGreedyFusedStep's packed
// orderable key).  It is the portable reference path of the library; the
// tensor-core step kernel is the fast one.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTile = 128;
constexpr int kRowGroup = 16;
constexpr int kW2Pitch = 528;  // bytes per staged w2 row: 512 + 16 (no bank conflicts)

__global__ void anchor_kernel(const int32_t* __restrict__ input_ids, const int64_t* __restrict__ anchor_idx,
                              unsigned long long* __restrict__ slots, unsigned int* __restrict__ counters,
                              unsigned int* __restrict__ abort_word, int rows, int steps, int max_rows) {
  // The next kernel (a step launched with programmatic dependent launch) may
  // start its prologue and its w2 prefetch now; it reads what this kernel
  // writes only after griddepcontrol.wait, which waits for this grid.
  pdl_launch_dependents();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < rows) {
    const int32_t token = input_ids[anchor_idx[r]];
    slots[r] = static_cast<unsigned long long>(~static_cast<uint32_t>(token));
    for (int s = 1; s <= steps; ++s) slots[static_cast<int64_t>(s) * max_rows + r] = 0ull;
  }
  if (blockIdx.x == 0) {
    for (int s = threadIdx.x; s < steps; s += blockDim.x) counters[s] = 0u;
    if (threadIdx.x == 0) *abort_word = 0u;
  }
}

// The soft-capped transform of every BF16 sum (bits i): the step kernels'
// epilogue looks the cached value up instead of evaluating tanh per element.
__global__ void xform_lut_kernel(uint16_t* __restrict__ lut, float mult, float inv_cap, float cap) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 65536) {
    float l;
    lut[i] = transform_sum<true>(bf16_bits_to_float(static_cast<uint32_t>(i)), mult, inv_cap, cap, &l);
  }
}

__device__ __forceinline__ void unpack8(const uint4 w, float* f) {
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  f[4] = __uint_as_float(w.z << 16);
  f[5] = __uint_as_float(w.z & 0xFFFF0000u);
  f[6] = __uint_as_float(w.w << 16);
  f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

template <bool kHasCap>
__global__ void __launch_bounds__(128) step_simple_kernel(const StepParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* w2s = smem;
  float* embs = reinterpret_cast<float*>(smem + kTile * kW2Pitch);
  RowInfo* infos = reinterpret_cast<RowInfo*>(embs + kRowGroup * kRank);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(infos + kRowGroup);
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int64_t v = v0 + tid;
  const bool in = v < p.vocab;

  // Everything below reads the previous step's slots or writes outputs.
  pdl_wait();

  for (int idx = tid; idx < kTile * 32; idx += 128) {
    const int row = idx >> 5, ch = idx & 31;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (v0 + row < p.vocab) val = ldg_nc_v4(p.w2 + (v0 + row) * kRank + ch * 8);
    *reinterpret_cast<uint4*>(w2s + row * kW2Pitch + ch * 16) = val;
  }
  for (int r = tid; r < p.rows; r += 128) best[r] = 0ull;

  const uint64_t last_row = static_cast<uint64_t>(p.w1_rows - 1);
  for (int rg = 0; rg < p.rows; rg += kRowGroup) {
    const int nr = min(kRowGroup, p.rows - rg);
    for (int idx = tid; idx < nr * 32; idx += 128) {
      const int i = idx >> 5, ch = idx & 31;
      const int64_t tok = slot_token(__ldcg(p.slots_prev + rg + i));
      const uint64_t row = static_cast<uint64_t>(tok) < last_row ? static_cast<uint64_t>(tok) : last_row;
      float f[8];
      unpack8(ldg_nc_v4(p.w1 + row * kRank + ch * 8), f);
      float4* e = reinterpret_cast<float4*>(embs + i * kRank + ch * 8);
      e[0] = make_float4(f[0], f[1], f[2], f[3]);
      e[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    if (tid < nr) infos[tid] = row_info(p, rg + tid);
    __syncthreads();

    float acc[kRowGroup];
#pragma unroll
    for (int i = 0; i < kRowGroup; ++i) acc[i] = 0.0f;
    const unsigned char* wrow = w2s + tid * kW2Pitch;
    for (int ch = 0; ch < 32; ++ch) {
      float w[8];
      unpack8(*reinterpret_cast<const uint4*>(wrow + ch * 16), w);
#pragma unroll
      for (int i = 0; i < kRowGroup; ++i) {
        if (i < nr) {
          const float4 e0 = *reinterpret_cast<const float4*>(embs + i * kRank + ch * 8);
          const float4 e1 = *reinterpret_cast<const float4*>(embs + i * kRank + ch * 8 + 4);
          float a = acc[i];
          a = __fmaf_rn(w[0], e0.x, a);
          a = __fmaf_rn(w[1], e0.y, a);
          a = __fmaf_rn(w[2], e0.z, a);
          a = __fmaf_rn(w[3], e0.w, a);
          a = __fmaf_rn(w[4], e1.x, a);
          a = __fmaf_rn(w[5], e1.y, a);
          a = __fmaf_rn(w[6], e1.z, a);
          a = __fmaf_rn(w[7], e1.w, a);
          acc[i] = a;
        }
      }
    }

#pragma unroll
    for (int i = 0; i < kRowGroup; ++i) {
      if (i < nr) {
        const int r = rg + i;
        const RowInfo ri = infos[i];
        unsigned long long cand = 0ull;
        if (in) {
          const __nv_bfloat16 b16 = __float2bfloat16_rn(acc[i]);
          if (p.bias_out)
            p.bias_out[(static_cast<int64_t>(r) * p.steps + p.step) * p.vocab + v] = __bfloat16_as_ushort(b16);
          const float basef = bf16_bits_to_float(p.base[static_cast<int64_t>(r) * p.base_s0 + v]);
          float l;
          const uint16_t c = transform_logit<kHasCap>(basef, __bfloat162float(b16), p.mult, p.inv_cap, p.cap, &l);
          if (ri.valid) p.cache[ri.cache_off + v] = c;
          float key = l;
          if (ri.temp != 0.0f) key = noised_key(l, ri.temp, murmur_finish(ri.prefix, static_cast<uint32_t>(v)));
          cand = pack_key(key, static_cast<uint32_t>(v));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, cand, off);
          cand = o > cand ? o : cand;
        }
        if (lane == 0) atomicMax(&best[r], cand);
      }
    }
    __syncthreads();
  }

  if (p.partials) {  // the select launch reduces the CTAs' maxima
    for (int r = tid; r < p.rows; r += 128)
      p.partials[static_cast<int64_t>(r) * gridDim.x + blockIdx.x] = best[r];
    return;
  }
  for (int r = tid; r < p.rows; r += 128) atomicMax(p.slots_out + r, best[r]);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int r = tid; r < p.rows; r += 128) {
      const unsigned long long sv = atomicAdd(p.slots_out + r, 0ull);
      p.tokens[static_cast<int64_t>(r) * p.tokens_s0 + p.step] = slot_token(sv);
    }
  }
}

// Select ([P2] _markov_select_kernel): one CTA per row reduces the row's
// per-CTA packed maxima under the total order (the u64 maximum: first NaN,
// else the lowest id of the largest key), then writes the step's token and
// the next step's previous token.
__global__ void __launch_bounds__(256) select_kernel(const unsigned long long* __restrict__ partials, int nparts,
                                                     unsigned long long* __restrict__ slots_out,
                                                     int64_t* __restrict__ tokens, int64_t tokens_s0, int step) {
  __shared__ unsigned long long s_warp[8];
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const unsigned long long* row = partials + static_cast<int64_t>(r) * nparts;
  unsigned long long m = 0ull;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
    const unsigned long long x = row[i];
    m = x > m ? x : m;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, m, off);
    m = o > m ? o : m;
  }
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = s_warp[w] > m ? s_warp[w] : m;
    slots_out[r] = m;
    tokens[static_cast<int64_t>(r) * tokens_s0 + step] = slot_token(m);
  }
}

size_t simple_smem_bytes() {
  return kTile * kW2Pitch + kRowGroup * kRank * sizeof(float) + kRowGroup * sizeof(RowInfo) +
         kMaxRows * sizeof(unsigned long long);
}

}  // namespace

cudaError_t launch_anchor(const int32_t* input_ids, const int64_t* anchor_idx, unsigned long long* slots,
                          unsigned int* counters, unsigned int* abort_word, int rows, int steps, int max_rows,
                          cudaStream_t stream) {
  anchor_kernel<<<(rows + 127) / 128, 128, 0, stream>>>(input_ids, anchor_idx, slots, counters, abort_word, rows,
                                                         steps, max_rows);
  return cudaGetLastError();
}

cudaError_t launch_xform_lut(uint16_t* lut, float mult, float cap, cudaStream_t stream) {
  xform_lut_kernel<<<256, 256, 0, stream>>>(lut, mult, cap != 0.0f ? 1.0f / cap : 0.0f, cap);
  return cudaGetLastError();
}

int simple_step_grid(int64_t vocab) { return static_cast<int>((vocab + kTile - 1) / kTile); }

cudaError_t launch_select(const unsigned long long* partials, int nparts, unsigned long long* slots_out,
                          int64_t* tokens, int64_t tokens_s0, int step, int rows, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, select_kernel, partials, nparts, slots_out, tokens, tokens_s0, step);
}

cudaError_t setup_step_simple() {
  const int smem = static_cast<int>(simple_smem_bytes());
  cudaError_t e = cudaFuncSetAttribute(step_simple_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(step_simple_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_step_simple(const StepParams& p, bool has_cap, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(simple_step_grid(p.vocab));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = simple_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (has_cap) return cudaLaunchKernelEx(&cfg, step_simple_kernel<true>, p);
  return cudaLaunchKernelEx(&cfg, step_simple_kernel<false>, p);
}

}  // namespace dspark
