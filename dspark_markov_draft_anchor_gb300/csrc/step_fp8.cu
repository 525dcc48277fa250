// step_fp8.cu -- the fused Markov step with w2 as E4M3 bytes and one FP16
// scale per row ([P1] dsparkMarkovGreedyFusedStepFp8: the FP8-w2 variant of
// the fused step, hardware fp8x2 -> half2 conversion), with this library's
// sampler and outputs.
//
// The CTA layout is the CUDA-core step's: one CTA of 128 threads per
// 128-entry vocabulary tile and every request row.  The tile's E4M3 rows
// (256 bytes each) are staged in shared memory; each thread decodes its row
// sixteen values at a time and accumulates sum_j e_j * decode(q_j) in FP32
// (any order), then applies the row scale once: bias = RN_bf16(RN(acc *
// scale)).  The epilogue (BF16 add, multiplier, soft cap, cache store,
// Gumbel key, packed argmax, last-arriving CTA) is the CUDA-core step's.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTile = 128;
constexpr int kRowGroup = 16;
constexpr int kQPitch = 272;  // bytes per staged E4M3 row: 256 + 16 (no bank conflicts)

size_t fp8_smem_bytes() {
  return kTile * kQPitch + kRowGroup * kRank * sizeof(float) + kRowGroup * sizeof(RowInfo) +
         kMaxRows * sizeof(unsigned long long);
}

// Sixteen E4M3 values (bytes in id order) as floats, two at a time through
// the hardware conversion to half2 (exact: every E4M3 value is an FP16 value).
__device__ __forceinline__ void decode16(const uint4 w, float* f) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 lo(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] & 0xFFFFu), __NV_E4M3));
    const __half2 hi(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] >> 16), __NV_E4M3));
    const float2 a = __half22float2(lo), b = __half22float2(hi);
    f[4 * k] = a.x;
    f[4 * k + 1] = a.y;
    f[4 * k + 2] = b.x;
    f[4 * k + 3] = b.y;
  }
}

__device__ __forceinline__ void unpack8_bf16(const uint4 w, float* f) {
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
__global__ void __launch_bounds__(128)
    step_fp8_kernel(const StepParams p, const uint8_t* __restrict__ w2q, const uint16_t* __restrict__ w2s) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* qs = smem;
  float* embs = reinterpret_cast<float*>(smem + kTile * kQPitch);
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

  for (int idx = tid; idx < kTile * 16; idx += 128) {
    const int row = idx >> 4, ch = idx & 15;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (v0 + row < p.vocab) val = ldg_nc_v4(w2q + (v0 + row) * kRank + ch * 16);
    *reinterpret_cast<uint4*>(qs + row * kQPitch + ch * 16) = val;
  }
  const float scale = in ? __half2float(__ushort_as_half(w2s[v])) : 0.0f;
  for (int r = tid; r < p.rows; r += 128) best[r] = 0ull;

  const uint64_t last_row = static_cast<uint64_t>(p.w1_rows - 1);
  for (int rg = 0; rg < p.rows; rg += kRowGroup) {
    const int nr = min(kRowGroup, p.rows - rg);
    for (int idx = tid; idx < nr * 32; idx += 128) {
      const int i = idx >> 5, ch = idx & 31;
      const int64_t tok = slot_token(__ldcg(p.slots_prev + rg + i));
      const uint64_t row = static_cast<uint64_t>(tok) < last_row ? static_cast<uint64_t>(tok) : last_row;
      float f[8];
      unpack8_bf16(ldg_nc_v4(p.w1 + row * kRank + ch * 8), f);
      float4* e = reinterpret_cast<float4*>(embs + i * kRank + ch * 8);
      e[0] = make_float4(f[0], f[1], f[2], f[3]);
      e[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    if (tid < nr) infos[tid] = row_info(p, rg + tid);
    __syncthreads();

    float acc[kRowGroup];
#pragma unroll
    for (int i = 0; i < kRowGroup; ++i) acc[i] = 0.0f;
    const unsigned char* qrow = qs + tid * kQPitch;
    for (int ch = 0; ch < 16; ++ch) {
      float w[16];
      decode16(*reinterpret_cast<const uint4*>(qrow + ch * 16), w);
#pragma unroll
      for (int i = 0; i < kRowGroup; ++i) {
        if (i < nr) {
          const float* e = embs + i * kRank + ch * 16;
          float a = acc[i];
#pragma unroll
          for (int k = 0; k < 16; k += 4) {
            const float4 ek = *reinterpret_cast<const float4*>(e + k);
            a = __fmaf_rn(w[k], ek.x, a);
            a = __fmaf_rn(w[k + 1], ek.y, a);
            a = __fmaf_rn(w[k + 2], ek.z, a);
            a = __fmaf_rn(w[k + 3], ek.w, a);
          }
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
          const __nv_bfloat16 b16 = __float2bfloat16_rn(__fmul_rn(acc[i], scale));
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

}  // namespace

cudaError_t setup_step_fp8() {
  const int smem = static_cast<int>(fp8_smem_bytes());
  cudaError_t e = cudaFuncSetAttribute(step_fp8_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(step_fp8_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_step_fp8(const StepParams& p, const uint8_t* w2q, const uint16_t* w2s, bool has_cap, bool pdl,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(simple_step_grid(p.vocab));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = fp8_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (has_cap) return cudaLaunchKernelEx(&cfg, step_fp8_kernel<true>, p, w2q, w2s);
  return cudaLaunchKernelEx(&cfg, step_fp8_kernel<false>, p, w2q, w2s);
}

}  // namespace dspark
