// fp8_quant.cu -- [P1] dsparkQuantizeMarkovW2Fp8: markov_w2 as E4M3 bytes
// with one FP16 scale per row, behind the C ABI of include/dspark_markov.h.
//
// Per row: rowAbsMax over the non-NaN BF16 values, scale = RN(rowAbsMax /
// 448) in FP32 then to FP16 (nearest even, saturating at 65504), and
// q = E4M3(RN(w / scale)) nearest even with saturation to +-448 (NaN stays
// NaN); a row whose scale is 0 stores zeros.  One warp per row, 16-byte
// loads of eight BF16 values a lane.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark_markov.h"

namespace dspark {
namespace {

constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    quantize_w2_fp8_kernel(const uint16_t* __restrict__ w2, uint8_t* __restrict__ q, uint16_t* __restrict__ scale,
                           int64_t vocab, int32_t rank) {
  const int lane = threadIdx.x & 31;
  const int64_t v = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (v >= vocab) return;
  const uint4* row = reinterpret_cast<const uint4*>(w2 + v * rank);
  const int groups = rank / 8;
  float amax = 0.0f;
  for (int g = lane; g < groups; g += 32) {
    const uint4 x = row[g];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[k] & 0xFFFFu)));  // fmaxf drops NaN
      amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[k] >> 16)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const float s32 = __fdiv_rn(amax, 448.0f);
  const uint16_t s16 = s32 >= 65504.0f ? static_cast<uint16_t>(0x7BFF) : __half_as_ushort(__float2half_rn(s32));
  const float s = __half2float(__ushort_as_half(s16));
  if (lane == 0) scale[v] = s16;
  uint2* qrow = reinterpret_cast<uint2*>(q + v * rank);
  for (int g = lane; g < groups; g += 32) {
    const uint4 x = row[g];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t packed[2] = {0u, 0u};
    if (s != 0.0f) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = __nv_cvt_float_to_fp8(__fdiv_rn(bf16_bits_to_float(w[k] & 0xFFFFu), s), __NV_SATFINITE,
                                                  __NV_E4M3);
        const uint32_t hi =
            __nv_cvt_float_to_fp8(__fdiv_rn(bf16_bits_to_float(w[k] >> 16), s), __NV_SATFINITE, __NV_E4M3);
        packed[k >> 1] |= (lo | (hi << 8)) << (16 * (k & 1));
      }
    }
    qrow[g] = make_uint2(packed[0], packed[1]);
  }
}

}  // namespace
}  // namespace dspark

extern "C" int dspark_quantize_w2_fp8(const uint16_t* w2_bf16, uint8_t* w2_fp8, uint16_t* scale_f16, int64_t vocab,
                                      int32_t rank, cudaStream_t stream) {
  if (vocab < 0 || rank < 8 || rank % 8 != 0) return DSPARK_ERR_INVALID_ARG;
  if (vocab == 0) return DSPARK_OK;
  if (!w2_bf16 || !w2_fp8 || !scale_f16) return DSPARK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w2_bf16) & 15u) || (reinterpret_cast<uintptr_t>(w2_fp8) & 7u) ||
      (reinterpret_cast<uintptr_t>(scale_f16) & 1u))
    return DSPARK_ERR_MISALIGNED;
  const int64_t blocks = (vocab + dspark::kRowsPerBlock - 1) / dspark::kRowsPerBlock;
  if (blocks > 0x7FFFFFFF) return DSPARK_ERR_INVALID_ARG;
  dspark::quantize_w2_fp8_kernel<<<static_cast<unsigned>(blocks), 32 * dspark::kRowsPerBlock, 0, stream>>>(
      w2_bf16, w2_fp8, scale_f16, vocab, rank);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
