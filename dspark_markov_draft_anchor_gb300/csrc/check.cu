// check.cu -- elementwise kernels over the step kernel's own device functions
// (include/dspark_markov_check.h), for exhaustive bit-exact tests.
#include <cuda_runtime.h>

#include "dspark_markov.h"
#include "dspark_markov_check.h"
#include "kernels.h"
#include "markov_math.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t n) {
  const int64_t g = (n + kThreads - 1) / kThreads;
  return static_cast<int>(g < 152 * 64 ? g : 152 * 64);
}

#define GRID_STRIDE(i, n) \
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < (n); \
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)

__global__ void noise_range_kernel(uint32_t h0, float* L, int64_t n) {
  GRID_STRIDE(i, n) { L[i] = noise_L(h0 + static_cast<uint32_t>(i)); }
}

__global__ void hash_kernel(uint64_t seed, int32_t step, int64_t pos, uint32_t salt, const uint32_t* ids,
                            uint32_t* out, int64_t n) {
  const uint32_t prefix = murmur_prefix(seed, step, pos, salt);
  GRID_STRIDE(i, n) { out[i] = murmur_finish(prefix, ids[i]); }
}

template <bool kHasCap>
__global__ void logit_kernel(const uint16_t* base, const uint16_t* bias, uint16_t* c, float* l, int64_t n,
                             float mult, float inv_cap, float cap) {
  GRID_STRIDE(i, n) {
    float lv;
    c[i] = transform_logit<kHasCap>(bf16_bits_to_float(base[i]), bf16_bits_to_float(bias[i]), mult, inv_cap,
                                    cap, &lv);
    l[i] = lv;
  }
}

__global__ void key_kernel(const float* l, float temp, const uint32_t* h, float* key, int64_t n) {
  GRID_STRIDE(i, n) { key[i] = temp != 0.0f ? noised_key(l[i], temp, h[i]) : l[i]; }
}

__global__ void logf_kernel(const float* x, float* y, int64_t n) {
  GRID_STRIDE(i, n) { y[i] = own_logf(x[i]); }
}

__global__ void tanhf_kernel(const float* x, float* y, int64_t n) {
  GRID_STRIDE(i, n) { y[i] = own_tanhf(x[i]); }
}

__global__ void expf_kernel(const float* x, float* y, int64_t n) {
  GRID_STRIDE(i, n) { y[i] = own_exp_nonpos(x[i]); }
}

__global__ void div_kernel(const float* x, float d, float* y, int64_t n) {
  const Divider D = make_divider(d);
  GRID_STRIDE(i, n) { y[i] = div_rn(x[i], D); }
}

// Every float x with bits in [lo, lo + n): count the x whose div_rn(x, d)
// differs in its bits from the IEEE quotient (two NaNs count as equal) and
// keep the smallest such bit pattern.
__global__ void div_sweep_kernel(float d, uint32_t lo, int64_t n, unsigned long long* out) {
  const Divider D = make_divider(d);
  unsigned long long bad = 0;
  uint32_t first = 0xFFFFFFFFu;
  GRID_STRIDE(i, n) {
    const uint32_t b = lo + static_cast<uint32_t>(i);
    const float x = __uint_as_float(b);
    const float got = div_rn(x, D), want = __fdiv_rn(x, d);
    if (__float_as_uint(got) != __float_as_uint(want) && !(got != got && want != want)) {
      ++bad;
      first = b < first ? b : first;
    }
  }
  if (bad) {
    atomicAdd(out, bad);
    atomicMin(out + 1, static_cast<unsigned long long>(first));
  }
}

int done() { return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

}  // namespace
}  // namespace dspark

extern "C" {

int dspark_check_noise_range(uint32_t h0, float* L, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && !L)) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::noise_range_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(h0, L, n);
  return dspark::done();
}

int dspark_check_hash(int64_t seed, int32_t step, int64_t pos, uint32_t salt, const uint32_t* ids, uint32_t* out,
                      int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!ids || !out))) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::hash_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(static_cast<uint64_t>(seed), step, pos,
                                                                           salt, ids, out, n);
  return dspark::done();
}

int dspark_check_logit(const uint16_t* base, const uint16_t* bias, uint16_t* c, float* l, int64_t n, float mult,
                       float cap, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!base || !bias || !c || !l))) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  const float inv_cap = cap != 0.0f ? 1.0f / cap : 0.0f;
  if (cap != 0.0f)
    dspark::logit_kernel<true><<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(base, bias, c, l, n, mult,
                                                                                     inv_cap, cap);
  else
    dspark::logit_kernel<false><<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(base, bias, c, l, n, mult,
                                                                                      inv_cap, cap);
  return dspark::done();
}

int dspark_check_key(const float* l, float temp, const uint32_t* h, float* key, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!l || !h || !key))) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::key_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(l, temp, h, key, n);
  return dspark::done();
}

int dspark_check_logf(const float* x, float* y, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::logf_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(x, y, n);
  return dspark::done();
}

int dspark_check_tanhf(const float* x, float* y, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::tanhf_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(x, y, n);
  return dspark::done();
}

int dspark_check_expf(const float* x, float* y, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::expf_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(x, y, n);
  return dspark::done();
}

int dspark_check_div(const float* x, float d, float* y, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::div_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(x, d, y, n);
  return dspark::done();
}

int dspark_check_div_sweep(float d, uint32_t lo, int64_t n, unsigned long long* out, cudaStream_t stream) {
  if (n < 0 || n > (int64_t{1} << 32) || !out) return DSPARK_ERR_INVALID_ARG;
  if (n == 0) return DSPARK_OK;
  dspark::div_sweep_kernel<<<dspark::grid_for(n), dspark::kThreads, 0, stream>>>(d, lo, n, out);
  return dspark::done();
}

int dspark_noise_bound_tables(float* ub, float* lb, int32_t n) {
  if (!ub || !lb || n < dspark::kNoiseBuckets) return DSPARK_ERR_INVALID_ARG;
  dspark::noise_bound_tables(ub, lb);
  return dspark::kNoiseBuckets;
}

}  // extern "C"
