// step_common.cuh -- parameters and small device helpers shared by the
// anchor and step kernels of the Markov loop.
#pragma once

#include <stdint.h>

#include "markov_math.cuh"

namespace dspark {

constexpr int kRank = 256;           // Markov rank supported by the kernels
constexpr int kMaxRows = 256;        // rows per loop call
constexpr int kMaxSteps = 64;        // draft steps per loop call

// Device status codes (mirrors of the DSPARK_ERR_* values).
constexpr int kStatusTimeout = -7;

// Everything one step launch needs.  Strides are in elements.
struct StepParams {
  const uint16_t* w1;   // [w1_rows, 256] BF16
  const uint16_t* w2;   // [V, 256] BF16
  const uint16_t* base; // base logits, step column already applied: base + step*base_s1
  int64_t base_s0;
  uint16_t* cache;      // cache, step column already applied: cache + step*cache_s1 (or null)
  int64_t cache_s0;
  const int64_t* req_idx;  // [rows, steps] or null
  int64_t req_s0;
  const int64_t* sample_pos;
  int64_t pos_s0;
  int64_t num_req;
  const int64_t* seeds;
  const float* temperature;
  int64_t* tokens;
  int64_t tokens_s0;
  uint16_t* bias_out;   // [rows, steps, V] or null; step applied by the kernel
  const unsigned long long* slots_prev;  // [rows] previous token (packed)
  unsigned long long* slots_out;         // [rows] this step's packed argmax
  unsigned int* counter;                 // this step's arrival counter
  int* status;
  int64_t vocab;
  int64_t w1_rows;
  int32_t rows;
  int32_t steps;
  int32_t step;
  float mult;
  float inv_cap;
  float cap;
  uint32_t salt;
  int32_t finish;      // this launch writes its own tokens (the last CTA to arrive)
  int32_t write_prev;  // CTA 0 writes the previous step's tokens from slots_prev
  // Several steps in one launch (the tensor-core kernel only): steps
  // step .. step_end - 1; step j's base, cache, slots and counter are those of
  // `step` advanced by (j - step) times the strides below.
  int32_t step_end;
  int64_t base_s1;
  int64_t cache_s1;
  int64_t slots_s;            // elements between consecutive steps' argmax slots
  unsigned int* abort_word;   // set by a CTA whose bounded wait gave up; cleared by the anchor kernel
  // Two-launch select: each CTA writes its row maxima to partials[r * grid +
  // block] and a separate select launch reduces them (null: one atomicMax per
  // row into slots_out).
  unsigned long long* partials;
  int32_t test_stall;  // checking aid (host side: picks the kernel whose first grid wait cannot end)
  // With a soft cap: the cached BF16 of every BF16 sum x (x's bits index it),
  // built by the anchor for this call's multiplier and cap.
  const uint16_t* xform_lut;
  // E4M3 w2 on the tensor-core step: the FP16 row scales [V] (else null).
  const uint16_t* w2_scale;
  // One rank of a vocabulary-sharded loop ([P3] markov_step with a
  // vocab-parallel w2): the step covers global ids vocab_offset .. +vocab-1
  // (the noise hashes the global id), the cache is rank-local [rows, steps,
  // shard] indexed by row and written for every row, and the launch's last
  // CTA writes packets[r * 4 .. +3] = (key bits, global id, 0, 0) instead of
  // the token (tensor-core step, one step per launch).
  int32_t sharded;
  int64_t vocab_offset;
  int32_t* packets;
  // One-launch loop without the anchor launch: step 0's previous tokens are
  // read from input_ids[anchor_idx[r]], and the loop leaves its slots and
  // counters zero for the next call (the last CTA to arrive at step j >= 1
  // clears step j - 1's counter and the slots step j read; at the last step
  // it clears the rest after writing the tokens).
  int32_t self_reset;
  const int32_t* input_ids;
  const int64_t* anchor_idx;
};

// PTX griddepcontrol (programmatic dependent launch): wait for the grids this
// one depends on to complete and flush; a no-op without a dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Per-row, per-step sampling state ([P3] _StepKernel.kernel): request,
// validity, temperature, seed and the Murmur3 prefix.
struct RowInfo {
  uint32_t prefix;
  float temp;
  int32_t valid;
  int32_t pad;
  int64_t cache_off;  // req * cache_s0 (valid rows)
};

__device__ __forceinline__ RowInfo row_info(const StepParams& p, int r, int step) {
  RowInfo ri;
  const int64_t req = p.req_idx ? p.req_idx[static_cast<int64_t>(r) * p.req_s0 + step] : r;
  const bool valid = req >= 0 && req < p.num_req;
  const float temp = valid ? p.temperature[req] : 0.0f;
  const uint64_t seed = valid ? static_cast<uint64_t>(p.seeds[req]) : 0ull;
  const int64_t pos = p.sample_pos[static_cast<int64_t>(r) * p.pos_s0 + step];
  ri.prefix = murmur_prefix(seed, step, pos, p.salt);
  ri.temp = temp;
  if (p.sharded) {  // a rank-local cache row per request row, written whatever the row's request
    ri.valid = p.cache != nullptr;
    ri.cache_off = static_cast<int64_t>(r) * p.cache_s0;
  } else {
    ri.valid = valid && p.cache != nullptr;
    ri.cache_off = valid ? req * p.cache_s0 : 0;
  }
  ri.pad = 0;
  return ri;
}

__device__ __forceinline__ RowInfo row_info(const StepParams& p, int r) { return row_info(p, r, p.step); }

}  // namespace dspark
