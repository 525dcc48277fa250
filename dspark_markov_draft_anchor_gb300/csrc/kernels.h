// kernels.h -- host-side launchers of the library's kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "step_common.cuh"

namespace dspark {

// Anchor: slots_prev row 0 <- the anchor tokens, later step slots and the
// arrival counters cleared ([P3] anchor_embed, _AnchorKernel).
cudaError_t launch_anchor(const int32_t* input_ids, const int64_t* anchor_idx, unsigned long long* slots,
                          unsigned int* counters, unsigned int* abort_word, int rows, int steps, int max_rows,
                          cudaStream_t stream);

// The soft-capped transform of all 65536 BF16 sums into lut (cap != 0).
cudaError_t launch_xform_lut(uint16_t* lut, float mult, float cap, cudaStream_t stream);

// Two-launch select: reduce each row's per-CTA maxima (partials [rows,
// nparts]) into slots_out and tokens[:, step] (one CTA per row).
cudaError_t launch_select(const unsigned long long* partials, int nparts, unsigned long long* slots_out,
                          int64_t* tokens, int64_t tokens_s0, int step, int rows, bool pdl, cudaStream_t stream);

// Sharded loop: the winner of the gathered packets [tp, rows, 4] per row
// (one warp a row) into tokens[:, step] and slot_next.
cudaError_t launch_pick(const int32_t* packets, int tp, int rows, int64_t* tokens, int64_t tokens_s0, int step,
                        unsigned long long* slot_next, cudaStream_t stream);

// Simple fused step: one CTA per 128-entry vocabulary tile, FP32 FMA bias.
int simple_step_grid(int64_t vocab);
cudaError_t setup_step_simple();
cudaError_t launch_step_simple(const StepParams& p, bool has_cap, bool pdl, cudaStream_t stream);

// The same step with w2 as E4M3 bytes [V, 256] and FP16 row scales [V]
// (CUDA-core FMA bias, the scale applied to each row's sum).
cudaError_t setup_step_fp8();
cudaError_t launch_step_fp8(const StepParams& p, const uint8_t* w2q, const uint16_t* w2s, bool has_cap, bool pdl,
                            cudaStream_t stream);

// Tensor-core fused step: persistent CTAs over vocabulary ranges, TMA-fed w2
// and base, tcgen05 bias into TMEM.
cudaError_t setup_step_tc();
int tc_step_grid(int64_t vocab, int sm_count);
int tc_smem_bytes(int rows);
// box_rows: 32 (any tile) or 128 (whole tiles, one copy per stage).
bool encode_w2_map(CUtensorMap* map, const void* w2, int64_t vocab, int box_rows);
// The same over E4M3 w2 [V, 256] bytes: boxes of 128 K bytes x box_rows.
bool encode_w2_fp8_map(CUtensorMap* map, const void* w2_fp8, int64_t vocab, int box_rows);
// The most rows the tensor-core step takes with E4M3 w2 (its shared memory
// holds the FP16 operand stages beside the E4M3 ones).
int tc_fp8_max_rows();
// Steps p.step .. p.step_end - 1 in one launch; more than one step needs a
// cooperative launch (its CTAs wait for one another between steps).  With
// fp8 the maps are E4M3 maps (encode_w2_fp8_map) and p.w2_scale is set.
// Returns cudaErrorInvalidValue, launching nothing, when the base logits'
// strides cannot form the kernel's tensor map or the rows do not fit.
cudaError_t launch_step_tc(const StepParams& p, const CUtensorMap& w2_map, const CUtensorMap& w2_tile_map, int grid,
                           bool pdl, bool cooperative, cudaStream_t stream, bool fp8 = false);
// The grid's CTAs can all be resident at once (a cooperative launch is possible).
bool tc_cooperative_ok(int grid);

// The unique id of the calling thread's current CUDA context (a driver
// context id, never reused within a process), or 0 when no context is
// current or the driver cannot say.  One-time set-up that lives in a context
// (a kernel attribute, a looked-up symbol address) is keyed on it, so that a
// device reset or a new context makes the next call redo it.
unsigned long long current_context_id();

// Bounds of the Gumbel noise -L(h) used to skip elements that cannot win:
// bucket 16 k + m of g = h | 1 (k: the position of g's leading one, m: the
// 4 bits after it); ub[b] >= -L(h) >= lb[b] for every h of bucket b (host
// code, no GPU).
constexpr int kNoiseBuckets = 32 * 16;
void noise_bound_tables(float* ub, float* lb);

}  // namespace dspark
