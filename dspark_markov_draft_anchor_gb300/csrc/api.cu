// api.cu -- the C ABI of libdspark_markov.so (declared in include/dspark_markov.h):
// argument validation, the context's scratch, and the launch sequence of the
// Markov loop ([P2] FusedMarkov.run; [P3] anchor_embed + markov_step).
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "dspark_markov.h"
#include "kernels.h"

struct dspark_markov_ctx {
  int device;
  int sm_count;
  dspark_markov_config cfg;
  const uint16_t* w1;
  const uint16_t* w2;
  unsigned long long* slots;  // [(max_steps + 1) * max_rows] packed argmax slots
  unsigned int* counters;     // [max_steps] arrival counters, then the loop's abort word
  unsigned long long* partials;  // [max_rows, max grid] per-CTA maxima of the two-launch select
  uint16_t* xform_lut;           // [65536] soft-capped transform of every BF16 sum (per call)
  int* status;                // device status word
  int grid_simple;
  int grid_tc;
  bool tc_ok;                 // tensor-core step available (tensor map encoded)
  bool fused_ok;              // the tensor-core kernel may run several steps in one cooperative launch
  CUtensorMap w2_map;         // TMA map over w2: boxes of 32 rows x 64 K, 128-byte swizzle
  CUtensorMap w2_tile_map;    // the same with boxes of 128 rows (whole vocabulary tiles)
  const uint8_t* w2_fp8;      // E4M3 w2 [V, 256] (caller-owned) or null: when set, every step takes
  const uint16_t* w2_scale;   // its bias from it and these FP16 row scales [V]
  bool tc8_ok;                // TMA maps over the E4M3 w2 encoded: the tensor-core step can read it
  CUtensorMap w2f8_map;       // boxes of 32 rows x 128 K bytes, 128-byte swizzle
  CUtensorMap w2f8_tile_map;  // the same with boxes of 128 rows
  // The slots, counters and abort word are as the anchor leaves them (zero):
  // a one-launch loop then needs no anchor launch, and leaves them so again.
  // Any other launch on them, or a reported device error, clears this.
  bool state_clean;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rows up to which the CUDA-core kernel forms the bias by default; above,
// tensor cores.  Zero: the tensor-core loop is faster at every row count on
// sm_103a (its MMA pipe idles most of a step, so padding the rows to N = 16
// costs nothing, and it streams w2 through a pipelined persistent launch).
constexpr int kFmaMaxRows = 0;

// The TMA-fed kernel reads base rows as tensor tiles: 16-byte aligned rows.
bool tma_base_ok(const dspark_markov_loop_args* a) {
  return aligned16(a->base) && (a->base_s0 % 8) == 0 && (a->base_s1 % 8) == 0;
}

int check_args(const dspark_markov_ctx* ctx, const dspark_markov_loop_args* a) {
  if (!ctx || !a) return DSPARK_ERR_INVALID_ARG;
  if (a->rows < 1 || a->steps < 1) return DSPARK_ERR_INVALID_ARG;
  if (a->rows > ctx->cfg.max_rows || a->steps > ctx->cfg.max_steps) return DSPARK_ERR_TOO_MANY_ROWS;
  if (!a->base || !a->input_ids || !a->anchor_idx || !a->sample_pos || !a->tokens) return DSPARK_ERR_INVALID_ARG;
  if (a->num_req < 0 || (a->num_req > 0 && (!a->seeds || !a->temperature))) return DSPARK_ERR_INVALID_ARG;
  if (!isfinite(a->mult) || !isfinite(a->cap)) return DSPARK_ERR_INVALID_ARG;
  if (a->base_s0 < 0 || a->base_s1 < 0 || a->tokens_s0 < a->steps || a->pos_s0 < a->steps)
    return DSPARK_ERR_INVALID_ARG;
  if (a->req_idx && a->req_s0 < a->steps) return DSPARK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a->base) & 1u) return DSPARK_ERR_MISALIGNED;
  if (a->cache) {
    if (a->cache_s0 < 0 || a->cache_s1 < 0) return DSPARK_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(a->cache) & 1u) return DSPARK_ERR_MISALIGNED;
  }
  return DSPARK_OK;
}

dspark::StepParams make_params(const dspark_markov_ctx* ctx, const dspark_markov_loop_args* a, int step) {
  dspark::StepParams p;
  p.w1 = ctx->w1;
  p.w2 = ctx->w2;
  p.base = static_cast<const uint16_t*>(a->base) + static_cast<int64_t>(step) * a->base_s1;
  p.base_s0 = a->base_s0;
  p.cache = a->cache ? static_cast<uint16_t*>(a->cache) + static_cast<int64_t>(step) * a->cache_s1 : nullptr;
  p.cache_s0 = a->cache_s0;
  p.req_idx = a->req_idx;
  p.req_s0 = a->req_s0;
  p.sample_pos = a->sample_pos;
  p.pos_s0 = a->pos_s0;
  p.num_req = a->num_req;
  p.seeds = a->seeds;
  p.temperature = a->temperature;
  p.tokens = a->tokens;
  p.tokens_s0 = a->tokens_s0;
  p.bias_out = static_cast<uint16_t*>(a->bias_out);
  const int64_t mr = ctx->cfg.max_rows;
  p.slots_prev = ctx->slots + static_cast<int64_t>(step) * mr;
  p.slots_out = ctx->slots + static_cast<int64_t>(step + 1) * mr;
  p.counter = ctx->counters + step;
  p.status = ctx->status;
  p.vocab = ctx->cfg.vocab;
  p.w1_rows = ctx->cfg.w1_rows;
  p.rows = a->rows;
  p.steps = a->steps;
  p.step = step;
  p.mult = a->mult;
  p.cap = a->cap;
  p.inv_cap = a->cap != 0.0f ? 1.0f / a->cap : 0.0f;
  p.salt = a->salt;
  p.finish = 1;
  p.write_prev = 0;
  p.step_end = step + 1;
  p.base_s1 = a->base_s1;
  p.cache_s1 = a->cache_s1;
  p.slots_s = mr;
  p.abort_word = ctx->counters + ctx->cfg.max_steps;
  p.partials = nullptr;
  p.test_stall = (ctx->cfg.flags & DSPARK_FLAG_TEST_STALL) != 0;
  p.xform_lut = ctx->xform_lut;
  p.w2_scale = nullptr;
  p.sharded = 0;
  p.vocab_offset = 0;
  p.packets = nullptr;
  p.self_reset = 0;
  p.input_ids = a->input_ids;
  p.anchor_idx = a->anchor_idx;
  return p;
}

}  // namespace

namespace dspark {

unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  struct Fns {
    GetCurrentFn get_current = nullptr;
    GetIdFn get_id = nullptr;
  };
  // looked up once (a function-local static is initialised by one thread)
  static const Fns fns = [] {
    Fns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<GetIdFn>(p);
    (void)cudaGetLastError();
    return f;
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!fns.get_current || !fns.get_id || fns.get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      fns.get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

}  // namespace dspark

extern "C" {

const char* dspark_strerror(int code) {
  switch (code) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID_ARG: return "invalid argument";
    case DSPARK_ERR_UNSUPPORTED_RANK: return "unsupported Markov rank (256 only)";
    case DSPARK_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case DSPARK_ERR_TOO_MANY_ROWS: return "rows or steps above the context's maximum";
    case DSPARK_ERR_CAPTURING: return "stream is capturing (init allocates)";
    case DSPARK_ERR_CUDA: return "CUDA error";
    case DSPARK_ERR_DEVICE_TIMEOUT: return "a bounded device wait gave up";
    case DSPARK_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (GB300)";
    case DSPARK_ERR_HOST_ALLOC: return "host memory allocation failed";
    default: return "unknown error";
  }
}

int dspark_markov_init(dspark_markov_ctx** out, const dspark_markov_config* cfg, const void* w1_bf16,
                       const void* w2_bf16, cudaStream_t stream) {
  if (!out || !cfg || !w1_bf16 || !w2_bf16) return DSPARK_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->rank != dspark::kRank) return DSPARK_ERR_UNSUPPORTED_RANK;
  if (cfg->vocab < 1 || cfg->w1_rows < 1) return DSPARK_ERR_INVALID_ARG;
  if (cfg->max_rows < 1 || cfg->max_rows > dspark::kMaxRows) return DSPARK_ERR_TOO_MANY_ROWS;
  if (cfg->max_steps < 1 || cfg->max_steps > dspark::kMaxSteps) return DSPARK_ERR_TOO_MANY_ROWS;
  if (!aligned16(w1_bf16) || !aligned16(w2_bf16)) return DSPARK_ERR_MISALIGNED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return DSPARK_ERR_CAPTURING;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (major != 10 || minor != 3) return DSPARK_ERR_UNSUPPORTED_DEVICE;
  if (dspark::setup_step_simple() != cudaSuccess || dspark::setup_step_fp8() != cudaSuccess) return DSPARK_ERR_CUDA;
  const bool tc_setup = dspark::setup_step_tc() == cudaSuccess;
  (void)cudaGetLastError();

  dspark_markov_ctx* ctx = static_cast<dspark_markov_ctx*>(calloc(1, sizeof(dspark_markov_ctx)));
  if (!ctx) return DSPARK_ERR_HOST_ALLOC;
  ctx->device = dev;
  ctx->sm_count = sms;
  ctx->cfg = *cfg;
  ctx->w1 = static_cast<const uint16_t*>(w1_bf16);
  ctx->w2 = static_cast<const uint16_t*>(w2_bf16);
  const size_t nslots = static_cast<size_t>(cfg->max_steps + 1) * cfg->max_rows;
  if (cudaMalloc(&ctx->slots, nslots * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMalloc(&ctx->counters, (cfg->max_steps + 1) * sizeof(unsigned int)) != cudaSuccess ||
      cudaMalloc(&ctx->status, 4 * sizeof(int)) != cudaSuccess) {
    dspark_markov_destroy(ctx);
    return DSPARK_ERR_CUDA;
  }
  if (cudaMemsetAsync(ctx->slots, 0, nslots * sizeof(unsigned long long), stream) != cudaSuccess ||
      cudaMemsetAsync(ctx->counters, 0, (cfg->max_steps + 1) * sizeof(unsigned int), stream) != cudaSuccess ||
      cudaMemsetAsync(ctx->status, 0, 4 * sizeof(int), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    dspark_markov_destroy(ctx);
    return DSPARK_ERR_CUDA;
  }
  ctx->grid_simple = dspark::simple_step_grid(cfg->vocab);
  ctx->grid_tc = dspark::tc_step_grid(cfg->vocab, sms);
  // the tensor-core kernel packs vocabulary ids into 24 bits
  ctx->tc_ok = tc_setup && cfg->vocab < (1 << 24) && dspark::encode_w2_map(&ctx->w2_map, w2_bf16, cfg->vocab, 32) &&
              dspark::encode_w2_map(&ctx->w2_tile_map, w2_bf16, cfg->vocab, 128);
  ctx->fused_ok = ctx->tc_ok && dspark::tc_cooperative_ok(ctx->grid_tc);
  const int max_grid = ctx->grid_simple > ctx->grid_tc ? ctx->grid_simple : ctx->grid_tc;
  if (cudaMalloc(&ctx->partials, static_cast<size_t>(cfg->max_rows) * max_grid * sizeof(unsigned long long)) !=
          cudaSuccess ||
      cudaMalloc(&ctx->xform_lut, 65536 * sizeof(uint16_t)) != cudaSuccess) {
    dspark_markov_destroy(ctx);
    return DSPARK_ERR_CUDA;
  }
  *out = ctx;
  return DSPARK_OK;
}

void dspark_markov_destroy(dspark_markov_ctx* ctx) {
  if (!ctx) return;
  if (ctx->slots) cudaFree(ctx->slots);
  if (ctx->counters) cudaFree(ctx->counters);
  if (ctx->status) cudaFree(ctx->status);
  if (ctx->partials) cudaFree(ctx->partials);
  if (ctx->xform_lut) cudaFree(ctx->xform_lut);
  free(ctx);
}

int32_t dspark_markov_bias_path(const dspark_markov_ctx* ctx, int32_t rows) {
  if (ctx && ctx->w2_fp8)
    return ctx->tc8_ok && !(ctx->cfg.flags & DSPARK_FLAG_FORCE_FMA) && rows <= dspark::tc_fp8_max_rows() ? 3 : 2;
  if (!ctx || !ctx->tc_ok || (ctx->cfg.flags & DSPARK_FLAG_FORCE_FMA)) return 0;
  if (ctx->cfg.flags & DSPARK_FLAG_FORCE_MMA) return 1;
  return rows > kFmaMaxRows ? 1 : 0;
}

int32_t dspark_markov_partial_count(const dspark_markov_ctx* ctx) {
  if (!ctx) return 0;
  const int32_t path = dspark_markov_bias_path(ctx, ctx->cfg.max_rows);
  return path == 1 || path == 3 ? ctx->grid_tc : ctx->grid_simple;
}

int dspark_markov_set_w2_fp8(dspark_markov_ctx* ctx, const void* w2_fp8, const void* w2_scale_f16) {
  if (!ctx || (!w2_fp8) != (!w2_scale_f16)) return DSPARK_ERR_INVALID_ARG;
  if (w2_fp8 && (!aligned16(w2_fp8) || (reinterpret_cast<uintptr_t>(w2_scale_f16) & 1u)))
    return DSPARK_ERR_MISALIGNED;
  ctx->w2_fp8 = static_cast<const uint8_t*>(w2_fp8);
  ctx->w2_scale = static_cast<const uint16_t*>(w2_scale_f16);
  // the tensor-core step reads E4M3 stages by TMA; without the maps the
  // CUDA-core FP8 step serves every call
  ctx->tc8_ok = w2_fp8 && ctx->tc_ok && dspark::encode_w2_fp8_map(&ctx->w2f8_map, w2_fp8, ctx->cfg.vocab, 32) &&
                dspark::encode_w2_fp8_map(&ctx->w2f8_tile_map, w2_fp8, ctx->cfg.vocab, 128);
  return DSPARK_OK;
}

int dspark_markov_anchor(dspark_markov_ctx* ctx, const dspark_markov_loop_args* a, cudaStream_t stream) {
  int rc = check_args(ctx, a);
  if (rc != DSPARK_OK) return rc;
  if (a->cap != 0.0f && dspark::launch_xform_lut(ctx->xform_lut, a->mult, a->cap, stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (dspark::launch_anchor(a->input_ids, a->anchor_idx, ctx->slots, ctx->counters,
                            ctx->counters + ctx->cfg.max_steps, a->rows, a->steps, ctx->cfg.max_rows,
                            stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  ctx->state_clean = true;
  return DSPARK_OK;
}

namespace {

// One step launch.  In a loop on the tensor-core path a step leaves its
// tokens in the argmax slots and the next step's CTA 0 writes them, so that
// no step but the last waits for a last-arriving CTA.  With the two-launch
// select the step writes per-CTA maxima and a select launch follows.
int launch_step(dspark_markov_ctx* ctx, const dspark_markov_loop_args* a, int32_t step, bool in_loop,
                cudaStream_t stream) {
  dspark::StepParams p = make_params(ctx, a, step);
  const bool pdl = (ctx->cfg.flags & DSPARK_FLAG_PDL) != 0;
  const bool select = (ctx->cfg.flags & DSPARK_FLAG_SELECT_2LAUNCH) != 0;
  if (select) p.partials = ctx->partials;
  cudaError_t e;
  int grid;
  const int32_t path = dspark_markov_bias_path(ctx, a->rows);
  if ((path == 1 || path == 3) && tma_base_ok(a)) {
    if (select) {
      p.finish = 0;
    } else if (in_loop) {
      p.finish = step == a->steps - 1;
      p.write_prev = step > 0;
    }
    grid = ctx->grid_tc;
    if (path == 3) {
      p.w2_scale = ctx->w2_scale;
      e = dspark::launch_step_tc(p, ctx->w2f8_map, ctx->w2f8_tile_map, grid, pdl, false, stream, true);
    } else {
      e = dspark::launch_step_tc(p, ctx->w2_map, ctx->w2_tile_map, grid, pdl, false, stream);
    }
  } else if (ctx->w2_fp8) {
    grid = ctx->grid_simple;
    e = dspark::launch_step_fp8(p, ctx->w2_fp8, ctx->w2_scale, a->cap != 0.0f, pdl, stream);
  } else {
    grid = ctx->grid_simple;
    e = dspark::launch_step_simple(p, a->cap != 0.0f, pdl, stream);
  }
  if (e == cudaSuccess && select)
    e = dspark::launch_select(ctx->partials, grid, p.slots_out, a->tokens, a->tokens_s0, step, a->rows, pdl, stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// The loop runs as one multi-step launch: tensor-core path, TMA-readable base,
// several steps, a cooperative launch possible and not switched off.
bool loop_fused(const dspark_markov_ctx* ctx, const dspark_markov_loop_args* a) {
  const int32_t path = dspark_markov_bias_path(ctx, a->rows);
  return ctx->fused_ok && !(ctx->cfg.flags & (DSPARK_FLAG_PER_STEP | DSPARK_FLAG_SELECT_2LAUNCH)) && a->steps > 1 &&
         (path == 1 || path == 3) && tma_base_ok(a);
}

}  // namespace

int dspark_markov_step(dspark_markov_ctx* ctx, const dspark_markov_loop_args* a, int32_t step,
                       cudaStream_t stream) {
  int rc = check_args(ctx, a);
  if (rc != DSPARK_OK) return rc;
  if (step < 0 || step >= a->steps) return DSPARK_ERR_INVALID_ARG;
  ctx->state_clean = false;
  return launch_step(ctx, a, step, false, stream);
}

int dspark_markov_shard_step(dspark_markov_ctx* ctx, const dspark_markov_loop_args* a, int32_t step,
                             int64_t vocab_offset, int32_t* packets, cudaStream_t stream) {
  int rc = check_args(ctx, a);
  if (rc != DSPARK_OK) return rc;
  if (step < 0 || step >= a->steps || vocab_offset < 0 || !packets) return DSPARK_ERR_INVALID_ARG;
  if (vocab_offset + ctx->cfg.vocab > (int64_t{1} << 31)) return DSPARK_ERR_INVALID_ARG;  // global ids are int32
  if (reinterpret_cast<uintptr_t>(packets) & 15u) return DSPARK_ERR_MISALIGNED;
  const int32_t path = dspark_markov_bias_path(ctx, a->rows);
  if (path != 1 && path != 3) return DSPARK_ERR_INVALID_ARG;  // the tensor-core step only
  if (!tma_base_ok(a)) return DSPARK_ERR_MISALIGNED;
  ctx->state_clean = false;
  dspark::StepParams p = make_params(ctx, a, step);
  p.sharded = 1;
  p.vocab_offset = vocab_offset;
  p.packets = packets;
  p.finish = 1;
  p.write_prev = 0;
  const bool pdl = (ctx->cfg.flags & DSPARK_FLAG_PDL) != 0;
  cudaError_t e;
  if (path == 3) {
    p.w2_scale = ctx->w2_scale;
    e = dspark::launch_step_tc(p, ctx->w2f8_map, ctx->w2f8_tile_map, ctx->grid_tc, pdl, false, stream, true);
  } else {
    e = dspark::launch_step_tc(p, ctx->w2_map, ctx->w2_tile_map, ctx->grid_tc, pdl, false, stream);
  }
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

int dspark_markov_pick(dspark_markov_ctx* ctx, const int32_t* packets, int32_t tp, int32_t rows, int64_t* tokens,
                       int64_t tokens_s0, int32_t step, cudaStream_t stream) {
  if (!ctx || !packets || !tokens || tp < 1 || tp > 32 || rows < 1 || step < 0) return DSPARK_ERR_INVALID_ARG;
  if (rows > ctx->cfg.max_rows || step >= ctx->cfg.max_steps) return DSPARK_ERR_TOO_MANY_ROWS;
  if (tokens_s0 <= step) return DSPARK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(packets) & 15u) return DSPARK_ERR_MISALIGNED;
  unsigned long long* slot_next = ctx->slots + static_cast<int64_t>(step + 1) * ctx->cfg.max_rows;
  ctx->state_clean = false;
  return dspark::launch_pick(packets, tp, rows, tokens, tokens_s0, step, slot_next, stream) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_ERR_CUDA;
}

int32_t dspark_markov_loop_kernels(const dspark_markov_ctx* ctx, const dspark_markov_loop_args* a) {
  if (check_args(ctx, a) != DSPARK_OK) return 0;
  const int32_t lut = a->cap != 0.0f ? 1 : 0;
  if (loop_fused(ctx, a)) return (ctx->state_clean ? 1 : 2) + lut;
  return 1 + lut + a->steps * ((ctx->cfg.flags & DSPARK_FLAG_SELECT_2LAUNCH) ? 2 : 1);
}

int dspark_markov_loop(dspark_markov_ctx* ctx, const dspark_markov_loop_args* a, cudaStream_t stream) {
  int rc = check_args(ctx, a);
  if (rc != DSPARK_OK) return rc;
  const bool fused = loop_fused(ctx, a);
  if (fused && ctx->state_clean) {
    // the loop state is zero: no anchor launch (the soft cap's table only)
    if (a->cap != 0.0f && dspark::launch_xform_lut(ctx->xform_lut, a->mult, a->cap, stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  } else {
    rc = dspark_markov_anchor(ctx, a, stream);
    if (rc != DSPARK_OK) return rc;
  }
  if (fused) {
    // every step in one cooperative launch; the last CTA to arrive at the
    // last step writes its tokens and leaves the loop state zero
    dspark::StepParams p = make_params(ctx, a, 0);
    p.step_end = a->steps;
    p.self_reset = 1;
    const bool pdl = (ctx->cfg.flags & DSPARK_FLAG_PDL) != 0;
    const bool fp8 = dspark_markov_bias_path(ctx, a->rows) == 3;
    if (fp8) p.w2_scale = ctx->w2_scale;
    const cudaError_t e = fp8 ? dspark::launch_step_tc(p, ctx->w2f8_map, ctx->w2f8_tile_map, ctx->grid_tc, pdl,
                                                       true, stream, true)
                              : dspark::launch_step_tc(p, ctx->w2_map, ctx->w2_tile_map, ctx->grid_tc, pdl, true,
                                                       stream);
    if (e == cudaSuccess) {
      ctx->state_clean = true;
      return DSPARK_OK;
    }
    ctx->state_clean = false;
    if (e != cudaErrorInvalidValue) return DSPARK_ERR_CUDA;
    // the base strides do not form the multi-step tensor map: step by step,
    // from the anchor's previous tokens
    rc = dspark_markov_anchor(ctx, a, stream);
    if (rc != DSPARK_OK) return rc;
  }
  ctx->state_clean = false;
  for (int s = 0; s < a->steps; ++s) {
    rc = launch_step(ctx, a, s, true, stream);
    if (rc != DSPARK_OK) return rc;
  }
  return DSPARK_OK;
}

int dspark_markov_get_status_detail(dspark_markov_ctx* ctx, cudaStream_t stream, int32_t* detail) {
  if (!ctx || !detail) return DSPARK_ERR_INVALID_ARG;
  int v[4] = {0, 0, 0, 0};
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaMemcpy(v, ctx->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaMemset(ctx->status, 0, sizeof(v)) != cudaSuccess) return DSPARK_ERR_CUDA;
  // a loop that gave up left its slots, counters and abort word set: the
  // next loop starts from the anchor
  if (v[0] != 0) ctx->state_clean = false;
  for (int i = 0; i < 4; ++i) detail[i] = v[i];
  return DSPARK_OK;
}

int dspark_markov_get_status(dspark_markov_ctx* ctx, cudaStream_t stream, int32_t* device_status) {
  if (!device_status) return DSPARK_ERR_INVALID_ARG;
  int32_t d[4];
  const int rc = dspark_markov_get_status_detail(ctx, stream, d);
  if (rc == DSPARK_OK) *device_status = d[0];
  return rc;
}

}  // extern "C"
