/*
 * dspark_markov.h -- C ABI of the GB300 (sm_103a) DSpark Markov draft-sampling
 * library, libdspark_markov.so.
 *
 * The operations follow these pages (cited as "page, section"):
 *   [P1] TensorRT Edge-LLM C++ API, "Dspark Kernels": dsparkMarkovPartialCount,
 *        dsparkBuildVerifyTokens, dsparkGreedyAccept.
 *   [P2] vLLM models.kimi_k3.nvidia.specialized_decode.drafter.markov: module
 *        docstring (exactness paragraph), FusedMarkov, _gumbel_key, _loop_rest.
 *   [P3] vLLM models.muse_spark.nvidia.specialized_decode.cutedsl.draft.markov:
 *        module docstring, anchor_embed, markov_step (_StepKernel.kernel,
 *        _finish, _logit, _gumbel, _murmur_prefix, _combine, _w1_row).
 *   [P4] vLLM models.deepseek_v41.amd.ops.fused_markov: module docstring.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to device memory of the
 *     current CUDA device; the caller owns them.  The library owns only the
 *     context's scratch.  Strides are in elements.
 *   - Return 0 (DSPARK_OK) or a negative DSPARK_ERR_* code; nothing throws.
 *     Launch-type entry points do not synchronise the host; they enqueue on
 *     `stream` and are safe to capture in a CUDA graph (fixed pointers, no
 *     allocation).  dspark_markov_init and dspark_markov_get_status are not.
 *   - BF16 tensors are passed as raw 16-bit storage (`const void *`).
 */
#ifndef DSPARK_MARKOV_H
#define DSPARK_MARKOV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes ------------------------------------------------------- */
#define DSPARK_OK 0
#define DSPARK_ERR_INVALID_ARG (-1)      /* null pointer, bad size, bad stride */
#define DSPARK_ERR_UNSUPPORTED_RANK (-2) /* Markov rank other than 256 */
#define DSPARK_ERR_MISALIGNED (-3)       /* a pointer breaks its required alignment */
#define DSPARK_ERR_TOO_MANY_ROWS (-4)    /* rows > max_rows or steps > max_steps */
#define DSPARK_ERR_CAPTURING (-5)        /* init called while `stream` is capturing */
#define DSPARK_ERR_CUDA (-6)             /* a CUDA runtime call or launch failed */
#define DSPARK_ERR_DEVICE_TIMEOUT (-7)   /* a bounded device wait gave up (status word) */
#define DSPARK_ERR_UNSUPPORTED_DEVICE (-8) /* not a compute capability 10.3 device */
#define DSPARK_ERR_HOST_ALLOC (-9)       /* a host memory allocation failed */

/* ---- config flags ------------------------------------------------------ */
#define DSPARK_FLAG_PDL 0x1        /* launch steps with programmatic dependent launch */
#define DSPARK_FLAG_FORCE_FMA 0x2  /* bias on CUDA-core FMA (one launch per step) for every row count */
#define DSPARK_FLAG_FORCE_MMA 0x4  /* bias on tcgen05 tensor cores for every row count */
#define DSPARK_FLAG_PER_STEP 0x8   /* loop: one launch per step even where one launch could run them all */
#define DSPARK_FLAG_TEST_STALL 0x100 /* checking aid, no counterpart in the pages: in the one-launch
                                        loop the first step boundary waits for one arrival more than
                                        the grid makes, so its bounded wait runs out (a few seconds)
                                        and the loop ends with DSPARK_ERR_DEVICE_TIMEOUT in the status
                                        word (site 9); tests use it to exercise the timeout path.
                                        Multiplier 1 without a soft cap only (else DSPARK_ERR_CUDA) */
#define DSPARK_FLAG_SELECT_2LAUNCH 0x10 /* each step as two launches: the step kernel writes its blocks'
                                           maxima, a select launch (one CTA per row) reduces them under the
                                           same total order and writes the token ([P2] _markov_select_kernel);
                                           implies one launch per step */

/* Opaque context: the Markov tables, the tensor maps over them and the
 * scratch of one loop (per-step argmax slots and arrival counters), sized
 * once for max_rows x max_steps so that captured graphs keep its addresses
 * ([P2] FusedMarkov: "scratch sized for its largest batch, allocated once").
 * A context serves one loop at a time: its slots, counters, status word and
 * soft-cap table belong to the call in flight, so calls on one context must
 * be ordered (one stream, or streams ordered by events).  Loops that should
 * run concurrently need one context each. */
typedef struct dspark_markov_ctx dspark_markov_ctx;

typedef struct {
  int32_t vocab;     /* V: rows of w2 and width of a logits row (>= 1) */
  int32_t rank;      /* Markov rank R of w1 and w2; must be 256 */
  int32_t w1_rows;   /* rows of w1 (>= 1); ids are clamped to w1_rows - 1 */
  int32_t max_rows;  /* largest `rows` a loop call may pass (1..256) */
  int32_t max_steps; /* largest `steps` a loop call may pass (1..64) */
  int32_t flags;     /* DSPARK_FLAG_* */
} dspark_markov_config;

/*
 * dspark_markov_init -- validate the tables and allocate the context
 * ([P2] FusedMarkov.__init__, why_not; [P3] MarkovKernels).
 *   w1_bf16: device, [w1_rows, rank] BF16, row-major, 16-byte aligned.
 *   w2_bf16: device, [vocab, rank] BF16, row-major, 16-byte aligned.
 * The tables are not copied: they must stay valid and unchanged while the
 * context is used.  Allocates with cudaMalloc, so it must not run while
 * `stream` is being captured (DSPARK_ERR_CAPTURING).  On success *out owns
 * the context; free it with dspark_markov_destroy.  DSPARK_ERR_HOST_ALLOC if
 * the context's host structure cannot be allocated, DSPARK_ERR_CUDA if a
 * device allocation or set-up call fails.
 */
DSPARK_API int dspark_markov_init(dspark_markov_ctx **out, const dspark_markov_config *cfg, const void *w1_bf16,
                       const void *w2_bf16, cudaStream_t stream);

/* Arguments of one loop call (all device pointers unless stated). */
typedef struct {
  int32_t rows;  /* request rows of this call, 1..max_rows */
  int32_t steps; /* draft steps k, 1..max_steps */
  /* Base logits [rows, steps, V] BF16: base[r, s, v] = base[r*base_s0 + s*base_s1 + v].
   * Any non-negative strides; the TMA-fed step kernel is used when the
   * pointer is 16-byte aligned and the strides are multiples of 8 elements
   * (the values are the same either way, [P3] vectorized). */
  const void *base;
  int64_t base_s0, base_s1;
  /* Draft-logits cache [num_req, steps, V] BF16 (pre-temperature logits),
   * written at [req, s, v] for valid rows ([P3] _StepKernel.kernel); NULL
   * stores nothing.  Must not overlap base. */
  void *cache;
  int64_t cache_s0, cache_s1;
  /* Step 0's previous token: sext(input_ids[anchor_idx[r]]) ([P3] anchor_embed). */
  const int32_t *input_ids;  /* int32 token ids */
  const int64_t *anchor_idx; /* [rows] int64 indices into input_ids */
  /* Request of (row, step): req_idx[r*req_s0 + s] (int64); NULL means req = r.
   * A request outside [0, num_req) marks the row invalid for that step: no
   * cache store, temperature and seed read as 0 (greedy). */
  const int64_t *req_idx;
  int64_t req_s0;
  const int64_t *sample_pos; /* [rows, steps] int64 at sample_pos[r*pos_s0 + s] */
  int64_t pos_s0;
  int64_t num_req;           /* length of seeds / temperature, rows of cache */
  const int64_t *seeds;      /* [num_req] int64 (a uint64 bit pattern) */
  const float *temperature;  /* [num_req] f32; 0 = greedy */
  float mult;                /* logit multiplier ([P3] _logit), finite */
  float cap;                 /* soft cap, finite; 0 = none */
  uint32_t salt;             /* draft noise salt; the pages use 1u << 30 */
  int64_t *tokens;           /* out: [rows, steps] int64 at tokens[r*tokens_s0 + s] */
  int64_t tokens_s0;
  /* Optional: the BF16 bias the kernel used, [rows, steps, V] contiguous;
   * NULL in production (a checking aid, costs one extra write per element). */
  void *bias_out;
} dspark_markov_loop_args;

/*
 * dspark_markov_loop -- the whole k-step loop ([P2] FusedMarkov.run,
 * _loop_rest; [P3] anchor_embed + markov_step per step): for each step s and
 * row r, embed the previous token (w1 row clamped to the last row), bias
 * GEMV against w2 in FP32 rounded once to BF16, BF16 add to the base logits,
 * multiplier and optional soft cap, cache store, Gumbel-max with
 * MurmurHash3 noise of (seed, step, position + salt, vocab id), and a
 * total-order argmax (first NaN, else lowest id of the maximum).  The
 * winner is tokens[r, s] and the next step's previous token.
 * Enqueues either one launch for all steps (tensor-core path, steps > 1,
 * TMA-readable base, a cooperative launch possible and DSPARK_FLAG_PER_STEP
 * not set: its CTAs, all resident at once, wait for one another between
 * steps with bounded waits) or the anchor kernel and one launch per step;
 * with a soft cap, the cap's table kernel first.  The one-launch loop reads
 * step 0's previous tokens itself and leaves the context's argmax slots and
 * step counters zero, so it needs the anchor kernel only when something
 * else used them last (the context's first call, a per-step, sharded or
 * select launch, or a device error read by dspark_markov_get_status*); see
 * dspark_markov_loop_kernels.  After a device error that nobody has read,
 * later loops on the context give up at once (the error stays recorded).
 * No host synchronisation.
 */
DSPARK_API int dspark_markov_loop(dspark_markov_ctx *ctx, const dspark_markov_loop_args *args,
                       cudaStream_t stream);

/* dspark_markov_anchor / dspark_markov_step -- the loop's kernels one at a
 * time ([P3] anchor_embed, markov_step): anchor first, then step 0 .. steps-1
 * in order, with the same args (with DSPARK_FLAG_SELECT_2LAUNCH a step call
 * enqueues the step and its select launch).  The results equal
 * dspark_markov_loop's. */
DSPARK_API int dspark_markov_anchor(dspark_markov_ctx *ctx, const dspark_markov_loop_args *args,
                         cudaStream_t stream);
DSPARK_API int dspark_markov_step(dspark_markov_ctx *ctx, const dspark_markov_loop_args *args, int32_t step,
                       cudaStream_t stream);

/* [P1] dsparkMarkovPartialCount: the number of vocabulary blocks the step
 * kernel partitions the vocabulary into (its grid size). */
DSPARK_API int32_t dspark_markov_partial_count(const dspark_markov_ctx *ctx);

/* Which bias path a call with `rows` rows takes: 0 = FMA, 1 = tcgen05,
 * 2 = FMA over the FP8 w2 attached by dspark_markov_set_w2_fp8 (forced, or
 * above 160 rows), 3 = tcgen05 over that FP8 w2.  (A base whose pointer or
 * strides a TMA cannot address takes the FMA form of the same path.) */
DSPARK_API int32_t dspark_markov_bias_path(const dspark_markov_ctx *ctx, int32_t rows);

/*
 * dspark_markov_set_w2_fp8 -- attach (or, with two NULLs, detach) an FP8 w2
 * ([P1] dsparkMarkovGreedyFusedStepFp8): w2_fp8 [vocab, 256] E4M3 bytes
 * (16-byte aligned) and w2_scale_f16 [vocab] FP16 row scales, device
 * pointers owned by the caller (e.g. from dspark_quantize_w2_fp8) and read by
 * every later step.  While attached, every step takes its bias as
 * RN_bf16(RN(scale * sum_j e_j * decode(q_j))) with the sum in FP32 (any
 * order; within 1 BF16 ulp of the exactly rounded s * sum(e * decode(q))
 * outside the FP32 accumulation bound); the rest of the step is unchanged.
 * Up to 160 rows the tensor-core loop serves it (E4M3 stages by TMA, turned
 * into FP16 operands in shared memory; the embeddings enter as FP16 of
 * e * 2^k per row, exact for every entry within 2^32 of the row's largest),
 * else one CUDA-core launch per step.  Enqueues nothing.  DSPARK_ERR_INVALID_ARG
 * for one NULL and one non-NULL pointer, DSPARK_ERR_MISALIGNED for a pointer
 * off its alignment.
 */
DSPARK_API int dspark_markov_set_w2_fp8(dspark_markov_ctx *ctx, const void *w2_fp8, const void *w2_scale_f16);

/*
 * Vocabulary-sharded loop ([P3] "muse_spark cutedsl draft markov": module
 * docstring -- with a vocab-parallel w2 each rank works on its vocab range,
 * its last block writes a packet instead of the token, markov_pick picks the
 * winner from the gathered per-rank packets, cache_fill scatters the gathered
 * draft-logits shards after the loop; _finish, markov_pick, cache_fill).
 * A rank's context is initialised over its w2 shard (cfg.vocab = the shard's
 * width, w2 = its [width, 256] rows) and the whole w1.  Per call: the anchor
 * (dspark_markov_anchor), then for each step s: dspark_markov_shard_step on
 * every rank, an all-gather of the ranks' packets into [tp, rows, 4] (rank
 * k's rows at offset k * rows * 4; the caller's collective, into local
 * memory), dspark_markov_pick on every rank; after the last step the
 * all-gather of the rank-local caches and dspark_cache_fill.  The tokens equal
 * the unsharded loop's (the total order makes the pick shard-invariant).
 *
 * dspark_markov_shard_step -- step `step` of this rank's shard: global ids
 *   vocab_offset .. vocab_offset + width - 1 (the noise hashes the global id;
 *   vocab_offset + width <= 2^31).  args->base is the rank's base shard
 *   [rows, steps, width] (TMA-readable: 16-byte aligned, strides multiples of
 *   8); args->cache, if not NULL, the rank-local cache [rows, steps, >= width]
 *   written at [r, step, v] for every row r whatever its request (the fill
 *   places the valid ones); the previous token comes from the anchor (step
 *   0) or the pick of step - 1.  Writes packets [rows, 4] int32 (device,
 *   16-byte aligned): (bits of the winner's noised key, its global id, 0, 0)
 *   -- args->tokens is not written.  The tensor-core step only (bias path 1 or
 *   3, else DSPARK_ERR_INVALID_ARG); one launch.
 */
DSPARK_API int dspark_markov_shard_step(dspark_markov_ctx *ctx, const dspark_markov_loop_args *args, int32_t step,
                                        int64_t vocab_offset, int32_t *packets, cudaStream_t stream);

/* dspark_markov_pick -- [P3] markov_pick: per row the winner over the
 * gathered packets [tp, rows, 4] int32 (device, 16-byte aligned; 1 <= tp <= 32)
 * under the total order (the first NaN, else the largest value, ties to the
 * lower global id); writes tokens[r * tokens_s0 + step] (int64) and makes it
 * the previous token of the context's next step.  One launch. */
DSPARK_API int dspark_markov_pick(dspark_markov_ctx *ctx, const int32_t *packets, int32_t tp, int32_t rows,
                                  int64_t *tokens, int64_t tokens_s0, int32_t step, cudaStream_t stream);

/* dspark_cache_fill -- [P3] cache_fill: src = the gathered rank-local caches,
 * BF16 [tp, rows, steps, shard] (rank stride src_s0 elements, >= rows * steps
 * * shard); for every (row r, step i) whose request req = req_idx[r * req_s0 +
 * i] (r when req_idx is NULL) lies in [0, num_req), cache[req * cache_s0 + i *
 * cache_s1 + v] = src[k * src_s0 + (r * steps + i) * shard + v - k * shard],
 * k = v / shard, for v < vocab (shard * tp >= vocab); other cache rows are
 * left alone.  16-byte copies when pointers, strides, shard and vocab allow.
 * One launch, nothing allocated. */
DSPARK_API int dspark_cache_fill(const void *src, int64_t src_s0, void *cache, int64_t cache_s0, int64_t cache_s1,
                                 const int64_t *req_idx, int64_t req_s0, int64_t num_req, int32_t rows,
                                 int32_t steps, int32_t shard, int32_t tp, int32_t vocab, cudaStream_t stream);

/* The number of kernels dspark_markov_loop would enqueue now for `args`:
 * when one launch runs every step, 1 (2 if the anchor is needed first, see
 * dspark_markov_loop); else 1 + 2 steps with DSPARK_FLAG_SELECT_2LAUNCH, else
 * 1 + steps; plus 1 with a soft cap (its table); 0 if the arguments are
 * invalid.  No counterpart in the pages: it tells a caller what a captured
 * loop holds. */
DSPARK_API int32_t dspark_markov_loop_kernels(const dspark_markov_ctx *ctx, const dspark_markov_loop_args *args);

/* Synchronise `stream`, then read and clear the device status word: 0, or a
 * DSPARK_ERR_* a kernel recorded (a bounded wait that gave up).  Returns
 * DSPARK_OK or DSPARK_ERR_CUDA. */
DSPARK_API int dspark_markov_get_status(dspark_markov_ctx *ctx, cudaStream_t stream, int32_t *device_status);

/* As dspark_markov_get_status, with where a bounded wait gave up:
 * detail[0] = status, detail[1] = wait site (1 w2 slot free, 2 base slot free,
 * 3 embeddings ready, 4 accumulator free, 5 w2 tile landed, 6 accumulator
 * ready, 7 base chunk landed, 9 other CTAs' step results), detail[2] = block,
 * detail[3] = the step within the launch << 24 | tile << 12 | sequence number
 * (low 12 bits).  Reading clears the record. */
DSPARK_API int dspark_markov_get_status_detail(dspark_markov_ctx *ctx, cudaStream_t stream, int32_t *detail);

DSPARK_API void dspark_markov_destroy(dspark_markov_ctx *ctx);

/*
 * dspark_build_verify_tokens -- [P1] dsparkBuildVerifyTokens:
 *   verify[b, 0] = last[b];  verify[b, j + 1] = draft[b * draft_stride + j], j < P.
 * last [batch] int64, draft [batch, draft_stride] int64, verify [batch, P + 1]
 * int64 contiguous (device).  batch >= 0, 0 <= P <= draft_stride.
 */
DSPARK_API int dspark_build_verify_tokens(const int64_t *last, const int64_t *draft, int64_t *verify,
                               int32_t batch, int32_t draft_stride, int32_t P, cudaStream_t stream);

/*
 * dspark_greedy_accept -- [P1] dsparkGreedyAccept: a_j = total-order argmax
 * of logits[b, j, :]; accept draft[b, j] while it equals a_j for
 * j < clamp(proposal_len[b], 0, P); then append the bonus a_n.
 *   logits: device BF16 [batch, P + 1, vocab], contiguous, 16-byte aligned,
 *           vocab a multiple of 8.
 *   draft [batch, draft_stride] int64; proposal_len [batch] int32.
 *   accepted: out [batch, P + 1] int64: a_0 .. a_n, then -1.
 *   accept_len: out [batch] int32 = n + 1 (drafts accepted plus the bonus).
 *   scratch: device, >= dspark_greedy_accept_scratch_bytes(batch, P, vocab)
 *            bytes (8 per verify row + 16), 16-byte aligned; its contents
 *            on entry do not matter.
 * Three kernels on `stream` (clear the slots, scan, walk the acceptance),
 * chained with programmatic dependent launch.
 * Positions after the last one the acceptance can reach are not scanned.
 */
DSPARK_API size_t dspark_greedy_accept_scratch_bytes(int32_t batch, int32_t P, int32_t vocab);
DSPARK_API int dspark_greedy_accept(const void *logits, const int64_t *draft, const int32_t *proposal_len,
                         int64_t *accepted, int32_t *accept_len, void *scratch, size_t scratch_bytes,
                         int32_t batch, int32_t draft_stride, int32_t P, int32_t vocab,
                         cudaStream_t stream);

/*
 * dspark_greedy_accept_noalloc -- dspark_greedy_accept with library-owned
 * scratch, for callers that cannot allocate device memory.  The pages have
 * no counterpart of this entry point; it exists for this library's users.
 *
 * Who needs it: a caller whose device memory belongs to someone else (an
 * inference engine that reserves nearly all of HBM at start-up for its KV
 * cache and gives a plugin no workspace), or a caller on a latency-critical
 * path where cudaMalloc/cudaFree must not run (cudaFree synchronises the
 * whole device, and a new allocation can stall as well).  Such a caller
 * still owns every input and output; only the scratch moves into the
 * library.
 *
 * Arguments, results and error codes are those of dspark_greedy_accept, less
 * `scratch` and `scratch_bytes`.  The scratch is a fixed device array of
 * DSPARK_NOALLOC_MAX_VERIFY_ROWS + 2 eight-byte words (64 KB + 16 bytes)
 * that every device which loads the library holds until the process exits.
 *   - batch * (P + 1) > DSPARK_NOALLOC_MAX_VERIFY_ROWS is rejected with
 *     DSPARK_ERR_TOO_MANY_ROWS before anything is launched; use
 *     dspark_greedy_accept with caller scratch for larger batches.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and keeps it for the
 *     device's current context; make that first call before any stream
 *     capture.  A device reset (cudaDeviceReset) or another context made
 *     current starts a new context, and the next call looks the address up
 *     again, so after a reset make one call before capturing again.  If the
 *     lookup fails the call returns DSPARK_ERR_CUDA and the next call tries
 *     again.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Every call shares the one array, which keeps the last call's contents.
 *     The slots, which must start at zero, are
 *     cleared by the call's first kernel, so stale contents do no harm.  Two
 *     calls whose kernels overlap on the GPU (different streams without an
 *     ordering between them) race on the array and may give wrong results:
 *     order them on one stream or with events.
 */
#define DSPARK_NOALLOC_MAX_VERIFY_ROWS 8192
DSPARK_API int dspark_greedy_accept_noalloc(const void *logits, const int64_t *draft, const int32_t *proposal_len,
                                 int64_t *accepted, int32_t *accept_len, int32_t batch,
                                 int32_t draft_stride, int32_t P, int32_t vocab, cudaStream_t stream);

/*
 * Confidence-scored proposal lengths -- [P1] "Dspark Kernels":
 * dsparkComputeConfidenceScores, dsparkComputeConfidenceAndProposalLengths and
 * dsparkComputeConfidenceAndSPSProposalLengths.  The pages give the inputs
 * and one-line contracts; what follows is this library's reading of them.
 *
 * The confidence that draft position j of request b (0 <= j < P) is accepted
 * is a logistic head over the feature that produced that draft:
 *   feature = hidden[b, j, 0 .. H)  ++  w1[prev_j, 0 .. rank)  (the second
 *             part only with with_markov), prev_0 = first_prev[b],
 *             prev_j = draft[b, j - 1]; an id outside [0, w1_rows) takes the
 *             last w1 row, as in the loop;
 *   z      = (weight . feature) + bias  -- products exact in FP32, summed in
 *            FP32 in a fixed order (within (H + rank + 2) 2^-24 of the sum of
 *            |products| and |bias| of the exactly rounded value), one FP32
 *            bias add;
 *   score  = sigmoid(z) = RN(1 / RN(1 + E)) for z >= 0, RN(E / RN(1 + E))
 *            below, E = exp(-|z|) by the library's own exp; NaN stays NaN.
 * Device pointers; BF16 values are raw 16-bit patterns.
 *   hidden: BF16; the feature of (b, j) starts at element
 *           hidden_offset + (b * P + j) * hidden_stride (hidden_stride 0 means
 *           hidden_size; otherwise >= hidden_size).
 *   w1 [w1_rows, rank] BF16 row-major (read only with with_markov).
 *   weight [hidden_size + rank] BF16 (rank counted only with with_markov);
 *   bias [1] FP32.
 *   first_prev [batch] int64; draft [batch, draft_s0] int64 (draft_s0 >= P;
 *   both read only with with_markov).
 *   scores: out [batch, P] FP32 contiguous; logits: optional out [batch, P]
 *   FP32 (z), NULL to skip.
 * When hidden (plus offset), w1 and weight start on 16 bytes, hidden_size,
 * rank and hidden_stride are multiples of 8 and (P + 1) (hidden_size + rank)
 * 2 bytes fit in 200 KB, a request's rows are bulk-copied into shared memory
 * (one mbarrier, bounded wait; a request whose wait gave up -- never in
 * correct operation -- gets NaN scores and length -1); otherwise the rows
 * load into registers (16-byte loads where aligned, else 2-byte loads).
 * batch >= 0, 0 <= P <= DSPARK_CONFIDENCE_MAX_P.  One kernel on `stream`,
 * one CTA per request; allocates nothing.
 */
#define DSPARK_CONFIDENCE_MAX_P 256
typedef struct dspark_confidence_args {
  const void *hidden;
  int64_t hidden_stride;
  int64_t hidden_offset;
  int32_t hidden_size;
  int32_t with_markov;
  const void *w1;
  int64_t w1_rows;
  int32_t rank;
  int32_t batch;
  int32_t proposal_len;     /* P */
  int32_t reserved;         /* 0 */
  const void *weight;
  const float *bias;
  const int64_t *first_prev;
  const int64_t *draft;
  int64_t draft_s0;
  float *scores;
  float *logits;
} dspark_confidence_args;

/* The scores alone (the pages keep this form for chain-side analysis). */
DSPARK_API int dspark_confidence_scores(const dspark_confidence_args *args, cudaStream_t stream);

/*
 * Scores and threshold-scheduled lengths: with S_j = RN(S_{j-1} * score_j)
 * (S_{-1} = 1, the chance that drafts 0..j are all accepted),
 * L = the number of leading positions whose S_j >= threshold, clamped to
 * [lo, hi]: hi = clamp(max_proposal_len, 0, P), lo = clamp(min_proposal_len,
 * 0, hi).  proposal_lengths: out [batch] int32.
 */
DSPARK_API int dspark_confidence_and_proposal_lengths(const dspark_confidence_args *args, float threshold,
                                                      int32_t min_proposal_len, int32_t max_proposal_len,
                                                      int32_t *proposal_lengths, cudaStream_t stream);

/*
 * Scores and SPS-scheduled lengths (draft-side confidence only): the length
 * L in [lo, hi] (as above) with the largest RN(T_L / verify_cost[L]),
 * T_L = 1 + S_0 + ... + S_{L-1} summed in that order in FP32 (the expected
 * tokens out of a verify of L drafts), ties to the shorter; a length L > lo
 * is considered only while S_{L-1} >= survival_floor (the scan stops at the
 * first that is below), and a cost that is not > 0 (or NaN) rules its
 * length out (lo if every one is ruled out).  verify_cost: [P + 1] FP32
 * device array, the caller's estimate of a verify of L + 1 tokens (the pages
 * use a B100 verify-bucket cost model that they do not give).
 * proposal_lengths: out [batch] int32.
 */
DSPARK_API int dspark_confidence_and_sps_proposal_lengths(const dspark_confidence_args *args,
                                                          float survival_floor, int32_t min_proposal_len,
                                                          int32_t max_proposal_len, const float *verify_cost,
                                                          int32_t *proposal_lengths, cudaStream_t stream);

/*
 * dspark_fill_uniforms -- [P1] dsparkFillUniforms: n deterministic uniforms
 * in [0, 1) into `uniforms` (device, float32).  Element i is word i % 4 of
 * Philox4x32-10 (Salmon et al., SC 2011) at counter offset + i / 4 (a 64-bit
 * number in the low two words, the high two zero) with key (lo32(seed),
 * hi32(seed)), its top 24 bits times 2^-24 (a reading: the pages name the
 * generator's seed and offset only).  n >= 0.  One kernel on `stream`.
 */
DSPARK_API int dspark_fill_uniforms(float *uniforms, int64_t n, uint64_t seed, uint64_t offset,
                                    cudaStream_t stream);

/*
 * dspark_probabilistic_accept -- [P1] dsparkProbabilisticAccept, speculative
 * sampling with residual sampling.  Device pointers:
 *   target_probs [batch, P+1, vocab] float32, draft_probs [batch, P, vocab]
 *   float32 (contiguous), draft [batch, draft_stride] int64, proposal_len
 *   [batch] int32 (clamped to [0, P]), uniforms [batch, 2P+1] float32:
 *   u[j] decides draft position j, u[P+j] the residual sample after a
 *   rejection at j, u[2P] the bonus sample after a full accept.
 * Position j accepts its draft token d when RN(u[j] * q) < t (t and q the
 * target and draft probabilities of d; an id outside [0, vocab) is rejected).
 * After a rejection at j the token is sampled from max(0, RN(t - q)) over the
 * vocabulary (from the target row if that weighs nothing); after a full
 * accept from target row P_b.  Sampling is an inverse CDF over fixed-point
 * weights (probabilities clamped to [0, 1], truncated to units of 2^-40):
 * U = floor(u 2^24), T = floor(U S / 2^24) for the total S, the smallest id
 * whose inclusive prefix exceeds T (id 0 if the row weighs nothing) -- exact
 * sums, so the id does not depend on any summation order (readings; the pages
 * give the uniforms' layout and the method).  Writes accepted [batch, P+1]
 * int64 (accepted drafts, the sample, then -1) and accept_len [batch] int32
 * (accepted drafts + 1).  batch, P >= 0, vocab >= 1, draft_stride >= P.
 * Allocates nothing; one kernel on `stream`.  A row whose bounded wait for a
 * shared-memory copy gave up (never in correct operation) gets accept_len 0
 * and its accepted entries are left unwritten.
 */
DSPARK_API int dspark_probabilistic_accept(const float *target_probs, const float *draft_probs,
                                           const int64_t *draft, const int32_t *proposal_len,
                                           const float *uniforms, int64_t *accepted, int32_t *accept_len,
                                           int32_t batch, int32_t draft_stride, int32_t P, int32_t vocab,
                                           cudaStream_t stream);

/*
 * dspark_logits_to_probs -- [P1] dsparkLogitsToProbabilities: dense
 * probability rows after temperature, top-k and top-p.  Device pointers:
 * logits [rows, vocab] float32 (contiguous), probs [rows, vocab] float32
 * (contiguous; may be the same buffer as logits).
 *   temperature <= 0 (or NaN): greedy, 1 at the lowest id of the largest
 *     non-NaN logit (all zeros if every logit is NaN).
 *   Otherwise z = RN(l / temperature) (-0 as +0); ids whose z is NaN get 0.
 *   top_k: 0 < top_k < (ids with a non-NaN z) keeps the top_k first ids in
 *     the order (z descending, id ascending); other values keep all.
 *   e = exp(z - m), m the largest z (exactly 1 where z == m, so infinite
 *     logits share their mass), by the library's own exp (within 2 ulp);
 *     fixed-point weights w = floor(e 2^40).
 *   top_p < 1 keeps the shortest prefix of the kept ids in the order
 *     (w descending, id ascending) whose weights reach max(1, ceil(top_p W)),
 *     W their total (top_p <= 0 keeps one id); top_p >= 1 or NaN keeps all.
 *   probs = RN(e / S) on the final ids, S = RN(sum of their w) 2^-40;
 *     0 elsewhere.
 * Every decision is an exact comparison (readings: the pages name the three
 * filters only).  rows >= 0, vocab >= 1.  Allocates nothing; one kernel on
 * `stream`: without top-k and top-p (temperature > 0), with 16-byte-aligned
 * rows and vocab a multiple of 4 up to 8 x 25600, a cluster of CTAs holds
 * each row in shared memory; otherwise one CTA per row.
 */
DSPARK_API int dspark_logits_to_probs(const float *logits, float *probs, int32_t rows, int32_t vocab,
                                      float temperature, int32_t top_k, float top_p, cudaStream_t stream);

/*
 * dspark_quantize_w2_fp8 -- [P1] dsparkQuantizeMarkovW2Fp8: markov_w2 as
 * E4M3 bytes with one FP16 scale per row.  Device pointers: w2_bf16
 * [vocab, rank] BF16 bits (16-byte aligned), w2_fp8 out [vocab, rank] E4M3
 * bytes (8-byte aligned), scale_f16 out [vocab] FP16 bits (2-byte aligned).
 * Per row: rowAbsMax over the non-NaN values, scale = RN(rowAbsMax / 448)
 * in FP32, then to FP16 nearest even, saturating at 65504 (the pages give
 * rowAbsMax / 448 only); q = E4M3(RN(w / scale)), nearest even, saturating
 * to +-448, NaN to 0x7F; a row whose scale is 0 stores zeros.
 * rank a multiple of 8 (>= 8), vocab >= 0.  DSPARK_ERR_MISALIGNED for a
 * pointer off its alignment.  Allocates nothing; one kernel on `stream`.
 */
DSPARK_API int dspark_quantize_w2_fp8(const uint16_t *w2_bf16, uint8_t *w2_fp8, uint16_t *scale_f16,
                                      int64_t vocab, int32_t rank, cudaStream_t stream);

/* A short English description of a DSPARK_* code (static storage). */
DSPARK_API const char *dspark_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_MARKOV_H */
