/*
 * dspark_oracle.h -- the CPU oracle's own declarations (test infrastructure
 * only; the CUDA library neither includes nor links this).  See
 * dspark_oracle.c for the definitions and the pages each one follows.
 */
#ifndef DSPARK_ORACLE_H
#define DSPARK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

float oracle_bf16_to_f32(uint16_t b);
uint16_t oracle_f32_to_bf16(float f);
float oracle_logf(float x);
float oracle_tanhf(float z);
uint16_t oracle_logit(uint16_t base, uint16_t bias, float mult, int has_cap, float inv_cap,
                      float cap, float *l_out);
uint32_t oracle_murmur_block(uint32_t h, uint32_t k);
uint32_t oracle_murmur_fmix(uint32_t h);
uint32_t oracle_noise_hash(int64_t seed, int32_t step, int64_t sample_pos, uint32_t salt,
                           uint32_t vocab_id);
float oracle_uniform(uint32_t h);
float oracle_log1m(float u);
float oracle_noise_L(uint32_t h);
float oracle_key(float l, float temp, uint32_t h);
int64_t oracle_argmax(const float *keys, int64_t n);
int oracle_combine_first_wins(float v1, int64_t i1, float v2, int64_t i2);
uint16_t oracle_dot_bf16(const uint16_t *a, const uint16_t *b, int n);

/* Arguments of one loop call; strides in elements. */
typedef struct {
  int64_t vocab;      /* V: rows of w2, width of base / cache rows */
  int32_t rank;       /* 256 on the pages */
  int64_t w1_rows;    /* rows of w1 (ids are clamped to w1_rows - 1) */
  const uint16_t *w1; /* [w1_rows, rank] BF16 */
  const uint16_t *w2; /* [vocab, rank] BF16 */
  int32_t rows;       /* R request rows */
  int32_t steps;      /* k draft steps */
  const uint16_t *base;
  int64_t base_s0, base_s1; /* base[r, s, v] = base[r*s0 + s*s1 + v] */
  uint16_t *cache;          /* may be NULL */
  int64_t cache_s0, cache_s1;
  const int32_t *input_ids;
  const int64_t *anchor_idx; /* [rows] */
  const int64_t *req_idx;    /* [rows, steps] (stride req_s0) or NULL = identity */
  int64_t req_s0;
  const int64_t *sample_pos; /* [rows, steps] (stride pos_s0) */
  int64_t pos_s0;
  int64_t num_req; /* length of seeds / temperature; cache rows */
  const int64_t *seeds;
  const float *temperature;
  float mult;
  float cap; /* 0: no soft cap */
  uint32_t salt;
  const uint16_t *fed_bias; /* [rows, steps, vocab] or NULL: computed exactly */
  int64_t *tokens;          /* [rows, steps] (stride tokens_s0) */
  int64_t tokens_s0;
  uint16_t *bias_out; /* optional [rows, steps, vocab] */
  float *keys_out;    /* optional [rows, steps, vocab] */
  int nthreads;
  const uint8_t *w2_fp8;   /* optional [vocab, rank] E4M3: the bias from it (and w2_scale) instead of w2 */
  const uint16_t *w2_scale; /* [vocab] FP16 row scales, with w2_fp8 */
  uint16_t *logits_out;     /* optional [rows, steps, vocab]: the cached BF16 logit c of every row,
                               valid or not (the rank-local cache of a vocabulary shard holds them all) */
} oracle_loop_args;

int oracle_markov_loop(const oracle_loop_args *a);
void oracle_build_verify_tokens(const int64_t *last, const int64_t *draft, int64_t *verify,
                                int32_t batch, int32_t draft_stride, int32_t P);
int oracle_greedy_accept(const uint16_t *logits, const int64_t *draft, const int32_t *proposal_len,
                         int64_t *accepted, int32_t *accept_len, int32_t batch,
                         int32_t draft_stride, int32_t P, int64_t vocab);

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void oracle_fill_uniforms(float *u, int64_t n, uint64_t seed, uint64_t offset);
uint64_t oracle_weight(float p);
int64_t oracle_sample_weights(const uint64_t *w, int64_t n, float u);
int oracle_probabilistic_accept(const float *target, const float *draft_probs, const int64_t *draft,
                                const int32_t *proposal_len, const float *uniforms, int64_t *accepted,
                                int32_t *accept_len, int32_t batch, int32_t draft_stride, int32_t P,
                                int64_t vocab);

float oracle_e4m3_value(uint8_t q);
uint8_t oracle_e4m3_from_f32(float x);
float oracle_f16_value(uint16_t h);
uint16_t oracle_f16_from_f32(float x);
void oracle_quantize_w2_fp8(const uint16_t *w2, uint8_t *q, uint16_t *scale, int64_t vocab, int rank);
uint16_t oracle_dot_fp8(const uint16_t *e, const uint8_t *q, uint16_t scale, int n);
void oracle_dot_fp8_rows(const uint16_t *e, const uint8_t *q, const uint16_t *scale, uint16_t *out, int64_t rows,
                         int n);
void oracle_e4m3_value_array(const uint8_t *q, float *out, int64_t n);
void oracle_e4m3_from_f32_array(const float *x, uint8_t *out, int64_t n);
void oracle_f16_value_array(const uint16_t *h, float *out, int64_t n);
void oracle_f16_from_f32_array(const float *x, uint16_t *out, int64_t n);
float oracle_expf_nonpos(float x);
void oracle_expf_nonpos_array(const float *x, float *out, int64_t n);
int oracle_logits_to_probs(const float *logits, float *probs, int32_t rows, int64_t vocab, float temperature,
                           int32_t top_k, float top_p);

/* Vocabulary-sharded loop ([P3] module docstring, _finish, markov_pick, cache_fill). */
void oracle_shard_packet(const float *keys, int64_t width, int64_t vocab_offset, uint32_t packet[4]);
void oracle_pick(const uint32_t *packets, int32_t tp, int32_t rows, int64_t *tokens);
float oracle_dot_bf16_f32(const uint16_t *a, const uint16_t *b, int n);
float oracle_sigmoid(float z);
void oracle_confidence(const uint16_t *hidden, int64_t hidden_stride, int64_t hidden_offset, const uint16_t *w1,
                       int64_t w1_rows, int32_t rank, const uint16_t *weight, float bias, const int64_t *first_prev,
                       const int64_t *draft, int64_t draft_stride, int32_t batch, int32_t P, int32_t hidden_size,
                       int32_t with_markov, const float *fed_logits, float *logits_out, float *scores);
int32_t oracle_threshold_length(const float *scores, int32_t P, float threshold, int32_t min_len, int32_t max_len);
int32_t oracle_sps_length(const float *scores, int32_t P, float survival_floor, int32_t min_len, int32_t max_len,
                          const float *cost);
void oracle_cache_fill(const uint16_t *src, int64_t src_s0, uint16_t *cache, int64_t cache_s0, int64_t cache_s1,
                       const int64_t *req_idx, int64_t req_s0, int64_t num_req, int32_t rows, int32_t steps,
                       int32_t shard, int32_t tp, int64_t vocab);

#ifdef __cplusplus
}
#endif
#endif
