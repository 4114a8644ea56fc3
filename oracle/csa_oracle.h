/*
 * CPU oracle for the compressed-sparse-attention KV Compressor.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow restatement of what the
 * compressor computes, used to check the CUDA library.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never does.  It shares no code with the CUDA library.
 *
 * Sources (web pages):
 *  [V41]  "DeepSeek V4.1 - Pool token pairs" (open-model-atlas), the pooling
 *         formula and the Compressor module excerpt (model.py 429-485):
 *         projection, group softmax pool, kv_state/score_state, prefill and
 *         decode branches, bf16 rounding before RMSNorm.
 *  [RUST] "Module compress" (metrale.ai DeepSeek-V4.1 CPU reference docs):
 *         precision contract, linear_f32, fp4_quant_e4m3_inplace,
 *         to_e2m1_rne, LATENT_BLOCK, yarn_freqs_cis.
 *  [CSA4] "Compressed Sparse Attention - ratio m = 4" (yiliu30 explainer):
 *         two branches x 512, 8 candidates, padded first entry, decode rule,
 *         RoPE after normalisation, released Flash configuration.
 *
 * All floating point is double unless the pages fix a precision; the values
 * the pages fix in float32 (projection outputs, the pooled result, the fp4
 * scale and value quotients) are rounded to float32 exactly where stated.
 */
#ifndef CSA_ORACLE_H
#define CSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int max_batch;     /* state slots */
  int rope_dim;      /* rotary slice at the end of the latent; 0 = no RoPE */
  double rope_base;  /* compress_rope_theta */
  double rope_factor;
  int rope_orig_len;
  double beta_fast, beta_slow;
  int fp4;           /* 1 = e2m1 values / e4m3 scales per 16 (the latent); 2 = e2m1 values /
                        power-of-two (e8m0) scales per 32 (the indexer's keys); 0 = off */
  double eps;        /* RMSNorm epsilon */
} oracle_options;

typedef struct oracle_compressor oracle_compressor;

/* ---- number formats ---- */
uint16_t oracle_bf16_from_f32(float v);            /* round to nearest even */
uint16_t oracle_bf16_from_f64(double v);           /* one rounding from double */
float oracle_bf16_to_f32(uint16_t h);
uint8_t oracle_e4m3_from_f32(float v);             /* RNE, saturating to +-448 */
double oracle_e4m3_to_f64(uint8_t bits);
uint8_t oracle_e2m1_from_f32(float v);             /* RNE ties to even code, sign kept, saturating to 6 */
double oracle_e2m1_to_f64(uint8_t code);
/* fp4 round trip of n consecutive blocks of 16 bf16 values. */
void oracle_fp4_e4m3(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out);
/* The indexer's fp4 round trip of n consecutive blocks of 32 bf16 values: codes [n][16],
 * scales [n] e8m0 bytes (2^(byte - 127)), out [n][32] bf16. */
void oracle_fp4_e8m0(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out);

/* ---- RoPE ---- */
/* corrected inverse frequencies f'_i, i < rope_dim/2 */
void oracle_yarn_freqs(int rope_dim, double base, double factor, int orig_len, double beta_fast,
                       double beta_slow, double* freqs);
/* ramp bounds (low, high) of the YaRN correction */
void oracle_yarn_bounds(int rope_dim, double base, int orig_len, double beta_fast, double beta_slow,
                        double* low, double* high);

/* ---- single steps, exposed for the pins ---- */
/* softmax pool of n candidates per feature: out[h] = sum_i w_i[h] kv_i[h]; weights optional [n][H] */
void oracle_pool(const float* kv, const float* score, int n, int H, float* out, double* weights);
/* bf16 round, RMSNorm, RoPE at pos (if rope_dim), into prequant bf16 [H] */
void oracle_epilogue(const oracle_compressor* c, const float* pooled, int64_t pos, uint16_t* prequant);
/* f32 x . w^T for M bf16 rows, out [M][C] */
void oracle_linear(const uint16_t* x, int64_t M, int dim, const float* w, int C, float* out, int nthreads);

/* ---- the compressor ---- */
oracle_compressor* oracle_create(int dim, int head_dim, int ratio, int overlap, const oracle_options* opt);
void oracle_destroy(oracle_compressor* c);
void oracle_set_weights(oracle_compressor* c, const float* wkv, const float* wgate, const float* gain);
/* Prefill (start_pos 0) of B sequences of N tokens (x [B][N][dim] bf16) into state slots
 * slot_offset..slot_offset+B-1.  Writes G = N / ratio entries per sequence to latent [B][G][H]
 * (bf16), codes [B][G][H/2], scales [B][G][H/16], prequant [B][G][H] (each may be NULL).
 * Returns G, or -1 on bad arguments. */
int oracle_prefill(oracle_compressor* c, const uint16_t* x, int B, int N, int slot_offset, uint16_t* latent,
                   uint8_t* codes, uint8_t* scales, uint16_t* prequant, int nthreads);
/* Prefill chunk at start_pos >= 0 shared by the B sequences (start_pos 0: oracle_prefill): the
 * entries of the groups completing in [start_pos, start_pos + N), G = (start_pos + N) / ratio -
 * start_pos / ratio per sequence, to latent [B][G][H] etc.; earlier candidates come from the
 * state; the state receives the new tokens of the unfinished group (and, overlapped, of the
 * last complete group).  Returns G, or -1 on bad arguments. */
int oracle_prefill_chunk(oracle_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                         uint16_t* latent, uint8_t* codes, uint8_t* scales, uint16_t* prequant, int nthreads);
/* Only the listed groups of one sequence x [N][dim]; outputs [ng][...].  State untouched. */
int oracle_prefill_groups(const oracle_compressor* c, const uint16_t* x, int N, const int* groups, int ng,
                          uint16_t* latent, uint8_t* codes, uint8_t* scales, uint16_t* prequant, int nthreads);
/* One decode step for B sequences (slots 0..B-1) at per-sequence positions start_pos[B].
 * Rows of the outputs [B][...] are written only where emitted[b] = 1.  Returns the count. */
int oracle_decode(oracle_compressor* c, const uint16_t* x_tok, int B, const int32_t* start_pos,
                  uint16_t* latent, uint8_t* codes, uint8_t* scales, uint16_t* prequant, uint8_t* emitted,
                  int nthreads);
void oracle_state_reset(oracle_compressor* c);
/* Gate positional bias ([CSA4] "wgate(x) + positional bias"): ape [ratio][C] f32 (C = (1 +
 * overlap) * H, branch A then B), added to the gate logits of a token at position p as
 * ape[p % ratio]; NULL removes it. */
void oracle_set_gate_bias(oracle_compressor* c, const float* ape);
/* state layout: non-overlap [max_batch][ratio][H]; overlap [max_batch][2][4][2H] */
int64_t oracle_state_elems(const oracle_compressor* c);
void oracle_state_export(const oracle_compressor* c, float* kv, float* score);

#ifdef __cplusplus
}
#endif
#endif
