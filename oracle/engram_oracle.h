/*
 * engram_oracle.h -- plain CPU oracle of the Engram hashed n-gram memory lookup.
 *
 * TEST INFRASTRUCTURE ONLY.  This code is the parity reference for the CUDA
 * library: only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load or call it.  It shares no code, header, table or constant with the
 * CUDA path and never calls it.  Slow on purpose: one token at a time, fp64
 * arithmetic, no blocking, no fusion.
 *
 * What it computes (the Engram lookup as described on the VeOmni PR page
 * "support DeepSeek-V4.1-Flash in SeedOmni": tid2eid compression, hashed 2/3/4-gram
 * tables with row-wise FP8 dequantisation, hash ids [batch, sequence, hash_heads],
 * a gated residual write into the four mHC streams; with the hash, mean, gate and
 * add fixed by the workload spec: splitmix64 seeds of n*16+j, the
 * xor-multiply-xorshift fold, row = h mod rows_n, m = mean of the 3H dequantised
 * rows, g = sigmoid(<rmsnorm(stream0), rmsnorm(m)> / sqrt(D)),
 * out_s = stream_s + g * alpha_s * m).
 */
#ifndef ENGRAM_ORACLE_H
#define ENGRAM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error flags, OR-ed into the return value (0 = every output written). */
#define ORC_BAD_TOKEN 1 /* token id outside [0, vocab) */
#define ORC_BAD_EID 2   /* map value outside [0, n_eids], or a negative eid in a window */
#define ORC_BAD_ROW 4   /* row id outside [0, rows_n) */
#define ORC_BAD_ARG 16  /* unusable sizes */

#define ORC_FP8_E4M3FN 0
#define ORC_BF16 1
#define ORC_FP8_E8M0_B32 2 /* FP8 e4m3fn + one e8m0 exponent per row per 32 columns */

/* A dead position (an image span): compresses to this marker, blocks every
 * n-gram that would span it, and its token's row ids are all ORC_DEAD. */
#define ORC_DEAD (-1)

uint64_t orc_splitmix64(uint64_t x);
uint64_t orc_seed(int n, int j);
uint64_t orc_ngram_hash(const int32_t *window, int n, int j);
double orc_e4m3fn_decode(uint8_t byte);
double orc_bf16_decode(uint16_t bits);
double orc_e8m0_decode(uint8_t e);
uint16_t orc_bf16_round(double y);

int orc_compress(const int32_t *token_ids, int64_t n, const int32_t *tid2eid, int32_t vocab,
                 int32_t n_eids, int32_t *eids_out);

int orc_compress_masked(const int32_t *token_ids, int64_t n, const int32_t *tid2eid,
                        int32_t vocab, int32_t n_eids, const uint8_t *dead, int32_t *eids_out);

int orc_hash(const int32_t *eids, int32_t B, int32_t S, const int32_t *history,
             int32_t n_heads, const int64_t rows[3], int32_t *row_ids_out,
             int32_t *history_out);

int orc_hash_packed(const int32_t *eids, int32_t B, int32_t S, const int32_t *positions,
                    const int32_t *history, int32_t n_heads, const int64_t rows[3],
                    int32_t *row_ids_out, int32_t *history_out);

int orc_bucket_primes(int32_t n_layers, int32_t max_ngram, int32_t n_heads, int64_t hash_vocab,
                      int64_t *primes_out);

int orc_hash_bucketed(const int32_t *eids, int32_t B, int32_t S, const int32_t *positions,
                      const int32_t *history, int32_t n_heads, const int64_t *primes,
                      int32_t *row_ids_out, int32_t *history_out);

int orc_lookup(const int32_t *row_ids, int64_t n_tokens, int32_t n_heads, int32_t dtype,
               int32_t D, const void *const tables[3], const void *const scales[3],
               const int64_t rows[3], const uint16_t *streams_in, const float *alpha,
               double eps, uint16_t *streams_out, double *gate_out, double *mem_out);

int orc_connection(const int32_t *row_ids, int64_t n_tokens, int32_t n_heads, int32_t dtype,
                   int32_t d, const void *const tables[3], const void *const scales[3],
                   const int64_t rows[3], const uint16_t *wkv, int32_t D,
                   const uint16_t *streams_in, const float *alpha, double eps,
                   uint16_t *streams_out, double *gate_out, double *k_out);

int orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
