/*
 * engram_oracle.c -- plain CPU oracle of the Engram hashed n-gram memory lookup.
 *
 * TEST INFRASTRUCTURE ONLY (parity reference; see engram_oracle.h).  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares
 * nothing with the CUDA library.  Parity pins: tests/test_oracle_pins.py.
 *
 * Built with -ffp-contract=off so that no a*b+c is fused: every fp64 operation
 * below rounds exactly as written, on x86-64 and on AArch64 alike.
 */
#include "engram_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The multiplier of the n-gram fold, fixed by the workload spec. */
#define ORC_FOLD_MUL 0x9E3779B97F4A7C15ull

/*
 * splitmix64 (S. Vigna, public domain): the first output of a generator whose
 * state is x.  The state is advanced by the golden-ratio increment, then mixed
 * with two xor-shift-multiply rounds and a final xor-shift, all mod 2^64.
 */
uint64_t orc_splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Seed of n-gram order n (2, 3 or 4) and hash head j: splitmix64 of n*16 + j. */
uint64_t orc_seed(int n, int j) { return orc_splitmix64((uint64_t)(n * 16 + j)); }

/*
 * The hash of one n-gram window (oldest id first), for head j:
 * h = seed(n, j); for each id e: h = (h xor e) * FOLD_MUL mod 2^64; h ^= h >> 29.
 * Ids are non-negative and zero-extended to 64 bits.  (VeOmni PR page, commit
 * "n-gram memory lookup": hash ids per n-gram order and head; the fold itself is
 * the workload spec's, the pages do not print one.)
 */
uint64_t orc_ngram_hash(const int32_t *window, int n, int j) {
  uint64_t h = orc_seed(n, j);
  for (int k = 0; k < n; ++k) {
    h = (h ^ (uint64_t)(uint32_t)window[k]) * ORC_FOLD_MUL;
    h ^= h >> 29;
  }
  return h;
}

/*
 * OCP 8-bit floating point, E4M3 "fn" flavour (the pages' fp8_e4m3fn): 1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN;
 * exponent field 0 is subnormal: m * 2^-9.  Normal: (1 + m/8) * 2^(e-7).
 */
double orc_e4m3fn_decode(uint8_t byte) {
  int s = byte >> 7;
  int e = (byte >> 3) & 0xF;
  int m = byte & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/*
 * OCP Microscaling E8M0 scale (the pages' e8m0 block exponents, VeOmni PR page,
 * checkpoint commits): an unsigned 8-bit exponent with bias 127 and no
 * mantissa, 2^(e-127); 0xFF is NaN.
 */
double orc_e8m0_decode(uint8_t e) {
  if (e == 0xFF) return NAN;
  return ldexp(1.0, (int)e - 127);
}

/* bfloat16 is the upper half of an IEEE binary32: widening is exact. */
double orc_bf16_decode(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * Round a double once to the nearest bfloat16, ties to even.  A bfloat16 has 8
 * significant bits, so inside the binade [2^(e-1), 2^e) its spacing is 2^(e-8);
 * below the smallest normal 2^-126 the spacing stays at 2^-133.  Scaling by a
 * power of two is exact, and nearbyint() rounds ties to even in the default
 * rounding mode.  Results beyond the largest finite bfloat16, (2 - 2^-7) * 2^127,
 * become infinities.
 */
uint16_t orc_bf16_round(double y) {
  if (isnan(y)) return 0x7FC0;
  if (isinf(y)) return signbit(y) ? 0xFF80 : 0x7F80;
  if (y == 0.0) return signbit(y) ? 0x8000 : 0x0000;
  int e;
  (void)frexp(fabs(y), &e); /* |y| = f * 2^e, f in [0.5, 1) */
  int ulp_exp = e - 8;
  if (ulp_exp < -133) ulp_exp = -133;
  double r = ldexp(nearbyint(ldexp(y, -ulp_exp)), ulp_exp);
  if (fabs(r) > 0x1.FEp127) return signbit(y) ? 0xFF80 : 0x7F80;
  if (r == 0.0) return signbit(y) ? 0x8000 : 0x0000;
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/*
 * tid2eid compression (VeOmni PR page, PR description and the "n-gram memory
 * lookup" commit: a persistent many-to-one token_map from tokenizer id to
 * compressed id).  eid = tid2eid[tid].  A token id outside [0, vocab) or a map
 * value outside [0, n_eids] leaves that output unwritten and sets a flag.
 */
int orc_compress(const int32_t *token_ids, int64_t n, const int32_t *tid2eid, int32_t vocab,
                 int32_t n_eids, int32_t *eids_out) {
  int flags = 0;
  if (n < 0 || vocab < 1 || n_eids < 0) return ORC_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    int32_t t = token_ids[i];
    if (t < 0 || t >= vocab) {
      flags |= ORC_BAD_TOKEN;
      continue;
    }
    int32_t e = tid2eid[t];
    if (e < 0 || e > n_eids) {
      flags |= ORC_BAD_EID;
      continue;
    }
    eids_out[i] = e;
  }
  return flags;
}

/*
 * tid2eid compression with a dead mask: a dead position (an image span, P3:
 * image-span tokens are dead and break n-grams; P1 pack_ngram_inputs commit: they
 * reach compression marked dead) becomes ORC_DEAD whatever its token id; the
 * others as orc_compress.
 */
int orc_compress_masked(const int32_t *token_ids, int64_t n, const int32_t *tid2eid,
                        int32_t vocab, int32_t n_eids, const uint8_t *dead, int32_t *eids_out) {
  int flags = 0;
  if (n < 0 || vocab < 1 || n_eids < 0) return ORC_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (dead && dead[i]) {
      eids_out[i] = ORC_DEAD;
      continue;
    }
    flags |= orc_compress(token_ids + i, 1, tid2eid, vocab, n_eids, eids_out + i);
  }
  return flags;
}

/*
 * The compressed id at position p of sequence b.  Positions before the start of
 * the call take the caller's history (the last three ids of the earlier
 * sequence, oldest first) when one is given, else the pad id 0: an n-gram never
 * reaches past position 0 (VeOmni PR page, "n-gram memory lookup" commit and the
 * commit on the incremental decode cache: a three-id tail is the whole cache; a
 * blocked lookback compresses to pad).
 */
static int32_t orc_eid_at(const int32_t *eids, int32_t S, const int32_t *history, int32_t b,
                          int32_t p) {
  if (p >= 0) return eids[(int64_t)b * S + p];
  if (history) return history[(int64_t)b * 3 + 3 + p];
  return 0;
}

/*
 * The 4-id window of token (b, s), oldest first (w4[3] is the token's own id),
 * with lookback blocking (VeOmni PR page, "n-gram memory lookup" commit: an
 * n-gram never spans an image span or reaches past position 0; the commit on
 * pack_ngram_inputs: a blocked lookback compresses to pad; the review on packed
 * batches: positions restart at 0 per sample and bound the lookback; the decode
 * cache commit: history sets how far back the walk can read, the start position
 * whether it has reached the true start).  The id k back (k = 1..3) is read only
 * if k <= limit, where limit = positions[b, s] when positions are given, else 3
 * with a history and s without, and only if no id 1..k back is ORC_DEAD; every
 * other slot is the pad id 0.
 * Returns 0, 1 when the token itself is dead, or ORC_BAD_EID for a read id
 * below ORC_DEAD.
 */
static int orc_window(const int32_t *eids, int32_t S, const int32_t *positions,
                      const int32_t *history, int32_t b, int32_t s, int32_t w4[4]) {
  const int32_t self = eids[(int64_t)b * S + s];
  if (self == ORC_DEAD) return 1;
  if (self < 0) return ORC_BAD_EID;
  w4[3] = self;
  int64_t limit = positions ? positions[(int64_t)b * S + s] : (history ? 3 : s);
  int blocked = 0;
  for (int k = 1; k <= 3; ++k) {
    int32_t e = 0;
    if (!blocked && k <= limit && (s - k >= 0 || history)) {
      e = orc_eid_at(eids, S, history, b, s - k);
      if (e == ORC_DEAD) {
        blocked = 1;
        e = 0;
      } else if (e < 0) {
        return ORC_BAD_EID;
      }
    }
    w4[3 - k] = e;
  }
  return 0;
}

/*
 * Hash ids [B, S, 3, H] (n-major: index ((b*S + s)*3 + (n-2))*H + j) for the
 * 2-, 3- and 4-gram ending at every position (NeMo AutoModel page,
 * DeepseekV41Block.forward: engram_hash_ids [batch, sequence, hash_heads]), with
 * positions (may be NULL) giving each token's index within its packed sample.
 * The window of order n is the last n ids of the token's blocked window.  row =
 * h mod rows_n, unsigned, on the full 64-bit h.  A dead token gets ORC_DEAD for
 * all its 3H ids.  A read id below ORC_DEAD leaves all 3H ids of that token
 * unwritten and sets a flag.  history_out (optional) receives the last three
 * ids of history ++ eids, oldest first, dead ones included: the next call's
 * history.
 */
int orc_hash_packed(const int32_t *eids, int32_t B, int32_t S, const int32_t *positions,
                    const int32_t *history, int32_t n_heads, const int64_t rows[3],
                    int32_t *row_ids_out, int32_t *history_out) {
  if (B < 0 || S < 0 || n_heads < 1) return ORC_BAD_ARG;
  for (int n = 0; n < 3; ++n)
    if (rows[n] < 1) return ORC_BAD_ARG;
  const int64_t T = (int64_t)B * S;
  const int R = 3 * n_heads;
  int flags = 0;
#pragma omp parallel for schedule(static) reduction(| : flags)
  for (int64_t t = 0; t < T; ++t) {
    int32_t b = (int32_t)(t / S), s = (int32_t)(t % S);
    int32_t w4[4];
    int st = orc_window(eids, S, positions, history, b, s, w4);
    if (st == ORC_BAD_EID) {
      flags |= ORC_BAD_EID;
      continue;
    }
    for (int r = 0; r < R; ++r) {
      int n = 2 + r / n_heads, j = r % n_heads;
      if (st == 1) {
        row_ids_out[t * R + r] = ORC_DEAD;
        continue;
      }
      uint64_t h = orc_ngram_hash(w4 + (4 - n), n, j); /* ids at s-n+1 .. s */
      row_ids_out[t * R + r] = (int32_t)(h % (uint64_t)rows[n - 2]);
    }
  }
  if (history_out) {
    for (int32_t b = 0; b < B; ++b) {
      int32_t tail[3];
      for (int k = 0; k < 3; ++k) tail[k] = orc_eid_at(eids, S, history, b, S - 3 + k);
      for (int k = 0; k < 3; ++k) history_out[(int64_t)b * 3 + k] = tail[k];
    }
  }
  return flags;
}

/* orc_hash_packed with every sequence starting at position 0 of its sample
 * (or continuing its history). */
int orc_hash(const int32_t *eids, int32_t B, int32_t S, const int32_t *history,
             int32_t n_heads, const int64_t rows[3], int32_t *row_ids_out,
             int32_t *history_out) {
  return orc_hash_packed(eids, B, S, NULL, history, n_heads, rows, row_ids_out, history_out);
}

/* n is prime: trial division by every d with d*d <= n. */
static int orc_is_prime(int64_t n) {
  if (n < 2) return 0;
  for (int64_t d = 2; d * d <= n; ++d)
    if (n % d == 0) return 0;
  return 1;
}

/*
 * The released prime-bucket layout (VeOmni PR page, "n-gram memory lookup"
 * commit: the bucket layout reproduces the release's prime draw by trial
 * division; the commit on hash_vocab_size: the primes are drawn above the hash
 * vocabulary; the review on validate_bucket_layout: a table needs at least the
 * sum of its layer's primes).  For every layer, every order n = 2..max_ngram and
 * every head j, in that order: the smallest prime >= hash_vocab + (the heads
 * already drawn for this order) that no earlier bucket uses; each order starts
 * again from hash_vocab.  primes_out gets n_layers * (max_ngram - 1) * n_heads
 * primes in draw order.
 */
int orc_bucket_primes(int32_t n_layers, int32_t max_ngram, int32_t n_heads, int64_t hash_vocab,
                      int64_t *primes_out) {
  if (n_layers < 1 || max_ngram < 2 || n_heads < 1 || hash_vocab < 1) return ORC_BAD_ARG;
  const int64_t total = (int64_t)n_layers * (max_ngram - 1) * n_heads;
  int64_t k = 0;
  for (int32_t l = 0; l < n_layers; ++l)
    for (int32_t n = 2; n <= max_ngram; ++n) {
      int64_t cand = hash_vocab - 1;
      for (int32_t j = 0; j < n_heads; ++j) {
        ++cand;
        for (;;) {
          int used = 0;
          for (int64_t q = 0; q < k && !used; ++q) used = primes_out[q] == cand;
          if (!used && orc_is_prime(cand)) break;
          ++cand;
        }
        primes_out[k++] = cand;
      }
    }
  return k == total ? 0 : ORC_BAD_ARG;
}

/*
 * Hash ids into one table cut into prime buckets: the bucket of order n, head j
 * (r = (n-2)*H + j) has primes[r] rows and starts at the sum of the buckets
 * before it in draw order; row = offset_r + (h mod primes[r]), h the n-gram hash
 * of orc_hash_packed's blocked window.  Dead tokens, flags and history_out as in
 * orc_hash_packed.
 */
int orc_hash_bucketed(const int32_t *eids, int32_t B, int32_t S, const int32_t *positions,
                      const int32_t *history, int32_t n_heads, const int64_t *primes,
                      int32_t *row_ids_out, int32_t *history_out) {
  if (B < 0 || S < 0 || n_heads < 1) return ORC_BAD_ARG;
  const int R = 3 * n_heads;
  for (int r = 0; r < R; ++r)
    if (primes[r] < 1) return ORC_BAD_ARG;
  const int64_t T = (int64_t)B * S;
  int flags = 0;
#pragma omp parallel for schedule(static) reduction(| : flags)
  for (int64_t t = 0; t < T; ++t) {
    int32_t b = (int32_t)(t / S), s = (int32_t)(t % S);
    int32_t w4[4];
    int st = orc_window(eids, S, positions, history, b, s, w4);
    if (st == ORC_BAD_EID) {
      flags |= ORC_BAD_EID;
      continue;
    }
    int64_t offset = 0;
    for (int r = 0; r < R; ++r) {
      int n = 2 + r / n_heads, j = r % n_heads;
      if (st == 1) {
        row_ids_out[t * R + r] = ORC_DEAD;
      } else {
        uint64_t h = orc_ngram_hash(w4 + (4 - n), n, j);
        row_ids_out[t * R + r] = (int32_t)(offset + (int64_t)(h % (uint64_t)primes[r]));
      }
      offset += primes[r];
    }
  }
  if (history_out) {
    for (int32_t b = 0; b < B; ++b) {
      int32_t tail[3];
      for (int k = 0; k < 3; ++k) tail[k] = orc_eid_at(eids, S, history, b, S - 3 + k);
      for (int k = 0; k < 3; ++k) history_out[(int64_t)b * 3 + k] = tail[k];
    }
  }
  return flags;
}

/*
 * The fused lookup for n_tokens tokens, one at a time, in fp64:
 *  1. gather + dequantise the 3H rows of the token: FP8 byte decoded exactly,
 *     times the row's fp32 scale (VeOmni PR page: FP8 tables with row-wise
 *     dequantisation on lookup), or times the e8m0 exponent of its row's
 *     32-column block (the release's (1, 32) blocking), or the BF16 value
 *     widened exactly;
 *  2. m = (sum of the 3H rows) / (3H)  (workload spec: the mean of the rows);
 *  3. with a = stream 0 of the token:
 *     g = sigmoid( sum(a*m) / (sqrt(mean(a^2)+eps) * sqrt(mean(m^2)+eps) * sqrt(D)) ),
 *     which is <rmsnorm(a), rmsnorm(m)> / sqrt(D) with unit RMSNorm weights;
 *  4. out_s = bf16_round(stream_s + g * alpha_s * m), rounded once, for the four
 *     streams [tokens, 4, D] (VeOmni PR page: the Engram write goes into the mHC
 *     streams before its layer; NeMo AutoModel page: streams [batch, sequence,
 *     streams, hidden]).
 * A row id outside [0, rows_n) leaves the token's outputs unwritten and sets a
 * flag; a token whose 3H ids are all ORC_DEAD passes through with g = 0 and
 * m = 0 (some but not all dead is a bad row).  gate_out [n_tokens] and mem_out
 * [n_tokens, D] are optional.
 */
int orc_lookup(const int32_t *row_ids, int64_t n_tokens, int32_t n_heads, int32_t dtype,
               int32_t D, const void *const tables[3], const void *const scales[3],
               const int64_t rows[3], const uint16_t *streams_in, const float *alpha,
               double eps, uint16_t *streams_out, double *gate_out, double *mem_out) {
  if (n_tokens < 0 || n_heads < 1 || D < 1) return ORC_BAD_ARG;
  if (dtype != ORC_FP8_E4M3FN && dtype != ORC_BF16 && dtype != ORC_FP8_E8M0_B32) return ORC_BAD_ARG;
  if (dtype == ORC_FP8_E8M0_B32 && D % 32) return ORC_BAD_ARG;
  const int R = 3 * n_heads;
  int flags = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : flags)
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int32_t *ids = row_ids + t * R;
    int bad = 0, dead = 0;
    for (int r = 0; r < R; ++r) {
      int n = r / n_heads;
      if (ids[r] == ORC_DEAD)
        ++dead;
      else if (ids[r] < 0 || (int64_t)ids[r] >= rows[n])
        bad = 1;
    }
    if (bad || (dead && dead != R)) {
      flags |= ORC_BAD_ROW;
      continue;
    }
    if (dead) {
      /* A dead token's gate is zeroed (vLLM page, DeepseekV4Model.forward: the
       * Engram mask keeps live tokens only): its streams pass through unchanged. */
      const uint16_t *xd = streams_in + t * 4 * (int64_t)D;
      uint16_t *yd = streams_out + t * 4 * (int64_t)D;
      if (yd != xd) memcpy(yd, xd, (size_t)4 * D * sizeof(uint16_t));
      if (gate_out) gate_out[t] = 0.0;
      if (mem_out)
        for (int i = 0; i < D; ++i) mem_out[t * D + i] = 0.0;
      continue;
    }
    double *m = (double *)calloc((size_t)D, sizeof(double));
    for (int r = 0; r < R; ++r) {
      int n = r / n_heads;
      int64_t row = ids[r];
      for (int i = 0; i < D; ++i) {
        double v;
        if (dtype == ORC_FP8_E4M3FN) {
          const uint8_t *tab = (const uint8_t *)tables[n];
          v = orc_e4m3fn_decode(tab[row * D + i]) * (double)((const float *)scales[n])[row];
        } else if (dtype == ORC_FP8_E8M0_B32) {
          /* (1, 32) blocks: one exponent per row per 32 columns (VeOmni PR page, the
           * commit on the tables' per-row block scales) */
          const uint8_t *tab = (const uint8_t *)tables[n];
          const uint8_t *sc = (const uint8_t *)scales[n];
          v = orc_e4m3fn_decode(tab[row * D + i]) * orc_e8m0_decode(sc[row * (D / 32) + i / 32]);
        } else {
          const uint16_t *tab = (const uint16_t *)tables[n];
          v = orc_bf16_decode(tab[row * D + i]);
        }
        m[i] += v;
      }
    }
    for (int i = 0; i < D; ++i) m[i] /= (double)R;

    const uint16_t *x = streams_in + t * 4 * (int64_t)D;
    double saa = 0.0, smm = 0.0, sam = 0.0;
    for (int i = 0; i < D; ++i) {
      double a = orc_bf16_decode(x[i]);
      saa += a * a;
      smm += m[i] * m[i];
      sam += a * m[i];
    }
    double rms_a = sqrt(saa / D + eps);
    double rms_m = sqrt(smm / D + eps);
    double logit = sam / (rms_a * rms_m * sqrt((double)D));
    double g = 1.0 / (1.0 + exp(-logit));

    uint16_t *y = streams_out + t * 4 * (int64_t)D;
    for (int s = 0; s < 4; ++s)
      for (int i = 0; i < D; ++i) {
        double xi = orc_bf16_decode(x[(int64_t)s * D + i]);
        y[(int64_t)s * D + i] = orc_bf16_round(xi + g * (double)alpha[s] * m[i]);
      }
    if (gate_out) gate_out[t] = g;
    if (mem_out)
      for (int i = 0; i < D; ++i) mem_out[t * D + i] = m[i];
    free(m);
  }
  return flags;
}

/*
 * The Engram connection with a wkv projection (VeOmni PR page, "n-gram memory
 * lookup" commit and the layer commit: the other half of Engram, wkv and the
 * gate, reads the mHC streams; the rows cross to it as n-gram embeddings).  The
 * pages give no shapes or formula; the reading implemented here: per token,
 *  1. e = the 3H dequantised rows of width d concatenated in (order, head)
 *     order, K = 3H*d values (FP8 with e8m0 blocks or BF16: exact in bf16);
 *  2. k = wkv e, wkv bf16 [D, K] (row j holds output j's weights), in fp64;
 *  3. g = sigmoid(<rmsnorm(stream0), rmsnorm(k)> / sqrt(D)), the spec's gate
 *     with k in place of the mean;
 *  4. out_s = bf16_round(stream_s + g * alpha_s * k), rounded once.
 * Bad rows and dead tokens as in orc_lookup.  gate_out [n_tokens] and k_out
 * [n_tokens, D] are optional.
 */
int orc_connection(const int32_t *row_ids, int64_t n_tokens, int32_t n_heads, int32_t dtype,
                   int32_t d, const void *const tables[3], const void *const scales[3],
                   const int64_t rows[3], const uint16_t *wkv, int32_t D,
                   const uint16_t *streams_in, const float *alpha, double eps,
                   uint16_t *streams_out, double *gate_out, double *k_out) {
  if (n_tokens < 0 || n_heads < 1 || d < 1 || D < 1) return ORC_BAD_ARG;
  if (dtype != ORC_BF16 && dtype != ORC_FP8_E8M0_B32) return ORC_BAD_ARG;
  if (dtype == ORC_FP8_E8M0_B32 && d % 32) return ORC_BAD_ARG;
  const int R = 3 * n_heads;
  const int64_t K = (int64_t)R * d;
  int flags = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : flags)
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int32_t *ids = row_ids + t * R;
    int bad = 0, dead = 0;
    for (int r = 0; r < R; ++r) {
      if (ids[r] == ORC_DEAD)
        ++dead;
      else if (ids[r] < 0 || (int64_t)ids[r] >= rows[r / n_heads])
        bad = 1;
    }
    if (bad || (dead && dead != R)) {
      flags |= ORC_BAD_ROW;
      continue;
    }
    const uint16_t *x = streams_in + t * 4 * (int64_t)D;
    uint16_t *y = streams_out + t * 4 * (int64_t)D;
    if (dead) {
      if (y != x) memcpy(y, x, (size_t)4 * D * sizeof(uint16_t));
      if (gate_out) gate_out[t] = 0.0;
      if (k_out)
        for (int i = 0; i < D; ++i) k_out[t * D + i] = 0.0;
      continue;
    }
    double *e = (double *)malloc((size_t)K * sizeof(double));
    double *k = (double *)calloc((size_t)D, sizeof(double));
    for (int r = 0; r < R; ++r) {
      const int n = r / n_heads;
      const int64_t row = ids[r];
      for (int i = 0; i < d; ++i) {
        double v;
        if (dtype == ORC_FP8_E8M0_B32)
          v = orc_e4m3fn_decode(((const uint8_t *)tables[n])[row * d + i]) *
              orc_e8m0_decode(((const uint8_t *)scales[n])[row * (d / 32) + i / 32]);
        else
          v = orc_bf16_decode(((const uint16_t *)tables[n])[row * d + i]);
        e[(int64_t)r * d + i] = v;
      }
    }
    for (int j = 0; j < D; ++j) {
      double acc = 0.0;
      for (int64_t i = 0; i < K; ++i) acc += orc_bf16_decode(wkv[(int64_t)j * K + i]) * e[i];
      k[j] = acc;
    }
    double saa = 0.0, skk = 0.0, sak = 0.0;
    for (int i = 0; i < D; ++i) {
      double a = orc_bf16_decode(x[i]);
      saa += a * a;
      skk += k[i] * k[i];
      sak += a * k[i];
    }
    double logit = sak / (sqrt(saa / D + eps) * sqrt(skk / D + eps) * sqrt((double)D));
    double g = 1.0 / (1.0 + exp(-logit));
    for (int s = 0; s < 4; ++s)
      for (int i = 0; i < D; ++i)
        y[(int64_t)s * D + i] =
            orc_bf16_round(orc_bf16_decode(x[(int64_t)s * D + i]) + g * (double)alpha[s] * k[i]);
    if (gate_out) gate_out[t] = g;
    if (k_out)
      for (int i = 0; i < D; ++i) k_out[t * D + i] = k[i];
    free(e);
    free(k);
  }
  return flags;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
