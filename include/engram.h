/*
 * engram.h -- C ABI of libengram, the GB300 (sm_103a) Engram hashed n-gram memory
 * lookup.
 *
 * The Engram lookup, as the pages describe it (VeOmni PR "support
 * DeepSeek-V4.1-Flash in SeedOmni", PR description and commit "n-gram memory
 * lookup"; NeMo AutoModel page, DeepseekV41Block.forward; vLLM page,
 * DeepseekV4Model.forward): token ids are compressed through a many-to-one
 * tid2eid map; the 2-, 3- and 4-gram windows of compressed ids are hashed into
 * row ids [batch, sequence, hash_heads]; the rows are gathered from three tables
 * (FP8 e4m3fn with a per-row scale, dequantised on lookup, or BF16); and a gated
 * memory is added into the four mHC residual streams [batch, sequence, 4, hidden]
 * before the layer.  The pages leave the hash, the combine and the gate open; this
 * library implements them as follows:
 *   seed(n, j)  = splitmix64(n*16 + j)            (first output, state n*16+j)
 *   h           = seed; for each id e of the window, oldest first:
 *                 h = (h ^ e) * 0x9E3779B97F4A7C15 mod 2^64;  h ^= h >> 29
 *   row(n, j)   = h mod rows_n                     (unsigned, full 64-bit h)
 *   m           = mean of the 3H dequantised rows  (fp32 accumulation)
 *   g           = sigmoid( <rmsnorm(stream0), rmsnorm(m)> / sqrt(D) ),
 *                 rmsnorm(x) = x / sqrt(mean(x^2) + eps), no learned weight
 *   out_s       = bf16_rne(stream_s + g * alpha_s * m),  s = 0..3
 *
 * Conventions for every call:
 *  - Pointers named *_host are host memory; every other data pointer is device
 *    memory on the current CUDA device, except the members of engram_layout,
 *    whose memory the struct's comment states per call.  All memory is owned
 *    and allocated by the caller; the library allocates nothing and keeps no
 *    pointer after a call.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous on it; the library never synchronises
 *    except in engram_read_status.
 *  - Host-side argument errors are returned synchronously, before any launch:
 *    nothing is written.  engram_last_error() then describes the argument.
 *  - Data errors found on the device (a token id outside the vocabulary, a map
 *    value or id out of range, a row id outside its table) never trap: the
 *    kernel OR-s an ENGRAM_FLAG_* bit into *status (optional device int32; may be
 *    NULL) and leaves that element's outputs unwritten.  Read the word with
 *    engram_read_status or any device-to-host copy.
 *  - bf16 values travel as their uint16 bit patterns.
 *  - Requires a compute-capability 10.3 device (GB300); others get
 *    ENGRAM_ERR_UNSUPPORTED.
 */
#ifndef ENGRAM_H
#define ENGRAM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ENGRAM_API __attribute__((visibility("default")))
#else
#define ENGRAM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t engram_status;

#define ENGRAM_OK 0
#define ENGRAM_ERR_INVALID_ARG 1  /* null, size, alignment, aliasing, range of an argument */
#define ENGRAM_ERR_UNSUPPORTED 2  /* device is not sm_103, or a size beyond the limits below */
#define ENGRAM_ERR_CUDA 3         /* a CUDA runtime call or kernel launch failed */
#define ENGRAM_ERR_OUT_OF_RANGE 4 /* engram_read_status: a data range flag was set */
#define ENGRAM_ERR_TIMEOUT 5      /* engram_read_status: a bounded device wait gave up */

/* Bits of the device status word. */
#define ENGRAM_FLAG_BAD_TOKEN 1 /* token id outside [0, vocab) */
#define ENGRAM_FLAG_BAD_EID 2   /* tid2eid value outside [0, n_eids], or a negative id */
#define ENGRAM_FLAG_BAD_ROW 4   /* row id outside [0, rows_n) */
#define ENGRAM_FLAG_TIMEOUT 8   /* a bounded wait inside a kernel gave up */

#define ENGRAM_MAX_HEADS 32   /* hash heads per n-gram order */
#define ENGRAM_MAX_D 4096     /* row width = hidden size; D % 16 == 0 */

#define ENGRAM_TABLE_FP8_E4M3FN 0
#define ENGRAM_TABLE_BF16 1
#define ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 2
#define ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS 3

/* Bytes of one row of an ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS table of width D. */
#define ENGRAM_E8M0_ROW_BYTES(D) ((((int64_t)(D) + (int64_t)(D) / 32) + 15) / 16 * 16)

/*
 * Dead positions (image spans: vLLM page, DeepseekV4Model.forward, they break
 * n-grams and their gate is zeroed; VeOmni PR page, pack_ngram_inputs commit,
 * a blocked lookback compresses to pad): a dead position's compressed id is
 * ENGRAM_EID_DEAD; an n-gram never spans it (the ids at and before it read as
 * the pad id 0, as before a sequence start); the dead token's own 3H row ids
 * are ENGRAM_ROW_DEAD, and engram_lookup_fused passes such a token's streams
 * through unchanged (g = 0).
 */
#define ENGRAM_EID_DEAD (-1)
#define ENGRAM_ROW_DEAD (-1)

/*
 * The three n-gram tables (index 0, 1, 2 = orders 2, 3, 4), row-major
 * [rows[n], D], each 16-byte aligned, in one of three formats:
 *  - ENGRAM_TABLE_FP8_E4M3FN: one byte per element (OCP E4M3, "fn": bias 7, max
 *    448, no infinities); scale[n] = float [rows[n]], the row's dequantisation
 *    factor (VeOmni PR page: FP8 tables with row-wise dequantisation on lookup).
 *  - ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32: the same bytes; scale[n] = uint8
 *    [rows[n], D/32], one OCP E8M0 exponent per row per 32 columns (value
 *    2^(e-127), 0xFF NaN), 16-byte aligned; D % 32 == 0 (VeOmni PR page: the
 *    release blocks its tables (1, 32)).  The products are exact powers of two
 *    times the FP8 value, within the fp32 range.
 *  - ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS: the values of the previous format with
 *    each row's exponents stored right after its bytes: row r of table[n] is
 *    ENGRAM_E8M0_ROW_BYTES(D) bytes, its D e4m3fn bytes, its D/32 e8m0
 *    exponents, then zero padding to a multiple of 16 bytes; scale[n] unused
 *    (may be NULL); D % 32 == 0.  Not on the pages: a storage layout of this
 *    library, made by engram_pack_e8m0_rows, in which a lookup reads a row
 *    and its exponents as one contiguous run.  Every call gives the same
 *    results for it as for ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32.
 *  - ENGRAM_TABLE_BF16: two bytes per element; scale[n] ignored.
 * 1 <= rows[n] <= 2^31 - 1.  The struct itself is read on the host during the
 * call only.
 */
typedef struct engram_tables {
  int32_t dtype; /* ENGRAM_TABLE_* */
  int32_t D;     /* row width, multiple of 16 (32 for E8M0 blocks), 16..ENGRAM_MAX_D */
  int64_t rows[3];
  const void *table[3];
  const void *scale[3];
} engram_tables;

/*
 * engram_compress -- tid2eid canonical token compression (VeOmni PR page, PR
 * description and commit "n-gram memory lookup": a persistent many-to-one
 * token_map baked at conversion time; the pad id 0 is what an unhashable
 * position compresses to).
 *   eids_out[i] = tid2eid[token_ids[i]],  i < n_tokens
 * token_ids, eids_out: int32 [n_tokens] (may alias each other: in place is
 * allowed); tid2eid: int32 [vocab], values expected in [0, n_eids].
 * A token outside [0, vocab) sets ENGRAM_FLAG_BAD_TOKEN, a map value outside
 * [0, n_eids] sets ENGRAM_FLAG_BAD_EID; that eids_out[i] is not written.
 * n_tokens == 0 launches nothing and returns ENGRAM_OK.
 */
ENGRAM_API engram_status engram_compress(const int32_t *token_ids, int64_t n_tokens,
                                         const int32_t *tid2eid, int32_t vocab, int32_t n_eids,
                                         int32_t *eids_out, int32_t *status, void *stream);

/*
 * engram_compress_masked -- engram_compress with a dead mask: dead[i] != 0
 * (uint8 [n_tokens], device) makes eids_out[i] = ENGRAM_EID_DEAD whatever the
 * token id (no range check for it); dead may be NULL (then as engram_compress).
 */
ENGRAM_API engram_status engram_compress_masked(const int32_t *token_ids, int64_t n_tokens,
                                                const int32_t *tid2eid, int32_t vocab,
                                                int32_t n_eids, const uint8_t *dead,
                                                int32_t *eids_out, int32_t *status,
                                                void *stream);

/*
 * engram_hash -- n-gram hash ids per order and head (VeOmni PR page, commit
 * "n-gram memory lookup" and the commit on the incremental decode cache: a
 * window never reaches past position 0; a three-id tail of history is the whole
 * cache and is exact; NeMo AutoModel page: engram_hash_ids [batch, sequence,
 * hash_heads]).
 *   eids        int32 [batch, seq] compressed ids (>= 0, or ENGRAM_EID_DEAD)
 *   history     int32 [batch, 3] or NULL: the three ids before position 0,
 *               oldest first; NULL means every sequence starts here (positions
 *               before 0 are the pad id 0)
 *   history_out int32 [batch, 3] or NULL: receives the last three ids of
 *               history ++ eids, oldest first (the next call's history).  It
 *               may be the same buffer as history; it must not overlap eids or
 *               row_ids_out.
 *   rows_host   host int64 [3]: rows of the 2-, 3-, 4-gram tables, 1..2^31-1
 *   row_ids_out int32 [batch, seq, 3, n_heads], n-major: the row for order n,
 *               head j of token (b, s) is at ((b*seq + s)*3 + n-2)*n_heads + j
 * The window of order n at (b, s) is ids s-n+1 .. s, read back from s until
 * the lookback limit (s without a history, 3 with one) or a dead id, whichever
 * comes first; the slots beyond read as the pad id 0.  A dead token gets
 * ENGRAM_ROW_DEAD for all its ids.  A read id below ENGRAM_EID_DEAD sets
 * ENGRAM_FLAG_BAD_EID and leaves that token's 3*n_heads ids unwritten.
 * history_out carries dead ids like any other.  1 <= n_heads <= ENGRAM_MAX_HEADS.
 */
ENGRAM_API engram_status engram_hash(const int32_t *eids, int32_t batch, int32_t seq,
                                     const int32_t *history, int32_t *history_out,
                                     int32_t n_heads, const int64_t *rows_host,
                                     int32_t *row_ids_out, int32_t *status, void *stream);

/*
 * engram_hash_packed -- engram_hash for packed batches and resumed sequences:
 * positions (int32 [batch, seq], device; may be NULL) gives every token's index
 * within its own sample, restarting at 0 where a new sample starts (VeOmni PR
 * page, review of pack_ngram_inputs: n-gram hashes never cross sample
 * boundaries in a packed micro-batch).  The lookback limit of (b, s) is
 * positions[b, s]: a window never reaches before its sample's start, in the
 * batch or in the history (decode cache commit: the history sets how far back
 * the walk can read, the start position whether it reached the true start).
 * NULL positions is engram_hash.
 */
ENGRAM_API engram_status engram_hash_packed(const int32_t *eids, int32_t batch, int32_t seq,
                                            const int32_t *positions, const int32_t *history,
                                            int32_t *history_out, int32_t n_heads,
                                            const int64_t *rows_host, int32_t *row_ids_out,
                                            int32_t *status, void *stream);

/*
 * engram_bucket_primes -- the released table layout's bucket sizes (VeOmni PR
 * page: "n-gram memory lookup" commit, the bucket layout reproduces the
 * release's prime draw, giving 384006168 / 384016682 rows for its two Engram
 * layers; the commit on hash_vocab_size: primes drawn above the hash vocabulary;
 * the review on validate_bucket_layout: 462 for 1 layer, max n-gram 4, 2 heads,
 * vocabulary 64).  For every layer, every order n = 2..max_ngram and every head,
 * in that order, the smallest prime >= hash_vocab, counting up from the last
 * prime of the same order, that no earlier bucket took; every order starts
 * again from hash_vocab.  Host-only: writes n_layers * (max_ngram-1) * n_heads
 * int64 primes to primes_out_host in draw order (at most 65536).
 */
ENGRAM_API engram_status engram_bucket_primes(int32_t n_layers, int32_t max_ngram, int32_t n_heads,
                                              int64_t hash_vocab, int64_t *primes_out_host);

/*
 * engram_hash_bucketed -- engram_hash_packed into one table cut into prime
 * buckets (the released layout): the bucket of order n and head j has
 * primes_host[(n-2)*n_heads + j] rows and starts after the buckets before it in
 * that order; its row id is offset + (h mod prime).  primes_host: host int64
 * [3 * n_heads] (one layer's orders 2..4 from engram_bucket_primes); their sum
 * must be <= 2^31 - 1 and at most the table's rows.  For engram_lookup_fused,
 * pass that one table as table[0..2] (with its scales) and its rows as
 * rows[0..2].
 */
ENGRAM_API engram_status engram_hash_bucketed(const int32_t *eids, int32_t batch, int32_t seq,
                                              const int32_t *positions, const int32_t *history,
                                              int32_t *history_out, int32_t n_heads,
                                              const int64_t *primes_host, int32_t *row_ids_out,
                                              int32_t *status, void *stream);

/*
 * engram_compress_hash -- engram_compress_masked then engram_hash_packed (or
 * engram_hash_bucketed) as one launch: the hash compresses the ids of every
 * window itself (the map is small and stays cached), so the compressed ids make
 * no round trip through memory.  For valid input the row ids, history_out and
 * (when eids_out is given) the compressed ids equal those of the two calls.
 *   token_ids   int32 [batch, seq] (device); tid2eid, vocab, n_eids as for
 *               engram_compress
 *   history, history_out, n_heads, row_ids_out as for engram_hash
 *   rows_host   as for engram_hash; not read when layout_host->primes is given
 *   layout_host positions and dead mask in DEVICE memory, bucket primes on the
 *               host (engram_layout, below); NULL for the plain case
 *   eids_out    int32 [batch, seq] or NULL: the compressed ids
 * A token id outside [0, vocab) sets ENGRAM_FLAG_BAD_TOKEN, a map value outside
 * [0, n_eids] ENGRAM_FLAG_BAD_EID; that token's compressed id and row ids stay
 * unwritten, as do the row ids of every token whose window reaches it
 * (ENGRAM_FLAG_BAD_EID) and history_out of a sequence whose last three ids
 * hold it.  None of the outputs may overlap an input.
 */
struct engram_layout;
ENGRAM_API engram_status engram_compress_hash(
    const int32_t *token_ids, int32_t batch, int32_t seq, const int32_t *tid2eid, int32_t vocab,
    int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const int64_t *rows_host, const struct engram_layout *layout_host, int32_t *eids_out,
    int32_t *row_ids_out, int32_t *status, void *stream);

/*
 * engram_lookup_fused -- gather + dequantise the 3*n_heads rows of every token,
 * average them into m, gate with g = sigmoid(<rmsnorm(stream0), rmsnorm(m)> /
 * sqrt(D)) and add g * alpha_s * m into the four mHC streams (VeOmni PR page:
 * FP8 row-wise dequantisation on lookup, the Engram write goes into the streams
 * before its layer; NeMo AutoModel page: streams [batch, sequence, streams,
 * hidden]).  One pass over HBM: rows, stream 0..3 in, stream 0..3 out.
 *   row_ids     int32 [n_tokens, 3*n_heads] as written by engram_hash
 *   tables_host host struct describing the device tables (above)
 *   streams_in  bf16 bits [n_tokens, 4, D], 16-byte aligned
 *   streams_out bf16 bits [n_tokens, 4, D], 16-byte aligned; either exactly
 *               streams_in (in place) or not overlapping it
 *   alpha       fp32 [4] device: per-stream scale of the memory
 *   eps         RMSNorm epsilon, finite, >= 0
 *   gate_out    fp32 [n_tokens] or NULL: g per token
 *   mem_out     fp32 [n_tokens, D] or NULL (16-byte aligned): m per token
 * A row id outside its table sets ENGRAM_FLAG_BAD_ROW and leaves the token's
 * outputs unwritten.  A token whose 3*n_heads ids are all ENGRAM_ROW_DEAD is a
 * dead token: nothing is gathered, its streams are copied through unchanged
 * (nothing is written in place), g = 0 and m = 0; some dead and some live ids
 * is a bad row.
 */
ENGRAM_API engram_status engram_lookup_fused(const int32_t *row_ids, int64_t n_tokens,
                                             int32_t n_heads, const engram_tables *tables_host,
                                             const uint16_t *streams_in, uint16_t *streams_out,
                                             const float *alpha, float eps, float *gate_out,
                                             float *mem_out, int32_t *status, void *stream);

/*
 * engram_connection -- the Engram connection with a wkv projection in place of
 * the mean: the other half of Engram, "wkv and the gate", which reads the mHC
 * streams (VeOmni PR page, "n-gram memory lookup" commit and the DeepSeek-V4.1
 * layer commit; the gathered rows cross to it as n-gram embeddings, about 24 KB
 * a token = 3 orders x 8 heads x 256 columns x 2 layers x 2 bytes).  The pages give
 * no formula; this library reads it as, per token with K = 3*n_heads*d:
 *   e     = the 3*n_heads dequantised rows concatenated in (order, head) order,
 *           K values, each exact in bf16 (BF16 tables, or FP8 e4m3fn with
 *           (1, 32) e8m0 block exponents, apart or after each row)
 *   k     = wkv e, fp32 accumulation on the tensor cores (wkv bf16 [D, K],
 *           row j = output j's weights)
 *   g     = sigmoid(<rmsnorm(stream0), rmsnorm(k)> / sqrt(D)), as above with k
 *           in place of m
 *   out_s = bf16_rne(stream_s + g * alpha_s * k)
 * Three launches on `stream`: the rows into E (bf16 [n_tokens, K], workspace),
 * k = E wkv^T (tcgen05 tensor cores, TMA, fp32 in tensor memory), then the gate
 * and the add.
 *   row_ids      int32 [n_tokens, 3*n_heads], as for engram_lookup_fused
 *   tables_host  dtype ENGRAM_TABLE_BF16, ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 or
 *                ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS; D (the row width d) a
 *                multiple of 32
 *   wkv          bf16 bits [D, K], 16-byte aligned; D a multiple of 256 in
 *                [256, 8192] and K a multiple of 64
 *   streams_in / streams_out / alpha / eps / gate_out as engram_lookup_fused
 *   workspace    device, 256-byte aligned, at least
 *                engram_connection_workspace_bytes(n_tokens, n_heads, d, D)
 *                bytes, owned by the caller, busy until the call's kernels end
 *   k_out        fp32 [n_tokens, D] or NULL (16-byte aligned): k per token (0
 *                for a dead or bad token); NULL keeps k in the workspace
 * Dead tokens and bad rows as engram_lookup_fused.  A projection that does not
 * complete within the wait limit sets ENGRAM_FLAG_TIMEOUT and leaves k
 * unwritten for its tile.  Other table types give ENGRAM_ERR_UNSUPPORTED.
 */
ENGRAM_API size_t engram_connection_workspace_bytes(int64_t n_tokens, int32_t n_heads, int32_t d,
                                                    int32_t D);
ENGRAM_API engram_status engram_connection(const int32_t *row_ids, int64_t n_tokens,
                                           int32_t n_heads, const engram_tables *tables_host,
                                           const uint16_t *wkv, int32_t D,
                                           const uint16_t *streams_in, uint16_t *streams_out,
                                           const float *alpha, float eps, void *workspace,
                                           size_t workspace_bytes, float *gate_out, float *k_out,
                                           int32_t *status, void *stream);

/*
 * The three stages of engram_connection as calls of their own (the same kernels,
 * for callers that keep E or k, and for timing the projection alone):
 *
 * engram_concat_rows -- E[t] = the token's 3*n_heads dequantised rows in (order,
 *   head) order, bf16 bits [n_tokens, K], K = 3*n_heads*d (e_out 16-byte
 *   aligned), and state_out uint8 [n_tokens]: 0 live, 1 dead (every id
 *   ENGRAM_ROW_DEAD; E[t] = 0), 2 bad row (ENGRAM_FLAG_BAD_ROW raised; E[t] = 0).
 *   Tables as for engram_connection.
 * engram_wkv_project -- k = E wkv^T: e bf16 bits [n_tokens, K], wkv bf16 bits [D,
 *   K], k_out fp32 [n_tokens, D]; all 16-byte aligned; D a multiple of 256 in
 *   [256, 8192], K a multiple of 64.  tcgen05 tensor cores, fp32 accumulation.
 * engram_gate_add -- per token with state 0: g = sigmoid(<rmsnorm(stream0),
 *   rmsnorm(k)> / sqrt(D)), out_s = bf16_rne(stream_s + g * alpha_s * k); state
 *   1: streams copied through, g = 0; state 2: nothing written.  k fp32 [n_tokens,
 *   D] (16-byte aligned), D a multiple of 16 in [16, 8192]; streams, alpha, eps
 *   and gate_out as engram_lookup_fused.
 */
ENGRAM_API engram_status engram_concat_rows(const int32_t *row_ids, int64_t n_tokens,
                                            int32_t n_heads, const engram_tables *tables_host,
                                            uint16_t *e_out, uint8_t *state_out, int32_t *status,
                                            void *stream);
ENGRAM_API engram_status engram_wkv_project(const uint16_t *e, int64_t n_tokens, int32_t K,
                                            const uint16_t *wkv, int32_t D, float *k_out,
                                            int32_t *status, void *stream);
ENGRAM_API engram_status engram_gate_add(const float *k, const uint8_t *state, int64_t n_tokens,
                                         int32_t D, const uint16_t *streams_in,
                                         uint16_t *streams_out, const float *alpha, float eps,
                                         float *gate_out, void *stream);

/*
 * engram_layout -- how a batch is packed and how the tables are cut, for the
 * whole-path calls below.  A NULL struct, or NULL members, mean the plain case:
 * every sequence is one sample from position 0, nothing is dead, and order n
 * has its own table of tables_host->rows[n-2] rows.
 *   positions  int32 [batch, seq]: each token's index within its own sample,
 *              as for engram_hash_packed (VeOmni PR page, review of
 *              pack_ngram_inputs: no n-gram crosses a sample boundary)
 *   dead       uint8 [batch*seq]: non-zero marks a dead token, as for
 *              engram_compress_masked
 *   primes     HOST int64 [3*n_heads]: one table cut into prime buckets, as
 *              for engram_hash_bucketed (the released layout); tables_host
 *              then names that one table for all three orders, and the
 *              buckets' sum must be at most each of its rows[n]
 * positions and dead are device memory for engram_forward and
 * engram_forward_static, host memory (like the token ids) for the *_host
 * calls.  The struct itself is read on the host during the call only.
 */
typedef struct engram_layout {
  const int32_t *positions;
  const uint8_t *dead;
  const int64_t *primes;
} engram_layout;

/*
 * engram_forward -- the whole path in one call on device buffers:
 * engram_compress_masked, engram_hash_packed (or engram_hash_bucketed) and
 * engram_lookup_fused back to back on `stream`, with the compressed ids and
 * row ids kept in `workspace` (device memory of at least
 * engram_forward_workspace_bytes(batch, seq, n_heads) bytes, 16-byte aligned,
 * owned by the caller, not read after the call's kernels end).
 * A decode step (seq == 1) whose rows the bulk lookup takes (D a multiple of
 * 512, a token's rows within shared memory) runs as one fused launch instead:
 * each slot's block compresses its token, hashes its window into row ids kept
 * on chip, and looks them up, with results identical to the three calls; a bad
 * token id, map value or history id then flags the status word and leaves all
 * of that slot's outputs (streams, history_out) unwritten.  That launch allows
 * programmatic dependent launch: its blocks may be scheduled while the kernel
 * before it on `stream` finishes, and wait for that kernel to complete before
 * touching memory, so the ordering on `stream` is as for any launch.
 *   token_ids int32 [batch, seq] (device); history / history_out as in
 *   engram_hash; layout_host as above (may be NULL); streams as in
 *   engram_lookup_fused ([batch*seq, 4, D]).
 */
ENGRAM_API size_t engram_forward_workspace_bytes(int32_t batch, int32_t seq, int32_t n_heads);
ENGRAM_API engram_status engram_forward(const int32_t *token_ids, int32_t batch, int32_t seq,
                                        const int32_t *tid2eid, int32_t vocab, int32_t n_eids,
                                        const int32_t *history, int32_t *history_out,
                                        int32_t n_heads, const engram_tables *tables_host,
                                        const engram_layout *layout_host,
                                        const uint16_t *streams_in, uint16_t *streams_out,
                                        const float *alpha, float eps, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream);

/*
 * engram_forward_host -- the whole path with the token ids, the layout's
 * positions and dead mask, and the streams in HOST memory (pinned for overlap;
 * pageable works but serialises the copies).  The call copies the ids (and
 * positions, dead mask) in, runs compress + hash, then pipelines the streams
 * in chunks of `chunk_tokens` tokens (0 = 2048): host->device copies on one
 * internal copy stream, the fused lookup on `stream`, device->host copies on a
 * second copy stream, with three chunk buffers per direction in `workspace`
 * (device memory of at least engram_forward_host_workspace_bytes(...) bytes).
 * A decode step (seq == 1) that engram_forward would run as one fused launch
 * runs each chunk of slots as that launch instead of compress + hash + lookup.
 * Returns once everything is enqueued; `stream` is ordered after the last
 * device->host copy, so synchronising `stream` means streams_out_host is final.
 * The two copy streams and their events are created on first use per device
 * and kept for the life of the process; calls on one device take turns on
 * them.  tid2eid, history, history_out, the tables, alpha and status are device
 * memory as in the calls above.
 */
ENGRAM_API size_t engram_forward_host_workspace_bytes(int32_t batch, int32_t seq,
                                                      int32_t n_heads, int32_t D,
                                                      int32_t chunk_tokens);
ENGRAM_API engram_status engram_forward_host(
    const int32_t *token_ids_host, int32_t batch, int32_t seq, const int32_t *tid2eid,
    int32_t vocab, int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const engram_tables *tables_host, const engram_layout *layout_host,
    const uint16_t *streams_in_host, uint16_t *streams_out_host, const float *alpha, float eps,
    int32_t chunk_tokens, void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/*
 * engram_connection_host -- the connection's whole path (engram_compress_masked,
 * the hash, then engram_connection) with the token ids, the layout's positions
 * and dead mask, and the streams in HOST memory, pipelined as
 * engram_forward_host does: the ids are copied in and hashed on `stream`, then
 * the streams move in chunks of `chunk_tokens` tokens (0 = 8192, enough
 * 256-row projection tiles to fill every SM pair), each chunk's connection (rows
 * into E, k = wkv e on the tensor cores, gate and add) running on `stream`
 * between its two copies.  D is the stream width (wkv is bf16 [D, 3*n_heads*d],
 * d = tables_host->D); tables and wkv as for engram_connection.  workspace:
 * device, 256-byte aligned, at least engram_connection_host_workspace_bytes(...)
 * bytes.  Returns once everything is enqueued; synchronising `stream` means
 * streams_out_host is final.  It shares engram_forward_host's copy streams.
 */
ENGRAM_API size_t engram_connection_host_workspace_bytes(int32_t batch, int32_t seq,
                                                         int32_t n_heads, int32_t d, int32_t D,
                                                         int32_t chunk_tokens);
ENGRAM_API engram_status engram_connection_host(
    const int32_t *token_ids_host, int32_t batch, int32_t seq, const int32_t *tid2eid,
    int32_t vocab, int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const engram_tables *tables_host, const engram_layout *layout_host, const uint16_t *wkv,
    int32_t D, const uint16_t *streams_in_host, uint16_t *streams_out_host, const float *alpha,
    float eps, int32_t chunk_tokens, void *workspace, size_t workspace_bytes, int32_t *status,
    void *stream);

/*
 * engram_forward_static -- engram_forward without a workspace argument, for
 * callers that cannot call cudaMalloc: a plugin or kernel library loaded into a
 * host program that owns all device memory and hands it only input and output
 * buffers, a runtime whose memory pool forbids allocations outside it, or code
 * that must not allocate after start-up (an allocation can synchronise the
 * device or fail at an awkward time).  The pages have no counterpart; it is a
 * calling convenience.
 *
 * Instead of a caller workspace it uses one file-scope device array of
 * ENGRAM_STATIC_WORKSPACE_BYTES (16 MiB).  A device reserves it when the
 * library's code is loaded there, at the latest on the first call of this
 * function on that device (with lazy module loading, CUDA's default), and holds
 * it until the process exits; a first call can therefore fail with
 * ENGRAM_ERR_CUDA when the device is out of memory.  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.  Outside
 * a stream capture every call looks up the array's device address
 * (cudaGetSymbolAddress, with the calling device current), so a context made
 * anew after cudaDeviceReset gets its own; a call inside a capture reuses the
 * address the last call outside one found on that device, and returns
 * ENGRAM_ERR_INVALID_ARG if there was none.  So make one call per device at
 * start-up, outside any capture, and again after a device reset: a call with
 * batch = 0 or seq = 0 does the set-up and launches nothing.
 * Requests needing more than the array, engram_forward_workspace_bytes(batch,
 * seq, n_heads) > ENGRAM_STATIC_WORKSPACE_BYTES (100 bytes a token at 8 heads:
 * 167,772 tokens), return ENGRAM_ERR_UNSUPPORTED with a message and launch
 * nothing.  All calls share the one array, which keeps the last call's
 * contents; each call that uses it clears the part it uses on `stream` first (a
 * decode step, seq = 1 on the fused launch, keeps its ids on chip and uses none
 * of it).  Calls that overlap on the GPU (on different streams or host threads,
 * on one device) race on the array: order them.  Other arguments and results
 * are exactly those of engram_forward.
 */
#define ENGRAM_STATIC_WORKSPACE_BYTES (16u << 20)
ENGRAM_API engram_status engram_forward_static(
    const int32_t *token_ids, int32_t batch, int32_t seq, const int32_t *tid2eid, int32_t vocab,
    int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const engram_tables *tables_host, const engram_layout *layout_host,
    const uint16_t *streams_in, uint16_t *streams_out, const float *alpha, float eps,
    int32_t *status, void *stream);

/*
 * engram_pack_e8m0_rows -- builds an ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS table
 * from an ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 one: packed row r = table row r (D
 * bytes), then exps row r (D/32 bytes), then zeros up to
 * ENGRAM_E8M0_ROW_BYTES(D).
 *   table  uint8 [rows, D] (device, 16-byte aligned);
 *   exps   uint8 [rows, D/32] (device);
 *   packed uint8 [rows, ENGRAM_E8M0_ROW_BYTES(D)] (device, 16-byte aligned,
 *          caller-allocated; must not overlap the inputs).
 * D % 32 == 0, 32 <= D <= ENGRAM_MAX_D, rows >= 0.  Asynchronous on `stream`;
 * argument errors return before any launch.
 */
ENGRAM_API engram_status engram_pack_e8m0_rows(const uint8_t *table, const uint8_t *exps,
                                               int64_t rows, int32_t D, uint8_t *packed,
                                               void *stream);

/*
 * engram_read_status -- waits for `stream`, copies the device status word into
 * *flags_host and returns ENGRAM_OK (no flag), ENGRAM_ERR_TIMEOUT
 * (ENGRAM_FLAG_TIMEOUT set) or ENGRAM_ERR_OUT_OF_RANGE (a range flag set).  The
 * word is not cleared.
 */
ENGRAM_API engram_status engram_read_status(const int32_t *status, int32_t *flags_host,
                                            void *stream);

/*
 * Kernel choice of engram_lookup_fused for this process:
 *   ENGRAM_LOOKUP_AUTO    the library picks (default: BULK where it applies);
 *   ENGRAM_LOOKUP_GATHER  register-direct gathers, one token per thread group,
 *                         rows loaded in batches of 8 (any D);
 *   ENGRAM_LOOKUP_BULK    a token's 3H rows staged in shared memory by 1-D bulk
 *                         copies (TMA) on an mbarrier while the threads load
 *                         the scales and streams: for D % 512 == 0 a token a
 *                         block of D/16 threads (a few tokens in turn a block
 *                         when a token's rows exceed 56 KB), for D < 512 with
 *                         D/16 a power of two several tokens a block; the
 *                         token's rows must fit ~227 KB of shared memory,
 *                         otherwise the call falls back to GATHER.
 * Both give identical results.  Returns the previous setting, or -1 for an
 * unknown value (nothing changed).  Not synchronised with calls in flight on
 * other host threads.
 */
#define ENGRAM_LOOKUP_AUTO 0
#define ENGRAM_LOOKUP_GATHER 1
#define ENGRAM_LOOKUP_BULK 2
ENGRAM_API int32_t engram_set_lookup_kernel(int32_t which);

/*
 * Kernel choice of the wkv projection (engram_wkv_project, engram_connection)
 * for this process:
 *   ENGRAM_PROJECTION_AUTO    the library picks (default: PAIR);
 *   ENGRAM_PROJECTION_SINGLE  one CTA per SM, 128 x 256 tiles of k, each CTA
 *                             staging its slices of E and wkv;
 *   ENGRAM_PROJECTION_PAIR    CTA pairs (2-CTA clusters, tcgen05 cta_group::2),
 *                             256 x 256 tiles, each CTA staging its rows of E and
 *                             half of the wkv slice.
 * Both add the same products in the same order (identical results).  Returns
 * the previous setting, or -1 for an unknown value.  Not synchronised with
 * calls in flight on other host threads.
 */
#define ENGRAM_PROJECTION_AUTO 0
#define ENGRAM_PROJECTION_SINGLE 1
#define ENGRAM_PROJECTION_PAIR 2
ENGRAM_API int32_t engram_set_projection_kernel(int32_t which);

/*
 * Every wait inside a kernel on data another warp produces (an mbarrier phase)
 * gives up after this many nanoseconds, sets ENGRAM_FLAG_TIMEOUT and ends the
 * kernel early instead of hanging.  Default 250 ms; values below 1 ms are
 * raised to 1 ms.  Returns the previous limit.
 */
ENGRAM_API int64_t engram_set_wait_limit_ns(int64_t ns);

/*
 * Test hook for the timeout path: the next `launches` launches of the BULK
 * lookup kernels or of the fused decode step (engram_forward with seq = 1)
 * withhold one row copy in every block (the mbarrier still expects its bytes),
 * so the block's bounded wait runs out, the block skips its token or slot, and
 * the launch reports ENGRAM_FLAG_TIMEOUT.  For tests only; 0 turns it off.
 */
ENGRAM_API void engram_debug_withhold_copies(int32_t launches);

/* Static, human-readable name of a status code. */
ENGRAM_API const char *engram_status_string(engram_status code);

/* Description of the last failed call on this host thread ("" if none). */
ENGRAM_API const char *engram_last_error(void);

/* ABI version of this header (incremented on any incompatible change). */
#define ENGRAM_ABI_VERSION 4
ENGRAM_API int32_t engram_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* ENGRAM_H */
