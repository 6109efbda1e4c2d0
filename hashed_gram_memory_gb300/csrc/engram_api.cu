// engram_api.cu -- the extern "C" entry points of libengram (include/engram.h):
// argument validation on the host, the device check, the launches, and the
// status-word read-back.  Every argument error is reported before any launch.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace {

thread_local char g_last_error[512] = "";

engram_status fail(engram_status code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

engram_status ok() {
  g_last_error[0] = '\0';
  return ENGRAM_OK;
}

engram_status cuda_fail(const char *what, cudaError_t e) {
  return fail(ENGRAM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return na && nb && x < y + nb && y < x + na;
}

// Per-device memo of the architecture check: 0 unknown, 1 sm_103, 2 other.
std::atomic<int> g_arch_ok[64];

std::atomic<int> g_lookup_kernel{ENGRAM_LOOKUP_AUTO};
std::atomic<int64_t> g_wait_limit_ns{250000000};
std::atomic<int> g_withhold{0};

engram_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  const int slot = dev & 63;
  int known = g_arch_ok[slot].load(std::memory_order_relaxed);
  if (known == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail("cudaDeviceGetAttribute", e);
    known = (major == 10 && minor == 3) ? 1 : 2;
    g_arch_ok[slot].store(known, std::memory_order_relaxed);
    if (known == 2)
      return fail(ENGRAM_ERR_UNSUPPORTED, "device %d is sm_%d%d; libengram is built for sm_103a",
                  dev, major, minor);
  }
  if (known == 2) return fail(ENGRAM_ERR_UNSUPPORTED, "device %d is not sm_103", dev);
  return ENGRAM_OK;
}

engram_status launched(const char *what, cudaError_t e) {
  if (e != cudaSuccess) return cuda_fail(what, e);
  return ok();
}

}  // namespace

engram_status engram::set_error(engram_status code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

extern "C" {

ENGRAM_API int32_t engram_abi_version(void) { return ENGRAM_ABI_VERSION; }

ENGRAM_API const char *engram_last_error(void) { return g_last_error; }

ENGRAM_API const char *engram_status_string(engram_status code) {
  switch (code) {
    case ENGRAM_OK: return "ENGRAM_OK";
    case ENGRAM_ERR_INVALID_ARG: return "ENGRAM_ERR_INVALID_ARG: invalid argument";
    case ENGRAM_ERR_UNSUPPORTED: return "ENGRAM_ERR_UNSUPPORTED: unsupported device or size";
    case ENGRAM_ERR_CUDA: return "ENGRAM_ERR_CUDA: CUDA runtime error";
    case ENGRAM_ERR_OUT_OF_RANGE: return "ENGRAM_ERR_OUT_OF_RANGE: an input id was out of range";
    case ENGRAM_ERR_TIMEOUT: return "ENGRAM_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "ENGRAM: unknown status code";
  }
}

ENGRAM_API engram_status engram_compress_masked(const int32_t *token_ids, int64_t n_tokens,
                                                const int32_t *tid2eid, int32_t vocab,
                                                int32_t n_eids, const uint8_t *dead,
                                                int32_t *eids_out, int32_t *status,
                                                void *stream) {
  ENGRAM_NVTX_RANGE("engram_compress_masked");
  if (n_tokens < 0) return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: n_tokens < 0");
  if (vocab < 1) return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: vocab < 1");
  if (n_eids < 0) return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: n_eids < 0");
  if (!tid2eid) return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: tid2eid is NULL");
  if (n_tokens > 0 && (!token_ids || !eids_out))
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: token_ids or eids_out is NULL");
  if (!aligned(token_ids, 4) || !aligned(tid2eid, 4) || !aligned(eids_out, 4) || !aligned(status, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: int32 pointers must be 4-byte aligned");
  if (token_ids != eids_out && overlap(token_ids, n_tokens * 4, eids_out, n_tokens * 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: token_ids and eids_out overlap partially");
  if (overlap(tid2eid, (size_t)vocab * 4, eids_out, n_tokens * 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: eids_out overlaps tid2eid");
  if (dead && overlap(dead, n_tokens, eids_out, n_tokens * 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_compress: eids_out overlaps the dead mask");
  if (n_tokens == 0) return ok();
  engram_status st = check_device();
  if (st != ENGRAM_OK) return st;
  engram::CompressParams p{token_ids, n_tokens, dead, tid2eid, vocab, n_eids, eids_out, status};
  return launched("engram_compress launch", engram::launch_compress(p, (cudaStream_t)stream));
}

ENGRAM_API engram_status engram_compress(const int32_t *token_ids, int64_t n_tokens,
                                         const int32_t *tid2eid, int32_t vocab, int32_t n_eids,
                                         int32_t *eids_out, int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_compress");
  return engram_compress_masked(token_ids, n_tokens, tid2eid, vocab, n_eids, nullptr, eids_out,
                                status, stream);
}

// The compression inputs of engram_compress_hash (the hash then reads token ids
// and compresses them itself instead of reading eids).
struct FusedCompress {
  const int32_t *token_ids;
  const int32_t *tid2eid;
  const uint8_t *dead;
  int32_t *eids_out;
  int32_t vocab, n_eids;
};

// Shared validation and launch of the hash: mod/off are the per-(order, head)
// modulus and offset of every row id (host arrays of 3 * n_heads).  With `fc`
// the ids come from token ids compressed in the kernel, and `eids` is unused.
static engram_status hash_common(const char *fn, const int32_t *eids, int32_t batch, int32_t seq,
                                 const int32_t *positions, const int32_t *history,
                                 int32_t *history_out, int32_t n_heads, const int64_t *mod,
                                 const int64_t *off, int32_t *row_ids_out, int32_t *status,
                                 void *stream, const FusedCompress *fc = nullptr) {
  if (batch < 0 || seq < 0) return fail(ENGRAM_ERR_INVALID_ARG, "%s: batch or seq < 0", fn);
  if (n_heads < 1 || n_heads > ENGRAM_MAX_HEADS)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_heads must be in [1, %d]", fn, ENGRAM_MAX_HEADS);
  for (int r = 0; r < 3 * n_heads; ++r)
    if (mod[r] < 1 || off[r] < 0 || off[r] + mod[r] - 1 > INT32_MAX)
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: row ids must fit [0, 2^31-1] (bucket %d)", fn, r);
  const int64_t T = (int64_t)batch * seq;
  const size_t R = 3 * (size_t)n_heads;
  if (fc) {
    // The compression's own checks; eids_out is an output beside the row ids.
    if (fc->vocab < 1 || fc->n_eids < 0 || !fc->tid2eid)
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: vocab < 1, n_eids < 0 or tid2eid NULL", fn);
    if (T > 0 && !fc->token_ids)
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: token_ids is NULL", fn);
    if (!aligned(fc->token_ids, 4) || !aligned(fc->tid2eid, 4) || !aligned(fc->eids_out, 4))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: int32 pointers must be 4-byte aligned", fn);
    const size_t tb = (size_t)T * 4;
    if (fc->eids_out && (overlap(fc->eids_out, tb, fc->token_ids, tb) ||
                         overlap(fc->eids_out, tb, fc->tid2eid, (size_t)fc->vocab * 4) ||
                         overlap(fc->eids_out, tb, fc->dead, (size_t)T) ||
                         overlap(fc->eids_out, tb, row_ids_out, T * R * 4) ||
                         overlap(fc->eids_out, tb, history_out, (size_t)batch * 12) ||
                         overlap(fc->eids_out, tb, history, (size_t)batch * 12) ||
                         overlap(fc->eids_out, tb, positions, tb)))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: eids_out overlaps another buffer", fn);
    const size_t mb = (size_t)fc->vocab * 4;
    if (overlap(row_ids_out, T * R * 4, fc->token_ids, tb) ||
        overlap(row_ids_out, T * R * 4, fc->dead, (size_t)T) ||
        overlap(row_ids_out, T * R * 4, fc->tid2eid, mb) ||
        (history_out && (overlap(history_out, (size_t)batch * 12, fc->token_ids, tb) ||
                         overlap(history_out, (size_t)batch * 12, fc->dead, (size_t)T) ||
                         overlap(history_out, (size_t)batch * 12, fc->tid2eid, mb))))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: an output overlaps token_ids, tid2eid or the dead mask",
                  fn);
    eids = nullptr;
  }
  if (T > 0 && ((!eids && !fc) || !row_ids_out))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: eids or row_ids_out is NULL", fn);
  if (!aligned(eids, 4) || !aligned(history, 4) || !aligned(history_out, 4) ||
      !aligned(row_ids_out, 4) || !aligned(status, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: int32 pointers must be 4-byte aligned", fn);
  if (overlap(eids, T * 4, row_ids_out, T * R * 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: row_ids_out overlaps eids", fn);
  if (history_out) {
    const size_t hb = (size_t)batch * 3 * 4;
    if (overlap(history_out, hb, eids, T * 4) || overlap(history_out, hb, row_ids_out, T * R * 4))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: history_out overlaps eids or row_ids_out", fn);
    if (history && history != history_out && overlap(history, hb, history_out, hb))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: history and history_out overlap partially", fn);
  }
  if (history && overlap(history, (size_t)batch * 12, row_ids_out, T * R * 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: row_ids_out overlaps history", fn);
  if (positions && (!aligned(positions, 4) || overlap(positions, T * 4, row_ids_out, T * R * 4) ||
                    (history_out && overlap(positions, T * 4, history_out, (size_t)batch * 12))))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: positions misaligned or overlapping outputs", fn);
  if (T == 0 && (!history_out || batch == 0)) return ok();
  engram_status st = check_device();
  if (st != ENGRAM_OK) return st;
  engram::HashParams p;
  memset(&p, 0, sizeof p);
  p.eids = eids;
  p.positions = positions;
  p.history = history;
  p.history_out = history_out;
  p.row_ids = row_ids_out;
  p.status = status;
  p.T = T;
  p.batch = batch;
  p.seq = seq;
  p.H = n_heads;
  if (fc) {
    p.token_ids = fc->token_ids;
    p.tid2eid = fc->tid2eid;
    p.dead = fc->dead;
    p.eids_out = fc->eids_out;
    p.vocab = fc->vocab;
    p.n_eids = fc->n_eids;
  }
  for (int n = 0; n < 3; ++n)
    for (int j = 0; j < n_heads; ++j) {
      const int r = n * n_heads + j;
      p.mod[n][j] = (uint64_t)mod[r];
      p.off[n][j] = (uint64_t)off[r];
      p.rmul[n][j] = UINT64_MAX / p.mod[n][j];
      p.seed[n][j] = engram::splitmix64((uint64_t)((n + 2) * 16 + j));
    }
  return launched("engram_hash launch", engram::launch_hash(p, (cudaStream_t)stream));
}

ENGRAM_API engram_status engram_hash_packed(const int32_t *eids, int32_t batch, int32_t seq,
                                            const int32_t *positions, const int32_t *history,
                                            int32_t *history_out, int32_t n_heads,
                                            const int64_t *rows_host, int32_t *row_ids_out,
                                            int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_hash_packed");
  if (n_heads < 1 || n_heads > ENGRAM_MAX_HEADS)
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_hash: n_heads must be in [1, %d]",
                ENGRAM_MAX_HEADS);
  if (!rows_host) return fail(ENGRAM_ERR_INVALID_ARG, "engram_hash: rows_host is NULL");
  int64_t mod[3 * ENGRAM_MAX_HEADS], off[3 * ENGRAM_MAX_HEADS];
  for (int n = 0; n < 3; ++n) {
    if (rows_host[n] < 1 || rows_host[n] > INT32_MAX)
      return fail(ENGRAM_ERR_INVALID_ARG, "engram_hash: rows[%d] must be in [1, 2^31-1]", n);
    for (int j = 0; j < n_heads; ++j) {
      mod[n * n_heads + j] = rows_host[n];
      off[n * n_heads + j] = 0;
    }
  }
  return hash_common("engram_hash", eids, batch, seq, positions, history, history_out, n_heads,
                     mod, off, row_ids_out, status, stream);
}

ENGRAM_API engram_status engram_hash_bucketed(const int32_t *eids, int32_t batch, int32_t seq,
                                              const int32_t *positions, const int32_t *history,
                                              int32_t *history_out, int32_t n_heads,
                                              const int64_t *primes_host, int32_t *row_ids_out,
                                              int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_hash_bucketed");
  if (n_heads < 1 || n_heads > ENGRAM_MAX_HEADS)
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_hash_bucketed: n_heads must be in [1, %d]",
                ENGRAM_MAX_HEADS);
  if (!primes_host) return fail(ENGRAM_ERR_INVALID_ARG, "engram_hash_bucketed: primes is NULL");
  int64_t off[3 * ENGRAM_MAX_HEADS];
  int64_t sum = 0;
  for (int r = 0; r < 3 * n_heads; ++r) {
    if (primes_host[r] < 1 || primes_host[r] > INT32_MAX)
      return fail(ENGRAM_ERR_INVALID_ARG, "engram_hash_bucketed: bucket %d size out of range", r);
    off[r] = sum;
    sum += primes_host[r];
  }
  if (sum - 1 > INT32_MAX)
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_hash_bucketed: %lld rows exceed 2^31-1",
                (long long)sum);
  return hash_common("engram_hash_bucketed", eids, batch, seq, positions, history, history_out,
                     n_heads, primes_host, off, row_ids_out, status, stream);
}

ENGRAM_API engram_status engram_compress_hash(
    const int32_t *token_ids, int32_t batch, int32_t seq, const int32_t *tid2eid, int32_t vocab,
    int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const int64_t *rows_host, const engram_layout *layout_host, int32_t *eids_out,
    int32_t *row_ids_out, int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_compress_hash");
  const char *fn = "engram_compress_hash";
  if (n_heads < 1 || n_heads > ENGRAM_MAX_HEADS)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_heads must be in [1, %d]", fn, ENGRAM_MAX_HEADS);
  const int64_t *primes = layout_host ? layout_host->primes : nullptr;
  int64_t mod[3 * ENGRAM_MAX_HEADS], off[3 * ENGRAM_MAX_HEADS];
  int64_t sum = 0;
  for (int n = 0; n < 3; ++n) {
    if (!primes && (!rows_host || rows_host[n] < 1 || rows_host[n] > INT32_MAX))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: rows must be in [1, 2^31-1]", fn);
    for (int j = 0; j < n_heads; ++j) {
      const int r = n * n_heads + j;
      if (primes) {
        if (primes[r] < 1 || primes[r] > INT32_MAX)
          return fail(ENGRAM_ERR_INVALID_ARG, "%s: bucket %d size out of range", fn, r);
        mod[r] = primes[r];
        off[r] = sum;
        sum += primes[r];
      } else {
        mod[r] = rows_host[n];
        off[r] = 0;
      }
    }
  }
  const FusedCompress fc{token_ids, tid2eid, layout_host ? layout_host->dead : nullptr, eids_out,
                         vocab, n_eids};
  return hash_common(fn, nullptr, batch, seq, layout_host ? layout_host->positions : nullptr,
                     history, history_out, n_heads, mod, off, row_ids_out, status, stream, &fc);
}

// Trial division: no divisor d with d*d <= n.
static bool is_prime_u64(int64_t n) {
  if (n < 2) return false;
  if (n % 2 == 0) return n == 2;
  for (int64_t d = 3; d * d <= n; d += 2)
    if (n % d == 0) return false;
  return true;
}

ENGRAM_API engram_status engram_bucket_primes(int32_t n_layers, int32_t max_ngram, int32_t n_heads,
                                              int64_t hash_vocab, int64_t *primes_out_host) {
  if (n_layers < 1 || max_ngram < 2 || n_heads < 1 || hash_vocab < 1 || !primes_out_host)
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_bucket_primes: bad arguments");
  if ((int64_t)n_layers * (max_ngram - 1) * n_heads > 65536)
    return fail(ENGRAM_ERR_UNSUPPORTED, "engram_bucket_primes: more than 65536 buckets");
  int64_t k = 0;
  for (int32_t l = 0; l < n_layers; ++l)
    for (int32_t n = 2; n <= max_ngram; ++n) {
      int64_t c = hash_vocab;  // every order starts again at the vocabulary
      for (int32_t j = 0; j < n_heads; ++j) {
        for (;; ++c) {
          bool taken = false;
          for (int64_t q = 0; q < k && !taken; ++q) taken = primes_out_host[q] == c;
          if (!taken && is_prime_u64(c)) break;
        }
        primes_out_host[k++] = c++;
      }
    }
  return ok();
}

ENGRAM_API engram_status engram_hash(const int32_t *eids, int32_t batch, int32_t seq,
                                     const int32_t *history, int32_t *history_out,
                                     int32_t n_heads, const int64_t *rows_host,
                                     int32_t *row_ids_out, int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_hash");
  return engram_hash_packed(eids, batch, seq, nullptr, history, history_out, n_heads, rows_host,
                            row_ids_out, status, stream);
}

}  // extern "C"

// The argument checks of engram_lookup_fused and the fill of its launch
// parameters; row_ids may be NULL when `need_row_ids` is false (the fused
// decode step makes them itself).  With n_tokens == 0 it returns OK without a
// device query and leaves p.T == 0.
engram_status engram::prepare_lookup(const char *fn, const int32_t *row_ids, bool need_row_ids,
                                     int64_t n_tokens, int32_t n_heads,
                                     const engram_tables *tables_host, const uint16_t *streams_in,
                                     uint16_t *streams_out, const float *alpha, float eps,
                                     float *gate_out, float *mem_out, int32_t *status,
                                     LookupParams &p) {
  memset(&p, 0, sizeof p);
  if (n_tokens < 0) return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_tokens < 0", fn);
  if (n_heads < 1 || n_heads > ENGRAM_MAX_HEADS)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_heads must be in [1, %d]", fn, ENGRAM_MAX_HEADS);
  if (!tables_host) return fail(ENGRAM_ERR_INVALID_ARG, "%s: tables is NULL", fn);
  const engram_tables &tb = *tables_host;
  const bool e8m0 = tb.dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 ||
                    tb.dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS;
  if (tb.dtype != ENGRAM_TABLE_FP8_E4M3FN && tb.dtype != ENGRAM_TABLE_BF16 && !e8m0)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: unknown table dtype %d", fn, tb.dtype);
  if (tb.D < 16 || tb.D % 16 != 0)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: D = %d must be a positive multiple of 16", fn, tb.D);
  if (e8m0 && tb.D % 32 != 0)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: E8M0 (1, 32) blocks need D %% 32 == 0", fn);
  if (tb.D > ENGRAM_MAX_D)
    return fail(ENGRAM_ERR_UNSUPPORTED, "%s: D = %d exceeds %d", fn, tb.D, ENGRAM_MAX_D);
  const int D = tb.D;
  const size_t table_row = engram::table_row_bytes(tb.dtype, D);
  for (int n = 0; n < 3; ++n) {
    if (tb.rows[n] < 1 || tb.rows[n] > INT32_MAX)
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: rows[%d] must be in [1, 2^31-1]", fn, n);
    if (!tb.table[n] || !aligned(tb.table[n], 16))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: table[%d] NULL or not 16-byte aligned", fn, n);
    if (tb.dtype == ENGRAM_TABLE_FP8_E4M3FN && (!tb.scale[n] || !aligned(tb.scale[n], 4)))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: scale[%d] NULL or not 4-byte aligned", fn, n);
    if (tb.dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 && (!tb.scale[n] || !aligned(tb.scale[n], 16)))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: scale[%d] NULL or not 16-byte aligned", fn, n);
  }
  if (!alpha || !aligned(alpha, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: alpha NULL or not 4-byte aligned", fn);
  if (!(eps >= 0.f) || !isfinite(eps))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: eps must be finite and >= 0", fn);
  const size_t R = 3 * (size_t)n_heads;
  const size_t sbytes = (size_t)n_tokens * 4 * D * 2;
  if (n_tokens > 0) {
    if ((need_row_ids && !row_ids) || !streams_in || !streams_out)
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: row_ids or streams is NULL", fn);
    if (!aligned(row_ids, 4) || !aligned(status, 4) || !aligned(gate_out, 4))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: row_ids/status/gate_out not 4-byte aligned", fn);
    if (!aligned(streams_in, 16) || !aligned(streams_out, 16) || !aligned(mem_out, 16))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: streams and mem_out must be 16-byte aligned", fn);
    if (streams_in != streams_out && overlap(streams_in, sbytes, streams_out, sbytes))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: streams_out overlaps streams_in partially", fn);
    const size_t ib = n_tokens * R * 4;
    if (overlap(streams_out, sbytes, row_ids, ib) ||
        (mem_out && overlap(mem_out, (size_t)n_tokens * D * 4, streams_out, sbytes)) ||
        (gate_out && overlap(gate_out, (size_t)n_tokens * 4, streams_out, sbytes)))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: output buffers overlap", fn);
    for (int n = 0; n < 3; ++n)
      if (overlap(streams_out, sbytes, tb.table[n], (size_t)tb.rows[n] * table_row))
        return fail(ENGRAM_ERR_INVALID_ARG, "%s: streams_out overlaps table[%d]", fn, n);
  }
  if (n_tokens == 0) return ok();
  engram_status st = check_device();
  if (st != ENGRAM_OK) return st;
  p.row_ids = row_ids;
  for (int n = 0; n < 3; ++n) {
    p.table[n] = static_cast<const uint8_t *>(tb.table[n]);
    p.scale[n] = tb.scale[n];
    p.rows[n] = tb.rows[n];
  }
  p.x = streams_in;
  p.y = streams_out;
  p.alpha = alpha;
  p.gate_out = gate_out;
  p.mem_out = mem_out;
  p.status = status;
  p.T = n_tokens;
  p.H = n_heads;
  p.D = D;
  p.eps = eps;
  p.inv_R = 1.f / (float)(3 * n_heads);
  p.inv_D = 1.f / (float)D;
  p.sqrt_D = sqrtf((float)D);
  p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  return ENGRAM_OK;
}

int engram::lookup_kernel_choice() { return g_lookup_kernel.load(std::memory_order_relaxed); }

bool engram::take_withheld_launch() {
  int w = g_withhold.load(std::memory_order_relaxed);
  while (w > 0 && !g_withhold.compare_exchange_weak(w, w - 1)) {
  }
  return w > 0;
}

extern "C" {

ENGRAM_API engram_status engram_lookup_fused(const int32_t *row_ids, int64_t n_tokens,
                                             int32_t n_heads, const engram_tables *tables_host,
                                             const uint16_t *streams_in, uint16_t *streams_out,
                                             const float *alpha, float eps, float *gate_out,
                                             float *mem_out, int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_lookup_fused");
  engram::LookupParams p;
  engram_status st =
      engram::prepare_lookup("engram_lookup_fused", row_ids, true, n_tokens, n_heads, tables_host,
                             streams_in, streams_out, alpha, eps, gate_out, mem_out, status, p);
  if (st != ENGRAM_OK || n_tokens == 0) return st;
  const engram_tables &tb = *tables_host;
  const int D = tb.D;
  const int which = g_lookup_kernel.load(std::memory_order_relaxed);
  const bool bulk_family = which == ENGRAM_LOOKUP_BULK || which == ENGRAM_LOOKUP_AUTO;
  const bool bulk = bulk_family && engram::bulk_supported(D, tb.dtype, n_heads);
  const bool small = bulk_family && !bulk && engram::bulk_small_supported(D, tb.dtype, n_heads);
  if (bulk || small) {
    p.withhold = engram::take_withheld_launch() ? 1 : 0;
    if (small)
      return launched("engram_lookup_fused launch (bulk, small rows)",
                      engram::launch_lookup_bulk_small(p, tb.dtype, (cudaStream_t)stream));
    return launched("engram_lookup_fused launch (bulk)",
                    engram::launch_lookup_bulk(p, tb.dtype, (cudaStream_t)stream));
  }
  return launched("engram_lookup_fused launch (gather)",
                  engram::launch_lookup(p, tb.dtype, (cudaStream_t)stream));
}

static size_t round256(size_t x) { return (x + 255) / 256 * 256; }

ENGRAM_API size_t engram_connection_workspace_bytes(int64_t n_tokens, int32_t n_heads, int32_t d,
                                                    int32_t D) {
  if (n_tokens < 0 || n_heads < 1 || d < 1 || D < 1) return 0;
  const size_t T = (size_t)n_tokens, K = 3 * (size_t)n_heads * d;
  return round256(T * K * 2) + round256(T * (size_t)D * 4) + round256(T);
}

static engram_status check_connection_tables(const char *fn, int32_t n_heads,
                                             const engram_tables *tables_host) {
  if (n_heads < 1 || n_heads > ENGRAM_MAX_HEADS)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_heads must be in [1, %d]", fn, ENGRAM_MAX_HEADS);
  if (!tables_host) return fail(ENGRAM_ERR_INVALID_ARG, "%s: tables is NULL", fn);
  const engram_tables &tb = *tables_host;
  if (tb.dtype != ENGRAM_TABLE_BF16 && tb.dtype != ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 &&
      tb.dtype != ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS)
    return fail(ENGRAM_ERR_UNSUPPORTED,
                "%s: the projection takes BF16 or FP8 + e8m0 tables (exact in bf16)", fn);
  if (tb.D < 32 || tb.D % 32 != 0 || tb.D > 65536)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: row width %d must be a multiple of 32", fn, tb.D);
  for (int n = 0; n < 3; ++n) {
    if (tb.rows[n] < 1 || tb.rows[n] > INT32_MAX || !tb.table[n] || !aligned(tb.table[n], 16))
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: table[%d] bad (rows, NULL or alignment)", fn, n);
    if (tb.dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 && !tb.scale[n])
      return fail(ENGRAM_ERR_INVALID_ARG, "%s: scale[%d] is NULL", fn, n);
  }
  return ENGRAM_OK;
}

static engram_status check_projection(const char *fn, int64_t K, int32_t D) {
  if (K < 64 || K > INT32_MAX || D < 256 || D > 8192 || !engram::wkv_gemm_supported(D, (int)K))
    return fail(ENGRAM_ERR_UNSUPPORTED,
                "%s: D must be a multiple of 256 in [256, 8192] and K (= 3*n_heads*d) of 64", fn);
  return ENGRAM_OK;
}

static engram_status check_gate_add(const char *fn, int64_t n_tokens, int32_t D,
                                    const uint16_t *streams_in, uint16_t *streams_out,
                                    const float *alpha, float eps, float *gate_out) {
  if (!alpha || !aligned(alpha, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: alpha NULL or misaligned", fn);
  if (!(eps >= 0.f) || !isfinite(eps))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: eps must be finite and >= 0", fn);
  if (n_tokens == 0) return ENGRAM_OK;
  if (!streams_in || !streams_out || !aligned(streams_in, 16) || !aligned(streams_out, 16) ||
      !aligned(gate_out, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: NULL or misaligned stream or gate buffer", fn);
  const size_t sbytes = (size_t)n_tokens * 4 * D * 2;
  if (streams_in != streams_out && overlap(streams_in, sbytes, streams_out, sbytes))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: streams_out overlaps streams_in partially", fn);
  return ENGRAM_OK;
}

ENGRAM_API engram_status engram_concat_rows(const int32_t *row_ids, int64_t n_tokens,
                                            int32_t n_heads, const engram_tables *tables_host,
                                            uint16_t *e_out, uint8_t *state_out, int32_t *status,
                                            void *stream) {
  ENGRAM_NVTX_RANGE("engram_concat_rows");
  const char *fn = "engram_concat_rows";
  if (n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_tokens out of range", fn);
  engram_status st = check_connection_tables(fn, n_heads, tables_host);
  if (st != ENGRAM_OK) return st;
  if (n_tokens == 0) return ok();
  if (!row_ids || !e_out || !state_out || !aligned(row_ids, 4) || !aligned(e_out, 16) ||
      !aligned(status, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: NULL or misaligned buffer", fn);
  if ((st = check_device()) != ENGRAM_OK) return st;
  return launched("engram_concat_rows launch",
                  engram::launch_concat_rows(row_ids, n_tokens, n_heads, *tables_host, e_out,
                                             state_out, status, (cudaStream_t)stream));
}

ENGRAM_API engram_status engram_wkv_project(const uint16_t *e, int64_t n_tokens, int32_t K,
                                            const uint16_t *wkv, int32_t D, float *k_out,
                                            int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_wkv_project");
  const char *fn = "engram_wkv_project";
  if (n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_tokens out of range", fn);
  engram_status st = check_projection(fn, K, D);
  if (st != ENGRAM_OK) return st;
  if (!wkv || !aligned(wkv, 16))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: wkv NULL or not 16-byte aligned", fn);
  if (n_tokens == 0) return ok();
  if (!e || !k_out || !aligned(e, 16) || !aligned(k_out, 16) || !aligned(status, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: NULL or misaligned buffer", fn);
  if ((st = check_device()) != ENGRAM_OK) return st;
  return launched("engram_wkv_project launch",
                  engram::launch_wkv_gemm(e, wkv, k_out, (int)n_tokens, D, K,
                                          g_wait_limit_ns.load(std::memory_order_relaxed), status,
                                          (cudaStream_t)stream));
}

ENGRAM_API engram_status engram_gate_add(const float *k, const uint8_t *state, int64_t n_tokens,
                                         int32_t D, const uint16_t *streams_in,
                                         uint16_t *streams_out, const float *alpha, float eps,
                                         float *gate_out, void *stream) {
  ENGRAM_NVTX_RANGE("engram_gate_add");
  const char *fn = "engram_gate_add";
  if (n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_tokens out of range", fn);
  if (D < 16 || D % 16 != 0 || D > 8192)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: D must be a multiple of 16 in [16, 8192]", fn);
  engram_status st = check_gate_add(fn, n_tokens, D, streams_in, streams_out, alpha, eps, gate_out);
  if (st != ENGRAM_OK) return st;
  if (n_tokens == 0) return ok();
  if (!k || !state || !aligned(k, 16))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: k or state NULL, or k misaligned", fn);
  if ((st = check_device()) != ENGRAM_OK) return st;
  return launched("engram_gate_add launch",
                  engram::launch_gate_add(k, state, n_tokens, D, streams_in, streams_out, alpha,
                                          eps, gate_out, (cudaStream_t)stream));
}

ENGRAM_API engram_status engram_connection(const int32_t *row_ids, int64_t n_tokens,
                                           int32_t n_heads, const engram_tables *tables_host,
                                           const uint16_t *wkv, int32_t D,
                                           const uint16_t *streams_in, uint16_t *streams_out,
                                           const float *alpha, float eps, void *workspace,
                                           size_t workspace_bytes, float *gate_out, float *k_out,
                                           int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_connection");
  const char *fn = "engram_connection";
  if (n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: n_tokens out of range", fn);
  engram_status st = check_connection_tables(fn, n_heads, tables_host);
  if (st != ENGRAM_OK) return st;
  const int d = tables_host->D;
  const int64_t K = 3 * (int64_t)n_heads * d;
  if ((st = check_projection(fn, K, D)) != ENGRAM_OK) return st;
  if (!wkv || !aligned(wkv, 16))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: wkv NULL or not 16-byte aligned", fn);
  st = check_gate_add(fn, n_tokens, D, streams_in, streams_out, alpha, eps, gate_out);
  if (st != ENGRAM_OK) return st;
  if (n_tokens == 0) return ok();
  const size_t need = engram_connection_workspace_bytes(n_tokens, n_heads, d, D);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
    return fail(ENGRAM_ERR_INVALID_ARG,
                "%s: workspace NULL, not 256-byte aligned or under %zu bytes", fn, need);
  if (!row_ids || !aligned(row_ids, 4) || !aligned(k_out, 16) || !aligned(status, 4))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: NULL or misaligned buffer", fn);
  if ((st = check_device()) != ENGRAM_OK) return st;
  char *w = static_cast<char *>(workspace);
  uint16_t *e = reinterpret_cast<uint16_t *>(w);
  w += round256((size_t)n_tokens * K * 2);
  float *k = k_out ? k_out : reinterpret_cast<float *>(w);
  w += round256((size_t)n_tokens * D * 4);
  uint8_t *state = reinterpret_cast<uint8_t *>(w);
  return launched("engram_connection launch",
                  engram::launch_connection(row_ids, n_tokens, n_heads, *tables_host, wkv, D,
                                            streams_in, streams_out, alpha, eps, e, k, state,
                                            gate_out, g_wait_limit_ns.load(std::memory_order_relaxed),
                                            status, (cudaStream_t)stream));
}

ENGRAM_API engram_status engram_pack_e8m0_rows(const uint8_t *table, const uint8_t *exps,
                                               int64_t rows, int32_t D, uint8_t *packed,
                                               void *stream) {
  ENGRAM_NVTX_RANGE("engram_pack_e8m0_rows");
  const char *fn = "engram_pack_e8m0_rows";
  if (rows < 0 || D < 32 || D % 32 != 0 || D > ENGRAM_MAX_D)
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: rows >= 0 and D a multiple of 32 in [32, %d]", fn,
                ENGRAM_MAX_D);
  if (rows == 0) return ok();
  if (!table || !exps || !packed || !aligned(table, 16) || !aligned(packed, 16))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: NULL pointer, or table / packed not 16-byte aligned",
                fn);
  const size_t nt = (size_t)rows * D, ne = (size_t)rows * (D / 32);
  const size_t np = (size_t)rows * (size_t)ENGRAM_E8M0_ROW_BYTES(D);
  if (overlap(packed, np, table, nt) || overlap(packed, np, exps, ne))
    return fail(ENGRAM_ERR_INVALID_ARG, "%s: packed overlaps an input", fn);
  engram_status st = check_device();
  if (st != ENGRAM_OK) return st;
  return launched("engram_pack_e8m0_rows launch",
                  engram::launch_pack_e8m0_rows(table, exps, rows, D, packed,
                                                static_cast<cudaStream_t>(stream)));
}

ENGRAM_API int32_t engram_set_lookup_kernel(int32_t which) {
  if (which != ENGRAM_LOOKUP_AUTO && which != ENGRAM_LOOKUP_GATHER && which != ENGRAM_LOOKUP_BULK)
    return -1;
  return g_lookup_kernel.exchange(which);
}

ENGRAM_API int32_t engram_set_projection_kernel(int32_t which) {
  if (which != ENGRAM_PROJECTION_AUTO && which != ENGRAM_PROJECTION_SINGLE &&
      which != ENGRAM_PROJECTION_PAIR)
    return -1;
  return engram::set_projection_kernel(which);
}

ENGRAM_API int64_t engram_set_wait_limit_ns(int64_t ns) {
  if (ns < 1000000) ns = 1000000;
  return g_wait_limit_ns.exchange(ns);
}

ENGRAM_API void engram_debug_withhold_copies(int32_t launches) {
  g_withhold.store(launches > 0 ? launches : 0);
}

ENGRAM_API engram_status engram_read_status(const int32_t *status, int32_t *flags_host,
                                            void *stream) {
  ENGRAM_NVTX_RANGE("engram_read_status");
  if (!status || !flags_host)
    return fail(ENGRAM_ERR_INVALID_ARG, "engram_read_status: NULL pointer");
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, status, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail("engram_read_status", e);
  *flags_host = v;
  if (v & ENGRAM_FLAG_TIMEOUT) return fail(ENGRAM_ERR_TIMEOUT, "status word 0x%x", v);
  if (v) return fail(ENGRAM_ERR_OUT_OF_RANGE, "status word 0x%x", v);
  return ok();
}

}  // extern "C"
