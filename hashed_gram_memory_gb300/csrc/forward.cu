// forward.cu -- the whole Engram path in one call: engram_forward on device
// buffers, and engram_forward_host, which takes the token ids and the four
// streams in host memory and overlaps the host<->device copies with the fused
// lookup in a three-buffer chunk pipeline over two copy streams.
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "engram_internal.cuh"

namespace {

constexpr size_t kAlign = 256;
constexpr int kBufs = 3;
constexpr int kDefaultChunk = 2048;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Copy streams and events of the host pipeline, one set per device, created on
// first use and kept (they are driver objects, not device memory).
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t in_done[kBufs], comp_done[kBufs], out_done[kBufs];
};
HostPipe g_pipes[64];

cudaError_t pipe_init(HostPipe &hp) {
  if (hp.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&hp.copy_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.copy_out, cudaStreamNonBlocking);
  for (int i = 0; i < kBufs && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.comp_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.out_done[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) hp.ready = true;
  return e;
}

engram_status fwd_fail(engram_status code, const char *msg) {
  return engram::set_error(code, "%s", msg);
}

bool misaligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) != 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || !na || !nb) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// One decode step (one new token a slot) in one launch: compression, window,
// hash and bulk lookup fused, with the same argument checks as the three
// calls it replaces.  The row ids are not written out.
engram_status decode_step(const int32_t *token_ids, int32_t batch, const int32_t *tid2eid,
                          int32_t vocab, int32_t n_eids, const int32_t *history,
                          int32_t *history_out, int32_t n_heads, const engram_tables *tables_host,
                          const uint16_t *streams_in, uint16_t *streams_out, const float *alpha,
                          float eps, int32_t *status, void *stream) {
  const char *fn = "engram_forward";
  if (!token_ids || !tid2eid || misaligned4(token_ids) || misaligned4(tid2eid))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: token_ids or tid2eid NULL or misaligned");
  if (vocab < 1 || n_eids < 0)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: vocab must be >= 1 and n_eids >= 0");
  if (misaligned4(history) || misaligned4(history_out))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: history pointers not 4-byte aligned");
  const size_t hb = (size_t)batch * 12;
  const size_t sb = (size_t)batch * 4 * tables_host->D * 2;
  if (history && history_out && history != history_out && overlaps(history, hb, history_out, hb))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: history and history_out overlap partially");
  if (history_out && (overlaps(history_out, hb, streams_out, sb) ||
                      overlaps(history_out, hb, token_ids, (size_t)batch * 4)))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: history_out overlaps another buffer");
  for (int n = 0; n < 3; ++n)
    if (tables_host->rows[n] < 1 || tables_host->rows[n] > INT32_MAX)
      return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: rows must be in [1, 2^31-1]");
  engram::DecodeParams p;
  memset(&p, 0, sizeof p);
  engram_status st =
      engram::prepare_lookup(fn, nullptr, false, batch, n_heads, tables_host, streams_in,
                             streams_out, alpha, eps, nullptr, nullptr, status, p.lk);
  if (st != ENGRAM_OK) return st;
  p.token_ids = token_ids;
  p.tid2eid = tid2eid;
  p.history = history;
  p.history_out = history_out;
  p.vocab = vocab;
  p.n_eids = n_eids;
  for (int n = 0; n < 3; ++n)
    for (int j = 0; j < n_heads; ++j) {
      p.mod[n][j] = (uint64_t)tables_host->rows[n];
      p.off[n][j] = 0;
      p.rmul[n][j] = UINT64_MAX / p.mod[n][j];
      p.seed[n][j] = engram::splitmix64((uint64_t)((n + 2) * 16 + j));
    }
  const cudaError_t e = engram::launch_decode_step(p, tables_host->dtype, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return engram::set_error(ENGRAM_ERR_CUDA, "engram_forward decode launch: %s",
                             cudaGetErrorString(e));
  return engram::set_error(ENGRAM_OK, "%s", "");  // success clears the last message
}

}  // namespace

extern "C" {

ENGRAM_API size_t engram_forward_workspace_bytes(int32_t batch, int32_t seq, int32_t n_heads) {
  if (batch < 0 || seq < 0 || n_heads < 1) return 0;
  const size_t T = (size_t)batch * seq;
  return round_up(T * 4) + round_up(T * 3 * (size_t)n_heads * 4);
}

ENGRAM_API engram_status engram_forward(const int32_t *token_ids, int32_t batch, int32_t seq,
                                        const int32_t *tid2eid, int32_t vocab, int32_t n_eids,
                                        const int32_t *history, int32_t *history_out,
                                        int32_t n_heads, const engram_tables *tables_host,
                                        const uint16_t *streams_in, uint16_t *streams_out,
                                        const float *alpha, float eps, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream) {
  if (batch < 0 || seq < 0 || n_heads < 1 || n_heads > ENGRAM_MAX_HEADS || !tables_host)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: bad sizes or NULL tables");
  const size_t need = engram_forward_workspace_bytes(batch, seq, n_heads);
  const int64_t T = (int64_t)batch * seq;
  if (T > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 15)))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG,
                    "engram_forward: workspace NULL, misaligned or smaller than "
                    "engram_forward_workspace_bytes()");
  if (seq == 1 && T > 0) {
    const int which = engram::lookup_kernel_choice();
    if ((which == ENGRAM_LOOKUP_AUTO || which == ENGRAM_LOOKUP_BULK) &&
        engram::bulk_supported(tables_host->D, tables_host->dtype, n_heads))
      return decode_step(token_ids, batch, tid2eid, vocab, n_eids, history, history_out, n_heads,
                         tables_host, streams_in, streams_out, alpha, eps, status, stream);
  }
  int32_t *eids = static_cast<int32_t *>(workspace);
  int32_t *rows = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + round_up(T * 4));
  engram_status st = engram_compress(token_ids, T, tid2eid, vocab, n_eids, eids, status, stream);
  if (st != ENGRAM_OK) return st;
  st = engram_hash(eids, batch, seq, history, history_out, n_heads, tables_host->rows, rows, status,
                   stream);
  if (st != ENGRAM_OK) return st;
  return engram_lookup_fused(rows, T, n_heads, tables_host, streams_in, streams_out, alpha, eps,
                             nullptr, nullptr, status, stream);
}

ENGRAM_API size_t engram_forward_host_workspace_bytes(int32_t batch, int32_t seq,
                                                      int32_t n_heads, int32_t D,
                                                      int32_t chunk_tokens) {
  if (batch < 0 || seq < 0 || n_heads < 1 || D < 1 || chunk_tokens < 0) return 0;
  const size_t T = (size_t)batch * seq;
  const size_t chunk = chunk_tokens ? (size_t)chunk_tokens : kDefaultChunk;
  const size_t buf = round_up(chunk * 4 * (size_t)D * 2);
  return round_up(T * 4) + engram_forward_workspace_bytes(batch, seq, n_heads) + 2 * kBufs * buf;
}

ENGRAM_API engram_status engram_forward_host(
    const int32_t *token_ids_host, int32_t batch, int32_t seq, const int32_t *tid2eid,
    int32_t vocab, int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const engram_tables *tables_host, const uint16_t *streams_in_host,
    uint16_t *streams_out_host, const float *alpha, float eps, int32_t chunk_tokens,
    void *workspace, size_t workspace_bytes, int32_t *status, void *stream) {
  if (!tables_host || batch < 0 || seq < 0 || n_heads < 1 || n_heads > ENGRAM_MAX_HEADS ||
      chunk_tokens < 0)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward_host: bad sizes or NULL tables");
  const int64_t T = (int64_t)batch * seq;
  const int D = tables_host->D;
  if (D < 16 || D % 16 || D > ENGRAM_MAX_D)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward_host: bad D");
  const size_t need = engram_forward_host_workspace_bytes(batch, seq, n_heads, D, chunk_tokens);
  if (T > 0 && (!token_ids_host || !streams_in_host || !streams_out_host))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward_host: NULL host buffer");
  if (T > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 15)))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG,
                    "engram_forward_host: workspace NULL, misaligned or smaller than "
                    "engram_forward_host_workspace_bytes()");
  if (T == 0)
    return engram_hash(nullptr, batch, seq, history, history_out, n_heads, tables_host->rows,
                       nullptr, status, stream);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fwd_fail(ENGRAM_ERR_CUDA, "engram_forward_host: cudaGetDevice");
  HostPipe &hp = g_pipes[dev & 63];
  std::lock_guard<std::mutex> lock(hp.mu);
  if ((e = pipe_init(hp)) != cudaSuccess)
    return fwd_fail(ENGRAM_ERR_CUDA, "engram_forward_host: creating copy streams/events failed");
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const int64_t chunk = chunk_tokens ? chunk_tokens : kDefaultChunk;
  const size_t tok_bytes = (size_t)4 * D * 2;
  const size_t buf = round_up(chunk * tok_bytes);
  char *w = static_cast<char *>(workspace);
  int32_t *ids_dev = reinterpret_cast<int32_t *>(w);
  w += round_up(T * 4);
  int32_t *eids = reinterpret_cast<int32_t *>(w);
  w += round_up(T * 4);
  int32_t *rows = reinterpret_cast<int32_t *>(w);
  w += round_up(T * 3 * (size_t)n_heads * 4);
  char *in_buf = w;
  char *out_buf = w + kBufs * buf;

  // ids in, then compress + hash over the whole batch on the caller's stream.
  e = cudaMemcpyAsync(ids_dev, token_ids_host, T * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fwd_fail(ENGRAM_ERR_CUDA, "engram_forward_host: ids copy");
  engram_status st = engram_compress(ids_dev, T, tid2eid, vocab, n_eids, eids, status, stream);
  if (st != ENGRAM_OK) return st;
  st = engram_hash(eids, batch, seq, history, history_out, n_heads, tables_host->rows, rows, status,
                   stream);
  if (st != ENGRAM_OK) return st;

  // Chunk c uses buffer c % kBufs in each direction.  Every wait names the most
  // recent record of its event at the time it is enqueued, so the waits below
  // refer to chunk c - kBufs, or the previous call (buffer free), or to chunk c
  // itself (data ready).
  const int64_t nchunks = (T + chunk - 1) / chunk;
  const int R = 3 * n_heads;
  for (int64_t c = 0; c < nchunks; ++c) {
    const int b = (int)(c % kBufs);
    const int64_t t0 = c * chunk;
    const int64_t n = (T - t0) < chunk ? (T - t0) : chunk;
    char *ib = in_buf + b * buf, *ob = out_buf + b * buf;
    // (an event never recorded makes its wait a no-op; a record from the previous
    // call keeps that call's readers of this buffer ahead of the new copy)
    e = cudaStreamWaitEvent(hp.copy_in, hp.comp_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ib, reinterpret_cast<const char *>(streams_in_host) + t0 * tok_bytes,
                          n * tok_bytes, cudaMemcpyHostToDevice, hp.copy_in);
    if (e == cudaSuccess) e = cudaEventRecord(hp.in_done[b], hp.copy_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.in_done[b], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.out_done[b], 0);
    if (e != cudaSuccess) return fwd_fail(ENGRAM_ERR_CUDA, "engram_forward_host: copy in");
    st = engram_lookup_fused(rows + t0 * R, n, n_heads, tables_host,
                             reinterpret_cast<const uint16_t *>(ib), reinterpret_cast<uint16_t *>(ob),
                             alpha, eps, nullptr, nullptr, status, stream);
    if (st != ENGRAM_OK) return st;
    e = cudaEventRecord(hp.comp_done[b], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.copy_out, hp.comp_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(reinterpret_cast<char *>(streams_out_host) + t0 * tok_bytes, ob,
                          n * tok_bytes, cudaMemcpyDeviceToHost, hp.copy_out);
    if (e == cudaSuccess) e = cudaEventRecord(hp.out_done[b], hp.copy_out);
    if (e != cudaSuccess) return fwd_fail(ENGRAM_ERR_CUDA, "engram_forward_host: copy out");
  }
  // The caller's stream is ordered after the last copy out.
  const int last = (int)((nchunks - 1) % kBufs);
  e = cudaStreamWaitEvent(s, hp.out_done[last], 0);
  if (e != cudaSuccess) return fwd_fail(ENGRAM_ERR_CUDA, "engram_forward_host: final wait");
  return ENGRAM_OK;
}

}  // extern "C"
