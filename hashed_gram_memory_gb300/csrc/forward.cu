// forward.cu -- the whole Engram path in one call: engram_forward on device
// buffers, and the host-buffer calls engram_forward_host and
// engram_connection_host, which take the token ids and the four streams in
// host memory and overlap the host<->device copies with the compute in a
// three-buffer chunk pipeline over two copy streams.
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "engram_internal.cuh"

namespace {

constexpr size_t kAlign = 256;
constexpr int kBufs = 3;
constexpr int kDefaultChunk = 2048;             // lookup: one chunk is ~0.1 ms of work
constexpr int kDefaultConnectionChunk = 8192;   // projection: enough 256-row tiles for every SM pair

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

// The hash moduli and bucket offsets a layout gives (order-major, as the hash
// calls number the row ids): per-order tables of rows[n] rows, or one table cut
// into prime buckets laid end to end in draw order, which must fit each rows[n]
// (the tables struct names the one table for every order).
engram_status layout_buckets(const char *fn, const engram_tables *t, const engram_layout *lay,
                             int32_t n_heads, uint64_t (&mod)[3][engram::kMaxHeads],
                             uint64_t (&off)[3][engram::kMaxHeads]) {
  for (int n = 0; n < 3; ++n)
    if (t->rows[n] < 1 || t->rows[n] > INT32_MAX)
      return engram::set_error(ENGRAM_ERR_INVALID_ARG, "%s: rows must be in [1, 2^31-1]", fn);
  const int64_t *primes = lay ? lay->primes : nullptr;
  int64_t sum = 0;
  for (int n = 0; n < 3; ++n)
    for (int j = 0; j < n_heads; ++j) {
      if (!primes) {
        mod[n][j] = (uint64_t)t->rows[n];
        off[n][j] = 0;
        continue;
      }
      const int64_t p = primes[n * n_heads + j];
      if (p < 1 || p > INT32_MAX)
        return engram::set_error(ENGRAM_ERR_INVALID_ARG, "%s: bucket %d size out of range", fn,
                                 n * n_heads + j);
      mod[n][j] = (uint64_t)p;
      off[n][j] = (uint64_t)sum;
      sum += p;
    }
  if (primes)
    for (int n = 0; n < 3; ++n)
      if (sum > t->rows[n])
        return engram::set_error(ENGRAM_ERR_INVALID_ARG,
                                 "%s: the buckets hold %lld rows, table %d has %lld", fn,
                                 (long long)sum, n, (long long)t->rows[n]);
  return ENGRAM_OK;
}

// Compression (with the dead mask) and the hash (packed positions, prime
// buckets) of a whole batch into row ids, on `stream`, as one launch.
engram_status ids_to_rows(const int32_t *token_ids, int32_t batch, int32_t seq,
                          const int32_t *tid2eid, int32_t vocab, int32_t n_eids,
                          const int32_t *history, int32_t *history_out, int32_t n_heads,
                          const engram_tables *tables_host, const int32_t *positions,
                          const uint8_t *dead, const int64_t *primes, int32_t *rows,
                          int32_t *status, void *stream) {
  const engram_layout lay = {positions, dead, primes};
  return engram_compress_hash(token_ids, batch, seq, tid2eid, vocab, n_eids, history, history_out,
                              n_heads, tables_host->rows, &lay, nullptr, rows, status, stream);
}

// One decode step (one new token a slot) in one launch: compression, window,
// hash and bulk lookup fused, with the same argument checks as the three
// calls it replaces.  The row ids are not written out.
engram_status decode_step(const int32_t *token_ids, int32_t batch, const int32_t *tid2eid,
                          int32_t vocab, int32_t n_eids, const int32_t *history,
                          int32_t *history_out, int32_t n_heads, const engram_tables *tables_host,
                          const engram_layout *layout, const uint16_t *streams_in,
                          uint16_t *streams_out, const float *alpha, float eps, int32_t *status,
                          void *stream) {
  const char *fn = "engram_forward";
  const int32_t *positions = layout ? layout->positions : nullptr;
  const uint8_t *dead = layout ? layout->dead : nullptr;
  if (!token_ids || !tid2eid || misaligned4(token_ids) || misaligned4(tid2eid))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: token_ids or tid2eid NULL or misaligned");
  if (vocab < 1 || n_eids < 0)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: vocab must be >= 1 and n_eids >= 0");
  if (misaligned4(history) || misaligned4(history_out) || misaligned4(positions))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG,
                    "engram_forward: history or positions pointers not 4-byte aligned");
  const size_t hb = (size_t)batch * 12;
  const size_t sb = (size_t)batch * 4 * tables_host->D * 2;
  if (history && history_out && history != history_out && overlaps(history, hb, history_out, hb))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: history and history_out overlap partially");
  if (history_out && (overlaps(history_out, hb, streams_out, sb) ||
                      overlaps(history_out, hb, token_ids, (size_t)batch * 4) ||
                      overlaps(history_out, hb, positions, (size_t)batch * 4) ||
                      overlaps(history_out, hb, dead, (size_t)batch)))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: history_out overlaps another buffer");
  engram::DecodeParams p;
  memset(&p, 0, sizeof p);
  engram_status st = layout_buckets(fn, tables_host, layout, n_heads, p.mod, p.off);
  if (st != ENGRAM_OK) return st;
  st = engram::prepare_lookup(fn, nullptr, false, batch, n_heads, tables_host, streams_in,
                              streams_out, alpha, eps, nullptr, nullptr, status, p.lk);
  if (st != ENGRAM_OK) return st;
  p.lk.withhold = engram::take_withheld_launch() ? 1 : 0;
  p.token_ids = token_ids;
  p.tid2eid = tid2eid;
  p.history = history;
  p.history_out = history_out;
  p.positions = positions;
  p.dead = dead;
  p.vocab = vocab;
  p.n_eids = n_eids;
  for (int n = 0; n < 3; ++n)
    for (int j = 0; j < n_heads; ++j) {
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

namespace engram {

// One new token a slot, and the bulk lookup family applies: engram_forward runs
// the step as the one fused decode launch, which needs no workspace.
bool forward_is_decode_step(int32_t batch, int32_t seq, int32_t n_heads,
                            const engram_tables *tables_host) {
  if (seq != 1 || batch < 1 || !tables_host) return false;
  const int which = lookup_kernel_choice();
  return (which == ENGRAM_LOOKUP_AUTO || which == ENGRAM_LOOKUP_BULK) &&
         decode_supported(tables_host->D, tables_host->dtype, n_heads);
}

}  // namespace engram

namespace {

// The chunk pipeline of the host-buffer calls.  Chunk c of the streams uses
// buffer c % kBufs in each direction: its host->device copy on copy_in, then
// `compute(t0, n, in, out)` on the caller's stream, then its device->host copy
// on copy_out.  Every wait names the most recent record of its event at the
// time it is enqueued, so a wait refers to chunk c - kBufs or the previous call
// (the buffer is free again) or to chunk c itself (its data is ready); an event
// never recorded makes its wait a no-op.  On return the caller's stream is
// ordered after the last copy out.
template <class Compute>
engram_status run_chunks(const char *fn, HostPipe &hp, cudaStream_t s, int64_t T, int64_t chunk,
                         size_t tok_bytes, char *in_buf, char *out_buf, size_t buf,
                         const void *in_host, void *out_host, Compute compute) {
  const int64_t nchunks = (T + chunk - 1) / chunk;
  cudaError_t e = cudaSuccess;
  for (int64_t c = 0; c < nchunks; ++c) {
    const int b = (int)(c % kBufs);
    const int64_t t0 = c * chunk;
    const int64_t n = (T - t0) < chunk ? (T - t0) : chunk;
    char *ib = in_buf + b * buf, *ob = out_buf + b * buf;
    e = cudaStreamWaitEvent(hp.copy_in, hp.comp_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ib, static_cast<const char *>(in_host) + t0 * tok_bytes, n * tok_bytes,
                          cudaMemcpyHostToDevice, hp.copy_in);
    if (e == cudaSuccess) e = cudaEventRecord(hp.in_done[b], hp.copy_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.in_done[b], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.out_done[b], 0);
    if (e != cudaSuccess)
      return engram::set_error(ENGRAM_ERR_CUDA, "%s: copy in: %s", fn, cudaGetErrorString(e));
    const engram_status st = compute(t0, n, ib, ob);
    if (st != ENGRAM_OK) return st;
    e = cudaEventRecord(hp.comp_done[b], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.copy_out, hp.comp_done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char *>(out_host) + t0 * tok_bytes, ob, n * tok_bytes,
                          cudaMemcpyDeviceToHost, hp.copy_out);
    if (e == cudaSuccess) e = cudaEventRecord(hp.out_done[b], hp.copy_out);
    if (e != cudaSuccess)
      return engram::set_error(ENGRAM_ERR_CUDA, "%s: copy out: %s", fn, cudaGetErrorString(e));
  }
  e = cudaStreamWaitEvent(s, hp.out_done[(nchunks - 1) % kBufs], 0);
  if (e != cudaSuccess)
    return engram::set_error(ENGRAM_ERR_CUDA, "%s: final wait: %s", fn, cudaGetErrorString(e));
  return ENGRAM_OK;
}

// Device copies of the per-token host inputs (ids, positions, dead mask) of a
// host-buffer call, carved from the front of its workspace, and the row ids the
// hash writes (eids: room for compressed ids, which the one-launch
// compress-hash does not need).
struct HostIds {
  int32_t *ids, *positions, *eids, *rows;
  uint8_t *dead;
  char *rest;  // the rest of the workspace
};

size_t host_ids_bytes(size_t T, int32_t n_heads) {
  return 3 * round_up(T * 4) + round_up(T) + round_up(T * 3 * (size_t)n_heads * 4);
}

HostIds carve_host_ids(void *workspace, int64_t T, int32_t n_heads) {
  HostIds h;
  char *w = static_cast<char *>(workspace);
  h.ids = reinterpret_cast<int32_t *>(w);
  w += round_up(T * 4);
  h.positions = reinterpret_cast<int32_t *>(w);
  w += round_up(T * 4);
  h.eids = reinterpret_cast<int32_t *>(w);
  w += round_up(T * 4);
  h.dead = reinterpret_cast<uint8_t *>(w);
  w += round_up(T);
  h.rows = reinterpret_cast<int32_t *>(w);
  w += round_up(T * 3 * (size_t)n_heads * 4);
  h.rest = w;
  return h;
}

// Copies the host ids (and the layout's host positions and dead mask) in on `s`.
engram_status copy_host_ids(const char *fn, const HostIds &h, const int32_t *token_ids_host,
                            int64_t T, const engram_layout *layout, cudaStream_t s) {
  const int32_t *pos_host = layout ? layout->positions : nullptr;
  const uint8_t *dead_host = layout ? layout->dead : nullptr;
  cudaError_t e = cudaMemcpyAsync(h.ids, token_ids_host, T * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && pos_host)
    e = cudaMemcpyAsync(h.positions, pos_host, T * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && dead_host)
    e = cudaMemcpyAsync(h.dead, dead_host, T, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess)
    return engram::set_error(ENGRAM_ERR_CUDA, "%s: ids copy: %s", fn, cudaGetErrorString(e));
  return ENGRAM_OK;
}

// Copies the host ids (and layout) in on `s`, then compresses and hashes the
// whole batch there.
engram_status host_ids_to_rows(const char *fn, const HostIds &h, const int32_t *token_ids_host,
                               int32_t batch, int32_t seq, const int32_t *tid2eid, int32_t vocab,
                               int32_t n_eids, const int32_t *history, int32_t *history_out,
                               int32_t n_heads, const engram_tables *tables_host,
                               const engram_layout *layout, int32_t *status, cudaStream_t s) {
  const int64_t T = (int64_t)batch * seq;
  const int32_t *pos_host = layout ? layout->positions : nullptr;
  const uint8_t *dead_host = layout ? layout->dead : nullptr;
  const engram_status st = copy_host_ids(fn, h, token_ids_host, T, layout, s);
  if (st != ENGRAM_OK) return st;
  return ids_to_rows(h.ids, batch, seq, tid2eid, vocab, n_eids, history, history_out, n_heads,
                     tables_host, pos_host ? h.positions : nullptr, dead_host ? h.dead : nullptr,
                     layout ? layout->primes : nullptr, h.rows, status, s);
}

// The per-device pipe, locked for the call; NULL (error set) if it cannot be made.
HostPipe *acquire_pipe(const char *fn, std::unique_lock<std::mutex> &lock) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    engram::set_error(ENGRAM_ERR_CUDA, "%s: cudaGetDevice", fn);
    return nullptr;
  }
  HostPipe &hp = g_pipes[dev];
  lock = std::unique_lock<std::mutex>(hp.mu);
  if ((e = pipe_init(hp)) != cudaSuccess) {
    engram::set_error(ENGRAM_ERR_CUDA, "%s: creating copy streams/events: %s", fn,
                      cudaGetErrorString(e));
    return nullptr;
  }
  return &hp;
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
                                        const engram_layout *layout_host,
                                        const uint16_t *streams_in, uint16_t *streams_out,
                                        const float *alpha, float eps, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_forward");
  if (batch < 0 || seq < 0 || n_heads < 1 || n_heads > ENGRAM_MAX_HEADS || !tables_host)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_forward: bad sizes or NULL tables");
  const size_t need = engram_forward_workspace_bytes(batch, seq, n_heads);
  const int64_t T = (int64_t)batch * seq;
  if (T > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 15)))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG,
                    "engram_forward: workspace NULL, misaligned or smaller than "
                    "engram_forward_workspace_bytes()");
  uint64_t mod[3][engram::kMaxHeads], off[3][engram::kMaxHeads];
  engram_status st = layout_buckets("engram_forward", tables_host, layout_host, n_heads, mod, off);
  if (st != ENGRAM_OK) return st;
  if (engram::forward_is_decode_step(batch, seq, n_heads, tables_host))
    return decode_step(token_ids, batch, tid2eid, vocab, n_eids, history, history_out, n_heads,
                       tables_host, layout_host, streams_in, streams_out, alpha, eps, status,
                       stream);
  int32_t *rows = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + round_up(T * 4));
  st = ids_to_rows(token_ids, batch, seq, tid2eid, vocab, n_eids, history,
                   history_out, n_heads, tables_host,
                   layout_host ? layout_host->positions : nullptr,
                   layout_host ? layout_host->dead : nullptr,
                   layout_host ? layout_host->primes : nullptr, rows, status, stream);
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
  return host_ids_bytes(T, n_heads) + 2 * kBufs * buf;
}

ENGRAM_API engram_status engram_forward_host(
    const int32_t *token_ids_host, int32_t batch, int32_t seq, const int32_t *tid2eid,
    int32_t vocab, int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const engram_tables *tables_host, const engram_layout *layout_host,
    const uint16_t *streams_in_host, uint16_t *streams_out_host, const float *alpha, float eps,
    int32_t chunk_tokens, void *workspace, size_t workspace_bytes, int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_forward_host");
  const char *fn = "engram_forward_host";
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
  uint64_t mod[3][engram::kMaxHeads], off[3][engram::kMaxHeads];
  engram_status st = layout_buckets(fn, tables_host, layout_host, n_heads, mod, off);
  if (st != ENGRAM_OK) return st;
  // The lookup's own checks of the tables, alpha and eps (a call of no tokens),
  // before anything is enqueued.
  st = engram_lookup_fused(nullptr, 0, n_heads, tables_host, nullptr, nullptr, alpha, eps,
                           nullptr, nullptr, status, stream);
  if (st != ENGRAM_OK) return st;
  if (T == 0)  // only the history moves (unchanged: no new ids)
    return engram_hash(nullptr, batch, seq, history, history_out, n_heads, tables_host->rows,
                       nullptr, status, stream);
  std::unique_lock<std::mutex> lock;
  HostPipe *hp = acquire_pipe(fn, lock);
  if (!hp) return ENGRAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const HostIds h = carve_host_ids(workspace, T, n_heads);
  const int64_t chunk = chunk_tokens ? chunk_tokens : kDefaultChunk;
  const size_t tok_bytes = (size_t)4 * D * 2;
  const size_t buf = round_up(chunk * tok_bytes);
  const int which = engram::lookup_kernel_choice();
  if (seq == 1 && (which == ENGRAM_LOOKUP_AUTO || which == ENGRAM_LOOKUP_BULK) &&
      engram::decode_supported(D, tables_host->dtype, n_heads)) {
    // A decode step: each chunk of slots is one fused launch (compression,
    // window, hash and lookup), as engram_forward runs it; only the ids move
    // in ahead of the streams.
    st = copy_host_ids(fn, h, token_ids_host, T, layout_host, s);
    if (st != ENGRAM_OK) return st;
    const int32_t *pos = layout_host && layout_host->positions ? h.positions : nullptr;
    const uint8_t *dead = layout_host && layout_host->dead ? h.dead : nullptr;
    const int64_t *primes = layout_host ? layout_host->primes : nullptr;
    return run_chunks(fn, *hp, s, T, chunk, tok_bytes, h.rest, h.rest + kBufs * buf, buf,
                      streams_in_host, streams_out_host,
                      [&](int64_t t0, int64_t n, char *ib, char *ob) {
                        const engram_layout lay = {pos ? pos + t0 : nullptr,
                                                   dead ? dead + t0 : nullptr, primes};
                        return decode_step(h.ids + t0, (int32_t)n, tid2eid, vocab, n_eids,
                                           history ? history + t0 * 3 : nullptr,
                                           history_out ? history_out + t0 * 3 : nullptr, n_heads,
                                           tables_host, &lay,
                                           reinterpret_cast<const uint16_t *>(ib),
                                           reinterpret_cast<uint16_t *>(ob), alpha, eps, status,
                                           stream);
                      });
  }
  st = host_ids_to_rows(fn, h, token_ids_host, batch, seq, tid2eid, vocab, n_eids, history,
                        history_out, n_heads, tables_host, layout_host, status, s);
  if (st != ENGRAM_OK) return st;
  const int R = 3 * n_heads;
  return run_chunks(fn, *hp, s, T, chunk, tok_bytes, h.rest, h.rest + kBufs * buf, buf,
                    streams_in_host, streams_out_host,
                    [&](int64_t t0, int64_t n, char *ib, char *ob) {
                      return engram_lookup_fused(h.rows + t0 * R, n, n_heads, tables_host,
                                                 reinterpret_cast<const uint16_t *>(ib),
                                                 reinterpret_cast<uint16_t *>(ob), alpha, eps,
                                                 nullptr, nullptr, status, stream);
                    });
}

ENGRAM_API size_t engram_connection_host_workspace_bytes(int32_t batch, int32_t seq,
                                                         int32_t n_heads, int32_t d, int32_t D,
                                                         int32_t chunk_tokens) {
  if (batch < 0 || seq < 0 || n_heads < 1 || d < 1 || D < 1 || chunk_tokens < 0) return 0;
  const size_t T = (size_t)batch * seq;
  const size_t chunk = chunk_tokens ? (size_t)chunk_tokens : kDefaultConnectionChunk;
  const size_t buf = round_up(chunk * 4 * (size_t)D * 2);
  return host_ids_bytes(T, n_heads) + 2 * kBufs * buf +
         round_up(engram_connection_workspace_bytes((int64_t)chunk, n_heads, d, D));
}

ENGRAM_API engram_status engram_connection_host(
    const int32_t *token_ids_host, int32_t batch, int32_t seq, const int32_t *tid2eid,
    int32_t vocab, int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const engram_tables *tables_host, const engram_layout *layout_host, const uint16_t *wkv,
    int32_t D, const uint16_t *streams_in_host, uint16_t *streams_out_host, const float *alpha,
    float eps, int32_t chunk_tokens, void *workspace, size_t workspace_bytes, int32_t *status,
    void *stream) {
  ENGRAM_NVTX_RANGE("engram_connection_host");
  const char *fn = "engram_connection_host";
  if (!tables_host || batch < 0 || seq < 0 || n_heads < 1 || n_heads > ENGRAM_MAX_HEADS ||
      chunk_tokens < 0 || D < 1)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_connection_host: bad sizes or NULL tables");
  const int64_t T = (int64_t)batch * seq;
  const int d = tables_host->D;
  const size_t need =
      engram_connection_host_workspace_bytes(batch, seq, n_heads, d, D, chunk_tokens);
  if (need == 0)
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_connection_host: bad row width");
  if (T > 0 && (!token_ids_host || !streams_in_host || !streams_out_host))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG, "engram_connection_host: NULL host buffer");
  if (T > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)))
    return fwd_fail(ENGRAM_ERR_INVALID_ARG,
                    "engram_connection_host: workspace NULL, not 256-byte aligned or smaller "
                    "than engram_connection_host_workspace_bytes()");
  uint64_t mod[3][engram::kMaxHeads], off[3][engram::kMaxHeads];
  engram_status st = layout_buckets(fn, tables_host, layout_host, n_heads, mod, off);
  if (st != ENGRAM_OK) return st;
  // The connection's own checks of the tables, wkv, D, alpha and eps (a call of
  // no tokens), before anything is enqueued.
  st = engram_connection(nullptr, 0, n_heads, tables_host, wkv, D, nullptr, nullptr, alpha, eps,
                         nullptr, 0, nullptr, nullptr, status, stream);
  if (st != ENGRAM_OK) return st;
  if (T == 0)
    return engram_hash(nullptr, batch, seq, history, history_out, n_heads, tables_host->rows,
                       nullptr, status, stream);
  std::unique_lock<std::mutex> lock;
  HostPipe *hp = acquire_pipe(fn, lock);
  if (!hp) return ENGRAM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const HostIds h = carve_host_ids(workspace, T, n_heads);
  st = host_ids_to_rows(fn, h, token_ids_host, batch, seq, tid2eid, vocab, n_eids, history,
                        history_out, n_heads, tables_host, layout_host, status, s);
  if (st != ENGRAM_OK) return st;
  const int64_t chunk = chunk_tokens ? chunk_tokens : kDefaultConnectionChunk;
  const size_t tok_bytes = (size_t)4 * D * 2;
  const size_t buf = round_up(chunk * tok_bytes);
  char *conn_ws = h.rest + 2 * kBufs * buf;
  const size_t conn_bytes = engram_connection_workspace_bytes(chunk, n_heads, d, D);
  const int R = 3 * n_heads;
  // One connection workspace serves every chunk: the chunks' connections run
  // one after another on the caller's stream.
  return run_chunks(fn, *hp, s, T, chunk, tok_bytes, h.rest, h.rest + kBufs * buf, buf,
                    streams_in_host, streams_out_host,
                    [&](int64_t t0, int64_t n, char *ib, char *ob) {
                      return engram_connection(h.rows + t0 * R, n, n_heads, tables_host, wkv, D,
                                               reinterpret_cast<const uint16_t *>(ib),
                                               reinterpret_cast<uint16_t *>(ob), alpha, eps,
                                               conn_ws, conn_bytes, nullptr, nullptr, status,
                                               stream);
                    });
}

}  // extern "C"
