// forward_static.cu -- engram_forward for callers that cannot allocate device
// memory.  The compressed ids and row ids that engram_forward keeps in a caller
// workspace live here in one file-scope device array instead, of a fixed size,
// which a device holds from the library's first use there until the process
// exits.
#include <cuda_runtime.h>

#include <mutex>

#include "engram_internal.cuh"

// The shared scratch.  In host code this name is only a host-side stand-in for
// the symbol, not a device address: the address comes from
// cudaGetSymbolAddress, with the device current, below.
static __device__ __align__(256) unsigned char g_engram_static_ws[ENGRAM_STATIC_WORKSPACE_BYTES];

namespace {

std::mutex g_static_mu;
void *g_static_addr[64];  // per device: the address found by the last call outside a capture

// True unless `stream` is known not to be capturing: a query that fails (the
// legacy stream while another stream captures) counts as capturing.
bool maybe_capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();  // the failed query leaves no sticky error
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

}  // namespace

extern "C" {

ENGRAM_API engram_status engram_forward_static(
    const int32_t *token_ids, int32_t batch, int32_t seq, const int32_t *tid2eid, int32_t vocab,
    int32_t n_eids, const int32_t *history, int32_t *history_out, int32_t n_heads,
    const engram_tables *tables_host, const engram_layout *layout_host,
    const uint16_t *streams_in, uint16_t *streams_out, const float *alpha, float eps,
    int32_t *status, void *stream) {
  ENGRAM_NVTX_RANGE("engram_forward_static");
  if (batch < 0 || seq < 0 || n_heads < 1 || n_heads > ENGRAM_MAX_HEADS || !tables_host)
    return engram::set_error(ENGRAM_ERR_INVALID_ARG, "engram_forward_static: bad sizes or NULL tables");
  const size_t need = engram_forward_workspace_bytes(batch, seq, n_heads);
  if (need > (size_t)ENGRAM_STATIC_WORKSPACE_BYTES)
    return engram::set_error(ENGRAM_ERR_UNSUPPORTED,
                             "engram_forward_static: batch %d x seq %d with %d heads needs %zu bytes "
                             "of scratch; the static workspace holds %zu (use engram_forward with "
                             "a caller workspace)",
                             batch, seq, n_heads, need, (size_t)ENGRAM_STATIC_WORKSPACE_BYTES);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return engram::set_error(ENGRAM_ERR_CUDA, "engram_forward_static: cudaGetDevice: %s",
                             cudaGetErrorString(e));
  if (dev < 0 || dev >= 64)
    return engram::set_error(ENGRAM_ERR_UNSUPPORTED, "engram_forward_static: device %d", dev);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  void *ws = nullptr;
  {
    // Outside a stream capture the address is looked up on every call, with
    // this device current, so a context created anew (after cudaDeviceReset)
    // gets its own; a call being captured reuses the last address looked up,
    // and there must be one.
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!maybe_capturing(s)) {
      void *addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_engram_static_ws);
      if (e != cudaSuccess || !addr)
        return engram::set_error(ENGRAM_ERR_CUDA,
                                 "engram_forward_static: cudaGetSymbolAddress: %s",
                                 cudaGetErrorString(e));
      g_static_addr[dev] = addr;
    } else if (!g_static_addr[dev]) {
      return engram::set_error(ENGRAM_ERR_INVALID_ARG,
                               "engram_forward_static: first call on device %d inside a stream "
                               "capture; make one call (batch 0 will do) before capturing",
                               dev);
    }
    ws = g_static_addr[dev];
  }
  // The array keeps the previous call's ids: clear the part this call uses, so
  // an element that a range error leaves unwritten reads as 0, never as stale.
  // A decode step runs as one fused launch that keeps its ids on chip and never
  // touches the array, so it needs no clear.
  if (need && !engram::forward_is_decode_step(batch, seq, n_heads, tables_host)) {
    e = cudaMemsetAsync(ws, 0, need, s);
    if (e != cudaSuccess)
      return engram::set_error(ENGRAM_ERR_CUDA, "engram_forward_static: clearing scratch: %s",
                               cudaGetErrorString(e));
  }
  return engram_forward(token_ids, batch, seq, tid2eid, vocab, n_eids, history, history_out,
                        n_heads, tables_host, layout_host, streams_in, streams_out, alpha, eps, ws,
                        (size_t)ENGRAM_STATIC_WORKSPACE_BYTES, status, stream);
}

}  // extern "C"
