// compress_hash.cu -- tid2eid compression and the 2/3/4-gram hash of the Engram
// lookup, for sm_103a.
//
// Both steps are a few bytes per token against the ~100 KB per token of the
// fused lookup, so they are written for simplicity and coalescing, not for
// bandwidth: one thread per token id (compression) and one thread per output
// row id (hash), with the 3H threads of a token in one block so that the ids of
// its window are read once from L1.
#include "engram_internal.cuh"
#include "hash_device.cuh"

namespace engram {
namespace {

__device__ __forceinline__ void flag_warp(int32_t *status, uint32_t flags) {
  // One atomic per warp instead of one per thread.
  const uint32_t all = __reduce_or_sync(0xffffffffu, flags);
  if (all && status && (threadIdx.x & 31) == 0) atomicOr(status, (int32_t)all);
}

// eids_out[i] = tid2eid[token_ids[i]] with range checks on both lookups.
__global__ void __launch_bounds__(256) compress_kernel(const __grid_constant__ CompressParams p) {
  uint32_t flags = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += stride) {
    if (p.dead && p.dead[i]) {
      p.eids_out[i] = ENGRAM_EID_DEAD;
      continue;
    }
    const int32_t tok = p.token_ids[i];
    if ((uint32_t)tok >= (uint32_t)p.vocab) {
      flags |= ENGRAM_FLAG_BAD_TOKEN;
      continue;
    }
    const int32_t e = __ldg(p.tid2eid + tok);
    if (e < 0 || e > p.n_eids) {
      flags |= ENGRAM_FLAG_BAD_EID;
      continue;
    }
    p.eids_out[i] = e;
  }
  flag_warp(p.status, flags);
}

// One thread per (token, order, head).  Thread r of a token computes row id r
// (n-major: r = (n-2)*H + j) from the token's window, read back from the token
// until its lookback limit (its position in its sample if positions are given,
// else 3 with a history and s without) or a dead id, whichever comes first;
// the slots beyond hold the pad id 0.  A dead token writes ENGRAM_ROW_DEAD.
__global__ void __launch_bounds__(256) hash_kernel(const __grid_constant__ HashParams p) {
  const int R = 3 * p.H;
  const int tl = threadIdx.x / R;
  const int r = threadIdx.x - tl * R;
  const int64_t t = (int64_t)blockIdx.x * p.tokens_per_block + tl;
  const bool valid = tl < p.tokens_per_block && t < p.T;
  uint32_t flags = 0;
  int32_t w[4] = {0, 0, 0, 0};  // oldest first, w[3] = the token's own id
  int32_t raw[4] = {0, 0, 0, 0};  // the ids s-3 .. s as stored (for history_out)
  int b = 0;
  if (valid) {
    b = (int)(t / p.seq);
    const int s = (int)(t - (int64_t)b * p.seq);
    const int64_t base = (int64_t)b * p.seq;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pos = s - 3 + k;
      if (pos >= 0)
        raw[k] = __ldg(p.eids + base + pos);
      else if (p.history)
        raw[k] = p.history[(int64_t)b * 3 + 3 + pos];  // plain load: history may be rewritten below
    }
    const int32_t self = raw[3];
    bool dead = self == ENGRAM_EID_DEAD, bad = self < ENGRAM_EID_DEAD;
    if (!dead && !bad) {
      // positions before 0 hold the history or 0 (raw), so the limit alone decides
      const int64_t limit = p.positions ? (int64_t)p.positions[base + s] : (p.history ? 3 : s);
      const int32_t before[3] = {raw[0], raw[1], raw[2]};
      bad = !make_window(before, self, limit, w);
    }
    if (bad) {
      flags = ENGRAM_FLAG_BAD_EID;
    } else if (dead) {
      p.row_ids[t * R + r] = ENGRAM_ROW_DEAD;
    } else {
      p.row_ids[t * R + r] = window_row(w, r, p.H, p.seed, p.mod, p.rmul, p.off);
    }
  }
  flag_warp(p.status, flags);
  if (p.history_inline) {
    // seq == 1: every reader of history[b] is a thread of this block.
    __syncthreads();
    if (valid && r == 0) {
#pragma unroll
      for (int k = 0; k < 3; ++k) p.history_out[(int64_t)b * 3 + k] = raw[k + 1];
    }
  }
}

// history_out[b] = last three ids of history[b] ++ eids[b]; one thread per
// sequence, all reads before any write (history_out may be history).
__global__ void history_kernel(const int32_t *eids, const int32_t *history, int32_t *history_out,
                               int32_t batch, int32_t seq) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  int32_t tail[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int pos = seq - 3 + k;
    tail[k] = pos >= 0 ? eids[(int64_t)b * seq + pos]
                       : (history ? history[(int64_t)b * 3 + 3 + pos] : 0);
  }
#pragma unroll
  for (int k = 0; k < 3; ++k) history_out[(int64_t)b * 3 + k] = tail[k];
}

}  // namespace

uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

cudaError_t launch_compress(const CompressParams &p, cudaStream_t stream) {
  if (p.n == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (p.n + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  compress_kernel<<<(unsigned)blocks, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_hash(const HashParams &p_in, cudaStream_t stream) {
  HashParams p = p_in;
  const int R = 3 * p.H;
  p.tokens_per_block = 256 / R > 0 ? 256 / R : 1;
  p.history_inline = (p.history_out != nullptr && p.seq == 1) ? 1 : 0;
  if (p.T > 0) {
    // Whole warps: flag_warp reduces over full warps; padding threads are invalid.
    const int threads = (p.tokens_per_block * R + 31) / 32 * 32;
    const int64_t blocks = (p.T + p.tokens_per_block - 1) / p.tokens_per_block;
    hash_kernel<<<(unsigned)blocks, threads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.history_out != nullptr && !p.history_inline && p.batch > 0) {
    history_kernel<<<(p.batch + 127) / 128, 128, 0, stream>>>(p.eids, p.history, p.history_out,
                                                               p.batch, p.seq);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace engram
