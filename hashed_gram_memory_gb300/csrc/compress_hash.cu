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

// The compressed id of position i when the hash compresses its own inputs: the
// dead id for a dead position (no range check), else the map's value, or
// kBadEid (below the dead id, so a window that reaches it is bad) with the
// reason in *why.
constexpr int32_t kBadEid = INT32_MIN;

__device__ __forceinline__ int32_t compress_at(const HashParams &p, int64_t i, uint32_t &why) {
  if (p.dead && p.dead[i]) return ENGRAM_EID_DEAD;
  const int32_t tok = __ldg(p.token_ids + i);
  if ((uint32_t)tok >= (uint32_t)p.vocab) {
    why = ENGRAM_FLAG_BAD_TOKEN;
    return kBadEid;
  }
  const int32_t e = __ldg(p.tid2eid + tok);
  if (e < 0 || e > p.n_eids) {
    why = ENGRAM_FLAG_BAD_EID;
    return kBadEid;
  }
  return e;
}

// One thread per token.  The thread reads the token's window once, back from
// the token until its lookback limit (its position in its sample if positions
// are given, else 3 with a history and s without) or a dead id, whichever comes
// first (the slots beyond hold the pad id 0), and computes its 3H row ids in a
// loop whose (order, head) index is the same in every lane: the per-(n, head)
// seeds, moduli and offsets are then warp-uniform parameter loads (an index
// that differs between lanes serialises them).  A dead token gets
// ENGRAM_ROW_DEAD.  The ids are staged in shared memory at an odd stride
// (conflict-free) and stored by the whole block, so that the stores are
// contiguous: the block's tokens own one contiguous range of row_ids.
// COMPRESS: the window's token ids are compressed here (the map is L2-resident,
// the neighbours' ids L1 hits), so no separate compression pass runs; a token
// whose own id or map value is out of range flags its reason, and every token
// whose window reaches it is left unwritten.
constexpr int kHashTokens = 64;

template <bool COMPRESS>
__global__ void __launch_bounds__(kHashTokens) hash_kernel(const __grid_constant__ HashParams p) {
  extern __shared__ int32_t s_rows[];  // [kHashTokens][stride], then [kHashTokens] skip flags
  const int R = 3 * p.H, stride = R | 1;
  int32_t *s_skip = s_rows + kHashTokens * stride;
  const int64_t t0 = (int64_t)blockIdx.x * kHashTokens;
  const int64_t t = t0 + threadIdx.x;
  uint32_t flags = 0;
  int skip = 1;
  if (t < p.T) {
    const int b = (int)(t / p.seq);
    const int s = (int)(t - (int64_t)b * p.seq);
    const int64_t base = (int64_t)b * p.seq;
    int32_t raw[4] = {0, 0, 0, 0};  // the ids s-3 .. s as stored (for history_out)
    uint32_t why = 0;               // COMPRESS: why the token's own id is bad
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pos = s - 3 + k;
      if (pos >= 0) {
        if (COMPRESS) {
          uint32_t w_k = 0;
          raw[k] = compress_at(p, base + pos, w_k);
          if (k == 3) why = w_k;
        } else {
          raw[k] = __ldg(p.eids + base + pos);
        }
      } else if (p.history) {
        raw[k] = p.history[(int64_t)b * 3 + 3 + pos];  // plain load: history may be rewritten below
      }
    }
    const int32_t self = raw[3];
    const bool dead = self == ENGRAM_EID_DEAD;
    const bool self_bad = COMPRESS && self == kBadEid;
    bool bad = self < ENGRAM_EID_DEAD;
    if (COMPRESS && !self_bad && p.eids_out) p.eids_out[t] = self;
    int32_t w[4] = {0, 0, 0, 0};  // oldest first, w[3] = the token's own id
    if (!dead && !bad) {
      // positions before 0 hold the history or 0 (raw), so the limit alone decides
      const int64_t limit = p.positions ? (int64_t)p.positions[base + s] : (p.history ? 3 : s);
      const int32_t before[3] = {raw[0], raw[1], raw[2]};
      bad = !make_window(before, self, limit, w);
    }
    int32_t *mine = s_rows + threadIdx.x * stride;
    if (bad) {
      flags = self_bad ? why : ENGRAM_FLAG_BAD_EID;
    } else if (dead) {
      for (int r = 0; r < R; ++r) mine[r] = ENGRAM_ROW_DEAD;
    } else {
      for (int r = 0; r < R; ++r) mine[r] = window_row(w, r, p.H, p.seed, p.mod, p.rmul, p.off);
    }
    skip = bad;
    if (p.history_inline && !self_bad) {
      // seq == 1: this thread is the only reader of history[b], and it is done.
#pragma unroll
      for (int k = 0; k < 3; ++k) p.history_out[(int64_t)b * 3 + k] = raw[k + 1];
    }
  }
  s_skip[threadIdx.x] = skip;
  flag_warp(p.status, flags);
  __syncthreads();
  // Contiguous stores: element i of the block's range is row r of token tl.
  const int64_t left = p.T - t0;
  const int n = left < kHashTokens ? (int)left : kHashTokens;
  int tl = (int)threadIdx.x / R, r = (int)threadIdx.x - tl * R;
  const int dq = kHashTokens / R, dr = kHashTokens - dq * R;  // kHashTokens = dq*R + dr
  for (int i = threadIdx.x; i < n * R; i += kHashTokens) {
    if (!s_skip[tl]) p.row_ids[t0 * R + i] = s_rows[tl * stride + r];
    tl += dq;
    r += dr;
    if (r >= R) {
      r -= R;
      ++tl;
    }
  }
}

// history_out[b] = last three ids of history[b] ++ eids[b]; one thread per
// sequence, all reads before any write (history_out may be history).
// COMPRESS: the last three ids are compressed here; a sequence whose tail holds
// a bad id keeps its history_out unwritten (the hash flagged it).
template <bool COMPRESS>
__global__ void history_kernel(const __grid_constant__ HashParams p) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.batch) return;
  int32_t tail[3];
  bool ok = true;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int pos = p.seq - 3 + k;
    if (pos >= 0) {
      if (COMPRESS) {
        uint32_t why = 0;
        tail[k] = compress_at(p, (int64_t)b * p.seq + pos, why);
        ok = ok && tail[k] != kBadEid;
      } else {
        tail[k] = p.eids[(int64_t)b * p.seq + pos];
      }
    } else {
      tail[k] = p.history ? p.history[(int64_t)b * 3 + 3 + pos] : 0;
    }
  }
  if (!ok) return;
#pragma unroll
  for (int k = 0; k < 3; ++k) p.history_out[(int64_t)b * 3 + k] = tail[k];
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
  const bool compress = p.token_ids != nullptr;
  p.tokens_per_block = kHashTokens;
  p.history_inline = (p.history_out != nullptr && p.seq == 1) ? 1 : 0;
  if (p.T > 0) {
    // kHashTokens is whole warps: flag_warp reduces over full warps.
    const size_t smem = (size_t)kHashTokens * ((R | 1) + 1) * sizeof(int32_t);
    const int64_t blocks = (p.T + kHashTokens - 1) / kHashTokens;
    if (compress)
      hash_kernel<true><<<(unsigned)blocks, kHashTokens, smem, stream>>>(p);
    else
      hash_kernel<false><<<(unsigned)blocks, kHashTokens, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.history_out != nullptr && !p.history_inline && p.batch > 0) {
    if (compress)
      history_kernel<true><<<(p.batch + 127) / 128, 128, 0, stream>>>(p);
    else
      history_kernel<false><<<(p.batch + 127) / 128, 128, 0, stream>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace engram
