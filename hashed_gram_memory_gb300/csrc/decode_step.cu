// decode_step.cu -- one decode step of the Engram path (one new token a slot) in
// one launch, for sm_103a: compression of the slot's token, its window from the
// slot's three-id history, the hash into row ids kept in shared memory, and the
// one-token-a-block bulk lookup body on them.
//
// The launch allows programmatic dependent launch: each block first waits for
// the previous grid on the stream to finish (griddepcontrol.wait, before any
// memory access, so the result never depends on what that grid wrote), then
// lets the next grid be scheduled into the room it leaves.  Back to back, a
// step's blocks are then resident when the previous step ends instead of being
// launched after it.
#include <atomic>

#include "bulk_copy.cuh"
#include "bulk_token.cuh"
#include "engram_internal.cuh"
#include "hash_device.cuh"

namespace engram {
namespace {

// A tid2eid entry, kept in L2 with the evict_last priority: the map (4 bytes a
// vocabulary entry) is read at random by every decode step, and its lines
// otherwise leave L2 between steps under the steps' own row and stream traffic
// (16.49 -> 16.28 us a step on 512 slots with cold ids and rows).
__device__ __forceinline__ int32_t ld_map_entry(const int32_t *p) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  int32_t v;
  asm volatile("ld.global.nc.L2::cache_hint.s32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
  return v;
}

// The decode step in one launch (one new token per slot, one slot a block):
// thread 0 compresses the slot's token id (a slot of the dead mask becomes the
// dead id), builds its window from the slot's history (the pad id 0 without
// one) back to its lookback limit (its position in its sample when positions
// are given), and writes the updated history; the first 3H threads hash the
// window into the row ids (the hash kernel's arithmetic, hash_device.cuh; a
// dead slot gets ENGRAM_ROW_DEAD), kept in shared memory; then the block looks
// them up as bulk_token does.  A bad token id, map value or history id flags
// the status word and leaves all of the slot's outputs unwritten.
template <int DT, bool AUX, bool EARLY>
__global__ void __launch_bounds__(256, EARLY ? 2 : 4)
    decode_step_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ int32_t s_ids[kMaxRows];
  __shared__ int32_t s_win[4];
  __shared__ int s_skip, s_dead;
  const int64_t b = blockIdx.x;
  const int H = p.lk.H, R = 3 * H;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The slot's streams do not depend on its token: their HBM reads start now,
  // under the dependent loads of the token and its map entry.
  if (threadIdx.x == 32) prefetch_l2(p.lk.x + b * 4 * p.lk.D, (uint32_t)(8 * p.lk.D));
  if (threadIdx.x == 0) {
    int32_t raw[3] = {0, 0, 0};
    if (p.history)
      for (int k = 0; k < 3; ++k) raw[k] = p.history[b * 3 + k];
    // A dead slot compresses to the dead id whatever its token (no range check).
    const bool dead = p.dead && p.dead[b];
    uint32_t flag = 0;
    int32_t e = ENGRAM_EID_DEAD, w[4];
    if (!dead) {
      const int32_t tok = p.token_ids[b];
      if ((uint32_t)tok >= (uint32_t)p.vocab) {
        flag = ENGRAM_FLAG_BAD_TOKEN;
      } else {
        e = ld_map_entry(p.tid2eid + tok);
        if (e < 0 || e > p.n_eids) flag = ENGRAM_FLAG_BAD_EID;
      }
      // lookback: the position in the sample if given, else the 3-id history or nothing
      const int64_t limit = p.positions ? (int64_t)p.positions[b] : (p.history ? 3 : 0);
      if (!flag && !make_window(raw, e, limit, w)) flag = ENGRAM_FLAG_BAD_EID;
    }
    if (!flag) {
      if (!dead)
        for (int k = 0; k < 4; ++k) s_win[k] = w[k];
      if (p.history_out) {
        p.history_out[b * 3 + 0] = raw[1];
        p.history_out[b * 3 + 1] = raw[2];
        p.history_out[b * 3 + 2] = e;
      }
    } else if (p.lk.status) {
      atomicOr(p.lk.status, (int32_t)flag);
    }
    s_skip = flag != 0;
    s_dead = dead;
  }
  __syncthreads();
  if (s_skip) return;  // block-uniform
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    int32_t id = ENGRAM_ROW_DEAD;
    if (!s_dead) {
      const int32_t w[4] = {s_win[0], s_win[1], s_win[2], s_win[3]};
      id = window_row(w, r, H, p.seed, p.mod, p.rmul, p.off);
    }
    s_ids[r] = id;
    if (p.row_ids_out) p.row_ids_out[b * R + r] = id;
  }
  __syncthreads();
  bulk_token<DT, AUX, EARLY>(p.lk, s_ids, b);
}

template <int DT, bool AUX, bool EARLY>
cudaError_t launch_decode_t(const DecodeParams &p, size_t smem, cudaStream_t stream) {
  auto kern = decode_step_kernel<DT, AUX, EARLY>;
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = raise_smem_ceiling(kern, configured);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.lk.T);
  cfg.blockDim = dim3((unsigned)(p.lk.D / 16));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int DT>
cudaError_t launch_decode_dt(const DecodeParams &p, size_t smem, bool aux, bool early,
                             cudaStream_t stream) {
  if (early)
    return aux ? launch_decode_t<DT, true, true>(p, smem, stream)
               : launch_decode_t<DT, false, true>(p, smem, stream);
  return aux ? launch_decode_t<DT, true, false>(p, smem, stream)
             : launch_decode_t<DT, false, false>(p, smem, stream);
}

}  // namespace

// The slot's block is the one-token-a-block lookup's: the same shape limits.
bool decode_supported(int D, int dtype, int H) { return bulk_supported(D, dtype, H); }

cudaError_t launch_decode_step(const DecodeParams &p, int dtype, cudaStream_t stream) {
  if (p.lk.T == 0) return cudaSuccess;
  const size_t smem = bulk_smem_bytes(p.lk.D, dtype, p.lk.H);
  const bool aux = p.lk.gate_out != nullptr || p.lk.mem_out != nullptr;
  const bool early = smem > 56 * 1024;
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN)
    return launch_decode_dt<ENGRAM_TABLE_FP8_E4M3FN>(p, smem, aux, early, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32)
    return launch_decode_dt<ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32>(p, smem, aux, early, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS)
    return launch_decode_dt<ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS>(p, smem, aux, early, stream);
  return launch_decode_dt<ENGRAM_TABLE_BF16>(p, smem, aux, early, stream);
}

}  // namespace engram
