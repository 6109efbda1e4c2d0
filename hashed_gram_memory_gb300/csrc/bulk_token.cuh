// bulk_token.cuh -- the bulk lookup of one token: a token's 3H row copies issued
// by warp 0 (one cp.async.bulk per row on one mbarrier), the row scales or block
// exponents staged in shared memory, the dequantise-and-accumulate of each
// thread's 16 columns, the gate reduction and the gated add into the four
// streams.  The phases are separate functions so that a block can also run
// several tokens in turn (the chained prefill kernel) with the next token's
// copies in flight under the current token's gate and stores; bulk_token runs
// them for one token (the one-token-a-block prefill kernel and the fused decode
// step).
#pragma once

#include "bulk_copy.cuh"
#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace engram {
namespace {

enum BulkState { kBulkLive = 0, kBulkDead = 1, kBulkBad = 2 };

// One token's staging in shared memory: its rows [R][row_bytes], their block
// exponents [R][exp_bytes] (e8m0 blocks apart from the rows), the mbarrier,
// the fp32 row scales [kMaxRows] and the gate's per-warp partial sums [8][3].
struct BulkSmem {
  uint8_t *rows;
  uint8_t *exps;
  uint64_t *bar;
  float *scale;
  float *red;
  uint32_t row_bytes, exp_bytes;
};

template <int DT>
__device__ __forceinline__ BulkSmem bulk_smem(uint8_t *sm, int R, int D) {
  constexpr bool kE8 = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32;
  BulkSmem s;
  s.row_bytes = table_row_bytes(DT, D);
  s.exp_bytes = kE8 ? (uint32_t)D / 32 : 0;
  s.rows = sm;
  s.exps = s.rows + (size_t)R * s.row_bytes;
  s.bar = reinterpret_cast<uint64_t *>(s.exps + (size_t)R * s.exp_bytes);
  s.scale = reinterpret_cast<float *>(s.bar + 1);
  s.red = s.scale + kMaxRows;
  return s;
}

// The token's state from its 3H ids, the same in every thread (thread r looks
// at row r, a loop when the block is narrower): live; dead (every id
// ENGRAM_ROW_DEAD); or bad (a mix, or an id outside its table), which flags
// the status word.  Contains a block-wide barrier.
__device__ __forceinline__ int bulk_state(const LookupParams &p, const int32_t *ids) {
  const int H = p.H, R = 3 * H;
  bool bad_here = false, dead_here = false, live_here = false;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int ni = (r >= H) + (r >= 2 * H);
    const int32_t id = ids[r];
    if (id == ENGRAM_ROW_DEAD) {
      dead_here = true;
    } else {
      live_here = true;
      bad_here |= (id < 0) | ((int64_t)id >= p.rows[ni]);
    }
  }
  if (!__syncthreads_or(bad_here || dead_here)) return kBulkLive;
  if (__syncthreads_and(!live_here)) return kBulkDead;
  if (threadIdx.x == 0 && p.status) atomicOr(p.status, ENGRAM_FLAG_BAD_ROW);
  return kBulkBad;
}

// Warp 0: every row copy of a live token on the barrier's current phase, lane r
// issuing the copies of rows r, r + 32, r + 64 from ids it loads itself (in
// parallel).  Without early streams, lane 0 then asks L2 for the token's
// streams, whose HBM reads start under the row copies.
template <bool EARLY>
__device__ __forceinline__ void bulk_issue_rows(const LookupParams &p, const int32_t *ids,
                                                int64_t t, const BulkSmem &s) {
  if (threadIdx.x >= 32) return;
  const int H = p.H, R = 3 * H, lane = threadIdx.x;
  if (lane == 0) mbar_arrive_expect_tx(s.bar, (uint32_t)R * s.row_bytes);
  __syncwarp();
  const int withheld = p.withhold != 0 ? 0 : -1;  // test hook: row 0's copy is never issued
  for (int r = lane; r < R; r += 32) {
    const int ni = (r >= H) + (r >= 2 * H);
    const int64_t id = ids[r];
    if (r != withheld)
      bulk_g2s(s.rows + (size_t)r * s.row_bytes, p.table[ni] + id * s.row_bytes, s.row_bytes, s.bar);
  }
  if (!EARLY && lane == 0) prefetch_l2(p.x + t * 4 * p.D, (uint32_t)(8 * p.D));
}

// The rows' (1, 32) block exponents (D/32 bytes each, a multiple of 16 here),
// 16 bytes per thread, coalesced.
__device__ __forceinline__ void bulk_load_exps(const LookupParams &p, const int32_t *ids,
                                               const BulkSmem &s) {
  const int H = p.H, R = 3 * H;
  const int per_row = (int)s.exp_bytes / 16;
  for (int i = threadIdx.x; i < R * per_row; i += blockDim.x) {
    const int r = i / per_row, c = i - r * per_row;
    const int ni = (r >= H) + (r >= 2 * H);
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(
        static_cast<const uint8_t *>(p.scale[ni]) + (int64_t)ids[r] * s.exp_bytes) + c);
    *reinterpret_cast<uint4 *>(s.exps + (size_t)r * s.exp_bytes + 16 * c) = v;
  }
}

// Row r's fp32 scale.
__device__ __forceinline__ float bulk_row_scale(const LookupParams &p, const int32_t *ids, int r) {
  const int ni = (r >= p.H) + (r >= 2 * p.H);
  return __ldg(static_cast<const float *>(p.scale[ni]) + ids[r]);
}

// What the accumulation reads besides the rows, staged in shared memory: the
// block exponents apart from the rows, or the fp32 row scales.
template <int DT>
__device__ __forceinline__ void bulk_load_scales(const LookupParams &p, const int32_t *ids,
                                                 const BulkSmem &s) {
  if constexpr (DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32) {
    bulk_load_exps(p, ids, s);
  } else if constexpr (DT == ENGRAM_TABLE_FP8_E4M3FN) {
    for (int r = threadIdx.x; r < 3 * p.H; r += blockDim.x) s.scale[r] = bulk_row_scale(p, ids, r);
  }
}

// The four stream slices of this thread (16 columns of each stream) into registers.
__device__ __forceinline__ void bulk_load_streams(const uint16_t *xrow, int D, uint4 (&xs)[4][2]) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    xs[s][0] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D));
    xs[s][1] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D + 8));
  }
}

// m over this thread's 16 columns: the mean of the token's dequantised rows,
// summed in row order from shared memory.
template <int DT>
__device__ __forceinline__ void bulk_accumulate(const LookupParams &p, const BulkSmem &s, int col0,
                                                float (&acc)[16]) {
  constexpr bool kFp8 = DT != ENGRAM_TABLE_BF16;
  constexpr bool kE8 = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32;
  constexpr bool kRows = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS;
  constexpr int kElt = kFp8 ? 1 : 2;
  const int R = 3 * p.H, D = p.D;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  const uint8_t *src = s.rows + (size_t)col0 * kElt;
#pragma unroll 4
  for (int r = 0; r < R; ++r) {
    const uint8_t *row = src + (size_t)r * s.row_bytes;
    if (kFp8) {
      const float scale = kRows ? e8m0_to_float(row[(D - col0) + (col0 >> 5)])
                          : kE8 ? e8m0_to_float(s.exps[(size_t)r * s.exp_bytes + (col0 >> 5)])
                                : s.scale[r];
      acc_fp8(acc, *reinterpret_cast<const uint4 *>(row), scale);
    } else {
      acc_bf16(acc, *reinterpret_cast<const uint4 *>(row));
      acc_bf16(acc + 8, *reinterpret_cast<const uint4 *>(row + 16));
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] *= p.inv_R;
}

// The gate of token t (its sums reduced over the block through s.red, one
// block-wide barrier) and the gated add into the four streams; without early
// streams the slices are loaded here, stream 0 first for the gate.  Then the
// gate and memory outputs when asked for.
template <bool AUX, bool EARLY>
__device__ __forceinline__ void bulk_gate_store(const LookupParams &p, int64_t t, const BulkSmem &s,
                                                uint4 (&xs)[4][2], const float (&acc)[16]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, D = p.D, col0 = tid * 16;
  const uint16_t *xrow = p.x + t * 4 * D + col0;
  if (!EARLY) {
    xs[0][0] = __ldcs(reinterpret_cast<const uint4 *>(xrow));
    xs[0][1] = __ldcs(reinterpret_cast<const uint4 *>(xrow + 8));
  }
  float saa = 0.f, smm = 0.f, sam = 0.f;
  gate_partials(xs[0][0], xs[0][1], acc, saa, smm, sam);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    saa += __shfl_xor_sync(0xffffffffu, saa, o);
    smm += __shfl_xor_sync(0xffffffffu, smm, o);
    sam += __shfl_xor_sync(0xffffffffu, sam, o);
  }
  if (lane == 0) {
    s.red[3 * warp + 0] = saa;
    s.red[3 * warp + 1] = smm;
    s.red[3 * warp + 2] = sam;
  }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  saa = smm = sam = 0.f;
  for (int w = 0; w < nw; ++w) {
    saa += s.red[3 * w + 0];
    smm += s.red[3 * w + 1];
    sam += s.red[3 * w + 2];
  }
  const float g = gate_value(saa, smm, sam, (float)D, p.eps, p.sqrt_D);

  uint16_t *yrow = p.y + t * 4 * D + col0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    if (!EARLY && s > 0) {
      xs[s][0] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D));
      xs[s][1] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D + 8));
    }
    const float c = g * __ldg(p.alpha + s);
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D), gated_add8(xs[s][0], acc, c));
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D + 8), gated_add8(xs[s][1], acc + 8, c));
  }
  if (AUX) {
    if (p.gate_out && tid == 0) p.gate_out[t] = g;
    if (p.mem_out) {
      float4 *mo = reinterpret_cast<float4 *>(p.mem_out + t * D + col0);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        mo[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
    }
  }
}

// A dead token's streams copied through (gate and memory outputs zero).
template <bool AUX>
__device__ __forceinline__ void bulk_pass_through(const LookupParams &p, int64_t t) {
  const int col0 = threadIdx.x * 16;
  pass_through16(p.x + t * 4 * p.D + col0, p.y + t * 4 * p.D + col0, p.D,
                 AUX && p.gate_out ? p.gate_out + t : nullptr,
                 AUX && p.mem_out ? p.mem_out + t * p.D + col0 : nullptr, threadIdx.x == 0);
}

// EARLY: the stream slices are loaded into registers before the rows arrive
// (two blocks per SM); otherwise after them, keeping the block within 64
// registers per thread so that four blocks share an SM (small tokens).
// Token t of a one-token-a-block launch, its 3H row ids at `ids` (global or
// shared memory).
template <int DT, bool AUX, bool EARLY>
__device__ __forceinline__ void bulk_token(const LookupParams &p, const int32_t *ids,
                                           const int64_t t) {
  constexpr bool kFp8 = DT != ENGRAM_TABLE_BF16;
  constexpr bool kE8 = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32;
  constexpr bool kRows = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS;
  extern __shared__ __align__(128) uint8_t sm[];
  const int R = 3 * p.H, tid = threadIdx.x;
  const BulkSmem s = bulk_smem<DT>(sm, R, p.D);

  if (tid == 0) {
    mbar_init(s.bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const int state = bulk_state(p, ids);  // its barrier also publishes the mbarrier's set-up
  if (state != kBulkLive) {
    if (state == kBulkDead) bulk_pass_through<AUX>(p, t);
    return;  // whole block: nothing issued
  }
  bulk_issue_rows<EARLY>(p, ids, t, s);
  // Meanwhile: the row scales into shared memory, the stream slices into registers.
  if constexpr (kE8) bulk_load_exps(p, ids, s);
  // fp32 row scales: thread r loads row r's scale; with the streams loaded
  // early it stores the scale only after issuing them (a store waits for its
  // load, and the stream loads should not wait behind it: 0.952 -> 0.961 on
  // the 8-head prefill; the same order for the e8m0 exponents measured 0.921 ->
  // 0.914, so they keep theirs).
  float sc = 0.f;
  if (kFp8 && !kE8 && !kRows && tid < R) {
    sc = bulk_row_scale(p, ids, tid);
    if (!EARLY) s.scale[tid] = sc;
  }
  uint4 xs[4][2];
  if (EARLY) bulk_load_streams(p.x + t * 4 * p.D + tid * 16, p.D, xs);
  if (kFp8 && !kE8 && !kRows) {
    if (EARLY && tid < R) s.scale[tid] = sc;
    for (int r = tid + blockDim.x; r < R; r += blockDim.x) s.scale[r] = bulk_row_scale(p, ids, r);
  }

  const bool landed = wait_bounded(s.bar, p.wait_limit_ns);
  // Block-uniform outcome (every wait above is bounded, so all threads get here);
  // the barrier also publishes the scales.
  if (__syncthreads_or(!landed)) {
    if (tid == 0) {
      if (p.status) atomicOr(p.status, ENGRAM_FLAG_TIMEOUT);
      wait_bounded(s.bar, p.wait_limit_ns);  // let the issued copies land before exit
    }
    return;
  }
  float acc[16];
  bulk_accumulate<DT>(p, s, tid * 16, acc);
  bulk_gate_store<AUX, EARLY>(p, t, s, xs, acc);
}

}  // namespace
}  // namespace engram
