// bulk_token.cuh -- the body of the one-token-a-block bulk lookup: a token's 3H
// row copies issued by warp 0 (one cp.async.bulk per row on one mbarrier), the
// row scales or block exponents staged in shared memory, the dequantise-and-
// accumulate of each thread's 16 columns, the gate reduction and the gated add
// into the four streams.  Used by the prefill lookup kernel and by the fused
// decode step.
#pragma once

#include "bulk_copy.cuh"
#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace engram {
namespace {

// EARLY: the stream slices are loaded into registers before the rows arrive
// (two blocks per SM); otherwise after them, keeping the block within 64
// registers per thread so that four blocks share an SM (small tokens).
// Token t of a one-token-a-block launch, its 3H row ids at `ids` (global or
// shared memory).
template <int DT, bool AUX, bool EARLY>
__device__ __forceinline__ void bulk_token(const LookupParams &p, const int32_t *ids,
                                           const int64_t t) {
  constexpr bool kFp8 = DT != ENGRAM_TABLE_BF16;                // FP8 bytes
  constexpr bool kE8 = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32;  // one exponent per 32 columns
  constexpr bool kRows = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS;  // the exponents after each row
  constexpr int kElt = kFp8 ? 1 : 2;
  extern __shared__ __align__(128) uint8_t sm[];

  const int H = p.H, R = 3 * H, D = p.D;
  const uint32_t row_bytes = table_row_bytes(DT, D);             // a row (+ its exponents)
  const uint32_t exp_bytes = kE8 ? (uint32_t)D / 32 : 0;         // a row's block exponents
  uint8_t *s_rows = sm;                                          // [R][row_bytes]
  uint8_t *s_exps = s_rows + (size_t)R * row_bytes;              // [R][exp_bytes]
  uint64_t *bar = reinterpret_cast<uint64_t *>(s_exps + (size_t)R * exp_bytes);
  float *s_scale = reinterpret_cast<float *>(bar + 1);           // [R]
  float *s_red = s_scale + kMaxRows;                             // [8][3]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int col0 = tid * 16;

  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Range checks: thread r looks at row r (a loop when the block is narrower).
  bool bad_here = false, dead_here = false, live_here = false;
  for (int r = tid; r < R; r += blockDim.x) {
    const int ni = (r >= H) + (r >= 2 * H);
    const int32_t id = ids[r];
    if (id == ENGRAM_ROW_DEAD) {
      dead_here = true;
    } else {
      live_here = true;
      bad_here |= (id < 0) | ((int64_t)id >= p.rows[ni]);
    }
  }
  if (__syncthreads_or(bad_here || dead_here)) {
    // A token whose ids are all dead passes through; any other mix is bad.
    if (__syncthreads_and(!live_here)) {
      pass_through16(p.x + t * 4 * D + col0, p.y + t * 4 * D + col0, D,
                     AUX && p.gate_out ? p.gate_out + t : nullptr,
                     AUX && p.mem_out ? p.mem_out + t * D + col0 : nullptr, tid == 0);
    } else if (tid == 0 && p.status) {
      atomicOr(p.status, ENGRAM_FLAG_BAD_ROW);
    }
    return;  // whole block: nothing issued
  }

  // Warp 0: every row copy of the token on the one barrier, lane r issuing the
  // copies of rows r, r + 32, r + 64 from ids it loads itself (in parallel).
  if (warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)R * row_bytes);
    __syncwarp();
    const int withheld = p.withhold != 0 ? 0 : -1;  // test hook: row 0's copy is never issued
    for (int r = lane; r < R; r += 32) {
      const int ni = (r >= H) + (r >= 2 * H);
      const int64_t id = ids[r];
      if (r != withheld)
        bulk_g2s(s_rows + (size_t)r * row_bytes, p.table[ni] + id * row_bytes, row_bytes, bar);
    }
    // Streams read after the rows: their HBM reads start now, under the row
    // copies, and the loads below find them in L2.
    if (!EARLY && lane == 0) prefetch_l2(p.x + t * 4 * D, (uint32_t)(8 * D));
  }
  // Meanwhile: the row scales into shared memory, the stream slices into registers.
  if constexpr (kE8) {
    // The rows' block exponents (D/32 bytes each, a multiple of 16 here), 16
    // bytes per thread, coalesced: their latency overlaps the row copies.
    const int per_row = (int)exp_bytes / 16;
    for (int i = tid; i < R * per_row; i += blockDim.x) {
      const int r = i / per_row, c = i - r * per_row;
      const int ni = (r >= H) + (r >= 2 * H);
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(
          static_cast<const uint8_t *>(p.scale[ni]) + (int64_t)ids[r] * exp_bytes) + c);
      *reinterpret_cast<uint4 *>(s_exps + (size_t)r * exp_bytes + 16 * c) = v;
    }
  }
  // fp32 row scales: thread r loads row r's scale; with the streams loaded
  // early it stores the scale only after issuing them (a store waits for its
  // load, and the stream loads should not wait behind it: 0.952 -> 0.961 on
  // the 8-head prefill; the same order for the e8m0 exponents measured 0.921 ->
  // 0.914, so they keep theirs).
  float sc = 0.f;
  if (kFp8 && !kE8 && !kRows && tid < R) {
    const int ni = (tid >= H) + (tid >= 2 * H);
    sc = __ldg(static_cast<const float *>(p.scale[ni]) + ids[tid]);
    if (!EARLY) s_scale[tid] = sc;
  }
  uint4 xs[4][2];
  const uint16_t *xrow = p.x + t * 4 * D + col0;
  if (EARLY) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      xs[s][0] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D));
      xs[s][1] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D + 8));
    }
  }
  if (kFp8 && !kE8 && !kRows) {
    if (EARLY && tid < R) s_scale[tid] = sc;
    for (int r = tid + blockDim.x; r < R; r += blockDim.x) {
      const int ni = (r >= H) + (r >= 2 * H);
      s_scale[r] = __ldg(static_cast<const float *>(p.scale[ni]) + ids[r]);
    }
  }

  const bool landed = wait_bounded(bar, p.wait_limit_ns);
  // Block-uniform outcome (every wait above is bounded, so all threads get here);
  // the barrier also publishes the scales.
  if (__syncthreads_or(!landed)) {
    if (tid == 0) {
      if (p.status) atomicOr(p.status, ENGRAM_FLAG_TIMEOUT);
      wait_bounded(bar, p.wait_limit_ns);  // let the issued copies land before exit
    }
    return;
  }

  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  const uint8_t *src = s_rows + (size_t)col0 * kElt;
#pragma unroll 4
  for (int r = 0; r < R; ++r) {
    const uint8_t *row = src + (size_t)r * row_bytes;
    if (kFp8) {
      const float scale = kRows ? e8m0_to_float(row[(D - col0) + (col0 >> 5)])
                          : kE8 ? e8m0_to_float(s_exps[(size_t)r * exp_bytes + (col0 >> 5)])
                                : s_scale[r];
      acc_fp8(acc, *reinterpret_cast<const uint4 *>(row), scale);
    } else {
      acc_bf16(acc, *reinterpret_cast<const uint4 *>(row));
      acc_bf16(acc + 8, *reinterpret_cast<const uint4 *>(row + 16));
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] *= p.inv_R;

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
    s_red[3 * warp + 0] = saa;
    s_red[3 * warp + 1] = smm;
    s_red[3 * warp + 2] = sam;
  }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  saa = smm = sam = 0.f;
  for (int w = 0; w < nw; ++w) {
    saa += s_red[3 * w + 0];
    smm += s_red[3 * w + 1];
    sam += s_red[3 * w + 2];
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

}  // namespace
}  // namespace engram
