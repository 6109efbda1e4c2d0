// lookup_fused.cu -- the fused Engram lookup for sm_103a: gather + dequantise the
// 3H rows of a token, average them into m, RMSNorm dot-product sigmoid gate
// against stream 0, and the gated add into the four bf16 mHC streams, in one
// pass over HBM.
//
// Work layout: a token is handled by tpt threads, each owning 16 consecutive
// columns (one 16-byte load per FP8 row, two per BF16 row, 32 bytes per bf16
// stream).  For D = 4096 a token is one 256-thread block; small D packs several
// tokens into a block.  Everything stays in registers: the four stream slices
// are loaded up front (they are needed for the gate and the add), the rows are
// loaded in batches so that ~32 KB per block is in flight, and the three sums
// of the gate are reduced with warp shuffles (plus one shared-memory step when a
// token spans several warps).  Rows are read with L1::no_allocate (no reuse
// inside an SM); streams with .cs (evict-first) so they do not push hot table
// rows out of L2.
#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace engram {
namespace {

__device__ __forceinline__ uint4 ld_row16(const uint8_t *ptr) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(ptr));
  return v;
}

template <int DT, bool AUX>
__global__ void __launch_bounds__(256, 2) lookup_kernel(const __grid_constant__ LookupParams p) {
  constexpr bool kFp8 = DT != ENGRAM_TABLE_BF16;           // FP8 bytes (row or block scales)
  constexpr bool kE8 = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32;  // one exponent per 32 columns
  constexpr bool kRows = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS;  // the exponents after each row
  constexpr int kElt = kFp8 ? 1 : 2;         // bytes per table element
  constexpr int kVecPerRow = kFp8 ? 1 : 2;   // 16-byte loads per row per thread
  constexpr int kBatch = kFp8 ? 8 : 4;       // rows in flight per thread

  extern __shared__ __align__(16) int32_t smem[];
  const int H = p.H, R = 3 * H;
  int32_t *s_ids = smem;
  float *s_red = reinterpret_cast<float *>(smem + p.tpb * R);

  const int tid = threadIdx.x;
  const int tl = tid / p.tpt;
  const int lane_t = tid - tl * p.tpt;
  const int64_t tok0 = (int64_t)blockIdx.x * p.tpb;

  // Row ids of the block's tokens, coalesced, into shared memory.
  for (int i = tid; i < p.tpb * R; i += blockDim.x) {
    const int64_t gi = tok0 * R + i;
    s_ids[i] = gi < p.T * R ? p.row_ids[gi] : 0;
  }
  __syncthreads();

  const int64_t t = tok0 + tl;
  const bool tok_valid = t < p.T;
  const int col0 = lane_t * 16;
  const int32_t *ids = s_ids + tl * R;
  bool bad = false;
  int ndead = 0;
  if (tok_valid) {
    for (int r = 0; r < R; ++r) {
      const int ni = (r >= H) + (r >= 2 * H);
      const int32_t id = ids[r];
      if (id == ENGRAM_ROW_DEAD)
        ++ndead;
      else
        bad |= (id < 0) | ((int64_t)id >= p.rows[ni]);
    }
    bad |= ndead > 0 && ndead < R;  // some dead, some live
    if (bad && lane_t == 0 && p.status) atomicOr(p.status, ENGRAM_FLAG_BAD_ROW);
  }
  const bool dead = tok_valid && !bad && ndead == R;
  const bool work = tok_valid && !bad && !dead && col0 < p.D;

  // The token's four stream slices, loaded first: stream 0 feeds the gate and
  // all four are rewritten at the end.
  uint4 xs[4][2];
  const uint16_t *xrow = p.x + t * 4 * p.D + col0;
  if (work) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      xs[s][0] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * p.D));
      xs[s][1] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * p.D + 8));
    }
  }

  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;

  if (work) {
    for (int r0 = 0; r0 < R; r0 += kBatch) {
      uint4 v[kBatch][kVecPerRow];
      float sc[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int r = r0 + k;
        if (r < R) {
          const int ni = (r >= H) + (r >= 2 * H);
          const int64_t row = ids[r];
          const uint8_t *rbase = p.table[ni] + row * (int64_t)table_row_bytes(DT, p.D);
          const uint8_t *base = rbase + col0 * kElt;
          v[k][0] = ld_row16(base);
          if (!kFp8) v[k][1] = ld_row16(base + 16);
          if (kRows)
            sc[k] = e8m0_to_float(__ldg(rbase + p.D + (col0 >> 5)));
          else if (kE8)
            sc[k] = e8m0_to_float(__ldg(static_cast<const uint8_t *>(p.scale[ni]) +
                                        row * (p.D >> 5) + (col0 >> 5)));
          else if (kFp8)
            sc[k] = __ldg(static_cast<const float *>(p.scale[ni]) + row);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (r0 + k < R) {
          if (kFp8) {
            acc_fp8(acc, v[k][0], sc[k]);
          } else {
            acc_bf16(acc, v[k][0]);
            acc_bf16(acc + 8, v[k][1]);
          }
        }
      }
    }
  }

  // m = mean of the rows; partial sums of the gate over this thread's columns.
  float saa = 0.f, smm = 0.f, sam = 0.f;
  if (work) {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= p.inv_R;
    gate_partials(xs[0][0], xs[0][1], acc, saa, smm, sam);
  }

  // Sum over the token's tpt threads.
  const int seg = p.tpt < 32 ? p.tpt : 32;
  for (int o = seg >> 1; o > 0; o >>= 1) {
    saa += __shfl_xor_sync(0xffffffffu, saa, o);
    smm += __shfl_xor_sync(0xffffffffu, smm, o);
    sam += __shfl_xor_sync(0xffffffffu, sam, o);
  }
  if (p.tpt > 32) {
    const int warp = tid >> 5;
    if ((tid & 31) == 0) {
      s_red[3 * warp + 0] = saa;
      s_red[3 * warp + 1] = smm;
      s_red[3 * warp + 2] = sam;
    }
    __syncthreads();
    const int nw = p.tpt >> 5, w0 = tl * nw;
    saa = smm = sam = 0.f;
    for (int k = 0; k < nw; ++k) {
      saa += s_red[3 * (w0 + k) + 0];
      smm += s_red[3 * (w0 + k) + 1];
      sam += s_red[3 * (w0 + k) + 2];
    }
  }

  if (!work) {
    if (dead && col0 < p.D)
      pass_through16(p.x + t * 4 * p.D + col0, p.y + t * 4 * p.D + col0, p.D,
                     AUX && p.gate_out ? p.gate_out + t : nullptr,
                     AUX && p.mem_out ? p.mem_out + t * p.D + col0 : nullptr, lane_t == 0);
    return;
  }

  const float g = gate_value(saa, smm, sam, (float)p.D, p.eps, p.sqrt_D);

  uint16_t *yrow = p.y + t * 4 * p.D + col0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float c = g * __ldg(p.alpha + s);
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * p.D), gated_add8(xs[s][0], acc, c));
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * p.D + 8), gated_add8(xs[s][1], acc + 8, c));
  }
  if (AUX) {
    if (p.gate_out && lane_t == 0) p.gate_out[t] = g;
    if (p.mem_out) {
      float4 *mo = reinterpret_cast<float4 *>(p.mem_out + t * p.D + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        mo[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    }
  }
}

template <int DT, bool AUX>
cudaError_t launch_t(const LookupParams &p, int threads, size_t smem, cudaStream_t stream) {
  const int64_t blocks = (p.T + p.tpb - 1) / p.tpb;
  lookup_kernel<DT, AUX><<<(unsigned)blocks, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lookup(const LookupParams &p_in, int dtype, cudaStream_t stream) {
  if (p_in.T == 0) return cudaSuccess;
  LookupParams p = p_in;
  const int chunks = p.D / 16;
  int tpt = 1;
  if (chunks <= 32) {
    while (tpt < chunks) tpt <<= 1;
  } else {
    tpt = (chunks + 31) / 32 * 32;
  }
  const int R = 3 * p.H;
  // Tokens per block: fill 256 threads, keep the staged row ids within 16 KB, and
  // keep the block a whole number of warps (the reduction shuffles full warps).
  int tpb = 256 / tpt;
  const int tpb_smem = 4096 / R;
  if (tpb > tpb_smem) tpb = tpb_smem;
  const int warp_tokens = tpt < 32 ? 32 / tpt : 1;
  tpb = tpb / warp_tokens * warp_tokens;
  if (tpb < warp_tokens) tpb = warp_tokens;
  p.tpt = tpt;
  p.tpb = tpb;
  const int threads = p.tpb * tpt;
  const size_t smem = (size_t)p.tpb * R * sizeof(int32_t) + 8 * 3 * sizeof(float);
  const bool aux = p.gate_out != nullptr || p.mem_out != nullptr;
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN)
    return aux ? launch_t<ENGRAM_TABLE_FP8_E4M3FN, true>(p, threads, smem, stream)
               : launch_t<ENGRAM_TABLE_FP8_E4M3FN, false>(p, threads, smem, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32)
    return aux ? launch_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32, true>(p, threads, smem, stream)
               : launch_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32, false>(p, threads, smem, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS)
    return aux ? launch_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS, true>(p, threads, smem, stream)
               : launch_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS, false>(p, threads, smem, stream);
  return aux ? launch_t<ENGRAM_TABLE_BF16, true>(p, threads, smem, stream)
             : launch_t<ENGRAM_TABLE_BF16, false>(p, threads, smem, stream);
}

}  // namespace engram
