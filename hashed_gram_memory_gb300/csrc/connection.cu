// connection.cu -- the Engram connection with a wkv projection: the token's 3H
// rows concatenated (exact bf16), projected by wkv on the tensor cores
// (wkv_gemm.cu), then the gate and the add into the four streams.
//
//   concat_rows_kernel : one token per block; dequantises its 3H rows (FP8 with
//                        e8m0 blocks, the exponents apart or after each row, or
//                        BF16) into E[t] = [row_0 | ... | row_3H-1]
//                        as bf16, 16-byte stores; records the token's state
//                        (live, dead, bad) for the last kernel.
//   wkv_gemm_kernel    : k = E wkv^T, fp32.
//   gate_add_kernel    : one token per block of D/16 threads; the RMSNorm
//                        dot-product sigmoid gate of k against stream 0 and
//                        out_s = bf16(stream_s + g alpha_s k); dead tokens copied
//                        through, bad tokens left unwritten.
#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace engram {
namespace {

constexpr uint8_t kLive = 0, kDead = 1, kBad = 2;

struct ConcatParams {
  const int32_t *row_ids;
  const uint8_t *table[3];
  const void *scale[3];
  int64_t rows[3];
  uint16_t *e;       // [T, K]
  uint8_t *state;    // [T]
  int32_t *status;
  int64_t T;
  int32_t H, d;
};

template <int DT>
__global__ void __launch_bounds__(256) concat_rows_kernel(const __grid_constant__ ConcatParams p) {
  constexpr bool kBf16 = DT == ENGRAM_TABLE_BF16;
  constexpr bool kRows = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS;  // the exponents after each row
  const int64_t t = blockIdx.x;
  const int H = p.H, R = 3 * H, d = p.d;
  const int64_t K = (int64_t)R * d;
  const int32_t *ids = p.row_ids + t * R;
  bool bad = false, dead = false, live = false;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int ni = (r >= H) + (r >= 2 * H);
    const int32_t id = ids[r];
    if (id == ENGRAM_ROW_DEAD) {
      dead = true;
    } else {
      live = true;
      bad |= (id < 0) | ((int64_t)id >= p.rows[ni]);
    }
  }
  const bool any_flag = __syncthreads_or(bad || dead);
  if (any_flag) {
    const bool all_dead = __syncthreads_and(!live);
    uint4 *erow = reinterpret_cast<uint4 *>(p.e + t * K);  // zero row: k = 0 for this token
    for (int64_t c = threadIdx.x; c < K / 8; c += blockDim.x) erow[c] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
      p.state[t] = all_dead ? kDead : kBad;
      if (!all_dead && p.status) atomicOr(p.status, ENGRAM_FLAG_BAD_ROW);
    }
    return;
  }
  // 16 output values (two 16-byte words of bf16) per step: one 16-byte load of
  // FP8 (two of BF16).
  const int chunks_per_row = d / 16;
  uint4 *erow = reinterpret_cast<uint4 *>(p.e + t * K);
  for (int c = threadIdx.x; c < R * chunks_per_row; c += blockDim.x) {
    const int r = c / chunks_per_row, col = (c - r * chunks_per_row) * 16;
    const int ni = (r >= H) + (r >= 2 * H);
    const int64_t row = ids[r];
    uint4 lo, hi;
    if (kBf16) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          reinterpret_cast<const uint16_t *>(p.table[ni]) + row * d + col);
      lo = __ldg(src);
      hi = __ldg(src + 1);
    } else {
      const uint8_t *rbase = p.table[ni] + row * (int64_t)table_row_bytes(DT, d);
      const uint4 b = __ldg(reinterpret_cast<const uint4 *>(rbase + col));
      const float s = e8m0_to_float(
          kRows ? __ldg(rbase + d + (col >> 5))
                : __ldg(static_cast<const uint8_t *>(p.scale[ni]) + row * (d >> 5) + (col >> 5)));
      float f[16];
      const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2_raw l2 =
            __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] & 0xFFFFu), __NV_E4M3);
        const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] >> 16), __NV_E4M3);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&l2));
        const float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
        // a power of two times a 4-bit value: exact, and exact in bf16 (signed zeros kept)
        f[4 * q + 0] = a.x * s;
        f[4 * q + 1] = a.y * s;
        f[4 * q + 2] = c.x * s;
        f[4 * q + 3] = c.y * s;
      }
      lo = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                      pack_bf16(f[6], f[7]));
      hi = make_uint4(pack_bf16(f[8], f[9]), pack_bf16(f[10], f[11]), pack_bf16(f[12], f[13]),
                      pack_bf16(f[14], f[15]));
    }
    uint4 *dst = erow + ((int64_t)r * d + col) / 8;
    dst[0] = lo;
    dst[1] = hi;
  }
  if (threadIdx.x == 0) p.state[t] = kLive;
}

struct GateAddParams {
  const float *k;        // [T, D]
  const uint8_t *state;  // [T]
  const uint16_t *x;
  uint16_t *y;
  const float *alpha;
  float *gate_out;
  int64_t T;
  int32_t D;
  float eps, sqrt_D;
};

__global__ void __launch_bounds__(512) gate_add_kernel(const __grid_constant__ GateAddParams p) {
  __shared__ float s_red[16 * 3];
  const int64_t t = blockIdx.x;
  const int D = p.D, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int col0 = tid * 16;
  const bool mine = col0 < D;
  const uint8_t state = p.state[t];  // block-uniform
  if (state == kBad) return;
  const uint16_t *xrow = p.x + t * 4 * D + col0;
  uint16_t *yrow = p.y + t * 4 * D + col0;
  if (state == kDead) {
    if (mine) pass_through16(xrow, yrow, D, p.gate_out ? p.gate_out + t : nullptr, nullptr, tid == 0);
    return;
  }
  float k[16];
  uint4 xs[4][2];
  float saa = 0.f, skk = 0.f, sak = 0.f;
  if (mine) {
    const float4 *kr = reinterpret_cast<const float4 *>(p.k + t * D + col0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = kr[q];
      k[4 * q] = v.x;
      k[4 * q + 1] = v.y;
      k[4 * q + 2] = v.z;
      k[4 * q + 3] = v.w;
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      xs[s][0] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D));
      xs[s][1] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D + 8));
    }
    gate_partials(xs[0][0], xs[0][1], k, saa, skk, sak);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    saa += __shfl_xor_sync(0xffffffffu, saa, o);
    skk += __shfl_xor_sync(0xffffffffu, skk, o);
    sak += __shfl_xor_sync(0xffffffffu, sak, o);
  }
  if (lane == 0) {
    s_red[3 * warp] = saa;
    s_red[3 * warp + 1] = skk;
    s_red[3 * warp + 2] = sak;
  }
  __syncthreads();
  saa = skk = sak = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    saa += s_red[3 * w];
    skk += s_red[3 * w + 1];
    sak += s_red[3 * w + 2];
  }
  if (!mine) return;
  const float g = gate_value(saa, skk, sak, (float)D, p.eps, p.sqrt_D);
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float c = g * __ldg(p.alpha + s);
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D), gated_add8(xs[s][0], k, c));
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D + 8), gated_add8(xs[s][1], k + 8, c));
  }
  if (p.gate_out && tid == 0) p.gate_out[t] = g;
}

}  // namespace

cudaError_t launch_concat_rows(const int32_t *row_ids, int64_t T, int H, const engram_tables &tb,
                               uint16_t *e, uint8_t *state, int32_t *status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  ConcatParams cp;
  cp.row_ids = row_ids;
  for (int n = 0; n < 3; ++n) {
    cp.table[n] = static_cast<const uint8_t *>(tb.table[n]);
    cp.scale[n] = tb.scale[n];
    cp.rows[n] = tb.rows[n];
  }
  cp.e = e;
  cp.state = state;
  cp.status = status;
  cp.T = T;
  cp.H = H;
  cp.d = tb.D;
  if (tb.dtype == ENGRAM_TABLE_BF16)
    concat_rows_kernel<ENGRAM_TABLE_BF16><<<(unsigned)T, 256, 0, stream>>>(cp);
  else if (tb.dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS)
    concat_rows_kernel<ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS><<<(unsigned)T, 256, 0, stream>>>(cp);
  else
    concat_rows_kernel<ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32><<<(unsigned)T, 256, 0, stream>>>(cp);
  return cudaGetLastError();
}

cudaError_t launch_gate_add(const float *k, const uint8_t *state, int64_t T, int D,
                            const uint16_t *x, uint16_t *y, const float *alpha, float eps,
                            float *gate_out, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  GateAddParams gp;
  gp.k = k;
  gp.state = state;
  gp.x = x;
  gp.y = y;
  gp.alpha = alpha;
  gp.gate_out = gate_out;
  gp.T = T;
  gp.D = D;
  gp.eps = eps;
  gp.sqrt_D = sqrtf((float)D);
  const int threads = (D / 16 + 31) / 32 * 32;
  gate_add_kernel<<<(unsigned)T, threads, 0, stream>>>(gp);
  return cudaGetLastError();
}

cudaError_t launch_connection(const int32_t *row_ids, int64_t T, int H, const engram_tables &tb,
                              const uint16_t *wkv, int D, const uint16_t *x, uint16_t *y,
                              const float *alpha, float eps, uint16_t *e, float *k,
                              uint8_t *state, float *gate_out, int64_t wait_limit_ns,
                              int32_t *status, cudaStream_t stream) {
  cudaError_t err = launch_concat_rows(row_ids, T, H, tb, e, state, status, stream);
  if (err != cudaSuccess) return err;
  err = launch_wkv_gemm(e, wkv, k, (int)T, D, 3 * H * tb.D, wait_limit_ns, status, stream);
  if (err != cudaSuccess) return err;
  return launch_gate_add(k, state, T, D, x, y, alpha, eps, gate_out, stream);
}

}  // namespace engram
