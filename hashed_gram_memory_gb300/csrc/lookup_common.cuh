// lookup_common.cuh -- device helpers shared by the two lookup kernels: the
// dequantisation of 16 columns of a row, the bf16 unpack / pack, and the gate.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "engram.h"

namespace engram {

// Bytes from one table row to the next: D (FP8), 2D (BF16), and D + D/32
// padded to 16 for FP8 rows carrying their e8m0 exponents after their bytes.
__host__ __device__ __forceinline__ uint32_t table_row_bytes(int dtype, int D) {
  if (dtype == ENGRAM_TABLE_BF16) return 2u * (uint32_t)D;
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS) return (uint32_t)ENGRAM_E8M0_ROW_BYTES(D);
  return (uint32_t)D;
}

// OCP E8M0 exponent -> fp32: 2^(e-127) (e = 0 is the subnormal 2^-127), 0xFF NaN.
// The hardware's ue8m0 -> bf16 conversion (exact: bf16 has fp32's exponent
// range), given e in both bytes so that either half of the result holds it,
// then the bf16 bits as the high half of an fp32: three instructions where a
// select chain on the special values took five (the e8m0 prefill 1.764 ->
// 1.701 ms, with the exponents after each row 1.737 -> 1.615 ms).
__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
  uint32_t r;
  asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(r) : "h"((unsigned short)(e * 0x101u)));
  return __uint_as_float(r & 0xFFFF0000u);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// (c0, c1) = fma((a0, a1), (s, s), (c0, c1)) by one packed instruction; each lane
// rounds exactly as fmaf.
__device__ __forceinline__ void fma2(float &c0, float &c1, float a0, float a1, float s) {
  unsigned long long av, sv, cv;
  asm("mov.b64 %0, {%1, %2};" : "=l"(av) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(sv) : "f"(s));
  asm("mov.b64 %0, {%1, %2};" : "=l"(cv) : "f"(c0), "f"(c1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(cv) : "l"(av), "l"(sv));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(c0), "=f"(c1) : "l"(cv));
}

// acc[0..16) += scale * e4m3(v[0..16)); e4m3 -> f16 -> f32 is exact.
__device__ __forceinline__ void acc_fp8(float (&acc)[16], const uint4 &v, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2_raw lo =
        __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    fma2(acc[4 * q + 0], acc[4 * q + 1], a.x, a.y, scale);
    fma2(acc[4 * q + 2], acc[4 * q + 3], b.x, b.y, scale);
  }
}

// acc[0..8) += bf16(v[0..8)).
__device__ __forceinline__ void acc_bf16(float *acc, const uint4 &v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q + 0] += bf16_lo(w[q]);
    acc[2 * q + 1] += bf16_hi(w[q]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Partial sums of the gate over 16 columns: sum a^2, sum m^2, sum a*m, with a =
// stream 0 (two 16-byte words of bf16) and m the memory.
__device__ __forceinline__ void gate_partials(const uint4 &a_lo, const uint4 &a_hi,
                                              const float (&m)[16], float &saa, float &smm,
                                              float &sam) {
  const uint32_t a32[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float a0 = bf16_lo(a32[q]), a1 = bf16_hi(a32[q]);
    const float m0 = m[2 * q], m1 = m[2 * q + 1];
    saa = fmaf(a0, a0, fmaf(a1, a1, saa));
    smm = fmaf(m0, m0, fmaf(m1, m1, smm));
    sam = fmaf(a0, m0, fmaf(a1, m1, sam));
  }
}

// g = sigmoid( sum(a m) / (rms(a) rms(m) sqrt(D)) ),  rms(x) = sqrt(mean(x^2) + eps).
__device__ __forceinline__ float gate_value(float saa, float smm, float sam, float Df, float eps,
                                            float sqrt_D) {
  const float rms_a = sqrtf(saa / Df + eps);
  const float rms_m = sqrtf(smm / Df + eps);
  const float logit = sam / (rms_a * rms_m * sqrt_D);
  return 1.f / (1.f + expf(-logit));
}

// out = bf16_rne(x + c * m) for 8 columns held as one 16-byte word of bf16.
__device__ __forceinline__ uint4 gated_add8(const uint4 &in, const float *m, float c) {
  uint4 out;
  out.x = pack_bf16(fmaf(c, m[0], bf16_lo(in.x)), fmaf(c, m[1], bf16_hi(in.x)));
  out.y = pack_bf16(fmaf(c, m[2], bf16_lo(in.y)), fmaf(c, m[3], bf16_hi(in.y)));
  out.z = pack_bf16(fmaf(c, m[4], bf16_lo(in.z)), fmaf(c, m[5], bf16_hi(in.z)));
  out.w = pack_bf16(fmaf(c, m[6], bf16_lo(in.w)), fmaf(c, m[7], bf16_hi(in.w)));
  return out;
}

// A dead token's four stream slices (16 columns each) copied through unchanged
// (nothing to do in place); its gate and memory outputs are zero.
__device__ __forceinline__ void pass_through16(const uint16_t *xrow, uint16_t *yrow, int D,
                                               float *gate_out, float *mem_row, bool lead) {
  if (yrow != xrow) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D));
      const uint4 b = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D + 8));
      __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D), a);
      __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D + 8), b);
    }
  }
  if (gate_out && lead) *gate_out = 0.f;
  if (mem_row) {
    float4 *mo = reinterpret_cast<float4 *>(mem_row);
#pragma unroll
    for (int i = 0; i < 4; ++i) mo[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

}  // namespace engram
