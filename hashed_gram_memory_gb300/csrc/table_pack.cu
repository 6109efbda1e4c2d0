// table_pack.cu -- builds the table layout in which every FP8 row carries its
// e8m0 block exponents (ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS) from the layout with
// the exponents apart (ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32): packed row r = the
// row's D bytes, its D/32 exponents, zeros up to a multiple of 16 bytes.  One
// thread writes one 16-byte word of the packed table (grid-stride): a word of
// the row's bytes is one 16-byte load, a word past them is put together from
// the exponents and zeros.
#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace engram {
namespace {

__global__ void __launch_bounds__(256) pack_e8m0_rows_kernel(const uint8_t *__restrict__ table,
                                                             const uint8_t *__restrict__ exps,
                                                             int64_t rows, int D,
                                                             uint8_t *__restrict__ packed) {
  const int64_t stride = ENGRAM_E8M0_ROW_BYTES(D);
  const int64_t words_per_row = stride / 16, n_exps = D / 32;
  const int64_t total = rows * words_per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / words_per_row, w = i - r * words_per_row;
    uint4 v;
    if (w * 16 < D) {
      v = __ldg(reinterpret_cast<const uint4 *>(table + r * D) + w);
    } else {
      uint32_t b[4] = {0, 0, 0, 0};
      for (int k = 0; k < 16; ++k) {
        const int64_t j = w * 16 + k - D;  // index among the row's exponents
        if (j < n_exps) b[k >> 2] |= (uint32_t)__ldg(exps + r * n_exps + j) << (8 * (k & 3));
      }
      v = make_uint4(b[0], b[1], b[2], b[3]);
    }
    reinterpret_cast<uint4 *>(packed + r * stride)[w] = v;
  }
}

}  // namespace

cudaError_t launch_pack_e8m0_rows(const uint8_t *table, const uint8_t *exps, int64_t rows, int D,
                                  uint8_t *packed, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t total = rows * (ENGRAM_E8M0_ROW_BYTES(D) / 16);
  const int64_t want = (total + 255) / 256;
  const int blocks = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  pack_e8m0_rows_kernel<<<blocks, 256, 0, stream>>>(table, exps, rows, D, packed);
  return cudaGetLastError();
}

}  // namespace engram
