// engram_internal.cuh -- launch parameters and launchers shared by the kernel
// translation units and the C ABI layer of libengram.  Not installed; the public
// interface is include/engram.h.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "engram.h"

namespace engram {

// A named NVTX range over a C-ABI call, so that a profiler's timeline shows
// each call and the kernels it launched; without a profiler attached the push
// and pop return at once.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};
#define ENGRAM_NVTX_RANGE(name) const ::engram::NvtxRange engram_nvtx_range_(name)

constexpr int kMaxHeads = ENGRAM_MAX_HEADS;
constexpr int kMaxRows = 3 * kMaxHeads;

struct CompressParams {
  const int32_t *token_ids;
  int64_t n;
  const uint8_t *dead;  // optional: dead positions become ENGRAM_EID_DEAD
  const int32_t *tid2eid;
  int32_t vocab;
  int32_t n_eids;
  int32_t *eids_out;
  int32_t *status;
};

struct HashParams {
  const int32_t *eids;
  const int32_t *positions;  // optional: index of each token within its sample
  const int32_t *history;
  int32_t *history_out;
  int32_t *row_ids;
  int32_t *status;
  int64_t T;
  int32_t batch, seq, H;
  int32_t tokens_per_block;  // tokens whose 3H outputs one block owns
  int32_t history_inline;    // 1: seq == 1 and the block writes history_out itself
  // Compression fused in (token_ids non-NULL): the ids of each window are
  // compressed where they are read (eids is then not read), and eids_out
  // (optional) receives each token's compressed id.
  const int32_t *token_ids;
  const int32_t *tid2eid;
  const uint8_t *dead;
  int32_t *eids_out;
  int32_t vocab, n_eids;
  // Row r = (n-2)*H + j of a token is off[n-2][j] + (h mod mod[n-2][j]):
  // one table per order (off 0, mod rows_n) or one table cut into prime buckets.
  uint64_t mod[3][kMaxHeads];
  uint64_t off[3][kMaxHeads];
  uint64_t rmul[3][kMaxHeads];  // floor((2^64 - 1) / mod): the reciprocal for h mod mod
  uint64_t seed[3][kMaxHeads];
};

struct LookupParams {
  const int32_t *row_ids;
  const uint8_t *table[3];
  const void *scale[3];  // float [rows] (FP8), uint8 [rows, D/32] (FP8 + E8M0 blocks)
  int64_t rows[3];
  const uint16_t *x;  // streams in  [T, 4, D]
  uint16_t *y;        // streams out [T, 4, D]
  const float *alpha;
  float *gate_out;
  float *mem_out;
  int32_t *status;
  int64_t T;
  int32_t H, D;
  int32_t tpt;  // gather kernel: threads per token (16 columns each)
  int32_t tpb;  // tokens per block (gather, small-row and chained bulk kernels)
  int32_t withhold; // test hook: withhold one row copy per block (bulk kernels, decode step)
  int64_t wait_limit_ns;
  float eps, inv_R, inv_D, sqrt_D;
};

// The fused decode step: compress + window + hash + bulk lookup, one slot a block.
struct DecodeParams {
  LookupParams lk;           // row_ids unused
  const int32_t *token_ids;  // [batch] (one new token a slot)
  const int32_t *tid2eid;
  const int32_t *history;    // [batch, 3] oldest first, or NULL (pad)
  int32_t *history_out;      // [batch, 3] or NULL; may be history
  int32_t *row_ids_out;      // [batch, 3H] or NULL
  const int32_t *positions;  // [batch] or NULL: the token's index within its sample
  const uint8_t *dead;       // [batch] or NULL: dead slots (every id ENGRAM_ROW_DEAD)
  int32_t vocab, n_eids;
  uint64_t mod[3][kMaxHeads];
  uint64_t off[3][kMaxHeads];
  uint64_t rmul[3][kMaxHeads];
  uint64_t seed[3][kMaxHeads];
};

cudaError_t launch_compress(const CompressParams &p, cudaStream_t stream);
cudaError_t launch_hash(const HashParams &p, cudaStream_t stream);
cudaError_t launch_lookup(const LookupParams &p, int dtype, cudaStream_t stream);
cudaError_t launch_lookup_bulk(const LookupParams &p, int dtype, cudaStream_t stream);
bool bulk_supported(int D, int dtype, int H);
size_t bulk_smem_bytes(int D, int dtype, int H);  // one token's rows, scales and barrier
bool decode_supported(int D, int dtype, int H);  // the fused decode step's shape limits
cudaError_t launch_decode_step(const DecodeParams &p, int dtype, cudaStream_t stream);
cudaError_t launch_lookup_bulk_small(const LookupParams &p, int dtype, cudaStream_t stream);
bool bulk_small_supported(int D, int dtype, int H);

cudaError_t launch_pack_e8m0_rows(const uint8_t *table, const uint8_t *exps, int64_t rows, int D,
                                  uint8_t *packed, cudaStream_t stream);

bool wkv_gemm_supported(int N, int K);
int set_projection_kernel(int which);  // returns the previous choice
cudaError_t launch_wkv_gemm(const uint16_t *e, const uint16_t *wkv, float *k_out, int T, int N, int K,
                            int64_t wait_limit_ns, int32_t *status, cudaStream_t stream);
cudaError_t launch_concat_rows(const int32_t *row_ids, int64_t T, int H, const engram_tables &tb,
                               uint16_t *e, uint8_t *state, int32_t *status, cudaStream_t stream);
cudaError_t launch_gate_add(const float *k, const uint8_t *state, int64_t T, int D,
                            const uint16_t *x, uint16_t *y, const float *alpha, float eps,
                            float *gate_out, cudaStream_t stream);
cudaError_t launch_connection(const int32_t *row_ids, int64_t T, int H, const engram_tables &tb,
                              const uint16_t *wkv, int D, const uint16_t *x, uint16_t *y,
                              const float *alpha, float eps, uint16_t *e, float *k,
                              uint8_t *state, float *gate_out, int64_t wait_limit_ns,
                              int32_t *status, cudaStream_t stream);

engram_status prepare_lookup(const char *fn, const int32_t *row_ids, bool need_row_ids,
                             int64_t n_tokens, int32_t n_heads, const engram_tables *tables_host,
                             const uint16_t *streams_in, uint16_t *streams_out, const float *alpha,
                             float eps, float *gate_out, float *mem_out, int32_t *status,
                             LookupParams &p);
int lookup_kernel_choice();
// The test hook of engram_debug_withhold_copies: true (and one launch fewer left)
// while launches are to withhold a row copy.
bool take_withheld_launch();
// engram_forward runs this call as the fused decode launch (no workspace used).
bool forward_is_decode_step(int32_t batch, int32_t seq, int32_t n_heads,
                            const engram_tables *tables_host);

// Records the message engram_last_error() returns on this thread; returns code.
engram_status set_error(engram_status code, const char *fmt, ...);

// splitmix64 first output for state x (S. Vigna, public domain), used for the
// per-(order, head) hash seeds on the host.
uint64_t splitmix64(uint64_t x);

}  // namespace engram
