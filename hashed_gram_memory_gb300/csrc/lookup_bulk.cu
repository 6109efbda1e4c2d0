// lookup_bulk.cu -- the fused Engram lookup with the table rows staged in shared
// memory by 1-D bulk copies (TMA), for sm_103a.
//
// A token is handled by a CTA of D/16 threads (16 columns each).  Warp 0 issues all 3H
// row copies of the token at once, lane r the copy of row r (one contiguous
// D*elt-byte run per row, one cp.async.bulk each, from an id the lane holds in a
// register), completing on a single mbarrier that expects their total byte
// count, while the other threads fetch the row scales (or the rows'
// 32-column block exponents, 16 coalesced bytes per thread) into shared memory
// and, for large tokens, the four 32-byte stream slices into registers with
// evict-first loads.  After the wait every thread reads its columns of the rows
// from shared memory, accumulates the dequantised rows in fp32, the gate sums
// are reduced across warps, and the four streams are written back with
// evict-first stores.  A whole token is in flight from one warp's issue and the
// rows cost no registers.  Two variants, chosen by the size of a token's
// rows: for large tokens (8 heads of FP8 at D = 4096: 96 KB of rows) two blocks
// per SM with the streams loaded early, each block running a few tokens in
// turn with the next token's copies issued under the current token's gate and
// stores (lookup_bulk_chain_kernel); for rows within 56 KB, one token a block,
// four blocks per SM within 64 registers with the streams loaded after the
// rows (lookup_bulk_kernel).
//
// The wait is bounded by the global timer: a copy that never lands makes the
// block set ENGRAM_FLAG_TIMEOUT, skip the token (and a chained block its later
// tokens), and exit only after thread 0 has waited (again bounded) for the
// copies warp 0 issued.  An id outside its table
// makes the block set ENGRAM_FLAG_BAD_ROW and skip the token before anything
// is copied; a dead token (all ids ENGRAM_ROW_DEAD) copies its streams through.
#include <atomic>

#include "bulk_copy.cuh"
#include "bulk_token.cuh"
#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace engram {
namespace {

template <int DT, bool AUX, bool EARLY>
__global__ void __launch_bounds__(256, EARLY ? 2 : 4)
    lookup_bulk_kernel(const __grid_constant__ LookupParams p) {
  const int64_t t = blockIdx.x;
  bulk_token<DT, AUX, EARLY>(p, p.row_ids + t * 3 * p.H, t);
}

// Large tokens (two blocks per SM, streams loaded early): p.tpb consecutive
// tokens a block, one after the other.  As soon as every thread has read a
// token's rows from shared memory, warp 0 issues the next token's row copies,
// which then fly under the current token's gate and stores; the next token's
// scales are loaded after those stores, under its copies.  A block thus keeps
// its rows in flight between tokens instead of ending and being replaced, and
// a few tokens a block leave the hardware scheduler room to even out the SMs.
// Each token's arithmetic is bulk_token's, so the results are the same bits.
template <int DT, bool AUX>
__global__ void __launch_bounds__(256, 2)
    lookup_bulk_chain_kernel(const __grid_constant__ LookupParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int R = 3 * p.H, tid = threadIdx.x;
  const BulkSmem s = bulk_smem<DT>(sm, R, p.D);
  if (tid == 0) {
    mbar_init(s.bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const int64_t t0 = (int64_t)blockIdx.x * p.tpb;
  const int64_t end = t0 + p.tpb < p.T ? t0 + p.tpb : p.T;
  uint32_t phase = 0;  // parity of the barrier phase the current token's copies complete
  int64_t t = t0;
  int state = bulk_state(p, p.row_ids + t * R);  // its barrier publishes the mbarrier's set-up
  if (state == kBulkLive) {
    bulk_issue_rows<true>(p, p.row_ids + t * R, t, s);
    bulk_load_scales<DT>(p, p.row_ids + t * R, s);
  }
  for (;;) {
    const int64_t tn = t + 1;
    const int32_t *ids_n = p.row_ids + tn * R;
    int next = kBulkBad;  // no next token
    if (state == kBulkLive) {
      uint4 xs[4][2];
      bulk_load_streams(p.x + t * 4 * p.D + tid * 16, p.D, xs);
      const bool landed = wait_bounded(s.bar, p.wait_limit_ns, phase);
      // Block-uniform outcome; the barrier also publishes the scales.
      if (__syncthreads_or(!landed)) {
        if (tid == 0) {
          if (p.status) atomicOr(p.status, ENGRAM_FLAG_TIMEOUT);
          wait_bounded(s.bar, p.wait_limit_ns, phase);  // let the issued copies land before exit
        }
        return;  // this token and the block's later ones stay unwritten
      }
      phase ^= 1;
      float acc[16];
      bulk_accumulate<DT>(p, s, tid * 16, acc);
      if (tn < end) {
        next = bulk_state(p, ids_n);  // its barrier: every thread is done with the rows
        if (next == kBulkLive) bulk_issue_rows<true>(p, ids_n, tn, s);
      }
      bulk_gate_store<AUX, true>(p, t, s, xs, acc);
      if (next == kBulkLive) bulk_load_scales<DT>(p, ids_n, s);
    } else {
      if (state == kBulkDead) bulk_pass_through<AUX>(p, t);
      if (tn < end) {
        next = bulk_state(p, ids_n);
        if (next == kBulkLive) {
          bulk_issue_rows<true>(p, ids_n, tn, s);
          bulk_load_scales<DT>(p, ids_n, s);
        }
      }
    }
    if (tn >= end) return;
    t = tn;
    state = next;
  }
}

// A row's e8m0 exponents, n = D/32 bytes with n in {1, 2, 4, 8} (the small-row
// kernel's widths), as one naturally aligned load and store.
__device__ __forceinline__ uint64_t load_exps(const uint8_t *e, uint32_t n) {
  if (n == 8) return __ldg(reinterpret_cast<const unsigned long long *>(e));
  if (n == 4) return __ldg(reinterpret_cast<const unsigned int *>(e));
  if (n == 2) return __ldg(reinterpret_cast<const unsigned short *>(e));
  return __ldg(e);
}

__device__ __forceinline__ void store_exps(uint8_t *se, uint64_t v, uint32_t n) {
  if (n == 8)
    *reinterpret_cast<uint64_t *>(se) = v;
  else if (n == 4)
    *reinterpret_cast<uint32_t *>(se) = (uint32_t)v;
  else if (n == 2)
    *reinterpret_cast<uint16_t *>(se) = (uint16_t)v;
  else
    *se = (uint8_t)v;
}

// Small rows (D < 512 with D/16 a power of two, e.g. the released 256-wide
// rows): several tokens per block, each handled by its tpt = D/16 threads, which
// issue the copies of the token's rows themselves (thread l of the token copies
// rows l, l + tpt, ...) into the token's slot of shared memory.  Every thread
// arrives once on the block's single mbarrier with the bytes it issued, so the
// wait covers exactly the copies made.  The gate sums are reduced over the
// token's threads with the same shuffles as the register-gather kernel, and
// rows are summed in the same order: the two give identical bits.
template <int DT, bool AUX>
__global__ void __launch_bounds__(256, 2)
    lookup_bulk_small_kernel(const __grid_constant__ LookupParams p) {
  constexpr bool kFp8 = DT != ENGRAM_TABLE_BF16;
  constexpr bool kE8 = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32;
  constexpr bool kRows = DT == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS;  // the exponents after each row
  constexpr int kElt = kFp8 ? 1 : 2;
  extern __shared__ __align__(128) uint8_t sm[];

  const int H = p.H, R = 3 * H, D = p.D, tpt = p.tpt, tpb = p.tpb;
  const uint32_t row_bytes = table_row_bytes(DT, D);
  const uint32_t exp_bytes = kE8 ? (uint32_t)D / 32 : 0;
  const size_t tok_bytes = (size_t)R * row_bytes;
  uint8_t *s_rows = sm;                                            // [tpb][R][row_bytes]
  uint8_t *s_exps = s_rows + (size_t)tpb * tok_bytes;              // [tpb][R][exp_bytes]
  float *s_scale = reinterpret_cast<float *>(
      s_exps + (((size_t)tpb * R * exp_bytes + 15) & ~(size_t)15));  // [tpb][R]
  uint64_t *bar = reinterpret_cast<uint64_t *>(s_scale + (((size_t)tpb * R + 1) & ~(size_t)1));

  const int tid = threadIdx.x;
  const int tl = tid / tpt, lane_t = tid - tl * tpt;
  const int64_t t = (int64_t)blockIdx.x * tpb + tl;
  const bool tok_valid = t < p.T;
  const int col0 = lane_t * 16;
  const int32_t *ids = p.row_ids + t * R;

  if (tid == 0) {
    mbar_init(bar, blockDim.x);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();  // the barrier is set up before any thread arrives on it

  // The token's state from its ids, OR-ed over its threads.
  int bad = 0, dead = 0, live = 0;
  if (tok_valid) {
    for (int r = lane_t; r < R; r += tpt) {
      const int ni = (r >= H) + (r >= 2 * H);
      const int32_t id = ids[r];
      if (id == ENGRAM_ROW_DEAD) {
        dead = 1;
      } else {
        live = 1;
        bad |= (id < 0) | ((int64_t)id >= p.rows[ni]);
      }
    }
  }
  for (int o = tpt >> 1; o > 0; o >>= 1) {
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    dead |= __shfl_xor_sync(0xffffffffu, dead, o);
    live |= __shfl_xor_sync(0xffffffffu, live, o);
  }
  const bool bad_tok = tok_valid && (bad || (dead && live));
  const bool dead_tok = tok_valid && !bad_tok && dead;
  const bool work = tok_valid && !bad_tok && !dead_tok;
  if (bad_tok && lane_t == 0 && p.status) atomicOr(p.status, ENGRAM_FLAG_BAD_ROW);

  // This thread's rows of its token: copies, and their scales or exponents.
  uint32_t my_bytes = 0;
  if (work)
    for (int r = lane_t; r < R; r += tpt) my_bytes += row_bytes;
  if (my_bytes)
    mbar_arrive_expect_tx(bar, my_bytes);
  else
    mbar_arrive(bar);
  // This thread's rows (r = lane_t + k*tpt): the copy, then the load of the
  // row's scale or exponents (1, 2, 4 or 8 bytes: one load), issued together.
  // The first four rows' words are stored to shared memory only after the
  // stream loads are issued (a store waits for its load); further rows' at once.
  uint64_t v[4] = {0, 0, 0, 0};
  bool withhold = work && p.withhold != 0 && tid == 0;  // test hook: one copy never issued
  uint8_t *dst = s_rows + (size_t)tl * tok_bytes;
  auto issue_row = [&](int r) -> uint64_t {
    const int ni = (r >= H) + (r >= 2 * H);
    const int64_t id = ids[r];
    if (withhold)
      withhold = false;
    else
      bulk_g2s(dst + (size_t)r * row_bytes, p.table[ni] + id * row_bytes, row_bytes, bar);
    if (kE8) return load_exps(static_cast<const uint8_t *>(p.scale[ni]) + id * exp_bytes, exp_bytes);
    if (kFp8 && !kRows) return __float_as_uint(__ldg(static_cast<const float *>(p.scale[ni]) + id));
    return 0;
  };
  auto store_row = [&](int r, uint64_t w) {
    if (kRows) return;
    if (kE8)
      store_exps(s_exps + ((size_t)tl * R + r) * exp_bytes, w, exp_bytes);
    else if (kFp8)
      s_scale[(size_t)tl * R + r] = __uint_as_float((uint32_t)w);
  };
  if (work) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (lane_t + k * tpt < R) v[k] = issue_row(lane_t + k * tpt);
    for (int r = lane_t + 4 * tpt; r < R; r += tpt) store_row(r, issue_row(r));
  }
  // The token's four stream slices, under the copies.
  uint4 xs[4][2];
  const uint16_t *xrow = p.x + t * 4 * D + col0;
  if (work) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      xs[s][0] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D));
      xs[s][1] = __ldcs(reinterpret_cast<const uint4 *>(xrow + (int64_t)s * D + 8));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (lane_t + k * tpt < R) store_row(lane_t + k * tpt, v[k]);
  }

  const bool landed = wait_bounded(bar, p.wait_limit_ns);
  // Block-uniform outcome; the barrier also publishes the scales and exponents.
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
  float saa = 0.f, smm = 0.f, sam = 0.f;
  if (work) {
    const uint8_t *src = s_rows + (size_t)tl * tok_bytes + (size_t)col0 * kElt;
    for (int r = 0; r < R; ++r) {
      const uint8_t *row = src + (size_t)r * row_bytes;
      if (kFp8) {
        const float scale =
            kRows ? e8m0_to_float(row[(D - col0) + (col0 >> 5)])
            : kE8 ? e8m0_to_float(s_exps[((size_t)tl * R + r) * exp_bytes + (col0 >> 5)])
                  : s_scale[(size_t)tl * R + r];
        acc_fp8(acc, *reinterpret_cast<const uint4 *>(row), scale);
      } else {
        acc_bf16(acc, *reinterpret_cast<const uint4 *>(row));
        acc_bf16(acc + 8, *reinterpret_cast<const uint4 *>(row + 16));
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= p.inv_R;
    gate_partials(xs[0][0], xs[0][1], acc, saa, smm, sam);
  }
  for (int o = tpt >> 1; o > 0; o >>= 1) {
    saa += __shfl_xor_sync(0xffffffffu, saa, o);
    smm += __shfl_xor_sync(0xffffffffu, smm, o);
    sam += __shfl_xor_sync(0xffffffffu, sam, o);
  }
  if (!work) {
    if (dead_tok)
      pass_through16(p.x + t * 4 * D + col0, p.y + t * 4 * D + col0, D,
                     AUX && p.gate_out ? p.gate_out + t : nullptr,
                     AUX && p.mem_out ? p.mem_out + t * D + col0 : nullptr, lane_t == 0);
    return;
  }
  const float g = gate_value(saa, smm, sam, (float)D, p.eps, p.sqrt_D);
  uint16_t *yrow = p.y + t * 4 * D + col0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float c = g * __ldg(p.alpha + s);
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D), gated_add8(xs[s][0], acc, c));
    __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D + 8), gated_add8(xs[s][1], acc + 8, c));
  }
  if (AUX) {
    if (p.gate_out && lane_t == 0) p.gate_out[t] = g;
    if (p.mem_out) {
      float4 *mo = reinterpret_cast<float4 *>(p.mem_out + t * D + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        mo[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    }
  }
}

template <int DT, bool AUX, bool EARLY>
cudaError_t launch_bulk_t(const LookupParams &p, size_t smem, cudaStream_t stream) {
  auto kern = lookup_bulk_kernel<DT, AUX, EARLY>;
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = raise_smem_ceiling(kern, configured);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)p.T, p.D / 16, smem, stream>>>(p);
  return cudaGetLastError();
}

// Tokens a block of the chained kernel: 4, fewer when that would leave part of
// the first wave of blocks empty.  Measured on the 8-head FP8 prefill (65,536
// tokens): 1 (a token a block) 1.649 ms; 4 1.625; 8 1.626; 16 1.636; 32 1.658;
// a single wave of blocks 1.649.  BF16 rows: 0.782 / 0.762 / 0.768 / 0.778 /
// 0.825 ms; the packed batch: 1.581 / 1.488 / 1.474 / 1.489 / 1.530 ms.
constexpr int kChainTokens = 4;

template <int DT, bool AUX>
cudaError_t launch_chain_t(const LookupParams &p_in, size_t smem, cudaStream_t stream) {
  auto kern = lookup_bulk_chain_kernel<DT, AUX>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = raise_smem_ceiling(kern, configured);
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, p_in.D / 16, smem);
  if (e != cudaSuccess) return e;
  LookupParams p = p_in;
  const int64_t wave = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  const int64_t fill = p.T / wave;  // tokens a block that still fill the first wave
  p.tpb = (int)(fill < 1 ? 1 : fill < kChainTokens ? fill : kChainTokens);
  const int64_t blocks = (p.T + p.tpb - 1) / p.tpb;
  kern<<<(unsigned)blocks, p.D / 16, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_bulk_dt(const LookupParams &p, size_t smem, bool aux, bool early,
                           cudaStream_t stream) {
  if (early)
    return aux ? launch_chain_t<DT, true>(p, smem, stream) : launch_chain_t<DT, false>(p, smem, stream);
  return aux ? launch_bulk_t<DT, true, false>(p, smem, stream)
             : launch_bulk_t<DT, false, false>(p, smem, stream);
}

template <int DT, bool AUX>
cudaError_t launch_small_t(const LookupParams &p, size_t smem, cudaStream_t stream) {
  auto kern = lookup_bulk_small_kernel<DT, AUX>;
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = raise_smem_ceiling(kern, configured);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (p.T + p.tpb - 1) / p.tpb;
  kern<<<(unsigned)blocks, p.tpb * p.tpt, smem, stream>>>(p);
  return cudaGetLastError();
}

// Shared memory of the small-row kernel for tpb tokens a block.
size_t small_smem_bytes(int D, int dtype, int H, int tpb) {
  const size_t rows = (size_t)tpb * 3 * H;
  const size_t exps = dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 ? rows * (D / 32) : 0;
  return rows * table_row_bytes(dtype, D) + ((exps + 15) & ~(size_t)15) +
         ((rows + 1) & ~(size_t)1) * 4 + 8;
}

// Tokens per block, a whole number of warps.  Measured on the released shape
// (256-wide FP8 rows with e8m0 blocks, 24 rows a token, 65,536 tokens): with the
// exponents apart, blocks of three warps, five to an SM, took 157 us; every
// other size tried, from one to seven warps a block and from two to sixteen
// blocks an SM (20 to 32 tokens resident), took 166-197 us, the three-warp size
// with only four blocks an SM among the slowest.  So: three warps when five
// such blocks fit in an SM's 228 KB of shared memory (1 KB of each block's is
// reserved); else the largest block of up to 256 threads within 56 KB (four
// blocks an SM).  With the exponents after each row, one warp a block measured
// best (131.9 us against 133.7 / 135.1 / 138.3 us for two, three and four warps).
int small_tokens_per_block(int D, int dtype, int H) {
  const int tpt = D / 16, warp_tokens = 32 / tpt;
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS) return warp_tokens;
  if (small_smem_bytes(D, dtype, H, 3 * warp_tokens) + 1024 <= 228 * 1024 / 5)
    return 3 * warp_tokens;
  int tpb = 256 / tpt;
  while (tpb > warp_tokens && small_smem_bytes(D, dtype, H, tpb) > 56 * 1024) tpb -= warp_tokens;
  return tpb;
}

}  // namespace

// D below 512 with D/16 a power of two (16 .. 256) and one warp of tokens within
// the 227 KB a block may use.
bool bulk_small_supported(int D, int dtype, int H) {
  if (D < 16 || D >= 512 || ((D / 16) & (D / 16 - 1)) != 0 || D % 16 != 0) return false;
  if ((dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 || dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS) &&
      D % 32 != 0)
    return false;
  return small_smem_bytes(D, dtype, H, small_tokens_per_block(D, dtype, H)) <= 227 * 1024;
}

cudaError_t launch_lookup_bulk_small(const LookupParams &p_in, int dtype, cudaStream_t stream) {
  if (p_in.T == 0) return cudaSuccess;
  LookupParams p = p_in;
  p.tpt = p.D / 16;
  p.tpb = small_tokens_per_block(p.D, dtype, p.H);
  const size_t smem = small_smem_bytes(p.D, dtype, p.H, p.tpb);
  const bool aux = p.gate_out != nullptr || p.mem_out != nullptr;
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN)
    return aux ? launch_small_t<ENGRAM_TABLE_FP8_E4M3FN, true>(p, smem, stream)
               : launch_small_t<ENGRAM_TABLE_FP8_E4M3FN, false>(p, smem, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32)
    return aux ? launch_small_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32, true>(p, smem, stream)
               : launch_small_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32, false>(p, smem, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS)
    return aux ? launch_small_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS, true>(p, smem, stream)
               : launch_small_t<ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS, false>(p, smem, stream);
  return aux ? launch_small_t<ENGRAM_TABLE_BF16, true>(p, smem, stream)
             : launch_small_t<ENGRAM_TABLE_BF16, false>(p, smem, stream);
}

size_t bulk_smem_bytes(int D, int dtype, int H) {
  const size_t exps = dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32 ? (size_t)3 * H * (D / 32) : 0;
  return (size_t)3 * H * table_row_bytes(dtype, D) + exps + 8 + kMaxRows * 4 + 24 * 4;
}

// D a multiple of 512 (whole warps of 16-column threads, at most 256 threads) and
// the token's rows within the 227 KB of shared memory a block may use.
bool bulk_supported(int D, int dtype, int H) {
  return D % 512 == 0 && D >= 512 && D <= ENGRAM_MAX_D &&
         bulk_smem_bytes(D, dtype, H) <= 227 * 1024;
}

cudaError_t launch_lookup_bulk(const LookupParams &p, int dtype, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  const size_t smem = bulk_smem_bytes(p.D, dtype, p.H);
  const bool aux = p.gate_out != nullptr || p.mem_out != nullptr;
  // Four blocks per SM when four tokens' rows fit in shared memory (streams
  // loaded after the rows); else two, with the streams loaded early.
  const bool early = smem > 56 * 1024;
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN)
    return launch_bulk_dt<ENGRAM_TABLE_FP8_E4M3FN>(p, smem, aux, early, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32)
    return launch_bulk_dt<ENGRAM_TABLE_FP8_E4M3FN_E8M0_B32>(p, smem, aux, early, stream);
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS)
    return launch_bulk_dt<ENGRAM_TABLE_FP8_E4M3FN_E8M0_ROWS>(p, smem, aux, early, stream);
  return launch_bulk_dt<ENGRAM_TABLE_BF16>(p, smem, aux, early, stream);
}

}  // namespace engram
