// wkv_gemm.cu -- k = E wkv^T on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// E [T, K] bf16 (the tokens' concatenated rows) times wkv [N, K] bf16 (one row of
// weights per output) gives k [T, N] fp32.  Two persistent kernels walk the
// tiles of k in order, N tiles fastest (the CTAs resident at one time share a
// few row slices of E, read from HBM once, and sweep wkv, which stays in L2):
//
//   wkv_gemm_pair_kernel (default): CTA pairs (2-CTA clusters), 256 x 256 tiles,
//     tcgen05.mma.cta_group::2 with M 256 -- each CTA stages its 128 rows of E
//     and its half of the wkv slice, a third less shared-memory traffic per MMA
//     than one CTA staging a whole 256-row slice;
//   wkv_gemm_kernel: one CTA per SM, 128 x 256 tiles, cta_group::1.
//
// Six warps per CTA in both:
//   warp 0, one thread : TMA producer -- fills a ring of shared-memory stages,
//                        each a 64-wide K slice of E and of wkv (one 128-byte
//                        swizzle atom along K), completing on an mbarrier;
//   warp 1             : allocates the 512 TMEM columns; one thread (of the
//                        pair's even CTA) issues the tcgen05.mma instructions
//                        (K 16, bf16 in, fp32 accumulated) into one of two
//                        256-column accumulators, frees each stage through an
//                        mbarrier once its MMAs have read it, and hands a
//                        finished accumulator to the epilogue through another;
//   warps 2..5         : the epilogue -- each reads its 32 TMEM lanes (tcgen05.ld)
//                        and stores fp32 rows of k, then returns the accumulator,
//                        so a tile's epilogue runs under the next tile's MMAs.
//
// Every mbarrier wait is bounded (SM clock cycles): a wait that gives up sets
// ENGRAM_FLAG_TIMEOUT and a shared abort flag, after which no warp issues more
// work and the tiles not yet stored stay unwritten; the issued copies and MMAs
// are waited for (bounded) and the TMEM columns freed before the block exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "engram_internal.cuh"

namespace engram {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kThreads = 192;                // producer, MMA, four epilogue warps
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kAccCols = 256;           // one fp32 accumulator: a column per output
constexpr uint32_t kTmemCols = 2 * kAccCols;  // two accumulators: all 512 columns
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + 256;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase of `bar` with parity `parity`, giving up after about
// limit_ns (SM cycles at 2.1 GHz, checked every 32 polls) or as soon as another
// thread raised the abort flag.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           int64_t limit_ns, int32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long limit = limit_ns * 21 / 10;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit) {
        *abort_flag = 1;
        if (status) atomicOr(status, ENGRAM_FLAG_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (draining work already issued).
__device__ __forceinline__ void drain_phase(uint64_t *bar, uint32_t parity, int64_t limit_ns) {
  const long long limit = limit_ns * 21 / 10;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return;
}

// 2-D TMA tile load (coordinates: x = K offset, y = row) completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row atoms 1024 bytes apart): start
// address, stride between 8-row groups 1024 B, descriptor version 1, layout
// SWIZZLE_128B (2).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 256, M = 128.
constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                                ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a_desc), "l"(b_desc), "r"(kInstrDesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    wkv_gemm_kernel(const __grid_constant__ CUtensorMap map_e, const __grid_constant__ CUtensorMap map_w,
                    float *__restrict__ k_out, int T, int N, int K, int64_t wait_limit_ns,
                    int32_t *status) {
  extern __shared__ uint8_t sm_raw[];
  // 1024-byte alignment for the swizzled tiles.
  uint8_t *sm = sm_raw + ((1024 - (smem_u32(sm_raw) & 1023)) & 1023);
  uint8_t *stage_base = sm;
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + kStages * kStageBytes);
  uint64_t *empty = full + kStages;
  uint64_t *acc_full = empty + kStages;  // [2] MMA -> epilogue
  uint64_t *acc_empty = acc_full + 2;    // [2] epilogue -> MMA (one arrive per epilogue warp)
  uint64_t *mma_done = acc_empty + 2;    // every MMA issued has completed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kblocks = K / kBK;
  const int n_tiles_n = N / kBN;
  const int64_t n_tiles = (int64_t)((T + kBM - 1) / kBM) * n_tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full + a, 1);
      mbar_init(acc_empty + a, 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // the whole warp allocates the accumulators' TMEM columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- TMA producer
      uint32_t it = 0;  // k-blocks issued, over all of this CTA's tiles
      for (int64_t tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
        const int m0 = (int)(tile / n_tiles_n) * kBM, n0 = (int)(tile % n_tiles_n) * kBN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!(ok = wait_phase(empty + s, ph ^ 1, abort_flag, wait_limit_ns, status))) break;
          uint8_t *a = stage_base + s * kStageBytes;
          mbar_arrive_expect_tx(full + s, kStageBytes);
          tma_load_2d(a, &map_e, kb * kBK, m0, full + s);
          tma_load_2d(a + kABytes, &map_w, kb * kBK, n0, full + s);
        }
        if (!ok) break;
      }
      // Loads issued into shared memory land before the block can exit.
      for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0; j < it; ++j)
        drain_phase(full + j % kStages, (j / kStages) & 1, wait_limit_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      uint32_t it = 0, local = 0;
      for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
        const uint32_t acc = local & 1, use = local >> 1;
        if (!wait_phase(acc_empty + acc, (use & 1) ^ 1, abort_flag, wait_limit_ns, status)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d_tmem = tmem + acc * kAccCols;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!(ok = wait_phase(full + s, ph, abort_flag, wait_limit_ns, status))) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t a = smem_u32(stage_base + s * kStageBytes);
          const uint32_t b = a + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)  // advance 16 bf16 = 32 bytes along K per MMA
            umma_bf16(d_tmem, smem_desc_sw128(a + 32 * k), smem_desc_sw128(b + 32 * k),
                      (kb | k) != 0 ? 1u : 0u);
          umma_commit(empty + s);  // the stage is free once these MMAs have read it
        }
        if (!ok) break;
        umma_commit(acc_full + acc);  // the accumulator is complete once they have run
      }
      umma_commit(mma_done);  // arrives when every MMA issued above has completed
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // this warp may read TMEM lanes 32*quad .. 32*quad+31
    uint32_t local = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
      const uint32_t acc = local & 1, use = local >> 1;
      const bool ok = wait_phase(acc_full + acc, use & 1, abort_flag, wait_limit_ns, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int m0 = (int)(tile / n_tiles_n) * kBM, n0 = (int)(tile % n_tiles_n) * kBN;
      const int row = m0 + quad * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + acc * kAccCols + c * 32;
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
            "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
              "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
              "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
              "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
              "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
              "=r"(v[31])
            : "r"(taddr)
            : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (row < T) {
          float4 *dst = reinterpret_cast<float4 *>(k_out + (int64_t)row * N + n0 + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + acc);
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) drain_phase(mma_done, 0, wait_limit_ns);
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// The CTA-pair variant: two CTAs of a cluster compute one 256 x 256 tile with
// tcgen05.mma.cta_group::2 (M 256).  Each CTA stages its own 128 rows of E and
// its half (128 rows) of the wkv slice, so a stage is 32 KB a CTA instead of
// 48 KB for the same MMAs; the even CTA (the leader) issues the MMAs, which
// read both CTAs' shared memory and write each CTA's 128 rows of the
// accumulator into that CTA's TMEM.
//
// Barriers: full[s] lives in the leader (one arrival, the leader's, expecting
// both CTAs' bytes; both CTAs' loads complete on it -- the peer's may land
// before the leader's arrival, which the barrier's signed transaction count
// allows, and the phase cannot complete before that arrival); empty[s],
// acc_full[a] and mma_done
// exist in both CTAs and are arrived on by the leader's commits, multicast to
// the pair; acc_empty[a] lives in the leader and takes one arrival from each of
// the eight epilogue warps of the pair.

constexpr int kPairStages = 6;
constexpr uint32_t kPairBBytes = (kBN / 2) * kBK * 2;  // 16 KB: this CTA's half of the slice
constexpr uint32_t kPairStageBytes = kABytes + kPairBBytes;
constexpr size_t kPairSmemBytes = 1024 + kPairStages * kPairStageBytes + 256;

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 256, M = 256 (the pair).
constexpr uint32_t kPairInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                    ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of `local` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(local), "r"(rank));
  return out;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// 2-D TMA load into this CTA's shared memory completing on a barrier of either
// CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a_desc), "l"(b_desc), "r"(kPairInstrDesc), "r"(accumulate)
      : "memory");
}

// Arrive (once each) on the barrier at `bar`'s offset in both CTAs of the pair
// when every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    wkv_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_e,
                         const __grid_constant__ CUtensorMap map_w, float *__restrict__ k_out,
                         int T, int N, int K, int64_t wait_limit_ns, int32_t *status) {
  extern __shared__ uint8_t sm_raw[];
  // 1024-byte alignment for the swizzled tiles (the same offset in both CTAs).
  uint8_t *sm = sm_raw + ((1024 - (smem_u32(sm_raw) & 1023)) & 1023);
  uint8_t *stage_base = sm;
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + kPairStages * kPairStageBytes);  // leader's
  uint64_t *empty = full + kPairStages;
  uint64_t *acc_full = empty + kPairStages;  // [2]
  uint64_t *acc_empty = acc_full + 2;        // [2] leader's, 8 arrivals
  uint64_t *mma_done = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int kblocks = K / kBK;
  const int n_tiles_n = N / kBN;
  const int64_t pair_tiles = (int64_t)((T + 2 * kBM - 1) / (2 * kBM)) * n_tiles_n;
  const int64_t cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full + a, 1);
      mbar_init(acc_empty + a, 8);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's TMEM columns together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  cluster_sync();  // both CTAs' barriers are initialised before either uses the other's
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const uint32_t full_lead = map_to_rank(smem_u32(full), 0);
  const uint32_t acc_empty_lead = map_to_rank(smem_u32(acc_empty), 0);

  if (warp == 0) {
    if (lane == 0) {
      // ----------------------------------------------- TMA producer (both CTAs)
      uint32_t it = 0;
      for (int64_t tile = cluster; tile < pair_tiles && !*abort_flag; tile += n_clusters) {
        const int m0 = (int)(tile / n_tiles_n) * 2 * kBM + (int)rank * kBM;
        const int n0 = (int)(tile % n_tiles_n) * kBN + (int)rank * (kBN / 2);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1;
          if (!(ok = wait_phase(empty + s, ph ^ 1, abort_flag, wait_limit_ns, status))) break;
          uint8_t *a = stage_base + s * kPairStageBytes;
          const uint32_t bar = full_lead + 8u * s;
          if (rank == 0) mbar_arrive_expect_tx(full + s, 2 * kPairStageBytes);
          tma_load_2d_pair(a, &map_e, kb * kBK, m0, bar);
          tma_load_2d_pair(a + kABytes, &map_w, kb * kBK, n0, bar);
        }
        if (!ok) break;
      }
      // The leader's full barriers count both CTAs' bytes: once they complete,
      // every load of the pair has landed.
      if (rank == 0)
        for (uint32_t j = it > (uint32_t)kPairStages ? it - kPairStages : 0; j < it; ++j)
          drain_phase(full + j % kPairStages, (j / kPairStages) & 1, wait_limit_ns);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------- MMA issuer (leader)
      uint32_t it = 0, local = 0;
      for (int64_t tile = cluster; tile < pair_tiles; tile += n_clusters, ++local) {
        const uint32_t acc = local & 1, use = local >> 1;
        if (!wait_phase(acc_empty + acc, (use & 1) ^ 1, abort_flag, wait_limit_ns, status)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d_tmem = tmem + acc * kAccCols;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1;
          if (!(ok = wait_phase(full + s, ph, abort_flag, wait_limit_ns, status))) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t a = smem_u32(stage_base + s * kPairStageBytes);
          const uint32_t b = a + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16_pair(d_tmem, smem_desc_sw128(a + 32 * k), smem_desc_sw128(b + 32 * k),
                           (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair(empty + s);  // both CTAs' stage s is free once these have run
        }
        if (!ok) break;
        umma_commit_pair(acc_full + acc);
      }
      umma_commit_pair(mma_done);
    }
  } else {
    // ------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;
    uint32_t local = 0;
    for (int64_t tile = cluster; tile < pair_tiles; tile += n_clusters, ++local) {
      const uint32_t acc = local & 1, use = local >> 1;
      const bool ok = wait_phase(acc_full + acc, use & 1, abort_flag, wait_limit_ns, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int m0 = (int)(tile / n_tiles_n) * 2 * kBM + (int)rank * kBM;
      const int n0 = (int)(tile % n_tiles_n) * kBN;
      const int row = m0 + quad * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + acc * kAccCols + c * 32;
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
            "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
              "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
              "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
              "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
              "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
              "=r"(v[31])
            : "r"(taddr)
            : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (row < T) {
          float4 *dst = reinterpret_cast<float4 *>(k_out + (int64_t)row * N + n0 + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_lead + 8u * acc);
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1 && lane == 0) drain_phase(mma_done, 0, wait_limit_ns);  // the pair's MMAs ran
  __syncwarp();
  cluster_sync();  // no CTA leaves while the other may still signal it
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// A row-major bf16 matrix [rows, cols] (cols contiguous) as a 2-D tiled map with
// box [64 cols, box_rows], 128-byte swizzle, zero fill outside.
bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool wkv_gemm_supported(int N, int K) { return N % kBN == 0 && K % kBK == 0 && K > 0 && N > 0; }

namespace {

// Per device: SM count and how many CTA pairs of the pair kernel fit at once
// (clusters need both CTAs in one GPC, so an odd SM in a GPC stays out).
struct GemmDeviceInfo {
  bool ready = false;
  int sms = 0, pair_clusters = 0;
};
GemmDeviceInfo g_gemm_info[64];
std::mutex g_gemm_info_mu;

cudaError_t gemm_device_info(int dev, GemmDeviceInfo &out) {
  std::lock_guard<std::mutex> lock(g_gemm_info_mu);
  GemmDeviceInfo &gi = g_gemm_info[dev & 63];
  if (!gi.ready) {
    cudaError_t err = cudaDeviceGetAttribute(&gi.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(wkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(wkv_gemm_pair_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmemBytes);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (gi.sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    err = cudaOccupancyMaxActiveClusters(&gi.pair_clusters, wkv_gemm_pair_kernel, &cfg);
    if (err != cudaSuccess) return err;
    gi.ready = true;
  }
  out = gi;
  return cudaSuccess;
}

std::atomic<int> g_projection_kernel{ENGRAM_PROJECTION_AUTO};

}  // namespace

int set_projection_kernel(int which) { return g_projection_kernel.exchange(which); }

cudaError_t launch_wkv_gemm(const uint16_t *e, const uint16_t *wkv, float *k_out, int T, int N, int K,
                            int64_t wait_limit_ns, int32_t *status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  GemmDeviceInfo gi;
  if (err == cudaSuccess) err = gemm_device_info(dev, gi);
  if (err != cudaSuccess) return err;
  const int which = g_projection_kernel.load(std::memory_order_relaxed);
  const bool pair = which != ENGRAM_PROJECTION_SINGLE && gi.pair_clusters > 0;
  CUtensorMap map_e, map_w;
  if (!make_map(&map_e, e, (uint64_t)T, (uint64_t)K, kBM) ||
      !make_map(&map_w, wkv, (uint64_t)N, (uint64_t)K, pair ? kBN / 2 : kBN))
    return cudaErrorInvalidValue;
  if (pair) {
    // persistent: as many CTA pairs as fit at once, each walking 256 x 256 tiles
    const int64_t pair_tiles = (int64_t)((T + 2 * kBM - 1) / (2 * kBM)) * (N / kBN);
    const int clusters = (int)(pair_tiles < gi.pair_clusters ? pair_tiles : gi.pair_clusters);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, wkv_gemm_pair_kernel, map_e, map_w, k_out, T, N, K,
                              wait_limit_ns, status);
  }
  const int64_t tiles = (int64_t)((T + kBM - 1) / kBM) * (N / kBN);
  const int grid = (int)(tiles < gi.sms ? tiles : gi.sms);  // persistent: one CTA per SM
  wkv_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_e, map_w, k_out, T, N, K,
                                                          wait_limit_ns, status);
  return cudaGetLastError();
}

}  // namespace engram
