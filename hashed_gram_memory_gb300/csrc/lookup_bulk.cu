// lookup_bulk.cu -- the fused Engram lookup as a persistent, warp-specialised
// sm_103a kernel fed by 1-D bulk copies (TMA).
//
// One CTA per SM.  Warp NW (the producer) walks the CTA's tokens and, for each,
// copies the token's four streams (one contiguous 4*D*2-byte run) into a stream
// stage and its 3H table rows (one contiguous D*elt-byte run each) into a ring of
// row slots with cp.async.bulk, each copy completing on an mbarrier with its
// byte count.  It also writes the token's row scales and a bad-id flag into the
// stage.  Warps 0..NW-1 (the consumers, D/16 threads, 16 columns each) take the
// rows from shared memory in order, accumulate the dequantised rows in fp32
// registers, reduce the three gate sums across warps through shared memory, and
// write the four updated streams straight to global memory.  The producer runs
// up to a ring (~1.5 tokens of rows) and two stream stages ahead, so ~200 KB per
// SM is in flight without holding a register per byte.
//
// Every wait is bounded: an mbarrier wait that outlives the wait limit sets
// ENGRAM_FLAG_TIMEOUT and a shared abort flag, every warp then leaves its loop,
// and the producer waits (again bounded) for the copies it issued before the
// block exits.  No named barrier is used after the roles split, so a warp that
// leaves early cannot strand the others.
#include "engram_internal.cuh"
#include "lookup_common.cuh"

namespace engram {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
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

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits, with the whole warp, for the phase of `bar` with parity `parity`.
// Every lane polls the barrier (so every lane acquires the data it guards); the
// decision to give up is taken by lane 0 and broadcast, so the result is the
// same on all 32 lanes and the warp never splits.  Returns false when another
// warp has aborted, or when the wait outlives limit_ns, in which case it raises
// the abort flag and the timeout status bit.  All 32 lanes must call it.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           int64_t limit_ns, int32_t *status) {
  bool done = mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, done)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (!done) done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((i & 15) == 0) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        if (*abort_flag) {
          give_up = 1;
        } else if ((int64_t)(global_ns() - t0) > limit_ns) {
          *abort_flag = 1;
          if (status) atomicOr(status, ENGRAM_FLAG_TIMEOUT);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
  }
}

// Bounded wait that ignores the abort flag (used to drain copies in flight).
__device__ __forceinline__ void drain_phase(uint64_t *bar, uint32_t parity, int64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if ((int64_t)(global_ns() - t0) > limit_ns) return;
  }
}

// Per-token metadata the producer leaves in a stream stage.
struct StageMeta {
  float scale[kMaxRows];
  int32_t bad;
  int32_t pad[3];
};

template <int DT, bool AUX>
__global__ void __launch_bounds__(288, 1) lookup_bulk_kernel(const __grid_constant__ LookupParams p) {
  constexpr bool kFp8 = DT == ENGRAM_TABLE_FP8_E4M3FN;
  constexpr int kElt = kFp8 ? 1 : 2;
  extern __shared__ __align__(128) uint8_t sm[];

  const int nw = p.nw;
  const int H = p.H, R = 3 * H, D = p.D;
  const uint32_t row_bytes = (uint32_t)D * kElt;
  const uint32_t st_bytes = (uint32_t)D * 4 * 2;
  const int nslot = p.nslot, nstage = p.nstage;

  uint8_t *s_rows = sm;
  uint8_t *s_st = s_rows + (size_t)nslot * row_bytes;
  StageMeta *s_meta = reinterpret_cast<StageMeta *>(s_st + (size_t)nstage * st_bytes);
  uint64_t *full_row = reinterpret_cast<uint64_t *>(s_meta + nstage);
  uint64_t *empty_row = full_row + nslot;
  uint64_t *full_st = empty_row + nslot;
  uint64_t *empty_st = full_st + nstage;
  uint64_t *red_bar = empty_st + nstage;
  float *red = reinterpret_cast<float *>(red_bar + 1);  // [2][nw][3]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(red + 2 * nw * 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nslot; ++i) {
      mbar_init(full_row + i, 1);
      mbar_init(empty_row + i, nw);
    }
    for (int i = 0; i < nstage; ++i) {
      mbar_init(full_st + i, 1);
      mbar_init(empty_st + i, nw);
    }
    mbar_init(red_bar, nw);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == nw) {
    // ------------------------------------------------------------ producer
    // Per token: publish the stage (scales + bad flag, then the stream copy),
    // then issue the 3H row copies into the ring.  Publishing first lets the
    // consumers start on the token while its rows are still being issued, so
    // any 3H works with any ring size.  Row ids are prefetched two tokens ahead
    // and scales one token ahead, so the publish does not wait on a load.
    uint32_t k = 0, q = 0;
    bool withhold = p.withhold != 0;
    const int64_t stride = gridDim.x;
    auto load_ids = [&](int64_t tok, int32_t (&dst)[3]) {
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int r = lane + 32 * i;
        dst[i] = (tok < p.T && r < R) ? p.row_ids[tok * R + r] : 0;
      }
    };
    auto check_ids = [&](const int32_t (&ids)[3]) {
      bool bad_lane = false;
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int r = lane + 32 * i;
        if (r < R) {
          const int ni = (r >= H) + (r >= 2 * H);
          bad_lane |= (ids[i] < 0) | ((int64_t)ids[i] >= p.rows[ni]);
        }
      }
      return __any_sync(0xffffffffu, bad_lane);
    };
    auto load_scales = [&](int64_t tok, const int32_t (&ids)[3], bool bad, float (&dst)[3]) {
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int r = lane + 32 * i;
        dst[i] = 1.f;
        if (kFp8 && !bad && tok < p.T && r < R) {
          const int ni = (r >= H) + (r >= 2 * H);
          dst[i] = __ldg(p.scale[ni] + ids[i]);
        }
      }
    };
    int64_t t = blockIdx.x;
    int32_t id0[3], id1[3], id2[3];
    float sc0[3], sc1[3];
    load_ids(t, id0);
    load_ids(t + stride, id1);
    bool bad0 = check_ids(id0);
    load_scales(t, id0, bad0, sc0);
    for (; t < p.T; t += stride) {
      load_ids(t + 2 * stride, id2);
      const bool bad1 = check_ids(id1);
      load_scales(t + stride, id1, bad1, sc1);

      const uint32_t si = q % nstage, sph = (q / nstage) & 1;
      if (!wait_phase(empty_st + si, sph ^ 1, abort_flag, p.wait_limit_ns, p.status)) break;
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int r = lane + 32 * i;
        if (r < R) s_meta[si].scale[r] = sc0[i];
      }
      if (lane == 0) s_meta[si].bad = bad0 ? 1 : 0;
      __threadfence_block();  // every lane's metadata before lane 0's releasing arrive
      __syncwarp();
      if (lane == 0) {
        if (!bad0) {
          mbar_arrive_expect_tx(full_st + si, st_bytes);
          bulk_g2s(s_st + (size_t)si * st_bytes, p.x + t * 4 * D, st_bytes, full_st + si);
        } else {
          mbar_arrive(full_st + si);
        }
      }
      ++q;
      bool aborted = false;
      if (!bad0) {
        for (int r = 0; r < R; ++r) {
          const int32_t mine = r < 32 ? id0[0] : (r < 64 ? id0[1] : id0[2]);
          const int32_t row = __shfl_sync(0xffffffffu, mine, r & 31);
          const int ni = (r >= H) + (r >= 2 * H);
          const uint32_t slot = k % nslot, ph = (k / nslot) & 1;
          if (!wait_phase(empty_row + slot, ph ^ 1, abort_flag, p.wait_limit_ns, p.status)) {
            aborted = true;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(full_row + slot, row_bytes);
            if (withhold)
              withhold = false;  // test hook: this copy is never issued
            else
              bulk_g2s(s_rows + (size_t)slot * row_bytes, p.table[ni] + (int64_t)row * row_bytes,
                       row_bytes, full_row + slot);
          }
          ++k;
        }
      }
      if (aborted) break;
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        id0[i] = id1[i];
        id1[i] = id2[i];
        sc0[i] = sc1[i];
      }
      bad0 = bad1;
    }
    {
      // Copies issued into shared memory must land before the block exits, even
      // if the consumers gave up on them (bounded; returns at once when landed).
      const uint32_t nk = k < (uint32_t)nslot ? k : (uint32_t)nslot;
      for (uint32_t j = k - nk; j < k; ++j)
        if (lane == 0) drain_phase(full_row + (j % nslot), (j / nslot) & 1, p.wait_limit_ns);
      const uint32_t nq = q < (uint32_t)nstage ? q : (uint32_t)nstage;
      for (uint32_t j = q - nq; j < q; ++j)
        if (lane == 0) drain_phase(full_st + (j % nstage), (j / nstage) & 1, p.wait_limit_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int col0 = (warp * 32 + lane) * 16;
  const float Df = (float)D;
  uint32_t k = 0, q = 0, it = 0;
  for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, ++it) {
    const uint32_t si = q % nstage, sph = (q / nstage) & 1;
    if (!wait_phase(full_st + si, sph, abort_flag, p.wait_limit_ns, p.status)) break;
    const StageMeta &meta = s_meta[si];
    const uint8_t *xs = s_st + (size_t)si * st_bytes + (size_t)col0 * 2;  // stream s at + s*D*2
    if (meta.bad) {
      if (warp == 0 && lane == 0 && p.status) atomicOr(p.status, ENGRAM_FLAG_BAD_ROW);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_st + si);
      ++q;
      // keep the reduction barrier's phase count in step with the other warps
      if (lane == 0) mbar_arrive(red_bar);
      if (!wait_phase(red_bar, it & 1, abort_flag, p.wait_limit_ns, p.status)) break;
      continue;
    }
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int r = 0; r < R; ++r) {
      const uint32_t slot = k % nslot, ph = (k / nslot) & 1;
      if (!wait_phase(full_row + slot, ph, abort_flag, p.wait_limit_ns, p.status)) {
        ok = false;
        break;
      }
      const uint8_t *src = s_rows + (size_t)slot * row_bytes + (size_t)col0 * kElt;
      if (kFp8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(src);
        acc_fp8(acc, v, meta.scale[r]);
      } else {
        const uint4 v0 = *reinterpret_cast<const uint4 *>(src);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(src + 16);
        acc_bf16(acc, v0);
        acc_bf16(acc + 8, v1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_row + slot);
      ++k;
    }
    if (!ok) break;

#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= p.inv_R;
    const uint4 a_lo = *reinterpret_cast<const uint4 *>(xs);
    const uint4 a_hi = *reinterpret_cast<const uint4 *>(xs + 16);
    float saa = 0.f, smm = 0.f, sam = 0.f;
    gate_partials(a_lo, a_hi, acc, saa, smm, sam);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      saa += __shfl_xor_sync(0xffffffffu, saa, o);
      smm += __shfl_xor_sync(0xffffffffu, smm, o);
      sam += __shfl_xor_sync(0xffffffffu, sam, o);
    }
    float *rb = red + (it & 1) * nw * 3;
    if (lane == 0) {
      rb[3 * warp + 0] = saa;
      rb[3 * warp + 1] = smm;
      rb[3 * warp + 2] = sam;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(red_bar);
    if (!wait_phase(red_bar, it & 1, abort_flag, p.wait_limit_ns, p.status)) break;
    saa = smm = sam = 0.f;
    for (int w = 0; w < nw; ++w) {
      saa += rb[3 * w + 0];
      smm += rb[3 * w + 1];
      sam += rb[3 * w + 2];
    }
    const float g = gate_value(saa, smm, sam, Df, p.eps, p.sqrt_D);

    uint16_t *yrow = p.y + t * 4 * D + col0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const float c = g * __ldg(p.alpha + s);
      const uint4 x0 = *reinterpret_cast<const uint4 *>(xs + (size_t)s * D * 2);
      const uint4 x1 = *reinterpret_cast<const uint4 *>(xs + (size_t)s * D * 2 + 16);
      __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D), gated_add8(x0, acc, c));
      __stcs(reinterpret_cast<uint4 *>(yrow + (int64_t)s * D + 8), gated_add8(x1, acc + 8, c));
    }
    if (AUX) {
      if (p.gate_out && warp == 0 && lane == 0) p.gate_out[t] = g;
      if (p.mem_out) {
        float4 *mo = reinterpret_cast<float4 *>(p.mem_out + t * D + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mo[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_st + si);
    ++q;
  }
}

template <int DT, bool AUX>
cudaError_t launch_bulk_t(const LookupParams &p, size_t smem, int blocks, cudaStream_t stream) {
  auto kern = lookup_bulk_kernel<DT, AUX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<blocks, (p.nw + 1) * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t bulk_smem_bytes(int D, int dtype, int nslot, int nstage) {
  const size_t elt = dtype == ENGRAM_TABLE_FP8_E4M3FN ? 1 : 2;
  const int nw = D / 512;
  return (size_t)nslot * D * elt + (size_t)nstage * D * 8 + (size_t)nstage * sizeof(StageMeta) +
         (2 * (size_t)nslot + 2 * (size_t)nstage + 1) * 8 + 2 * (size_t)nw * 3 * 4 + 16;
}

bool bulk_supported(int D) { return D % 512 == 0 && D >= 512 && D <= ENGRAM_MAX_D; }

cudaError_t launch_lookup_bulk(const LookupParams &p_in, int dtype, int num_sms,
                               cudaStream_t stream) {
  LookupParams p = p_in;
  p.nw = p.D / 512;
  p.nstage = 2;
  // Fill ~200 KB of shared memory: two stream stages, the rest row slots.
  const size_t budget = 200 * 1024;
  const size_t elt = dtype == ENGRAM_TABLE_FP8_E4M3FN ? 1 : 2;
  int nslot = 64;
  while (nslot > 4 && bulk_smem_bytes(p.D, dtype, nslot, p.nstage) > budget) --nslot;
  (void)elt;
  p.nslot = nslot;
  const size_t smem = bulk_smem_bytes(p.D, dtype, nslot, p.nstage);
  int64_t blocks = num_sms;
  if (blocks > p.T) blocks = p.T;
  const bool aux = p.gate_out != nullptr || p.mem_out != nullptr;
  if (dtype == ENGRAM_TABLE_FP8_E4M3FN)
    return aux ? launch_bulk_t<ENGRAM_TABLE_FP8_E4M3FN, true>(p, smem, (int)blocks, stream)
               : launch_bulk_t<ENGRAM_TABLE_FP8_E4M3FN, false>(p, smem, (int)blocks, stream);
  return aux ? launch_bulk_t<ENGRAM_TABLE_BF16, true>(p, smem, (int)blocks, stream)
             : launch_bulk_t<ENGRAM_TABLE_BF16, false>(p, smem, (int)blocks, stream);
}

}  // namespace engram
