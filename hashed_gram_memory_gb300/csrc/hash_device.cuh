// hash_device.cuh -- the device side of the Engram n-gram hash, shared by the
// hash kernel and the fused decode step: the window of a token (oldest id
// first, its own id last), the fold of its last n ids from the per-(n, head)
// seed, and the row in the (n, head) table or bucket.
#pragma once

#include <stdint.h>

#include "engram_internal.cuh"

namespace engram {

constexpr uint64_t kFold = 0x9E3779B97F4A7C15ull;

// x mod d for d >= 1, with m = floor((2^64 - 1) / d).  q = umulhi(x, m) is
// floor(x/d) or one less (d*m lies within d of 2^64, so x*m/2^64 > x/d - 1), so
// x - q*d is in [0, 2d) and one conditional subtraction finishes it.
__device__ __forceinline__ uint64_t mod_by_reciprocal(uint64_t x, uint64_t d, uint64_t m) {
  const uint64_t q = __umul64hi(x, m);
  const uint64_t r = x - q * d;
  return r >= d ? r - d : r;
}

// The window w[0..3] (oldest first, w[3] = the token's own id `self`, not dead)
// from the ids before it as stored, raw[0..2] (raw[2] the newest), read back no
// further than `limit` ids: slots beyond the limit or at and before a dead id
// hold the pad id 0.  Returns false when an id in reach is negative but not
// dead (a bad id).
__device__ __forceinline__ bool make_window(const int32_t (&raw)[3], int32_t self, int64_t limit,
                                            int32_t (&w)[4]) {
  w[3] = self;
  bool blocked = false, ok = true;
#pragma unroll
  for (int k = 1; k <= 3; ++k) {
    int32_t e = 0;
    if (!blocked && k <= limit) {
      e = raw[3 - k];
      if (e == ENGRAM_EID_DEAD) {
        blocked = true;
        e = 0;
      } else if (e < 0) {
        ok = false;
      }
    }
    w[3 - k] = e;
  }
  return ok;
}

// Row id r (n-major: r = (n-2)*H + j) of a window: h = seed(n, j); for each of
// the last n ids, oldest first, h = (h ^ e) * kFold, h ^= h >> 29; row =
// off + h mod m.
__device__ __forceinline__ int32_t window_row(const int32_t (&w)[4], int r, int H,
                                              const uint64_t (&seed)[3][kMaxHeads],
                                              const uint64_t (&mod)[3][kMaxHeads],
                                              const uint64_t (&rmul)[3][kMaxHeads],
                                              const uint64_t (&off)[3][kMaxHeads]) {
  const int ni = (r >= H) + (r >= 2 * H);  // n - 2
  const int j = r - ni * H;
  uint64_t h = seed[ni][j];
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // the last n = ni + 2 ids, oldest first
    if (k >= 2 - ni) {
      h = (h ^ (uint64_t)(uint32_t)w[k]) * kFold;
      h ^= h >> 29;
    }
  }
  return (int32_t)(off[ni][j] + mod_by_reciprocal(h, mod[ni][j], rmul[ni][j]));
}

}  // namespace engram
