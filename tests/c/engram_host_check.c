/*
 * engram_host_check.c -- the C ABI used from plain C99 with no GPU: links
 * against libengram.so, calls the host-only entry points and a few argument
 * errors, and prints one line per check.  Exit status 0 when all pass.
 */
#include <stdio.h>
#include <string.h>

#include "engram.h"

static int failures = 0;

static void check(int ok, const char *what) {
  printf("%s %s\n", ok ? "ok  " : "FAIL", what);
  if (!ok) ++failures;
}

int main(void) {
  check(engram_abi_version() == ENGRAM_ABI_VERSION, "ABI version matches the header");
  check(strlen(engram_status_string(ENGRAM_ERR_INVALID_ARG)) > 0, "status strings");

  /* The released layout's bucket draw (host only): one layer, orders 2..4, two
   * heads, hash vocabulary 64 sums to 462. */
  int64_t primes[6];
  check(engram_bucket_primes(1, 4, 2, 64, primes) == ENGRAM_OK, "bucket primes");
  int64_t sum = 0;
  for (int i = 0; i < 6; ++i) sum += primes[i];
  check(sum == 462, "bucket primes sum to 462");

  /* Argument errors come back before any device is touched. */
  int64_t rows[3] = {11, 13, 17};
  check(engram_hash((const int32_t *)0x1000, 1, 4, NULL, NULL, 0, rows, (int32_t *)0x2000, NULL,
                    NULL) == ENGRAM_ERR_INVALID_ARG,
        "n_heads 0 is an argument error");
  check(strlen(engram_last_error()) > 0, "the last error names the argument");
  check(engram_compress(NULL, 8, NULL, 100, 50, NULL, NULL, NULL) == ENGRAM_ERR_INVALID_ARG,
        "NULL map is an argument error");
  const int64_t empty_bucket[6] = {7, 11, 0, 13, 17, 19};
  engram_layout lay = {NULL, NULL, empty_bucket};
  check(engram_compress_hash((const int32_t *)0x1000, 1, 4, (const int32_t *)0x8000, 100, 50,
                             NULL, NULL, 2, rows, &lay, NULL, (int32_t *)0x20000, NULL,
                             NULL) == ENGRAM_ERR_INVALID_ARG,
        "a bucket of no rows is refused");
  check(engram_forward_workspace_bytes(2, 8, 4) >= (size_t)(2 * 8 * 4 + 2 * 8 * 12 * 4),
        "workspace size covers ids and row ids");
  check(engram_set_lookup_kernel(7) == -1, "unknown lookup kernel refused");
  return failures ? 1 : 0;
}
