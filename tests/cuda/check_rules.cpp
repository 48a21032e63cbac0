// Host test of the checked build's rules (checks.h): every predicate against
// cases written from the rules themselves, plus exhaustive sweeps of the
// coordinates and columns a kernel can pass. Prints FAIL lines, then ALL OK.
#include <stdio.h>

#include <initializer_list>

#include "checks.h"

static int fails = 0;
#define EXPECT(cond)                                         \
  do {                                                       \
    if (!(cond)) {                                           \
      printf("FAIL line %d: %s\n", __LINE__, #cond);         \
      ++fails;                                               \
    }                                                        \
  } while (0)

int main() {
  using namespace fa;
  // TMA loads: x a non-negative multiple of 8 elements, 1024-byte aligned destination
  for (int x = -64; x <= 512; ++x) EXPECT(tma_load_ok(x, 0) == (x >= 0 && x % 8 == 0));
  for (unsigned a = 0; a < 65536; a += 16) EXPECT(tma_load_ok(64, a) == (a % 1024 == 0));
  EXPECT(tma_load_ok(0, 16384) && tma_load_ok(192, 3 * 16384 + 8192));
  // TMA stores: x a non-negative multiple of 8, no negative start, 16-byte aligned source
  for (int x = -64; x <= 512; ++x) EXPECT(tma_store_ok(x, 0, 0, 0) == (x >= 0 && x % 8 == 0));
  EXPECT(!tma_store_ok(16, -1, 0, 0) && !tma_store_ok(16, 0, -1, 0) && tma_store_ok(16, 5000, 7, 0));
  for (unsigned a = 0; a < 4096; ++a) EXPECT(tma_store_ok(0, 0, 0, a) == (a % 16 == 0));
  // bulk copies: 16-byte aligned addresses, size a positive multiple of 16
  for (unsigned b = 0; b <= 4096; ++b) EXPECT(bulk_ok(0, 0, b) == (b > 0 && b % 16 == 0));
  for (unsigned a = 0; a < 256; ++a) {
    EXPECT(bulk_ok(a, 0, 512) == (a % 16 == 0));
    EXPECT(bulk_ok(0, 0x10000ull + a, 512) == (a % 16 == 0));
  }
  // TMEM: the warp's lane quarter, columns within the 512 of the allocation
  for (unsigned warp = 0; warp < 16; ++warp)
    for (unsigned lane = 0; lane < 128; lane += 32)
      for (unsigned n : {16u, 32u, 64u, 128u})
        for (unsigned col = 0; col <= 520; ++col) {
          const unsigned taddr = (lane << 16) | col;
          EXPECT(tmem_ok(taddr, n, warp) == (lane == 32 * (warp % 4) && col + n <= 512));
        }
  if (fails == 0) printf("ALL OK\n");
  return fails != 0;
}
