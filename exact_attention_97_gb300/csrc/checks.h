// checks.h -- the rules the checked build (FA_CHECKED) tests before it issues
// a TMA copy, a bulk copy or a TMEM access. Pure integer predicates on the
// instruction's arguments; sm103.cuh applies them in its wrappers. The header
// compiles as plain C++ too, so a CPU test checks the rules themselves.
//
// The rules, for the 16-bit tensors and maps of this library:
//   * a tiled TMA load starts at an innermost coordinate x >= 0 that is a
//     multiple of 8 elements (16 bytes), into a 1024-byte aligned shared
//     address (the tiles are 128-byte swizzled);
//   * a tiled TMA store also starts at x a multiple of 8, and at no negative
//     coordinate, from a 16-byte aligned shared address;
//   * a bulk copy has 16-byte aligned addresses and a size that is a positive
//     multiple of 16;
//   * a 32x32b tcgen05.ld / st of n columns addresses the lane quarter of the
//     issuing warp (warp index mod 4) and columns [c, c + n) within the 512 of
//     the allocation (a TMEM address holds the lane in bits 31..16 and the
//     column in bits 15..0).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define FA_CHECK_HD __host__ __device__ __forceinline__
#else
#define FA_CHECK_HD inline
#endif

namespace fa {

FA_CHECK_HD bool tma_load_ok(int x, uint32_t smem_dst) { return x >= 0 && (x & 7) == 0 && (smem_dst & 1023u) == 0; }

FA_CHECK_HD bool tma_store_ok(int x, int y, int z, uint32_t smem_src) {
  return x >= 0 && (x & 7) == 0 && y >= 0 && z >= 0 && (smem_src & 15u) == 0;
}

FA_CHECK_HD bool bulk_ok(uint32_t smem_dst, uint64_t global_src, uint32_t bytes) {
  return (smem_dst & 15u) == 0 && (global_src & 15u) == 0 && bytes > 0 && (bytes & 15u) == 0;
}

FA_CHECK_HD bool tmem_ok(uint32_t taddr, uint32_t cols, uint32_t warp) {
  return (taddr >> 16) == 32u * (warp & 3u) && (taddr & 0xFFFFu) + cols <= 512u;
}

}  // namespace fa
