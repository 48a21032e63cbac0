// sm103.cuh -- thin inline-PTX wrappers for the Blackwell (sm_103a) features
// the attention kernels use: mbarriers, TMA tensor loads, tensor memory
// (TMEM) allocation / loads / stores, and tcgen05 MMAs.
//
// Every wait on an mbarrier is bounded: after FA_WAIT_LIMIT_CYCLES it raises
// the CTA's abort flag (in shared memory) and returns false, so a broken
// pipeline ends the kernel instead of hanging the GPU. Kernels copy a raised
// flag into the caller-visible device status word before they exit.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "checks.h"
#include "kernels.h"

#ifndef FA_WAIT_LIMIT_CYCLES
#define FA_WAIT_LIMIT_CYCLES (4ll * 1000 * 1000 * 1000)  // ~2 s at 2 GHz
#endif

namespace fa {

// Checked build (FA_CHECKED): the TMA, bulk-copy and TMEM wrappers below test
// their arguments against the rules of their instruction first. A failed test
// sets a bit in this translation unit's check word and skips the instruction
// (nothing traps); every kernel copies a non-zero word into the status word
// (kErrCheck) at its end. Without FA_CHECKED the tests compile to nothing.
// The rules are the predicates of checks.h.
enum : uint32_t { kCheckTmaLoad = 1, kCheckTmaStore = 2, kCheckBulk = 4, kCheckTmem = 8 };
#ifdef FA_CHECKED
static __device__ uint32_t g_check_word;
#define FA_CHECK(cond, bit)              \
  do {                                   \
    if (!(cond)) {                       \
      atomicOr(&::fa::g_check_word, (bit)); \
      return;                            \
    }                                    \
  } while (0)
// For loads into a register array: the skipped load leaves zeros, so that
// the registers' earlier values need not stay live across the test.
#define FA_CHECK_LD(cond, bit, r, n)         \
  do {                                       \
    if (!(cond)) {                           \
      atomicOr(&::fa::g_check_word, (bit)); \
      _Pragma("unroll") for (int i_ = 0; i_ < (n); ++i_) r[i_] = 0u; \
      return;                                \
    }                                        \
  } while (0)
#else
#define FA_CHECK(cond, bit) \
  do {                      \
  } while (0)
#define FA_CHECK_LD(cond, bit, r, n) \
  do {                               \
  } while (0)
#endif

// The end of every kernel (after its closing barrier): a tripped check becomes
// the caller-visible status.
__device__ __forceinline__ void report_checks(int *status) {
#ifdef FA_CHECKED
  if (threadIdx.x == 0 && *reinterpret_cast<volatile uint32_t *>(&g_check_word) != 0u) atomicExch(status, kErrCheck);
#else
  (void)status;
#endif
}

// A 32x32b TMEM access of `cols` columns at taddr by the calling warp.
__device__ __forceinline__ bool tmem_access_ok(uint32_t taddr, uint32_t cols) {
  return tmem_ok(taddr, cols, threadIdx.x >> 5);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false
// (and raises the CTA abort flag) on timeout, or
// immediately once another thread of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *abort_flag) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (*reinterpret_cast<volatile int *>(abort_flag)) return false;
    if (clock64() - t0 > FA_WAIT_LIMIT_CYCLES) {
      *reinterpret_cast<volatile int *>(abort_flag) = 1;
      return false;
    }
  }
}

// Teardown wait: ignores the abort flag (it drains work already issued) but is
// still bounded in time. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > FA_WAIT_LIMIT_CYCLES) return false;
  }
  return true;
}

// Warp-collective form for roles whose next step is a .sync.aligned
// instruction: every lane gets the same answer, so a timeout seen by one lane
// never strands the others at a collective.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, int *abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

// ------------------------------------------------------------- CTA pairs
// A kernel launched with clusters of two CTAs (cluster rank 0 and 1) can run
// tcgen05 MMAs with M = 256 over both SMs: rank 0 issues them, each CTA holds
// half of A (its 128 rows) and half of B (N/2 rows or columns) at the same
// shared-memory offsets, and each CTA's tensor memory receives its 128 rows of
// the result. Barriers that gate the MMAs live in rank 0; the other CTA's
// copies and threads arrive on them through shared::cluster addresses.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the object at the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Every thread of both CTAs: release this CTA's prior writes (barrier
// initialisation included), acquire the other's.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on a barrier given by its shared::cluster address: this CTA's or the
// other's. Default (release, CTA-scope) semantics, like the waits: what a
// waiter needs from the arriving thread is its tensor-memory stores, which
// the arriving thread completes (tcgen05.wait::st) and orders before the
// arrival (tcgen05.fence::before_thread_sync), and the waiter orders its
// MMAs after the wait (tcgen05.fence::after_thread_sync). Cluster-scope
// release/acquire would put a fence in every arrival and every poll.
__device__ __forceinline__ void mbar_arrive_cl(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cl_addr) : "memory");
}

// 3-D tiled load into this CTA's shared memory whose byte count completes on
// a barrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cl, int x, int y,
                                                 int z) {
  FA_CHECK(tma_load_ok(x, smem_u32(dst)), kCheckTmaLoad);
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cl), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Tensor memory of a pair: the same columns in both CTAs. One warp of each
// CTA (the same warp) executes these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem] over the pair (M = 256).
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem] over the pair (each CTA's A rows in its own
// tensor memory).
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when
// all previously issued pair MMAs of this thread have completed.
__device__ __forceinline__ void mma_commit_pair_both(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// The same, on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
  FA_CHECK(tma_load_ok(x, smem_u32(dst)), kCheckTmaLoad);
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tiled store shared -> global, tracked as a bulk group of the issuing
// thread. Box elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y, int z) {
  FA_CHECK(tma_store_ok(x, y, z, smem_u32(src)), kCheckTmaStore);
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Prefetch one tile of a 3-D tensor map into L2 (no shared-memory copy, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  FA_CHECK(bulk_ok(smem_u32(dst), reinterpret_cast<uintptr_t>(src), bytes), kCheckBulk);
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk groups (the TMA stores): commit, then wait for the sources to be read.
// Groups are per issuing thread; the waits cover that thread's groups only.
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor-core reads of a tile written by threads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ tensor memory

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// TMEM addresses: lane in bits 31..16, column in bits 15..0.
// 32 lanes x 32 consecutive columns of 32 bits: lane i of the warp receives
// row (lane base + i), columns [col, col+32). Waits for completion.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  FA_CHECK_LD(tmem_access_ok(taddr, 32), kCheckTmem, r, 32);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 16 columns per lane; waits for completion.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  FA_CHECK_LD(tmem_access_ok(taddr, 16), kCheckTmem, r, 16);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Store 32 columns (32 x 32 bit per lane) and wait for completion.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  FA_CHECK(tmem_access_ok(taddr, 32), kCheckTmem);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 64 consecutive columns per lane in one instruction; waits for completion.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  FA_CHECK_LD(tmem_access_ok(taddr, 64), kCheckTmem, r, 64);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// 128 consecutive columns per lane in one instruction; waits for completion.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  FA_CHECK_LD(tmem_access_ok(taddr, 128), kCheckTmem, r, 128);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

// Store 64 consecutive columns per lane in one instruction and wait.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  FA_CHECK(tmem_access_ok(taddr, 64), kCheckTmem);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}

// Packed fp32 pairs (two lanes of one 64-bit register), sm_100+ only.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------------- tcgen05

// Instruction descriptor for kind::f16 with 16-bit A and B, fp32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format and 10-12 B format (0 = f16,
//   1 = bf16; A and B always share it), bit 15 A is MN-major, bit 16 B is
//   MN-major, bits 17-22 N/8, 24-28 M/16.
__host__ __device__ constexpr uint32_t idesc_16(int M, int N, bool a_mn_major, bool b_mn_major,
                                                bool f16) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte aligned buffer).
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 descriptor version (1),
//   61-63 layout (2 = 128-byte swizzle).
// K-major operand: rows of 128 bytes along K, SBO = 1024 (8-row groups),
//   LBO unused; stepping K by 16 elements adds 32 bytes to the start.
// MN-major operand: 64 MN-contiguous elements per 128-byte row, rows along
//   K; LBO = distance between 64-wide MN blocks, SBO = distance between
//   8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; A is M rows (lanes) x K, two bf16 per column.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 MMAs of this thread
// have completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// --------------------------------------------------------------- arithmetic

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float f16_to_f32(uint32_t h) {
  float f;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(f) : "r"(h));
  return f;
}

// The 16-bit element type of a kernel instance: bf16 (F16 = false) or f16.
// pack() rounds two floats to a packed pair (nearest even), lo()/hi() widen
// the low / high half of a packed pair back to float.
template <bool F16>
struct Elt;
template <>
struct Elt<false> {
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16x2(lo, hi); }
  __device__ static __forceinline__ float lo(uint32_t v) { return __uint_as_float(v << 16); }
  __device__ static __forceinline__ float hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
};
template <>
struct Elt<true> {
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) { return pack_f16x2(lo, hi); }
  __device__ static __forceinline__ float lo(uint32_t v) { return f16_to_f32(v & 0xFFFFu); }
  __device__ static __forceinline__ float hi(uint32_t v) { return f16_to_f32(v >> 16); }
};

// ------------------------------------------------------------------ dropout

// Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and
// Shaw ("Parallel random numbers: as easy as 1, 2, 3", SC 2011): ten rounds,
// each two 32 x 32 -> 64-bit products of counter words 0 and 2 with the
// paper's multipliers, a swap-and-xor of the halves with the key, and a Weyl
// increment of the key.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one widening multiply per product gives both halves
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k0, static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k1, static_cast<uint32_t>(p0));
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Dropout on the attention probabilities (struct Dropout, kernels.h):
// element (i, j) of head h (query i, key j) is kept iff byte j mod 4 of word
// i mod 4 of philox4x32_10((j/4, i/4, head_base + h, offset), seed) is >= t.

// Bit order inside a 32-key keep word (in the shared keep-bit rings and in the
// saved buffer): key b of the word is bit keep_bit(b) = 8 (b mod 4) + b / 4, so
// byte i holds keys i, 4 + i, ..., 28 + i. A 4 x 4 Philox group (keys
// 4c .. 4c + 3) then fills bit c of every byte with one shift, and a left
// shift of the word by 7 - c brings that group's bits to the top bits of the
// four bytes, where prmt's sign replication turns them into byte masks.
__host__ __device__ constexpr int keep_bit(int b) { return 8 * (b & 3) + (b >> 2); }

// 32 x 32 bit-matrix transpose across a warp: lane r passes row r (bit c =
// element (r, c)) and gets column `lane` back (bit r = element (r, lane)).
// Stage s swaps the off-diagonal s x s blocks of every 2s x 2s block: each
// lane sends its partner (lane ^ s) the half it gives up, already shifted
// into place, and keeps the other half.
__device__ __forceinline__ uint32_t warp_transpose_bits(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const uint32_t m = s == 16 ? 0x0000FFFFu : s == 8 ? 0x00FF00FFu : s == 4 ? 0x0F0F0F0Fu
                                                     : s == 2 ? 0x33333333u : 0x55555555u;
    const bool hi = lane & s;
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, hi ? x << s : x >> s, s);
    const uint32_t keep = hi ? ~m : m;
    x = (x & keep) | (recv & ~keep);
  }
  return x;
}

// Top bit of each byte of the result: byte of x >= t (the other bits are
// zero). t7 = (t mod 128) replicated in the four bytes, HIGH: t >= 128.
// In d = (x | 0x80) - (t mod 128) no byte borrows from the next, and the top
// bit of a byte of d says whether the low seven bits of x reach those of t;
// x >= t is then (top bit of x) or that bit when t < 128, and when t >= 128.
template <bool HIGH>
__device__ __forceinline__ uint32_t keep_top_bits(uint32_t x, uint32_t t7) {
  const uint32_t d = (x | 0x80808080u) - t7;
  return (HIGH ? (x & d) : (x | d)) & 0x80808080u;
}

// 0xFF in byte n of the result where bit 7 of byte (nibble n of sel) & 7 of
// x is set, else 0 (prmt with sign replication, every selector nibble >= 8).
__device__ __forceinline__ uint32_t byte_signs(uint32_t x, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0u), "r"(sel));
  return r;
}

// Keep bits of the 4 x 32 block of rows i0..i0+3 (i0 a multiple of 4) and
// keys j0..j0+31 (j0 a multiple of 4), drawn by one thread with no exchange:
// eight Philox calls, one per 4 x 4 group of the block. Component k of the
// result is row i0 + k, bit keep_bit(b) key j0 + b. HIGH says t >= 128.
template <bool HIGH>
__device__ __forceinline__ uint4 dropout_block_bits(const Dropout &dr, uint32_t h, int i0, int j0) {
  const uint32_t t7 = (dr.t & 0x7Fu) * 0x01010101u;
  uint32_t acc[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(j0 / 4 + c), static_cast<uint32_t>(i0 / 4),
                                             dr.head_base + h, dr.offset),
                                  dr.k0, dr.k1);
    const uint32_t x[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] += keep_top_bits<HIGH>(x[k], t7) >> (7 - c);  // bit 8 b + c: key 4 c + b
  }
  return make_uint4(acc[0], acc[1], acc[2], acc[3]);
}

// Register rebalancing between warpgroups (all four warps of a warpgroup
// execute the same one). The CTA's pool is its threads times the registers
// per thread at launch; the requests of all warpgroups must fit in it.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// ------------------------------------------------------- row-segment stores
// An accumulator read from TMEM leaves each lane holding one row, and the
// rows of a warp are 32 consecutive rows of the output, so a plain store from
// every lane writes 32 cache lines per instruction. These helpers first
// exchange 16-byte chunks inside groups of NC lanes (an NC x NC transpose in
// log2(NC) xor-shuffle stages), so that lane p of a group holds chunk p of each
// of the group's NC rows; store i then writes row i of every group, 32 / NC
// rows of NC * 16 contiguous bytes, whole 128-byte lines when NC = 8.

// w[4c .. 4c+3] is chunk c of the calling lane's row, which starts at `row`;
// rows are `stride` elements apart, and only rows less than `rows_left` past
// the calling lane's own are written. All 32 lanes must call it.
template <int NC>
__device__ __forceinline__ void store_row_chunks(uint32_t (&w)[4 * NC], uint16_t *row, int stride,
                                                 int rows_left) {
  const int p = lane_id() & (NC - 1);
#pragma unroll
  for (int m = 1; m < NC; m <<= 1) {
    // after this stage a lane's chunk k has row bit m from k and chunk bit m
    // from the lane: the lanes whose bit m differs from k's swap chunk k
    const bool up = (p & m) != 0;
#pragma unroll
    for (int k0 = 0; k0 < NC; ++k0) {
      if (k0 & m) continue;
      const int k1 = k0 | m;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t send = up ? w[4 * k0 + t] : w[4 * k1 + t];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
        if (up)
          w[4 * k0 + t] = recv;
        else
          w[4 * k1 + t] = recv;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NC; ++i)
    if (i - p < rows_left)
      *reinterpret_cast<uint4 *>(row + (i - p) * stride + p * 8) =
          make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// Columns [C0, COLS) of this lane's TMEM row (fp32, from taddr + C0), times
// `mul`, packed to 16-bit by E and stored at row[C0 ..] as above, in pieces of
// 64, 32 or 16 columns. COLS - C0 must be a multiple of 16.
template <class E, int COLS, int C0 = 0>
__device__ __forceinline__ void store_tmem_rows(uint32_t taddr, float mul, uint16_t *row, int stride,
                                                int rows_left) {
  if constexpr (C0 < COLS) {
    constexpr int kRem = COLS - C0;
    constexpr int kNC = kRem >= 64 ? 8 : kRem >= 32 ? 4 : 2;  // 16-byte chunks in this piece
    uint32_t w[4 * kNC];
#pragma unroll
    for (int c = 0; c < 8 * kNC; c += 16) {
      uint32_t rr[16];
      tmem_ld16(taddr + C0 + c, rr);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        w[c / 2 + u] = E::pack(__uint_as_float(rr[2 * u]) * mul, __uint_as_float(rr[2 * u + 1]) * mul);
    }
    store_row_chunks<kNC>(w, row + C0, stride, rows_left);
    store_tmem_rows<E, COLS, C0 + 8 * kNC>(taddr, mul, row, stride, rows_left);
  }
}

}  // namespace fa
