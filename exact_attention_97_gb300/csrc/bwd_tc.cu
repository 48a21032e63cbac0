// bwd_tc.cu -- exact attention backward on the sm_103a tensor cores, for
// 16-bit inputs (bf16 or f16; the element type is a template parameter).
//
// What it computes (pages): backward by recomputation, "Flash Attention
// 原理与实现", section "Backward 的 Tiling 策略": the probabilities are rebuilt
// from Q, K and the saved statistic, p = exp(s - L) ("research-attention"
// tutorial, section 04), then
//     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D)  with D_i = sum_c dO_ic O_ic,
//     dQ = scale dS K,  dK = scale dS^T Q.
// The blog's pitfalls item 3 names two ways to gather dQ across key blocks:
// atomic adds, or local results reduced globally. On GB300 the fp32
// reduction rate of L2 (about 3 TB/s) caps an atomic dQ far below the tensor
// cores, so dQ is formed locally instead: a second pass walks the key blocks
// of each query tile and keeps dQ in tensor memory. Each pass recomputes S
// and dP for its own reduction; nothing is accumulated in global memory.
//
// Three kernels on one stream:
//   1. bwd_prep  per query row, padded to whole 128-row tiles:
//                -L*log2(e) (-inf past N) and D_i = dO_i . O_i (0 past N).
//   2. bwd_dkdv  per (batch*head, 128-key block) item; query tiles of 128
//                rows stream through a TMA ring. Keys on the TMEM lanes:
//                  S^T = K Q^T, dP^T = V dO^T          (TMEM)
//                  dV += P^T dO   (P^T written over S^T in 16 bits, A from TMEM)
//                  dK += dS^T Q   (dS^T written over dP^T in 16 bits, A from TMEM)
//   3. bwd_dq    per (batch*head, 128-row query tile) item; key blocks
//                stream through a TMA ring. Queries on the TMEM lanes:
//                  S = Q K^T (double-buffered), dP = dO V^T   (TMEM)
//                  dQ += dS K     (dS read from TMEM in 16 bits)
// In both passes two warpgroups split the 128 columns of S and dP (64 each)
// for the elementwise work, one warp loads (two in the dQ pass), and two
// threads issue the MMAs, so that the barrier waits of either leave the
// tensor pipe fed by the other: in the dK/dV pass one per chain of products that reuse TMEM columns
// (S^T and dV; dP^T and dK), in the dQ pass one for S and dP and one for dQ,
// where S_{j+2} waits for dQ_j to complete before overwriting dS_j. Both
// passes are persistent: at most one CTA per SM walks a static list of items
// (tile_sched.h), and the rings and barrier phases carry over from item to
// item, so the next item's loads and first MMAs overlap the current item's
// last products and its epilogue. The dK/dV pass writes its results through
// per-warp shared-memory boxes and TMA stores, the dQ pass with whole-line
// row-segment stores. Head sizes 64, 96 and 128.
// With dropout both passes take the keep bits of each tile before its scores
// arrive: in DROP = kDrawn instances four more warps draw them
// (Philox4x32-10, sm103.cuh) into shared slots, DROP = kSaved instances read
// the ones the forward saved (separate instances, so that each is compiled
// for its own path). Given room in the workspace, the drawn dK/dV pass also
// writes its bits there in the saved layout, and a kSaved dQ pass reads them. dV takes P o Z / (1 - p), and dP is scaled by
// Z / (1 - p) before dS.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "kernels.h"
#include "tile_sched.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kBlk = 128;       // keys per block and query rows per tile
constexpr int kNoDrop = 0, kDrawn = 1, kSaved = 2;  // DROP: no dropout, keep bits drawn, keep bits saved
constexpr int kThreads = 384;   // 12 warps
constexpr int kThreadsMask = 512;  // dK/dV pass with drawn keep bits: warps 12-15 draw them
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void load_rows(uint8_t *dst, const CUtensorMap *map, uint64_t *bar,
                                          int D, int row, int bh) {
  for (int x = 0; x < D; x += 64) tma_load_3d(dst + (x / 64) * (kBlk * 128), map, bar, x, row, bh);
}


// TMEM column of k-step kk (16 keys or queries) of a 16-bit A operand that the
// two warpgroups wrote as packed pairs: warpgroup h (operand columns
// 64h..64h+63) writes 32 columns at 64h, inside the 64 score columns it read.
__device__ __forceinline__ uint32_t a_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// ------------------------------------------------------------------ kernel 1
// Per query row of a head padded to Np = 128*ceil(N/128) rows:
//   Lp = -L * log2(e) (so the passes form p = 2^(s*c + Lp)), -inf past N;
//   Dp = sum_c dO_ic O_ic, 0 past N.
// One group of prep_tpr(D) threads per row (D/8 rounded up to a power of
// two), one 16-byte load of O and of dO per thread that has one.
__host__ __device__ constexpr int prep_tpr(int D) { return D / 8 <= 8 ? 8 : (D / 8 <= 16 ? 16 : 32); }

template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t *__restrict__ o,
                                                       const uint16_t *__restrict__ dO,
                                                       const float *__restrict__ lse,
                                                       float *__restrict__ Lp, float *__restrict__ Dp,
                                                       int N, int Np, int64_t prow_total) {
  constexpr int kTpr = prep_tpr(D);  // threads per row
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t pr = gid / kTpr;  // padded row index
  const int part = static_cast<int>(gid % kTpr);
  const int64_t bh = pr / Np;
  const int i = static_cast<int>(pr % Np);
  const bool real = pr < prow_total && i < N;
  const int64_t r = bh * N + i;  // unpadded row
  float s = 0.f;
  if (real && part < D / 8) {
    const uint4 a = *reinterpret_cast<const uint4 *>(o + r * D + part * 8);
    const uint4 b = *reinterpret_cast<const uint4 *>(dO + r * D + part * 8);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      s = fmaf(Elt<F16>::lo(av[t]), Elt<F16>::lo(bv[t]), s);
      s = fmaf(Elt<F16>::hi(av[t]), Elt<F16>::hi(bv[t]), s);
    }
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (pr < prow_total && part == 0) {
    Dp[pr] = real ? s : 0.f;
    Lp[pr] = real ? -lse[r] * kLog2e : -INFINITY;
  }
}

// ------------------------------------------------------------------ kernel 2
//
// PAIR (d = 128, no dropout): a two-CTA cluster runs key blocks 2u and 2u + 1
// with M = 256 MMAs. Q_t and dO_t are each B of two products with different
// splits, so a CTA (rank r) holds four 16 KB halves per query tile: the rows
// 64r..64r+63 of Q and of dO (K-major, for S^T = K Q^T and dP^T = V dO^T) and
// the head columns 64r..64r+63 of all 128 rows of Q and of dO (MN-major, for
// dK += dS^T Q and dV += P^T dO). Same 64 KB per stage as one whole Q and dO.
template <int D, bool PAIR = false>
struct DkdvCfg {
  static_assert(!PAIR || D == 128, "the pair kernel covers d = 128");
  static constexpr int kDP = (D + 63) / 64 * 64;  // whole 64-column TMA boxes per row
  static constexpr int kStages = (kDP == 128) ? 2 : 3;
  static constexpr int kTileBytes = kBlk * kDP * 2;
  static constexpr int kSubBytes = kBlk * 128;  // 128 rows x 64 16-bit elements
  static constexpr int kHalfSub = kSubBytes / 2;  // 64 rows x 64 16-bit elements
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;
  static constexpr int kDO = kQ + kStages * kTileBytes;
  // pair: offsets of the four halves inside a stage of 2 * kTileBytes at kQ
  static constexpr int kPairStage = 2 * kTileBytes;
  static constexpr int kQRows = 0, kQCols = kTileBytes / 2, kDORows = kTileBytes, kDOCols = kTileBytes + kTileBytes / 2;
  // epilogue staging: per storing warp, two 32-row x 16-column buffers
  static constexpr int kStgBuf = 32 * 16 * 2;
  static constexpr int kStg = kDO + kStages * kTileBytes;
  static constexpr int kBytes = kStg + 8 * 2 * kStgBuf;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t tS = 0, tDP = 128, tDV = 256, tDK = 256 + D;  // TMEM columns
};

template <int D, bool F16, int DROP, bool PAIR>
__global__ void __launch_bounds__(DROP == kDrawn ? kThreadsMask : kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                    const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmdOh,
                    const float *__restrict__ Lp, const float *__restrict__ Dp, int N, int Nk,
                    const __grid_constant__ TileSched sched, float scale, float scale_log2, int causal,
                    const Dropout drop, int *status) {
  static_assert(!(PAIR && DROP), "the pair kernel has no dropout");
  using C = DkdvCfg<D, PAIR>;
  using E = Elt<F16>;
  constexpr int NST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  // ld_full: the L and D rows of a stage (in each CTA; a pair's qd_full is rank 0's)
  __shared__ uint64_t k_full, k_empty, v_full, v_empty, qd_full[NST], qd_empty[NST], ld_full[NST], s_full, dp_full,
      p_ready, ds_ready, done, drain, drain_kv;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ __align__(16) float Lst[NST][kBlk], Dst[NST][kBlk];  // per stage, by bulk copy
  // with dropout: the stage's 2 KB block of keep bits (128 query rows x 4
  // words), saved ones by bulk copy with the stage, drawn ones by the mask
  // warps (mk_full: written, mk_empty: the elementwise warps have read it)
  __shared__ __align__(16) uint32_t Mst[DROP != kNoDrop ? NST : 1][DROP != kNoDrop ? kBlk * 4 : 4];
  __shared__ uint64_t mk_full[DROP == kDrawn ? NST : 1], mk_empty[DROP == kDrawn ? NST : 1];

  const int warp = warp_id(), lane = lane_id();
  const int n_tiles_all = (N + kBlk - 1) / kBlk;
  const int Np = n_tiles_all * kBlk;
  // N query rows, Nk >= N keys under the causal mask; key j is seen by the
  // queries i >= j - (Nk - N) (bottom-right alignment). Schedule rank r is
  // unit r (a key block, or with PAIR the block pair 2r, 2r + 1 whose block
  // 2r + c runs on cluster rank c): low blocks see the most query tiles.
  const int off = Nk - N;
  const uint32_t crank = PAIR ? cluster_rank() : 0u;
  const int cta = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  auto block_of = [&](int rank) { return PAIR ? 2 * rank + static_cast<int>(crank) : rank; };
  // first query tile a unit visits: a pair starts at its lower block's (the
  // upper block's keys see the tiles before their own first one masked)
  auto first_tile = [&](int rank) {
    const int kb = PAIR ? 2 * rank : rank;
    return causal ? max(0, kb * kBlk - off) / kBlk : 0;
  };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&k_full, 1);
    mbar_init(&k_empty, 1);
    mbar_init(&v_full, 1);
    mbar_init(&v_empty, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&qd_full[s], 1);
      mbar_init(&qd_empty[s], 2);  // the two issuing threads' last readers of the stage
      mbar_init(&ld_full[s], 1);
    }
    mbar_init(&s_full, 1);
    mbar_init(&dp_full, 1);
    mbar_init(&p_ready, PAIR ? 2 * 8 : 256);  // pair: one arrival per elementwise warp of each CTA
    mbar_init(&ds_ready, PAIR ? 2 * 8 : 256);
    mbar_init(&done, 2);  // dV and dK, from the two issuing threads
    mbar_init(&drain, 1);
    mbar_init(&drain_kv, 1);
    if constexpr (DROP == kDrawn) {
      for (int s = 0; s < NST; ++s) {
        mbar_init(&mk_full[s], 4 * 32);
        mbar_init(&mk_empty[s], 8 * 32);
      }
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&tmem_base_s, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_base_s, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();  // the other CTA arrives on this one's barriers only once they exist
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // a pair's copies complete on rank 0's barriers, which only rank 0 drains
  const bool drains = !PAIR || crank == 0;
  // this CTA's K or V block on `bar` (rank 0's for a pair)
  auto load_block = [&](uint32_t dst, const CUtensorMap *map, uint64_t *bar, int row, int bh) {
    if constexpr (PAIR) {
      if (crank == 0) mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
      const uint32_t b0 = cluster_addr(bar, 0);
      for (int x = 0; x < D; x += 64) tma_load_3d_pair(smem + dst + (x / 64) * C::kSubBytes, map, b0, x, row, bh);
    } else {
      mbar_arrive_expect_tx(bar, C::kTileBytes);
      load_rows(smem + dst, map, bar, D, row, bh);
    }
  };

  // Every role walks the same items (key blocks); query tiles are counted
  // across items (g) for the ring and the per-tile barriers, items (it) for
  // the K, V and `done` barriers.
  // With drawn keep bits the block has 512 threads at 128 registers, and each
  // warpgroup resizes its share at the top of its branch: 56 for warps 0-3
  // (one producer and two issuing lanes), 168 for the elementwise warps, 112
  // for the mask warps (64512 of the 65536).
  if (warp < 4) {
  if constexpr (DROP == kDrawn) setmaxnreg_dec<56>();
  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // K of the next block loads as soon as the last S^T MMA of the current
    // one has completed, V after its last dP^T (both prefetched into L2 one
    // block ahead); query tiles stream on.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      bool ok = true;
      int g = 0, it = 0, rank, bh, kb = 0;
      auto load_qd = [&](int row) -> bool {
        const int st = g % NST;
        if (g >= NST && !mbar_wait(&qd_empty[st], ((g / NST) & 1) ^ 1, &abort_flag)) return false;
        if constexpr (PAIR) {
          // rows 64r.. of Q and dO, and head columns 64r.. of all their rows,
          // on rank 0's barrier; this CTA's L and D rows on its own
          if (crank == 0) mbar_arrive_expect_tx(&qd_full[st], 2 * 2 * C::kTileBytes);
          const uint32_t b0 = cluster_addr(&qd_full[st], 0);
          uint8_t *stage = smem + C::kQ + st * C::kPairStage;
          const int r64 = 64 * static_cast<int>(crank);
          for (int x = 0; x < D; x += 64) {
            tma_load_3d_pair(stage + C::kQRows + (x / 64) * C::kHalfSub, &tmQh, b0, x, row + r64, bh);
            tma_load_3d_pair(stage + C::kDORows + (x / 64) * C::kHalfSub, &tmdOh, b0, x, row + r64, bh);
          }
          tma_load_3d_pair(stage + C::kQCols, &tmQ, b0, r64, row, bh);
          tma_load_3d_pair(stage + C::kDOCols, &tmdO, b0, r64, row, bh);
          mbar_arrive_expect_tx(&ld_full[st], 2 * kBlk * 4);
          const size_t prow = static_cast<size_t>(bh) * Np + row;
          bulk_load(Lst[st], Lp + prow, kBlk * 4, &ld_full[st]);
          bulk_load(Dst[st], Dp + prow, kBlk * 4, &ld_full[st]);
        } else {
          constexpr bool saved = DROP == kSaved;
          mbar_arrive_expect_tx(&qd_full[st], 2 * C::kTileBytes + 2 * kBlk * 4 + (saved ? kBlk * 16 : 0));
          load_rows(smem + C::kQ + st * C::kTileBytes, &tmQ, &qd_full[st], D, row, bh);
          load_rows(smem + C::kDO + st * C::kTileBytes, &tmdO, &qd_full[st], D, row, bh);
          const size_t prow = static_cast<size_t>(bh) * Np + row;
          bulk_load(Lst[st], Lp + prow, kBlk * 4, &qd_full[st]);
          bulk_load(Dst[st], Dp + prow, kBlk * 4, &qd_full[st]);
          if constexpr (saved)  // the keep bits of query tile row / 128 against this key block
            bulk_load(Mst[st], reinterpret_cast<const uint8_t *>(drop.mask) + dropout_block(drop, bh, row / kBlk, kb),
                      kBlk * 16, &qd_full[st]);
        }
        ++g;
        return true;
      };
      int kdone = 0, vdone = 0;  // K / V loads issued
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        kb = block_of(rank);
        const int i_first = first_tile(rank), n_tiles = n_tiles_all - i_first;
        {  // the next block's K and V are read once: start them towards L2 now
          int nr, nbh, ns, k2 = k + 1;
          while ((ns = sched_item(sched, cta, k2, nr, nbh)) == kSkip) ++k2;
          if (ns == kItem)
            for (int x = 0; x < D; x += 64) {
              tma_prefetch_l2_3d(&tmK, x, block_of(nr) * kBlk, nbh);
              tma_prefetch_l2_3d(&tmV, x, block_of(nr) * kBlk, nbh);
            }
        }
        if (it > 0 && !mbar_wait(&k_empty, (it - 1) & 1, &abort_flag)) break;
        load_block(C::kK, &tmK, &k_full, kb * kBlk, bh);
        ++kdone;
        if (!load_qd(i_first * kBlk)) break;
        if (it > 0 && !mbar_wait(&v_empty, (it - 1) & 1, &abort_flag)) break;
        load_block(C::kV, &tmV, &v_full, kb * kBlk, bh);
        ++vdone;
        for (int t = 1; t < n_tiles; ++t)
          if (!load_qd((i_first + t) * kBlk)) { ok = false; break; }
        ++it;
      }
      if (drains) {
        if (kdone > 0) mbar_wait_drain(&k_full, (kdone - 1) & 1);
        if (vdone > 0) mbar_wait_drain(&v_full, (vdone - 1) & 1);
        for (int t = max(0, g - NST); t < g; ++t) mbar_wait_drain(&qd_full[t % NST], (t / NST) & 1);
      }
      if constexpr (PAIR)  // this CTA's own L / D copies
        for (int t = max(0, g - NST); t < g; ++t) mbar_wait_drain(&ld_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer: S^T and dV
    // Two threads issue, one per chain of products that reuse TMEM columns:
    // this one S^T_t and dV_t (P_t is written over S^T_t's columns, and
    // S^T_{t+1} overwrites them after dV_t has read them), warp 2 dP^T_t and
    // dK_t (likewise with dS_t over dP^T_t). Within a thread, issue order is
    // execution order, so a product that overwrites columns follows their
    // reader without waiting for it to complete; the two chains share no
    // TMEM columns. Q and dO stages are released by both threads (qd_empty
    // counts two), and the block's accumulators are done once both are.
    // With PAIR only rank 0 issues (M = 256 over both CTAs), and commits
    // arrive on the barrier of that name in both CTAs.
    if (lane == 0 && (!PAIR || crank == 0)) {
      constexpr uint32_t id_s = idesc_16(PAIR ? 2 * kBlk : kBlk, kBlk, false, false, F16);  // S^T
      constexpr uint32_t id_kv = idesc_16(PAIR ? 2 * kBlk : kBlk, D, false, true, F16);     // dV
      const uint32_t k_addr = smem_u32(smem + C::kK);
      auto commit = [](uint64_t *bar) {
        if constexpr (PAIR) mma_commit_pair_both(bar);
        else mma_commit(bar);
      };
      auto issue_s = [&](int gt) -> bool {  // S^T = K Q^T of global tile gt
        const int st = gt % NST;
        if (!mbar_wait(&qd_full[st], (gt / NST) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t q_addr = PAIR ? smem_u32(smem + C::kQ + st * C::kPairStage + C::kQRows)
                                     : smem_u32(smem + C::kQ + st * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::kSubBytes + (kk % 4) * 32;
          const uint32_t boff = (kk / 4) * (PAIR ? C::kHalfSub : C::kSubBytes) + (kk % 4) * 32;
          if constexpr (PAIR)
            mma_ss_pair(tmem + C::tS, sdesc_sw128(k_addr + off, 16, 1024), sdesc_sw128(q_addr + boff, 16, 1024),
                        id_s, kk > 0);
          else
            mma_ss(tmem + C::tS, sdesc_sw128(k_addr + off, 16, 1024), sdesc_sw128(q_addr + boff, 16, 1024), id_s,
                   kk > 0);
        }
        commit(&s_full);
        return true;
      };
      bool ok = true;
      int g = 0, it = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int n_tiles = n_tiles_all - first_tile(rank);
        if (!mbar_wait(&k_full, it & 1, &abort_flag) || !issue_s(g)) break;
        if (n_tiles == 1) commit(&k_empty);
        for (int t = 0; t < n_tiles; ++t, ++g) {
          const int st = g % NST;
          const uint32_t do_addr = PAIR ? smem_u32(smem + C::kQ + st * C::kPairStage + C::kDOCols)
                                        : smem_u32(smem + C::kDO + st * C::kTileBytes);
          // dV += P^T dO
          if (!mbar_wait(&p_ready, g & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk) {
            const uint64_t bdesc = sdesc_sw128(do_addr + kk * 2048, C::kSubBytes, 1024);
            if constexpr (PAIR)
              mma_ts_pair(tmem + C::tDV, tmem + C::tS + a_col(kk), bdesc, id_kv, (t > 0 || kk > 0) ? 1u : 0u);
            else
              mma_ts(tmem + C::tDV, tmem + C::tS + a_col(kk), bdesc, id_kv, (t > 0 || kk > 0) ? 1u : 0u);
          }
          commit(&qd_empty[st]);  // S^T_t completed before P_t existed; dV_t read dO_t
          if (t + 1 < n_tiles) {  // over the columns dV_t has just read
            if (!issue_s(g + 1)) { ok = false; break; }
            if (t + 2 == n_tiles) commit(&k_empty);  // the block's last S^T
          }
        }
        if (!ok) break;
        commit(&done);
        ++it;
      }
      if constexpr (PAIR) mma_commit_pair_local(&drain);
      else mma_commit(&drain);
      mbar_wait_drain(&drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------ MMA issuer: dP^T and dK
    if (lane == 0 && (!PAIR || crank == 0)) {
      constexpr uint32_t id_s = idesc_16(PAIR ? 2 * kBlk : kBlk, kBlk, false, false, F16);  // dP^T
      constexpr uint32_t id_kv = idesc_16(PAIR ? 2 * kBlk : kBlk, D, false, true, F16);     // dK
      const uint32_t v_addr = smem_u32(smem + C::kV);
      auto commit = [](uint64_t *bar) {
        if constexpr (PAIR) mma_commit_pair_both(bar);
        else mma_commit(bar);
      };
      auto issue_dp = [&](int gt) -> bool {  // dP^T = V dO^T of global tile gt
        const int st = gt % NST;
        if (!mbar_wait(&qd_full[st], (gt / NST) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t do_addr = PAIR ? smem_u32(smem + C::kQ + st * C::kPairStage + C::kDORows)
                                      : smem_u32(smem + C::kDO + st * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::kSubBytes + (kk % 4) * 32;
          const uint32_t boff = (kk / 4) * (PAIR ? C::kHalfSub : C::kSubBytes) + (kk % 4) * 32;
          if constexpr (PAIR)
            mma_ss_pair(tmem + C::tDP, sdesc_sw128(v_addr + off, 16, 1024), sdesc_sw128(do_addr + boff, 16, 1024),
                        id_s, kk > 0);
          else
            mma_ss(tmem + C::tDP, sdesc_sw128(v_addr + off, 16, 1024), sdesc_sw128(do_addr + boff, 16, 1024), id_s,
                   kk > 0);
        }
        commit(&dp_full);
        return true;
      };
      bool ok = true;
      int g = 0, it = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int n_tiles = n_tiles_all - first_tile(rank);
        if (!mbar_wait(&v_full, it & 1, &abort_flag) || !issue_dp(g)) break;
        if (n_tiles == 1) commit(&v_empty);
        for (int t = 0; t < n_tiles; ++t, ++g) {
          const int st = g % NST;
          const uint32_t q_addr = PAIR ? smem_u32(smem + C::kQ + st * C::kPairStage + C::kQCols)
                                       : smem_u32(smem + C::kQ + st * C::kTileBytes);
          // dK += dS^T Q
          if (!mbar_wait(&ds_ready, g & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk) {
            const uint64_t bdesc = sdesc_sw128(q_addr + kk * 2048, C::kSubBytes, 1024);
            if constexpr (PAIR)
              mma_ts_pair(tmem + C::tDK, tmem + C::tDP + a_col(kk), bdesc, id_kv, (t > 0 || kk > 0) ? 1u : 0u);
            else
              mma_ts(tmem + C::tDK, tmem + C::tDP + a_col(kk), bdesc, id_kv, (t > 0 || kk > 0) ? 1u : 0u);
          }
          commit(&qd_empty[st]);  // dP^T_t completed before dS_t existed; dK_t read Q_t
          if (t + 1 < n_tiles) {  // over the columns dK_t has just read
            if (!issue_dp(g + 1)) { ok = false; break; }
            if (t + 2 == n_tiles) commit(&v_empty);  // the block's last dP^T
          }
        }
        if (!ok) break;
        commit(&done);
        ++it;
      }
      if constexpr (PAIR) mma_commit_pair_local(&drain_kv);
      else mma_commit(&drain_kv);
      mbar_wait_drain(&drain_kv, 0);
    }
  }
  } else if (DROP == kDrawn && warp >= 12) {
    setmaxnreg_dec<112>();
    // -------------------------------------------------------------- keep bits
    // Warp 12 + c draws keys 32c..32c+31 of the block for query rows
    // 4 lane..4 lane + 3 of every query tile, into the slot of that tile's
    // Q/dO stage, in the layout of the saved keep bits; given drop.mask, it
    // also writes them there for the dQ pass.
    auto draw = [&](auto high) {
      constexpr bool kHigh = decltype(high)::value;
      const int wc = warp - 12;
      bool ok = true;
      int g = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int kb = block_of(rank);
        const int i_first = first_tile(rank), n_tiles = n_tiles_all - i_first;
        for (int t = 0; t < n_tiles; ++t, ++g) {
          const int st = g % NST;
          if (g >= NST && !mbar_wait_warp(&mk_empty[st], ((g / NST) & 1) ^ 1, &abort_flag)) {
            ok = false;
            break;
          }
          const uint4 bits = dropout_block_bits<kHigh>(drop, static_cast<uint32_t>(bh), (i_first + t) * kBlk + 4 * lane,
                                                       kb * kBlk + 32 * wc);
          *reinterpret_cast<uint4 *>(&Mst[st][wc * kBlk + 4 * lane]) = bits;
          mbar_arrive(&mk_full[st]);
          if (drop.mask)  // for the dQ pass, in the saved layout
            *reinterpret_cast<uint4 *>(drop.mask + dropout_block(drop, bh, i_first + t, kb) / 4 + wc * kBlk + 4 * lane) =
                bits;
        }
      }
    };
    if (drop.t >= 128u) draw(std::true_type{});
    else draw(std::false_type{});
  } else if (warp >= 4) {
    if constexpr (DROP == kDrawn) setmaxnreg_inc<168>();
    // -------------------------------------------- P, dS (warpgroup h: queries 64h..64h+63)
    const int h = (warp >= 8) ? 1 : 0;
    const int wq = warp & 3;
    const int kr = wq * 32 + lane;  // key row within the block (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint64_t cc = f2_pack(scale_log2, scale_log2);
    bool ok = true;
    int g = 0, it = 0, rank, bh;
    for (int k = 0; ok; ++k) {
      const int step = sched_item(sched, cta, k, rank, bh);
      if (step == kDone) break;
      if (step == kSkip) continue;
      const int kb = block_of(rank);
      const int i_first = first_tile(rank), n_tiles = n_tiles_all - i_first;
      const int key = kb * kBlk + kr;
      // queries below qmin see nothing of this key (causal); keys past Nk see nothing
      const int qmin0 = causal ? key - off : 0;
      for (int t = 0; t < n_tiles; ++t, ++g) {
        const uint32_t ph = g & 1;
        const int st = g % NST;
        const int q0 = (i_first + t) * kBlk + h * 64;  // first query of this warpgroup's columns
        const int qmin = (key >= Nk) ? (q0 + 64) : qmin0;
        uint32_t keep[2];  // dropout: keep bits of this key for the 64 queries
        if (!mbar_wait_warp(PAIR ? &ld_full[st] : &qd_full[st], (g / NST) & 1, &abort_flag)) {
          ok = false;
          break;
        }
        if constexpr (DROP == kDrawn) {
          if (!mbar_wait_warp(&mk_full[st], (g / NST) & 1, &abort_flag)) {
            ok = false;
            break;
          }
        }
        if constexpr (DROP != kNoDrop) {
          // the block's bits are stored by query row, 32 keys a word: the
          // warp's keys are word wq of each row, and the words wq of the
          // warpgroup's 64 rows are consecutive. Lane r takes rows r and
          // 32 + r, a transpose gives lane c the bits of bit position c,
          // and the key of bit position keep_bit(lane) is this lane's.
          const uint32_t *rows = &Mst[st][wq * kBlk + 64 * h];
#pragma unroll
          for (int w = 0; w < 2; ++w)
            keep[w] = __shfl_sync(0xffffffffu, warp_transpose_bits(rows[32 * w + lane]), keep_bit(lane));
          if constexpr (DROP == kDrawn) mbar_arrive(&mk_empty[st]);
        }
        const float4 *L4 = reinterpret_cast<const float4 *>(Lst[st] + h * 64);
        const float4 *D4 = reinterpret_cast<const float4 *>(Dst[st] + h * 64);
        if (!mbar_wait_warp(&s_full, ph, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t pk[32];
        float pf[64];  // P in fp32, for dS
        {
          uint32_t r[64];
          tmem_ld64(tmem + lane_addr + C::tS + h * 64, r);
          // P of query columns q0 + 2u, q0 + 2u + 1; the mask test only where
          // some of this row's 64 columns are masked (diagonal tiles, padding)
          auto p_pairs = [&](auto masked) {
#pragma unroll
            for (int u2 = 0; u2 < 16; ++u2) {
              const float4 nl = L4[u2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int u = 2 * u2 + e;
                const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])), cc,
                                           e ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y));
                float x0, x1;
                f2_unpack(x2, x0, x1);
                float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                if constexpr (decltype(masked)::value) {
                  if (q0 + 2 * u < qmin) p0 = 0.f;
                  if (q0 + 2 * u + 1 < qmin) p1 = 0.f;
                }
                pf[2 * u] = p0;
                pf[2 * u + 1] = p1;
                if constexpr (DROP == kNoDrop) pk[u] = E::pack(p0, p1);
              }
            }
          };
          if (q0 < qmin)
            p_pairs(std::true_type{});
          else
            p_pairs(std::false_type{});
          if constexpr (DROP != kNoDrop) {  // dV takes P o Z / (1 - p); dS takes P
#pragma unroll
            for (int u = 0; u < 32; ++u) {
              const uint32_t kb = keep[u >> 4] >> ((2 * u) & 31);
              // P o Z; the 1 / (1 - p) of dV is applied once, in the epilogue
              pk[u] = E::pack((kb & 1u) ? pf[2 * u] : 0.f, (kb & 2u) ? pf[2 * u + 1] : 0.f);
            }
            tmem_st32(tmem + lane_addr + C::tS + h * 64, pk);
          } else {
            tmem_st32(tmem + lane_addr + C::tS + h * 64, pk);
          }
        }
        tc_fence_before();
        if constexpr (PAIR) {  // one arrival per warp, on rank 0's barrier
          __syncwarp();
          if (lane == 0) mbar_arrive_cl(cluster_addr(&p_ready, 0));
        } else {
          mbar_arrive(&p_ready);
        }
        // dS^T = P^T o (dP^T - D); written in 16 bits
        // pairs over the dP^T columns this warpgroup has just read
        if (!mbar_wait_warp(&dp_full, ph, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t r[64];
          tmem_ld64(tmem + lane_addr + C::tDP + h * 64, r);
          uint32_t ds[32];
#pragma unroll
          for (int u2 = 0; u2 < 16; ++u2) {
            const float4 dd = D4[u2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int u = 2 * u2 + e;
              float dp0 = __uint_as_float(r[2 * u]), dp1 = __uint_as_float(r[2 * u + 1]);
              if constexpr (DROP != kNoDrop) {  // dP = (dO V^T) o Z / (1 - p)
                const uint32_t kb = keep[u >> 4] >> ((2 * u) & 31);
                dp0 = (kb & 1u) ? dp0 * drop.inv_keep : 0.f;
                dp1 = (kb & 2u) ? dp1 * drop.inv_keep : 0.f;
              }
              float d0, d1;  // P (dP - D), two lanes at a time
              f2_unpack(f2_mul(f2_pack(pf[2 * u], pf[2 * u + 1]),
                               f2_sub(f2_pack(dp0, dp1), e ? f2_pack(dd.z, dd.w) : f2_pack(dd.x, dd.y))),
                        d0, d1);
              ds[u] = E::pack(d0, d1);
            }
          }
          tmem_st32(tmem + lane_addr + C::tDP + h * 64, ds);
        }
        tc_fence_before();
        if constexpr (PAIR) {
          __syncwarp();
          if (lane == 0) mbar_arrive_cl(cluster_addr(&ds_ready, 0));
        } else {
          mbar_arrive(&ds_ready);
        }
      }
      // epilogue: warpgroup 0 stores dV, warpgroup 1 stores dK (times scale).
      // Each warp stages 32 rows x 16 columns at a time in shared memory (the
      // layout of the store map's 32-byte swizzle: the two 16-byte halves of
      // row r swap when bit 2 of r is set) and one lane writes the box with a
      // TMA store, alternating two buffers; rows past Nk are not written.
      if (!ok || !mbar_wait_warp(&done, it & 1, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const uint32_t col = h ? C::tDK : C::tDV;
        const float mul = h ? scale : (DROP != kNoDrop ? drop.inv_keep : 1.f);  // dV takes the dropout's 1 / (1 - p) here
        const CUtensorMap *map = h ? &tmdK : &tmdV;
        uint8_t *stg = smem + C::kStg + (warp - 4) * 2 * C::kStgBuf;
        const int row0 = kb * kBlk + wq * 32;
        const int sw = (lane >> 2) & 1;
#pragma unroll 1
        for (int ch = 0; ch < D / 16; ++ch) {
          uint8_t *buf = stg + (ch & 1) * C::kStgBuf;
          if (lane == 0) {
            if (ch == 0) bulk_wait_read_all();  // the previous block's stores have read both buffers
            else bulk_wait_read_le1();          // the store of chunk ch - 2 has read this buffer
          }
          __syncwarp();
          uint32_t r[16];
          tmem_ld16(tmem + lane_addr + col + ch * 16, r);
          uint32_t pk2[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            pk2[u] = E::pack(__uint_as_float(r[2 * u]) * mul, __uint_as_float(r[2 * u + 1]) * mul);
          uint4 *row = reinterpret_cast<uint4 *>(buf + lane * 32);
          row[sw] = make_uint4(pk2[0], pk2[1], pk2[2], pk2[3]);
          row[sw ^ 1] = make_uint4(pk2[4], pk2[5], pk2[6], pk2[7]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < Nk) {
            tma_store_3d(map, buf, ch * 16, row0, bh);
            bulk_commit();
          }
        }
      }
      ++it;
    }
  }

  // the staged dK / dV stores complete before the CTA's shared memory goes
  if (warp >= 4 && lane == 0) bulk_wait_all();
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();  // rank 0 has drained every copy and MMA that touches either CTA
  else
    __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && abort_flag) atomicExch(status, kErrTimeout);
  report_checks(status);
}

// ------------------------------------------------------------------ kernel 3
// K_j is needed until dQ_j, V_j only until dP_j, so they have rings of their
// own (K one deeper) and loaders of their own: the next K blocks can be in
// flight while dQ of the current one runs.
//
// PAIR (d = 128, no dropout): a two-CTA cluster runs query tiles 2u and 2u + 1
// with M = 256 MMAs, and each CTA holds half of each key block's operands:
// for S = Q K^T its keys 64r..64r+63 (rank r; K-major, two 8 KB sub-tiles),
// for dQ += dS K all 128 keys of head columns 64r..64r+63 (MN-major, one
// 16 KB sub-tile) -- a K stage holds both, 32 KB -- and for dP = dO V^T the
// value rows 64r..64r+63 (16 KB).
// DRAWN (dropout with drawn keep bits): at 128 columns the K ring is one
// stage shorter, which leaves room for the mask warps' ring of keep bits.
template <int D, bool PAIR = false, bool DRAWN = false>
struct DqCfg {
  static_assert(!PAIR || D == 128, "the pair kernel covers d = 128");
  static constexpr int kDP = (D + 63) / 64 * 64;  // whole 64-column TMA boxes per row
  static constexpr int kKStages = (kDP == 128) ? (DRAWN ? 2 : 3) : 4;
  static constexpr int kVStages = PAIR ? 3 : ((kDP == 128) ? 2 : 3);
  static constexpr int kTileBytes = kBlk * kDP * 2;
  static constexpr int kSubBytes = kBlk * 128;
  static constexpr int kHalfSub = kSubBytes / 2;           // 64 rows x 64 columns
  static constexpr int kKRowsBytes = PAIR ? kTileBytes / 2 : kTileBytes;  // keys 64r.. (or the whole tile)
  static constexpr int kKStageBytes = PAIR ? kTileBytes : kTileBytes;     // pair: rows half + columns half
  static constexpr int kVStageBytes = PAIR ? kTileBytes / 2 : kTileBytes;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kTileBytes;
  static constexpr int kV = kK + kKStages * kKStageBytes;
  static constexpr int kBytes = kV + kVStages * kVStageBytes;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t tS = 0, tDP = 256, tDQ = 384;  // S buffers at 0 and 128
};

template <int D, bool F16, int DROP, bool PAIR>
__global__ void __launch_bounds__(DROP == kDrawn ? kThreadsMask : kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmKh, const __grid_constant__ CUtensorMap tmVh,
                  const float *__restrict__ Lp, const float *__restrict__ Dp,
                  uint16_t *__restrict__ dq, int N, int Nk, const __grid_constant__ TileSched sched, float scale,
                  float scale_log2, int causal, const Dropout drop, int *status) {
  static_assert(!(PAIR && DROP), "the pair kernel has no dropout");
  using C = DqCfg<D, PAIR, DROP == kDrawn>;
  using E = Elt<F16>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  // drawn keep bits: a ring of (query tile, key block) blocks from the mask
  // warps, in the layout of the saved bits (mk_full: written, mk_empty: read)
  constexpr int kMSlots = 4;
  __shared__ __align__(16) uint32_t Mst[DROP == kDrawn ? kMSlots : 1][DROP == kDrawn ? kBlk * 4 : 4];
  __shared__ uint64_t mk_full[DROP == kDrawn ? kMSlots : 1], mk_empty[DROP == kDrawn ? kMSlots : 1];
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t q_full, q_empty, do_full, do_empty, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
      s_full[2], dp_full, ds_ready[2], sfree[2], done, drain, drain_q;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int n_tiles = (N + kBlk - 1) / kBlk;
  const int Np = n_tiles * kBlk;
  const int off = Nk - N;  // bottom-right causal alignment, as in the forward
  const int n_kb_all = (Nk + kBlk - 1) / kBlk;
  // A schedule unit is a query tile, or with PAIR a tile pair whose tile
  // 2u + r runs on cluster rank r (both CTAs walk the same units). Schedule
  // rank 0 is a head's most expensive unit (the last one under the causal
  // mask).
  const uint32_t crank = PAIR ? cluster_rank() : 0u;
  const int cta = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  auto unit_of = [&](int rank) { return causal ? sched.nt - 1 - rank : rank; };
  auto qtile_of = [&](int rank) { return PAIR ? 2 * unit_of(rank) + static_cast<int>(crank) : unit_of(rank); };
  auto kblocks_q = [&](int qt) {
    return causal ? min(n_kb_all, (qt * kBlk + kBlk - 1 + off) / kBlk + 1) : n_kb_all;
  };
  // key blocks of a unit: a pair walks those of its upper tile (the rows of
  // the lower tile see the extra block fully masked: p = 0 there)
  auto kblocks = [&](int rank) { return kblocks_q(PAIR ? 2 * unit_of(rank) + 1 : unit_of(rank)); };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    mbar_init(&do_full, 1);
    mbar_init(&do_empty, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&dp_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ds_ready[b], PAIR ? 2 * 8 : 256);  // pair: one arrival per elementwise warp of each CTA
      mbar_init(&sfree[b], 1);
    }
    mbar_init(&done, 1);
    mbar_init(&drain, 1);
    mbar_init(&drain_q, 1);
    if constexpr (DROP == kDrawn) {
      for (int s = 0; s < kMSlots; ++s) {
        mbar_init(&mk_full[s], 4 * 32);
        mbar_init(&mk_empty[s], 8 * 32);
      }
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&tmem_base_s, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_base_s, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();  // the other CTA arrives on this one's barriers only once they exist
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // a pair's copies complete on rank 0's barriers, which only rank 0 drains
  const bool drains = !PAIR || crank == 0;
  // this CTA's rows tile: Q or dO of `row` into smem + dst, counted on `bar`
  auto load_tile = [&](uint32_t dst, const CUtensorMap *map, uint64_t *bar, int row, int bh) {
    if constexpr (PAIR) {
      if (crank == 0) mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
      const uint32_t b0 = cluster_addr(bar, 0);
      for (int x = 0; x < D; x += 64) tma_load_3d_pair(smem + dst + (x / 64) * C::kSubBytes, map, b0, x, row, bh);
    } else {
      mbar_arrive_expect_tx(bar, C::kTileBytes);
      load_rows(smem + dst, map, bar, D, row, bh);
    }
  };

  // Every role walks the same items (query tiles); key blocks are counted
  // across items (g) for the K/V rings, the S buffers and the per-block
  // barriers, items (it) for the Q, dO and `done` barriers.
  // With drawn keep bits the block has 512 threads at 128 registers, split as
  // in the dK/dV pass: 56 for warps 0-3, 168 for the elementwise warps, 112 for
  // the mask warps.
  if (warp < 4) {
  if constexpr (DROP == kDrawn) setmaxnreg_dec<56>();
  if (warp == 0) {
    // ------------------------------------------------------- loader: Q, dO, K
    // Q of the next tile loads once the last S MMA of the current one has
    // completed, dO once its last dP MMA has (both prefetched into L2 one
    // tile ahead); the K ring runs on.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmdO);
      bool ok = true;
      int g = 0, nq = 0, ndo = 0, rank, bh;  // K blocks, Q tiles, dO tiles issued
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int qt = qtile_of(rank), n_kb = kblocks(rank);
        {  // the next tile's Q and dO are read once: start them towards L2 now
          int nr, nbh, ns, k2 = k + 1;
          while ((ns = sched_item(sched, cta, k2, nr, nbh)) == kSkip) ++k2;
          if (ns == kItem)
            for (int x = 0; x < D; x += 64) {
              tma_prefetch_l2_3d(&tmQ, x, qtile_of(nr) * kBlk, nbh);
              tma_prefetch_l2_3d(&tmdO, x, qtile_of(nr) * kBlk, nbh);
            }
        }
        if (nq > 0 && !mbar_wait(&q_empty, (nq - 1) & 1, &abort_flag)) break;
        load_tile(C::kQ, &tmQ, &q_full, qt * kBlk, bh);
        ++nq;
        for (int j = 0; j < n_kb; ++j, ++g) {
          const int st = g % KS;
          if (g >= KS && !mbar_wait(&k_empty[st], ((g / KS) & 1) ^ 1, &abort_flag)) { ok = false; break; }
          if constexpr (PAIR) {
            // keys 64r..64r+63 (for S) and head columns 64r..64r+63 of all
            // the block's keys (for dQ), both on rank 0's barrier
            if (crank == 0) mbar_arrive_expect_tx(&k_full[st], 2 * C::kKStageBytes);
            const uint32_t b0 = cluster_addr(&k_full[st], 0);
            uint8_t *dst = smem + C::kK + st * C::kKStageBytes;
            for (int x = 0; x < D; x += 64)
              tma_load_3d_pair(dst + (x / 64) * C::kHalfSub, &tmKh, b0, x, j * kBlk + 64 * static_cast<int>(crank),
                               bh);
            tma_load_3d_pair(dst + C::kKRowsBytes, &tmK, b0, 64 * static_cast<int>(crank), j * kBlk, bh);
          } else {
            mbar_arrive_expect_tx(&k_full[st], C::kTileBytes);
            load_rows(smem + C::kK + st * C::kKStageBytes, &tmK, &k_full[st], D, j * kBlk, bh);
          }
          if (j == 0) {  // dO after the first K block: S_0 needs Q and K_0 first
            if (ndo > 0 && !mbar_wait(&do_empty, (ndo - 1) & 1, &abort_flag)) { ok = false; ++g; break; }
            load_tile(C::kDO, &tmdO, &do_full, qt * kBlk, bh);
            ++ndo;
          }
        }
      }
      // teardown: every issued copy must land before the CTA's memory is released
      if (drains) {
        if (nq > 0) mbar_wait_drain(&q_full, (nq - 1) & 1);
        if (ndo > 0) mbar_wait_drain(&do_full, (ndo - 1) & 1);
        for (int j = max(0, g - KS); j < g; ++j) mbar_wait_drain(&k_full[j % KS], (j / KS) & 1);
      }
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------------- loader: V
    if (lane == 0) {
      tma_prefetch_desc(&tmV);
      bool ok = true;
      int g = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int n_kb = kblocks(rank);
        for (int j = 0; j < n_kb; ++j, ++g) {
          const int st = g % VS;
          if (g >= VS && !mbar_wait(&v_empty[st], ((g / VS) & 1) ^ 1, &abort_flag)) { ok = false; break; }
          if constexpr (PAIR) {  // value rows 64r..64r+63, on rank 0's barrier
            if (crank == 0) mbar_arrive_expect_tx(&v_full[st], 2 * C::kVStageBytes);
            const uint32_t b0 = cluster_addr(&v_full[st], 0);
            for (int x = 0; x < D; x += 64)
              tma_load_3d_pair(smem + C::kV + st * C::kVStageBytes + (x / 64) * C::kHalfSub, &tmVh, b0, x,
                               j * kBlk + 64 * static_cast<int>(crank), bh);
          } else {
            mbar_arrive_expect_tx(&v_full[st], C::kTileBytes);
            load_rows(smem + C::kV + st * C::kVStageBytes, &tmV, &v_full[st], D, j * kBlk, bh);
          }
        }
      }
      if (drains)
        for (int j = max(0, g - VS); j < g; ++j) mbar_wait_drain(&v_full[j % VS], (j / VS) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer: S, dP
    // Per tile: S_0, dP_0, S_1, then per key block j: dP_{j+1}, S_{j+2}. The
    // dQ products come from warp 2, so neither thread's barrier waits leave
    // the tensor pipe idle. Two issuing threads give no order between their
    // MMAs: S_{g+2} reuses the buffer of dS_g and so waits for dQ_g to
    // complete (sfree), and dP_{g+1} reuses the dP columns, which the
    // elementwise warps have read once dS_g is ready.
    // With PAIR only rank 0 issues (M = 256 over both CTAs), and commits
    // arrive on the barrier of that name in both CTAs.
    if (lane == 0 && (!PAIR || crank == 0)) {
      constexpr uint32_t id_s = idesc_16(PAIR ? 2 * kBlk : kBlk, kBlk, false, false, F16);  // S, dP
      constexpr int kBSub = PAIR ? C::kHalfSub : C::kSubBytes;  // B operand sub-tile stride
      const uint32_t q_addr = smem_u32(smem + C::kQ), do_addr = smem_u32(smem + C::kDO);
      auto commit = [](uint64_t *bar) {
        if constexpr (PAIR) mma_commit_pair_both(bar);
        else mma_commit(bar);
      };
      auto mma = [](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (PAIR) mma_ss_pair(d, a, b, id, acc);
        else mma_ss(d, a, b, id, acc);
      };
      auto issue_s = [&](int gj) -> bool {  // S of global block gj = Q K^T into buffer gj&1
        if (gj >= 2 && !mbar_wait(&sfree[gj & 1], ((gj >> 1) - 1) & 1, &abort_flag)) return false;
        const int st = gj % KS;
        if (!mbar_wait(&k_full[st], (gj / KS) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + C::kK + st * C::kKStageBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk / 4) * C::kSubBytes + (kk % 4) * 32, boff = (kk / 4) * kBSub + (kk % 4) * 32;
          mma(tmem + C::tS + (gj & 1) * 128, sdesc_sw128(q_addr + aoff, 16, 1024),
              sdesc_sw128(k_addr + boff, 16, 1024), id_s, kk > 0);
        }
        commit(&s_full[gj & 1]);
        return true;
      };
      auto issue_dp = [&](int gj) -> bool {  // dP = dO V^T
        const int st = gj % VS;
        if (!mbar_wait(&v_full[st], (gj / VS) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + C::kV + st * C::kVStageBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk / 4) * C::kSubBytes + (kk % 4) * 32, boff = (kk / 4) * kBSub + (kk % 4) * 32;
          mma(tmem + C::tDP, sdesc_sw128(do_addr + aoff, 16, 1024), sdesc_sw128(v_addr + boff, 16, 1024), id_s,
              kk > 0);
        }
        commit(&dp_full);
        commit(&v_empty[st]);
        return true;
      };
      bool ok = true;
      int g = 0, it = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int n_kb = kblocks(rank);
        if (!mbar_wait(&q_full, it & 1, &abort_flag) || !issue_s(g)) break;
        if (n_kb == 1) commit(&q_empty);
        if (!mbar_wait(&do_full, it & 1, &abort_flag) || !issue_dp(g)) break;
        if (n_kb == 1) commit(&do_empty);
        if (n_kb > 1) {
          if (!issue_s(g + 1)) break;
          if (n_kb == 2) commit(&q_empty);
        }
        for (int j = 0; j < n_kb; ++j, ++g) {
          if (!mbar_wait(&ds_ready[g & 1], (g >> 1) & 1, &abort_flag)) { ok = false; break; }
          if (j + 1 < n_kb) {  // dP_j has been read into dS_j
            tc_fence_after();
            if (!issue_dp(g + 1)) { ok = false; break; }
            if (j + 2 == n_kb) commit(&do_empty);  // the tile's last dP
          }
          if (j + 2 < n_kb) {
            if (!issue_s(g + 2)) { ok = false; break; }
            if (j + 3 == n_kb) commit(&q_empty);  // the tile's last S
          }
        }
        if (!ok) break;
        ++it;
      }
      if constexpr (PAIR) mma_commit_pair_local(&drain);
      else mma_commit(&drain);
      mbar_wait_drain(&drain, 0);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------- MMA issuer: dQ
    // dQ += dS_j K_j per key block (A = dS_j, 16-bit in TMEM; B = K_j
    // MN-major). The first of a tile overwrites the accumulator: it waits for
    // dS_0, which the elementwise warps only produce after storing the
    // previous tile's dQ.
    if (lane == 0 && (!PAIR || crank == 0)) {
      constexpr uint32_t id_q = idesc_16(PAIR ? 2 * kBlk : kBlk, D, false, true, F16);
      bool ok = true;
      int g = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int n_kb = kblocks(rank);
        for (int j = 0; j < n_kb; ++j, ++g) {
          const int st = g % KS;
          if (!mbar_wait(&ds_ready[g & 1], (g >> 1) & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
          // the pair's B: this CTA's head columns of all the block's keys (MN-major)
          const uint32_t k_addr = smem_u32(smem + C::kK + st * C::kKStageBytes) + (PAIR ? C::kKRowsBytes : 0);
#pragma unroll
          for (int kk = 0; kk < kBlk / 16; ++kk) {
            const uint64_t bdesc = sdesc_sw128(k_addr + kk * 2048, C::kSubBytes, 1024);
            if constexpr (PAIR)
              mma_ts_pair(tmem + C::tDQ, tmem + C::tS + (g & 1) * 128 + a_col(kk), bdesc, id_q,
                          (j > 0 || kk > 0) ? 1u : 0u);
            else
              mma_ts(tmem + C::tDQ, tmem + C::tS + (g & 1) * 128 + a_col(kk), bdesc, id_q,
                     (j > 0 || kk > 0) ? 1u : 0u);
          }
          // S_g completed before dS_g existed, so K_g is free once dQ_g is
          if constexpr (PAIR) {
            mma_commit_pair_both(&k_empty[st]);
            mma_commit_pair_local(&sfree[g & 1]);  // only rank 0's S issuer waits on it
          } else {
            mma_commit(&k_empty[st]);
            mma_commit(&sfree[g & 1]);
          }
        }
        if (!ok) break;
        if constexpr (PAIR) mma_commit_pair_both(&done);
        else mma_commit(&done);
      }
      if constexpr (PAIR) mma_commit_pair_local(&drain_q);
      else mma_commit(&drain_q);
      mbar_wait_drain(&drain_q, 0);
    }
  }
  } else if (DROP == kDrawn && warp >= 12) {
    setmaxnreg_dec<112>();
    // -------------------------------------------------------------- keep bits
    // Warp 12 + c draws keys 32c..32c+31 of every key block for rows
    // 4 lane..4 lane + 3 of the query tile, into ring slot g mod kMSlots.
    auto draw = [&](auto high) {
      constexpr bool kHigh = decltype(high)::value;
      const int wc = warp - 12;
      bool ok = true;
      int g = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int qt = qtile_of(rank), n_kb = kblocks(rank);
        for (int j = 0; j < n_kb; ++j, ++g) {
          const int m = g % kMSlots;
          if (g >= kMSlots && !mbar_wait_warp(&mk_empty[m], ((g / kMSlots) & 1) ^ 1, &abort_flag)) {
            ok = false;
            break;
          }
          const uint4 bits = dropout_block_bits<kHigh>(drop, static_cast<uint32_t>(bh), qt * kBlk + 4 * lane,
                                                       j * kBlk + 32 * wc);
          *reinterpret_cast<uint4 *>(&Mst[m][wc * kBlk + 4 * lane]) = bits;
          mbar_arrive(&mk_full[m]);
        }
      }
    };
    if (drop.t >= 128u) draw(std::true_type{});
    else draw(std::false_type{});
  } else if (warp >= 4) {
    if constexpr (DROP == kDrawn) setmaxnreg_inc<168>();
    // ------------------------------------------ P, dS (warpgroup h: keys 64h..64h+63 of a block)
    const int h = (warp >= 8) ? 1 : 0;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row within the tile (TMEM lane)
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint64_t cc = f2_pack(scale_log2, scale_log2);
    // this row's -L log2(e) and D of item k (padded rows hold -inf and 0),
    // loaded one item ahead so the epilogue hides their latency
    auto row_terms = [&](int k, float &nl, float &drow) {
      int rk, hb, st;
      while ((st = sched_item(sched, cta, k, rk, hb)) == kSkip) ++k;
      if (st == kDone) return;
      const int qt = qtile_of(rk);
      if (qt >= n_tiles) {  // a pair's second tile past the last one: no rows
        nl = -INFINITY;
        drow = 0.f;
        return;
      }
      const size_t prow = static_cast<size_t>(hb) * Np + qt * kBlk + r;
      nl = Lp[prow];
      drow = Dp[prow];
    };
    float nl_next = 0.f, drow_next = 0.f;
    row_terms(0, nl_next, drow_next);
    bool ok = true;
    int g = 0, it = 0, rank, bh;
    for (int k = 0; ok; ++k) {
      const int step = sched_item(sched, cta, k, rank, bh);
      if (step == kDone) break;
      if (step == kSkip) continue;
      const int qt = qtile_of(rank), n_kb = kblocks(rank);
      const int q = qt * kBlk + r;
      const float nl = nl_next, drow = drow_next;
      const uint64_t nn = f2_pack(nl, nl), dd2 = f2_pack(drow, drow), ndd2 = f2_pack(-drow, -drow);
      const int kvis = causal ? min(Nk, q + 1 + off) : Nk;  // keys below kvis are visible
      for (int j = 0; j < n_kb; ++j, ++g) {
        const uint32_t sb = C::tS + (g & 1) * 128 + h * 64;
        const int limit = kvis - (j * kBlk + h * 64);  // columns at or past limit are masked
        uint32_t keep[2];  // dropout: keep bits of this row for the 64 keys, read while S is in flight
        // (bit keep_bit(b) of keep[w]: key j * 128 + 64 h + 32 w + b)
        if constexpr (DROP == kSaved) {  // saved by the forward: words 2h, 2h + 1 of this row in block (qt, j)
          const uint32_t *blk = drop.mask + dropout_block(drop, bh, qt, j) / 4 + r;
          keep[0] = __ldg(blk + (2 * h) * kBlk);
          keep[1] = __ldg(blk + (2 * h + 1) * kBlk);
        } else if constexpr (DROP == kDrawn) {  // from the mask warps: the same words of ring slot g mod kMSlots
          const int m = g % kMSlots;
          if (!mbar_wait_warp(&mk_full[m], (g / kMSlots) & 1, &abort_flag)) { ok = false; break; }
          keep[0] = Mst[m][(2 * h) * kBlk + r];
          keep[1] = Mst[m][(2 * h + 1) * kBlk + r];
          mbar_arrive(&mk_empty[m]);
        }
        if (!mbar_wait_warp(&s_full[g & 1], (g >> 1) & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        float p[64];
        {
          uint32_t rr[64];
          tmem_ld64(tmem + lane_addr + sb, rr);
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(rr[2 * u]), __uint_as_float(rr[2 * u + 1])), cc, nn);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            p[2 * u] = ex2_approx(x0);
            p[2 * u + 1] = ex2_approx(x1);
          }
          if (limit < 64) {
#pragma unroll
            for (int u = 0; u < 64; ++u)
              if (u >= limit) p[u] = 0.f;
          }
        }
        if (!mbar_wait_warp(&dp_full, g & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t rr[64];
          tmem_ld64(tmem + lane_addr + C::tDP + h * 64, rr);
          uint32_t ds[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float dp0 = __uint_as_float(rr[2 * u]), dp1 = __uint_as_float(rr[2 * u + 1]);
            float d0, d1;  // p (dP - D), two lanes at a time
            if constexpr (DROP != kNoDrop) {  // dP = (dO V^T) o Z / (1 - p): dP m - D with m = Z / (1 - p)
              // keys 2u, 2u + 1 (bytes e, e + 1 of the word, bit c): shifted
              // left by 7 - c they are byte tops, and prmt makes each a
              // 32-bit mask for the bits of 1 / (1 - p)
              const int b = (2 * u) & 31, c = b >> 2, e = b & 3;
              const uint32_t y = keep[u >> 4] << (7 - c), ik = __float_as_uint(drop.inv_keep);
              const uint64_t m2 = f2_pack(__uint_as_float(byte_signs(y, (8 + e) * 0x1111u) & ik),
                                          __uint_as_float(byte_signs(y, (9 + e) * 0x1111u) & ik));
              f2_unpack(f2_mul(f2_pack(p[2 * u], p[2 * u + 1]), f2_fma(f2_pack(dp0, dp1), m2, ndd2)), d0, d1);
            } else {
              f2_unpack(f2_mul(f2_pack(p[2 * u], p[2 * u + 1]), f2_sub(f2_pack(dp0, dp1), dd2)), d0, d1);
            }
            ds[u] = E::pack(d0, d1);
          }
          tmem_st32(tmem + lane_addr + sb, ds);  // over scores already read
        }
        tc_fence_before();
        if constexpr (PAIR) {  // one arrival per warp, on rank 0's barrier
          __syncwarp();
          if (lane == 0) mbar_arrive_cl(cluster_addr(&ds_ready[g & 1], 0));
        } else {
          mbar_arrive(&ds_ready[g & 1]);
        }
      }
      if (ok) row_terms(k + 1, nl_next, drow_next);
      // epilogue: dQ = scale * accumulator; warpgroup h stores head columns
      // [hD/2, hD/2 + D/2) with whole-line row-segment stores
      if (!ok || !mbar_wait_warp(&done, it & 1, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      store_tmem_rows<E, D / 2>(tmem + lane_addr + C::tDQ + h * (D / 2), scale,
                                dq + (static_cast<size_t>(bh) * N + q) * D + h * (D / 2), D, N - q);
      ++it;
    }
  }

  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync_all();  // rank 0 has drained every copy and MMA that touches either CTA
  else
    __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && abort_flag) atomicExch(status, kErrTimeout);
  report_checks(status);
}

// DROP is the dK/dV pass's dropout mode, DROPQ the dQ pass's: they differ
// (kDrawn, kSaved) when the dK/dV pass writes the bits it draws to
// drop.mask for the dQ pass to read.
template <int D, bool F16, int DROP, int DROPQ>
cudaError_t launch(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                   const CUtensorMap &tmdO, const CUtensorMap &tmdK, const CUtensorMap &tmdV, const HalfMaps *half,
                   const void *o, const void *dO, const float *lse, void *dq, void *dk, void *dv, float *Lp,
                   float *Dp, int B, int H, int N, int Nk, float scale, int causal, const Dropout &drop, int *status,
                   int num_sms, cudaStream_t stream, const BwdSide &side) {
  const int n_tiles = (N + kBlk - 1) / kBlk;
  const int Np = n_tiles * kBlk;
  const float scale_log2 = scale * kLog2e;
  {
    const int64_t prows = static_cast<int64_t>(B) * H * Np;
    const int64_t threads = prows * prep_tpr(D);
    bwd_prep_kernel<D, F16><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const uint16_t *>(o), static_cast<const uint16_t *>(dO), lse, Lp, Dp, N, Np,
        prows);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // persistent grids: at most one CTA per SM, each walking its static list of
  // key blocks (dK/dV pass) or query tiles (dQ pass); an item costs the tiles
  // it visits plus about one for its epilogue
  const int BH = B * H, off = Nk - N, n_kb_all = (Nk + kBlk - 1) / kBlk;
  auto kblocks_q = [&](int qt) {
    return causal ? std::min(n_kb_all, (qt * kBlk + kBlk - 1 + off) / kBlk + 1) : n_kb_all;
  };
  auto first_tile = [&](int kb) { return causal ? std::max(0, kb * kBlk - off) / kBlk : 0; };

  // Each pass as a launch on a given stream; `ctas` tells how many SMs its
  // grid takes.
  struct Pass {
    int ctas = 0;
    bool pair = false;
    TileSched sched{};
  };
  Pass kv, q;
  int clusters_kv = 0, clusters_q = 0;
  if constexpr (D == 128 && DROP == kNoDrop && FA_PAIR_KERNELS) {
    // two-CTA clusters (block / tile pairs, M = 256 MMAs) when the heads have
    // at least two key blocks / query tiles
    static SmemOnce smem_kvp, smem_qp;
    auto kpk = bwd_dkdv_kernel<D, F16, kNoDrop, true>;
    auto kpq = bwd_dq_kernel<D, F16, kNoDrop, true>;
    if (half && n_kb_all >= 2) {
      if ((e = set_smem_once(reinterpret_cast<const void *>(kpk), DkdvCfg<D, true>::kAlloc, &smem_kvp)) !=
          cudaSuccess)
        return e;
      clusters_kv = pair_grid(reinterpret_cast<const void *>(kpk), DkdvCfg<D, true>::kAlloc, kThreads, num_sms);
    }
    if (half && n_tiles >= 2) {
      if ((e = set_smem_once(reinterpret_cast<const void *>(kpq), DqCfg<D, true>::kAlloc, &smem_qp)) != cudaSuccess)
        return e;
      clusters_q = pair_grid(reinterpret_cast<const void *>(kpq), DqCfg<D, true>::kAlloc, kThreads, num_sms);
    }
  }
  if (clusters_kv >= 1) {
    const int np = (n_kb_all + 1) / 2;  // a pair visits the query tiles of its lower block
    kv.sched = sched_cached(5, BH, N, Nk, causal != 0, np, clusters_kv, [&](int r) {
      return static_cast<long long>(n_tiles - first_tile(2 * r)) + 1;
    });
    kv.pair = true;
    kv.ctas = 2 * kv.sched.G;
  } else {
    kv.sched = sched_cached(1, BH, N, Nk, causal != 0, n_kb_all, num_sms, [&](int kb) {
      return static_cast<long long>(n_tiles - first_tile(kb)) + 1;
    });
    kv.ctas = kv.sched.G;
  }
  if (clusters_q >= 1) {
    const int np = (n_tiles + 1) / 2;
    q.sched = sched_cached(4, BH, N, Nk, causal != 0, np, clusters_q, [&](int rank) {
      return static_cast<long long>(kblocks_q(2 * (np - 1 - rank) + 1)) + 1;
    });
    q.pair = true;
    q.ctas = 2 * q.sched.G;
  } else {
    q.sched = sched_cached(2, BH, N, Nk, causal != 0, n_tiles, num_sms, [&](int rank) {
      return static_cast<long long>(kblocks_q(n_tiles - 1 - rank)) + 1;
    });
    q.ctas = q.sched.G;
  }

  auto run_kv = [&](cudaStream_t st) -> cudaError_t {
    timing_begin(st);
    if constexpr (D == 128 && DROP == kNoDrop && FA_PAIR_KERNELS) {
      if (kv.pair) {
        cudaError_t r = launch_pair_grid(bwd_dkdv_kernel<D, F16, kNoDrop, true>, kv.sched.G, kThreads,
                                         DkdvCfg<D, true>::kAlloc, st, tmQ, tmK, tmV, tmdO, tmdK, tmdV, half->q,
                                         half->dO, Lp, Dp, N, Nk, kv.sched, scale, scale_log2, causal, drop, status);
        timing_end(st);
        return r != cudaSuccess ? r : cudaGetLastError();
      }
    }
    static SmemOnce smem_kv;
    auto kern = bwd_dkdv_kernel<D, F16, DROP, false>;
    cudaError_t r = set_smem_once(reinterpret_cast<const void *>(kern), DkdvCfg<D>::kAlloc, &smem_kv);
    if (r != cudaSuccess) return r;
    kern<<<kv.sched.G, DROP == kDrawn ? kThreadsMask : kThreads, DkdvCfg<D>::kAlloc, st>>>(tmQ, tmK, tmV, tmdO, tmdK, tmdV, tmQ, tmdO, Lp, Dp, N, Nk,
                                                           kv.sched, scale, scale_log2, causal, drop, status);
    timing_end(st);
    return cudaGetLastError();
  };
  auto run_q = [&](cudaStream_t st) -> cudaError_t {
    timing_begin(st);
    if constexpr (D == 128 && DROP == kNoDrop && FA_PAIR_KERNELS) {
      if (q.pair) {
        cudaError_t r = launch_pair_grid(bwd_dq_kernel<D, F16, kNoDrop, true>, q.sched.G, kThreads,
                                         DqCfg<D, true>::kAlloc, st, tmQ, tmK, tmV, tmdO, half->k, half->v, Lp, Dp,
                                         static_cast<uint16_t *>(dq), N, Nk, q.sched, scale, scale_log2, causal, drop,
                                         status);
        timing_end(st);
        return r != cudaSuccess ? r : cudaGetLastError();
      }
    }
    static SmemOnce smem_q;
    auto kern = bwd_dq_kernel<D, F16, DROPQ, false>;
    using CQ = DqCfg<D, false, DROPQ == kDrawn>;
    cudaError_t r = set_smem_once(reinterpret_cast<const void *>(kern), CQ::kAlloc, &smem_q);
    if (r != cudaSuccess) return r;
    kern<<<q.sched.G, DROPQ == kDrawn ? kThreadsMask : kThreads, CQ::kAlloc, st>>>(tmQ, tmK, tmV, tmdO, tmK, tmV, Lp, Dp,
                                                        static_cast<uint16_t *>(dq), N, Nk, q.sched, scale,
                                                        scale_log2, causal, drop, status);
    timing_end(st);
    return cudaGetLastError();
  };

  // Both passes only read what the row-term kernel and the forward wrote
  // (unless the dK/dV pass hands the keep bits on), so when their grids fit
  // on the GPU together (small problems, where each leaves SMs idle) the dQ
  // pass runs on the side stream alongside the dK/dV pass; otherwise one
  // after the other (each persistent grid fills the GPU).
  if (DROP == DROPQ && side.stream && kv.ctas + q.ctas <= num_sms) {
    if ((e = cudaEventRecord(side.fork, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(side.stream, side.fork, 0)) != cudaSuccess)
      return e;
    if ((e = run_kv(stream)) != cudaSuccess) return e;
    if ((e = run_q(side.stream)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(side.join, side.stream)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(stream, side.join, 0);
  }
  if ((e = run_kv(stream)) != cudaSuccess) return e;
  return run_q(stream);
}

template <int DROP, int DROPQ>
cudaError_t dispatch(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                     const CUtensorMap &tmdO, const CUtensorMap &tmdK, const CUtensorMap &tmdV, const HalfMaps *half,
                     const void *o, const void *dO, const float *lse, void *dq, void *dk, void *dv, float *Lp,
                     float *Dp, int B, int H, int N, int Nk, int d, float scale, int causal, bool f16,
                     const Dropout &drop, int *status, int num_sms, cudaStream_t stream, const BwdSide &side) {
#define FA_BWD_LAUNCH(DD, FF)                                                                                  \
  return launch<DD, FF, DROP, DROPQ>(tmQ, tmK, tmV, tmdO, tmdK, tmdV, half, o, dO, lse, dq, dk, dv, Lp, Dp, B, H, N,  \
                              Nk, scale, causal, drop, status, num_sms, stream, side)
  if (f16) {
    if (d == 64) FA_BWD_LAUNCH(64, true);
    if (d == 96) FA_BWD_LAUNCH(96, true);
    FA_BWD_LAUNCH(128, true);
  }
  if (d == 64) FA_BWD_LAUNCH(64, false);
  if (d == 96) FA_BWD_LAUNCH(96, false);
  FA_BWD_LAUNCH(128, false);
#undef FA_BWD_LAUNCH
}

}  // namespace

cudaError_t launch_bwd_16(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          const CUtensorMap &tmdO, const CUtensorMap &tmdK, const CUtensorMap &tmdV,
                          const HalfMaps *half, const void *o, const void *dO, const float *lse, void *dq, void *dk,
                          void *dv, float *Lp, float *Dp, int B, int H, int N, int Nk, int d, float scale, int causal,
                          bool f16, const Dropout *drop, int *status, int num_sms, cudaStream_t stream,
                          const BwdSide &side, int *launches) {
  *launches += 3;
#define FA_BWD_DISPATCH(M, MQ, DR)                                                                              \
  return dispatch<M, MQ>(tmQ, tmK, tmV, tmdO, tmdK, tmdV, half, o, dO, lse, dq, dk, dv, Lp, Dp, B, H, N, Nk, d, \
                         scale, causal, f16, DR, status, num_sms, stream, side)
  if (drop && drop->mask && drop->dkdv_writes_mask) FA_BWD_DISPATCH(kDrawn, kSaved, *drop);
  if (drop && drop->mask) FA_BWD_DISPATCH(kSaved, kSaved, *drop);
  if (drop) FA_BWD_DISPATCH(kDrawn, kDrawn, *drop);
  FA_BWD_DISPATCH(kNoDrop, kNoDrop, Dropout{});
#undef FA_BWD_DISPATCH
}

}  // namespace fa
