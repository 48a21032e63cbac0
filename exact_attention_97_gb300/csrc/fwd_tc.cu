// fwd_tc.cu -- exact attention forward on the sm_103a tensor cores, for 16-bit
// inputs (bf16 or f16; the element type is a template parameter).
//
// What it computes (pages): the tiled loop of "Flash Attention 原理与实现",
// section "Forward 的 Tiling 策略" -- for each block Q_i of query rows, walk
// the key/value blocks K_j, V_j, form S_ij = Q_i K_j^T, fold it into the
// running row state and divide by l once at the end -- with the state update
// of the "research-attention" tutorial, section 02:
//     m' = max(m, rowmax S),  alpha = exp(m - m'),  p = exp(s - m'),
//     l' = alpha l + rowsum p, u' = alpha u + p V,   o = u / l,
// and the saved statistic L = m + ln l of its section 04.
//
// GB300 design: a persistent grid, one CTA per SM, each CTA walking a static
// list of 128-row query tiles (tile_sched.h); within a CTA:
//   warp 0      loader: Q of each tile, then K_j into a ring of shared-memory
//               stages (128-byte swizzle, 3-D tensor maps so rows past N read
//               as zero). The rings and barrier phases run on across tiles,
//               so the next tile's loads and S MMAs overlap the current
//               tile's last P V products and its epilogue.
//   warp 2      loader of V_j (its own ring); also allocates and frees the
//               512 tensor-memory (TMEM) columns.
//   warp 1      MMA issuer for S_j = Q K_j^T into one of the TMEM score
//               buffers, so the next scores can run while row statistics of
//               S_j are computed.
//   warp 3      MMA issuer for O += P_j V_j, with P_j read straight from TMEM
//               (A operand in TMEM, B = V_j in shared memory). Two issuing
//               threads keep the tensor pipe fed while either waits.
//   warps 4-7   softmax: thread t owns row t of the tile (= TMEM lane t).
//               Loads its 128 scores, applies the mask, takes the row max,
//               writes P = 2^(s*c - m*c) (c = scale*log2 e) back as 16-bit
//               pairs over the S columns, and keeps l. The running max is only
//               moved when it grows by more than 2^8: any common base leaves
//               u/l unchanged (tutorial section 02), so the O rescale in TMEM
//               (ld, multiply, st) is skipped on most tiles. At the end of
//               a tile the epilogue divides by l and stores O with
//               whole-line row-segment stores (store_tmem_rows, sm103.cuh),
//               then L = m*scale + ln l.
//   warps 8-11  without dropout (one-CTA kernels): the epilogue warps. The
//               softmax warps hand l and m over in shared memory and start
//               the next tile; these write O and L once its last P V is done,
//               and free O for the next tile's first P V.
//               With dropout: draw each tile's keep bits (Philox4x32-10,
//               sm103.cuh) into a shared ring one tile ahead; the softmax
//               warps then zero the dropped P for P V, keep the undropped l
//               and write the epilogue themselves (1 / (1 - p) folded in).
//
// Head sizes 64, 96 and 128 use one K/V unit per key tile; 256 uses two
// (FwdSmem). TMEM columns: score buffers of 128 columns, then O.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "kernels.h"
#include "tile_sched.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kBlockM = 128;   // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;   // keys per tile
constexpr int kThreads = 256;      // 8 warps
constexpr int kMaskWarps = 4;  // with dropout, warps 8-11 draw the keep masks (32 keys of each tile each)
constexpr int kThreadsDrop = 256 + 32 * kMaskWarps;
// The one-CTA forward without dropout: warps 8-11 write each item's O and L
// (the epilogue warps), so the softmax warps start the next item at once.
template <bool DROP, bool PAIR>
__host__ __device__ constexpr bool fwd_epi_warps() {
  return !DROP && !PAIR;
}
template <bool DROP, bool PAIR>
__host__ __device__ constexpr int fwd_threads() {
  return DROP ? kThreadsDrop : (fwd_epi_warps<DROP, PAIR>() ? 384 : kThreads);
}
constexpr int kMaskSlots = 3;      // keep-mask ring (128 rows x 128 keys of bits each)
constexpr int kMaskSlotBytes = 128 * 128 / 8;
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};
constexpr float kRescaleLog2 = 8.0f;  // move the running max only past 2^8
constexpr float kLn2 = 0.69314718055994531f;

#ifndef FA_FWD_QBUF
#define FA_FWD_QBUF 2
#endif

// Shared memory and tensor memory by head size. A row of a tile is whole
// 64-column TMA boxes (columns past D read as zero). K and V stream in units
// of at most 128 columns: one unit per key tile up to d = 128, two at d = 256
// (the score product then accumulates over both K units, and P V runs as two
// N = 128 products, one per V unit). Shared memory holds kQBuf query tiles
// (two let the next tile's Q land while the current tile still runs), the K
// ring and the V ring, under the 227 KB limit: at d = 96 and 128, 2 Q + 3 K +
// 2 V tiles; at d = 256, 1 Q tile + 3 K + 2 V units. Tensor memory holds
// kSBuf score buffers of 128 columns and O after them (512 columns).
//
// PAIR (d = 128, no dropout): a cluster of two CTAs runs the two query tiles
// of a tile pair with M = 256 MMAs. Each CTA then holds only its half of each
// key tile's operands: for S = Q K^T the keys 64r..64r+63 (rank r; K-major,
// two 8 KB sub-tiles of 64 rows), for O += P V the head columns 64r..64r+63
// of all 128 keys (MN-major, one 16 KB sub-tile). Both rings hold 16 KB
// stages, four of each.
template <int D, bool DROP = false, bool PAIR = false>
struct FwdSmem {
  static_assert(!PAIR || (D == 128 && !DROP), "the pair kernel covers d = 128 without dropout");
  static constexpr int kDP = (D + 63) / 64 * 64;
  static constexpr int kUnits = kDP > 128 ? kDP / 128 : 1;  // K / V ring units per key tile
  static constexpr int kUnitCols = kDP / kUnits;
  static constexpr int kUnitBytes = kBlockN * kUnitCols * 2;
  static constexpr int kKBytes = PAIR ? kUnitBytes / 2 : kUnitBytes;  // one K ring stage
  static constexpr int kVBytes = PAIR ? kUnitBytes / 2 : kUnitBytes;  // one V ring stage
  static constexpr int kKSub = PAIR ? (kBlockN / 2) * 128 : kBlockN * 128;  // bytes of one K sub-tile
  static constexpr int kQBytes = kBlockM * kDP * 2;
  static constexpr int kSK = (kUnits == 1 ? D : kUnitCols) / 16;  // k-steps of S per unit
  static constexpr int kPVN = kUnits == 1 ? D : kUnitCols;         // N of one P V product
  static constexpr int kSBuf = kDP > 128 ? 2 : 3;
  // with dropout the keep-mask ring needs 6 KB: one Q buffer, and at d = 256
  // a K ring of two units
  static constexpr int kQBuf = PAIR ? 2 : ((kDP > 128 || DROP) ? 1 : FA_FWD_QBUF);
  static constexpr int kKStages = PAIR ? 4 : ((kDP > 128 && DROP) ? 2 : 3);
  static constexpr int kVStages = PAIR ? 4 : (kDP > 128 ? 2 : ((kDP == 128 && (kQBuf == 2 || DROP)) ? 2 : 3));
  static constexpr int kSubBytes = kBlockN * 128;  // one 128-row x 64-column sub-tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBuf * kQBytes;
  static constexpr int kV = kK + kKStages * kKBytes;
  static constexpr int kMask = kV + kVStages * kVBytes;
  static constexpr int kMaskBytes = DROP ? kMaskSlots * kMaskSlotBytes : 0;
  static constexpr int kBytes = kMask + kMaskBytes;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

// Columns [c0, c1) of 128 rows starting at `row`, as 64-column boxes into
// consecutive sub-tiles at dst.
__device__ __forceinline__ void load_cols(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                          int row, int bh) {
  for (int x = c0; x < c1; x += 64) tma_load_3d(dst + ((x - c0) / 64) * (kBlockN * 128), map, bar, x, row, bh);
}

template <int D, bool F16, bool DROP, bool PAIR>
__global__ void __launch_bounds__(fwd_threads<DROP, PAIR>(), 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, uint16_t *__restrict__ o,
                    float *__restrict__ lse, int N, int Nk, const __grid_constant__ TileSched sched, float scale,
                    float scale_log2, int causal, const Dropout drop, int *status) {
  using L = FwdSmem<D, DROP, PAIR>;
  using E = Elt<F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  constexpr int kQBuf = L::kQBuf, kStages = L::kKStages, kVStages = L::kVStages, kSBuf = L::kSBuf;
  constexpr int kUnits = L::kUnits, kUC = L::kUnitCols;
  __shared__ uint64_t q_full[kQBuf], q_empty[kQBuf], k_full[kStages], k_empty[kStages], v_full[kVStages],
      v_empty[kVStages], s_full[kSBuf], p_ready[kSBuf], pv_done[kSBuf], drain_s, drain_pv,
      mask_full[DROP ? kMaskSlots : 1], mask_empty[DROP ? kMaskSlots : 1];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  // epilogue warps: each row's sum l and max m of the item just finished
  // (stat_full: written by the softmax warps, stat_empty: read), and o_free:
  // O has been read out of TMEM, so the next item's first P V may overwrite it
  constexpr bool EPI = fwd_epi_warps<DROP, PAIR>();
  __shared__ float st_l[EPI ? kBlockM : 1], st_m[EPI ? kBlockM : 1];
  __shared__ uint64_t stat_full, stat_empty, o_free;

  const int warp = warp_id(), lane = lane_id();
  // A schedule unit is a query tile, or with PAIR a tile pair (2u, 2u + 1)
  // whose tile 2u + r runs on cluster rank r; both CTAs of a pair walk the
  // same units. Schedule rank 0 is a head's most expensive unit (the last one
  // under the causal mask).
  const uint32_t crank = PAIR ? cluster_rank() : 0u;
  const int cta = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  auto unit_of = [&](int rank) { return causal ? sched.nt - 1 - rank : rank; };
  auto qtile_of = [&](int rank) { return PAIR ? 2 * unit_of(rank) + static_cast<int>(crank) : unit_of(rank); };
  // N query rows, Nk >= N keys under the causal mask; query i sees keys up to
  // i + (Nk - N) (bottom-right alignment; with Nk = N the usual triangle)
  const int off = Nk - N;
  const int n_ktiles_all = (Nk + kBlockN - 1) / kBlockN;
  auto ktiles_q = [&](int qtile) {
    return causal ? min(n_ktiles_all, (qtile * kBlockM + kBlockM - 1 + off) / kBlockN + 1) : n_ktiles_all;
  };
  // key tiles of a unit: a pair walks those of its upper tile (the lower
  // tile's softmax masks the extra one out entirely)
  auto ktiles = [&](int rank) { return ktiles_q(PAIR ? 2 * unit_of(rank) + 1 : unit_of(rank)); };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int b = 0; b < kQBuf; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < kSBuf; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_ready[b], PAIR ? 2 * 4 : 4 * 32);  // pair: one arrival per softmax warp of each CTA
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(&drain_s, 1);
    mbar_init(&drain_pv, 1);
    if constexpr (EPI) {
      mbar_init(&stat_full, 4 * 32);
      mbar_init(&stat_empty, 4 * 32);
      mbar_init(&o_free, 4 * 32);
    }
    if constexpr (DROP) {
      for (int b = 0; b < kMaskSlots; ++b) {
        mbar_init(&mask_full[b], kMaskWarps * 32);
        mbar_init(&mask_empty[b], 4 * 32);
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
  const uint32_t tmem_O = tmem + kSBuf * 128;

  // Every role walks the same item sequence. Key tiles are counted across
  // items (kt), so the K/V rings, the S buffers and their barrier phases run
  // on without a break from one item to the next; `it` counts items (phase of
  // q_full / q_empty).
  auto role_k_loader = [&]() {
    // ------------------------------------------------------------ loader: Q, K
    // Q of item `it` goes into buffer it % kQBuf once every S MMA of the item
    // that used it before has completed (q_empty); it is also prefetched into
    // L2 one item ahead.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      bool ok = true;
      int kt = 0, it = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int qtile = qtile_of(rank);
        {  // L2 prefetch of the next item's Q
          int nr, nbh, ns, k2 = k + 1;
          while ((ns = sched_item(sched, cta, k2, nr, nbh)) == kSkip) ++k2;
          if (ns == kItem)
            for (int x = 0; x < D; x += 64) tma_prefetch_l2_3d(&tmQ, x, qtile_of(nr) * kBlockM, nbh);
        }
        const int qb = it % kQBuf;
        if (it >= kQBuf && !mbar_wait(&q_empty[qb], ((it / kQBuf) & 1) ^ 1, &abort_flag)) { ok = false; break; }
        if constexpr (PAIR) {  // both CTAs' Q tiles complete on rank 0's barrier
          if (crank == 0) mbar_arrive_expect_tx(&q_full[qb], 2 * L::kQBytes);
          const uint32_t bar = cluster_addr(&q_full[qb], 0);
          for (int x = 0; x < D; x += 64)
            tma_load_3d_pair(smem + L::kQ + qb * L::kQBytes + (x / 64) * L::kSubBytes, &tmQ, bar, x,
                             qtile * kBlockM, bh);
        } else {
          mbar_arrive_expect_tx(&q_full[qb], L::kQBytes);
          load_cols(smem + L::kQ + qb * L::kQBytes, &tmQ, &q_full[qb], 0, D, qtile * kBlockM, bh);
        }
        const int nk = ktiles(rank) * kUnits;  // K units of this item
        for (int j = 0; j < nk; ++j, ++kt) {
          const int st = kt % kStages, c0 = (j % kUnits) * kUC;
          if (kt >= kStages && !mbar_wait(&k_empty[st], ((kt / kStages) & 1) ^ 1, &abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (PAIR) {  // keys 64r..64r+63 of the tile (tmK has 64-row boxes)
            if (crank == 0) mbar_arrive_expect_tx(&k_full[st], 2 * L::kKBytes);
            const uint32_t bar = cluster_addr(&k_full[st], 0);
            for (int x = 0; x < D; x += 64)
              tma_load_3d_pair(smem + L::kK + st * L::kKBytes + (x / 64) * L::kKSub, &tmK, bar, x,
                               j * kBlockN + 64 * static_cast<int>(crank), bh);
          } else {
            mbar_arrive_expect_tx(&k_full[st], L::kKBytes);
            load_cols(smem + L::kK + st * L::kKBytes, &tmK, &k_full[st], c0, min(D, c0 + kUC),
                      (j / kUnits) * kBlockN, bh);
          }
        }
        ++it;  // this item's Q load was issued
      }
      // teardown: every issued copy must land before the CTA's memory is
      // released (a pair's copies all complete on rank 0's barriers, which
      // rank 0 drains before the pair's closing cluster barrier)
      if (!PAIR || crank == 0) {
        for (int i = max(0, it - kQBuf); i < it; ++i) mbar_wait_drain(&q_full[i % kQBuf], (i / kQBuf) & 1);
        for (int j = max(0, kt - kStages); j < kt; ++j)
          mbar_wait_drain(&k_full[j % kStages], (j / kStages) & 1);
      }
    }
  };
  auto role_v_loader = [&]() {
    // ---------------------------------------------------------------- loader: V
    if (lane == 0) {
      tma_prefetch_desc(&tmV);
      bool ok = true;
      int kt = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int nk = ktiles(rank) * kUnits;  // V units of this item
        for (int j = 0; j < nk; ++j, ++kt) {
          const int st = kt % kVStages, c0 = (j % kUnits) * kUC;
          if (kt >= kVStages && !mbar_wait(&v_empty[st], ((kt / kVStages) & 1) ^ 1, &abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (PAIR) {  // head columns 64r..64r+63 of all the tile's keys
            if (crank == 0) mbar_arrive_expect_tx(&v_full[st], 2 * L::kVBytes);
            tma_load_3d_pair(smem + L::kV + st * L::kVBytes, &tmV, cluster_addr(&v_full[st], 0),
                             64 * static_cast<int>(crank), j * kBlockN, bh);
          } else {
            mbar_arrive_expect_tx(&v_full[st], L::kVBytes);
            load_cols(smem + L::kV + st * L::kVBytes, &tmV, &v_full[st], c0, min(D, c0 + kUC),
                      (j / kUnits) * kBlockN, bh);
          }
        }
      }
      if (!PAIR || crank == 0)
        for (int j = max(0, kt - kVStages); j < kt; ++j)
          mbar_wait_drain(&v_full[j % kVStages], (j / kVStages) & 1);
    }
  };
  auto role_s_issuer = [&]() {
    // ------------------------------------------------------ MMA issuer: S = Q K^T
    // S of key tile kt goes to buffer kt % kSBuf once P V of tile kt - kSBuf
    // (which used that buffer) has completed; it accumulates over the tile's K
    // units (ring position ku).
    // With PAIR only rank 0 issues (M = 256 over both CTAs), and each commit
    // arrives on the barrier of that name in both CTAs.
    if (lane == 0 && (!PAIR || crank == 0)) {
      constexpr uint32_t idesc_s = idesc_16(PAIR ? 2 * kBlockM : kBlockM, kBlockN, false, false, F16);
      auto commit = [](uint64_t *bar) {
        if constexpr (PAIR) mma_commit_pair_both(bar);
        else mma_commit(bar);
      };
      bool ok = true;
      int kt = 0, it = 0, ku = 0;
      int rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int nk = ktiles(rank);
        const int qb = it % kQBuf;
        const uint32_t q_addr = smem_u32(smem + L::kQ + qb * L::kQBytes);
        if (!mbar_wait(&q_full[qb], (it / kQBuf) & 1, &abort_flag)) { ok = false; break; }
        for (int j = 0; j < nk; ++j, ++kt) {
          const int sb = kt % kSBuf;
          if (kt >= kSBuf && !mbar_wait(&pv_done[sb], ((kt / kSBuf) - 1) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          for (int u = 0; u < kUnits; ++u, ++ku) {
            const int st = ku % kStages;
            if (!mbar_wait(&k_full[st], (ku / kStages) & 1, &abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t k_addr = smem_u32(smem + L::kK + st * L::kKBytes);
            const uint32_t qu_addr = q_addr + u * (kUC / 64) * L::kSubBytes;
#pragma unroll
            for (int kk = 0; kk < L::kSK; ++kk) {
              const uint32_t qoff = (kk / 4) * L::kSubBytes + (kk % 4) * 32;
              const uint32_t koff = (kk / 4) * L::kKSub + (kk % 4) * 32;
              const uint64_t adesc = sdesc_sw128(qu_addr + qoff, 16, 1024), bdesc = sdesc_sw128(k_addr + koff, 16, 1024);
              if constexpr (PAIR) mma_ss_pair(tmem + sb * 128, adesc, bdesc, idesc_s, (u > 0 || kk > 0) ? 1u : 0u);
              else mma_ss(tmem + sb * 128, adesc, bdesc, idesc_s, (u > 0 || kk > 0) ? 1u : 0u);
            }
            commit(&k_empty[st]);
          }
          if (!ok) break;
          commit(&s_full[sb]);
        }
        commit(&q_empty[qb]);  // this Q buffer is free once the item's S MMAs are done
        ++it;
      }
      // teardown: all issued MMAs finish before TMEM is released
      if constexpr (PAIR) mma_commit_pair_local(&drain_s);
      else mma_commit(&drain_s);
      mbar_wait_drain(&drain_s, 0);
    }
  };
  auto role_pv_issuer = [&]() {
    // ---------------------------------------------------- MMA issuer: O += P V
    // A second issuing thread, so the tensor pipe always has one of the two
    // streams queued while the other waits on its barriers. The first P V of
    // an item overwrites O: with epilogue warps it waits for them to have read
    // the previous item's O out of TMEM (o_free); otherwise its P is only
    // marked ready after the softmax warps have done so.
    if (lane == 0 && (!PAIR || crank == 0)) {
      constexpr uint32_t idesc_o = idesc_16(PAIR ? 2 * kBlockM : kBlockM, L::kPVN, false, true, F16);
      auto commit = [](uint64_t *bar) {
        if constexpr (PAIR) mma_commit_pair_both(bar);
        else mma_commit(bar);
      };
      bool ok = true;
      int kt = 0, vu = 0, it = 0;
      int rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int nk = ktiles(rank);
        if constexpr (EPI) {
          if (it > 0 && !mbar_wait(&o_free, (it - 1) & 1, &abort_flag)) break;
        }
        ++it;
        for (int j = 0; j < nk; ++j, ++kt) {
          const int sb = kt % kSBuf;
          if (!mbar_wait(&p_ready[sb], (kt / kSBuf) & 1, &abort_flag)) { ok = false; break; }
          for (int u = 0; u < kUnits; ++u, ++vu) {  // O columns [u kUC, (u+1) kUC) from V unit u
            const int st = vu % kVStages;
            if (!mbar_wait(&v_full[st], (vu / kVStages) & 1, &abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t v_addr = smem_u32(smem + L::kV + st * L::kVBytes);
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {
              const uint64_t bdesc = sdesc_sw128(v_addr + kk * 2048, L::kSubBytes, 1024);
              if constexpr (PAIR)
                mma_ts_pair(tmem_O + u * kUC, tmem + sb * 128 + kk * 8, bdesc, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
              else
                mma_ts(tmem_O + u * kUC, tmem + sb * 128 + kk * 8, bdesc, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
            }
            commit(&v_empty[st]);
          }
          if (!ok) break;
          commit(&pv_done[sb]);
        }
      }
      if constexpr (PAIR) mma_commit_pair_local(&drain_pv);
      else mma_commit(&drain_pv);
      mbar_wait_drain(&drain_pv, 0);
    }
  };
  auto role_softmax = [&]() {
    // ----------------------------------------------------------------- softmax
    const int wq = warp - 4;                 // TMEM lane quarter of this warp
    const int r_local = wq * 32 + lane;      // row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    bool ok = true;
    int kt = 0, it = 0;
    int rank, bh;
    for (int k = 0; ok; ++k) {
      const int step = sched_item(sched, cta, k, rank, bh);
      if (step == kDone) break;
      if (step == kSkip) continue;
      const int qtile = qtile_of(rank);
      const int nk = ktiles(rank);
      const int row = qtile * kBlockM + r_local;
      float m_used = -INFINITY, l_sum = 0.f;
      for (int j = 0; j < nk; ++j, ++kt) {
        const int sb = kt % kSBuf;
        uint32_t keep[4];  // dropout: keep bits of this row's 128 keys, from the mask warps
        if constexpr (DROP) {
          const int ms = kt % kMaskSlots;
          if (!mbar_wait_warp(&mask_full[ms], (kt / kMaskSlots) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t *mw = reinterpret_cast<const uint32_t *>(smem + L::kMask + ms * kMaskSlotBytes) + r_local;
#pragma unroll
          for (int w = 0; w < 4; ++w) keep[w] = mw[w * kBlockM];
          mbar_arrive(&mask_empty[ms]);
        }
        if (!mbar_wait_warp(&s_full[sb], (kt / kSBuf) & 1, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kBlockN];
        tmem_ld128(tmem + lane_addr + sb * 128, sr);
        const int key0 = j * kBlockN;
        int limit = Nk - key0;                                  // keys >= Nk are masked
        if (causal) limit = min(limit, row + off - key0 + 1);   // keys > row + off are masked
        if (limit < kBlockN) {
#pragma unroll
          for (int t = 0; t < kBlockN; ++t)
            if (t >= limit) sr[t] = __float_as_uint(-INFINITY);
        }
        // row max: four independent chains of 3-input max
        float mx;
        {
          float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
          for (int t = 0; t < kBlockN; t += 8) {
            m0 = fmax3(m0, __uint_as_float(sr[t]), __uint_as_float(sr[t + 1]));
            m1 = fmax3(m1, __uint_as_float(sr[t + 2]), __uint_as_float(sr[t + 3]));
            m2 = fmax3(m2, __uint_as_float(sr[t + 4]), __uint_as_float(sr[t + 5]));
            m3 = fmax3(m3, __uint_as_float(sr[t + 6]), __uint_as_float(sr[t + 7]));
          }
          mx = fmax3(m0, m1, fmaxf(m2, m3));
        }
        if (j == 0) {
          m_used = mx;
        } else {
          const bool need = (mx - m_used) * scale_log2 > kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            // O must hold P_{kt-1} V_{kt-1} before it is rescaled. Wait on
            // that product's own buffer barrier: its previous phase (tile
            // kt - 4) is known complete because S of tile kt - 1 was only
            // issued after it, so a stale phase cannot match the parity.
            if (!mbar_wait_warp(&pv_done[(kt - 1) % kSBuf], ((kt - 1) / kSBuf) & 1, &abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float alpha = need ? ex2_approx((m_used - mx) * scale_log2) : 1.f;
            if (need) {
              l_sum *= alpha;
              m_used = mx;
            }
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t r[32];
              tmem_ld32(tmem_O + lane_addr + ch * 32, r);
#pragma unroll
              for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * alpha);
              tmem_st32(tmem_O + lane_addr + ch * 32, r);
            }
          }
        }
        // P = 2^(s*c - m*c), two columns at a time
        const float neg = -m_used * scale_log2;
        const uint64_t cc = f2_pack(scale_log2, scale_log2), nn = f2_pack(neg, neg);
        uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;  // packed partial row sums (+0.0f pairs)
        uint32_t pk[kBlockN / 2];
#pragma unroll
        for (int w = 0; w < kBlockN / 2; ++w) {
          const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[2 * w]), __uint_as_float(sr[2 * w + 1])), cc, nn);
          float x0, x1;
          f2_unpack(x2, x0, x1);
          const uint64_t p2 = f2_pack(ex2_approx(x0), ex2_approx(x1));
          switch (w & 3) {
            case 0: acc0 = f2_add(acc0, p2); break;
            case 1: acc1 = f2_add(acc1, p2); break;
            case 2: acc2 = f2_add(acc2, p2); break;
            default: acc3 = f2_add(acc3, p2); break;
          }
          float p0, p1;
          f2_unpack(p2, p0, p1);
          pk[w] = E::pack(p0, p1);
          if constexpr (DROP) {  // l keeps the undropped sum; P V gets P o Z (1 / (1 - p) in the epilogue)
            // keys 2w, 2w + 1 are bits c + 8 e, c + 8 (e + 1) of their word (c = (2w mod 32) / 4,
            // e = 2w mod 4); shifted left by 7 - c they are the top bits of bytes e, e + 1
            const int b = (2 * w) & 31, c = b >> 2;
            pk[w] &= byte_signs(keep[w >> 4] << (7 - c), (b & 3) ? 0xBBAAu : 0x9988u);
          }
        }
        tmem_st64(tmem + lane_addr + sb * 128, pk);
        float rs;
        {
          float a0, a1;
          f2_unpack(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)), a0, a1);
          rs = a0 + a1;
        }
        l_sum += rs;
        tc_fence_before();
        if constexpr (PAIR) {  // one arrival per warp, on rank 0's barrier
          __syncwarp();
          if (lane == 0) mbar_arrive_cl(cluster_addr(&p_ready[sb], 0));
        } else {
          mbar_arrive(&p_ready[sb]);
        }
      }
      // -------------------------------------------------------------- epilogue
      if constexpr (EPI) {
        // this row's l and m go to the epilogue warps; the next item starts now
        if (!ok) break;
        if (it > 0 && !mbar_wait_warp(&stat_empty, (it - 1) & 1, &abort_flag)) {
          ok = false;
          break;
        }
        st_l[r_local] = l_sum;
        st_m[r_local] = m_used;
        mbar_arrive(&stat_full);
        ++it;
      } else {
        // the item's last P V (and, issued in order before it, every other
        // one) is done; the next item's first P V waits for this warp's next
        // p_ready arrival, which comes after these TMEM reads
        if (!ok || !mbar_wait_warp(&pv_done[(kt - 1) % kSBuf], ((kt - 1) / kSBuf) & 1, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv_l = DROP ? drop.inv_keep / l_sum : 1.f / l_sum;
        // O = accumulator / l, whole-line row-segment stores
        store_tmem_rows<E, D>(tmem_O + lane_addr, inv_l, o + (static_cast<size_t>(bh) * N + row) * D, D, N - row);
        if (row < N) lse[static_cast<size_t>(bh) * N + row] = (m_used * scale_log2 + log2f(l_sum)) * kLn2;
      }
    }
  };
  auto role_epilogue = [&]() {
    // ------------------------------------------------------- O and L (EPI)
    // Warp 8 + q writes rows 32q..32q+31 of each item once its last P V is
    // done, from the l and m the softmax warps handed over, then frees O for
    // the next item's first P V. That wait cannot meet a later phase of the
    // buffer: the next use of it is a P V of the next item, issued after o_free.
    const int wq = warp & 3;
    const int r_local = wq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    bool ok = true;
    int kt = 0, it = 0, rank, bh;
    for (int k = 0; ok; ++k) {
      const int step = sched_item(sched, cta, k, rank, bh);
      if (step == kDone) break;
      if (step == kSkip) continue;
      const int row = qtile_of(rank) * kBlockM + r_local;
      kt += ktiles(rank);
      if (!mbar_wait_warp(&stat_full, it & 1, &abort_flag)) {
        ok = false;
        break;
      }
      const float l_sum = st_l[r_local], m_used = st_m[r_local];
      mbar_arrive(&stat_empty);
      if (!mbar_wait_warp(&pv_done[(kt - 1) % kSBuf], ((kt - 1) / kSBuf) & 1, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // O = accumulator / l, whole-line row-segment stores
      store_tmem_rows<E, D>(tmem_O + lane_addr, 1.f / l_sum, o + (static_cast<size_t>(bh) * N + row) * D, D, N - row);
      if (row < N) lse[static_cast<size_t>(bh) * N + row] = (m_used * scale_log2 + log2f(l_sum)) * kLn2;
      tc_fence_before();
      mbar_arrive(&o_free);
      ++it;
    }
  };
  auto role_masks = [&](auto high) {
      // ---------------------------------------------------------- keep masks
      // Warp 8 + c draws keys 32c .. 32c + 31 of every key tile for rows
      // 4 lane .. 4 lane + 3 (no exchange between lanes), one tile ahead of
      // the softmax warps at most kMaskSlots, into a slot laid out word-major
      // (word c * 128 + r = keys 32c .. 32c + 31 of row r, bit keep_bit(b)
      // key 32c + b): one 16-byte store per lane, 512 contiguous bytes per
      // warp, in the same layout as the saved keep bits.
      static_assert(kMaskWarps * 32 == kBlockN && 4 * 32 == kBlockM, "one 4 x 32 block of bits per mask lane");
      constexpr bool kHigh = decltype(high)::value;
      const int wc = warp - 8;
      bool ok = true;
      int kt = 0, rank, bh;
      for (int k = 0; ok; ++k) {
        const int step = sched_item(sched, cta, k, rank, bh);
        if (step == kDone) break;
        if (step == kSkip) continue;
        const int qtile = qtile_of(rank);
        const int nk = ktiles(rank), row0 = qtile * kBlockM + 4 * lane;
        for (int j = 0; j < nk; ++j, ++kt) {
          const int ms = kt % kMaskSlots;
          if (kt >= kMaskSlots &&
              !mbar_wait_warp(&mask_empty[ms], ((kt / kMaskSlots) & 1) ^ 1, &abort_flag)) {
            ok = false;
            break;
          }
          const uint4 bits = dropout_block_bits<kHigh>(drop, static_cast<uint32_t>(bh), row0, j * kBlockN + 32 * wc);
          *reinterpret_cast<uint4 *>(smem + L::kMask + ms * kMaskSlotBytes + wc * 512 + 16 * lane) = bits;
          mbar_arrive(&mask_full[ms]);
          if (drop.mask)  // saved for the backward
            *reinterpret_cast<uint4 *>(drop.mask + dropout_block(drop, bh, qtile, j) / 4 + wc * 128 + 4 * lane) = bits;
        }
      }
  };
  if constexpr (DROP) {
    // The warps share the block's registers (384 x 168 with 4 mask warps,
    // 512 x 128 with 8): each warpgroup resizes its share at the top of its
    // branch (loaders and issuers 56, softmax 232, keep masks 96 per thread:
    // 49152 of the 64512, or 61440 of the 65536)
    if (warp < 4) {
      setmaxnreg_dec<56>();
      if (warp == 0) role_k_loader();
      else if (warp == 2) role_v_loader();
      else if (warp == 1) role_s_issuer();
      else role_pv_issuer();
    } else if (warp < 8) {
      setmaxnreg_inc<232>();
      role_softmax();
    } else {
      setmaxnreg_dec<96>();
      if (drop.t >= 128) role_masks(BoolTag<true>{});
      else role_masks(BoolTag<false>{});
    }
  } else if constexpr (EPI) {
    // 384 x 168 registers, resized as with dropout: loaders and issuers 56,
    // softmax 232, epilogue warps 96 (49152 of the 64512)
    if (warp < 4) {
      setmaxnreg_dec<56>();
      if (warp == 0) role_k_loader();
      else if (warp == 2) role_v_loader();
      else if (warp == 1) role_s_issuer();
      else role_pv_issuer();
    } else if (warp < 8) {
      setmaxnreg_inc<232>();
      role_softmax();
    } else {
      setmaxnreg_dec<96>();
      role_epilogue();
    }
  } else {
    if (warp == 0) role_k_loader();
    else if (warp == 2) role_v_loader();
    else if (warp == 1) role_s_issuer();
    else if (warp == 3) role_pv_issuer();
    else role_softmax();
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

template <int D, bool F16, bool DROP>
cudaError_t launch(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap *tmKhalf,
                   const CUtensorMap &tmV, void *o, float *lse, int B, int H, int N, int Nk, float scale,
                   int causal, const Dropout &drop, int *status, int num_sms, cudaStream_t stream) {
  const int BH = B * H, nt = (N + kBlockM - 1) / kBlockM;
  const int n_ktiles_all = (Nk + kBlockN - 1) / kBlockN, off = Nk - N;
  auto ktiles_q = [&](int qtile) {
    return causal ? std::min(n_ktiles_all, (qtile * kBlockM + kBlockM - 1 + off) / kBlockN + 1) : n_ktiles_all;
  };
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e;
  if constexpr (D == 128 && !DROP && FA_PAIR_KERNELS) {
    // pairs of query tiles on two-CTA clusters with M = 256 MMAs, when the
    // heads have at least two tiles (a lone tile would waste half the pair)
    using LP = FwdSmem<D, false, true>;
    auto kpair = fwd_kernel<D, F16, false, true>;
    static SmemOnce smem_pair;
    if (tmKhalf && nt >= 2) {
      if ((e = set_smem_once(reinterpret_cast<const void *>(kpair), LP::kAlloc, &smem_pair)) != cudaSuccess)
        return e;
      const int clusters =
          pair_grid(reinterpret_cast<const void *>(kpair), LP::kAlloc, kThreads, num_sms);
      if (clusters >= 1) {
        const int np = (nt + 1) / 2;
        // a pair costs the key tiles of its upper tile plus about one for the epilogues
        const TileSched sched = sched_cached(3, BH, N, Nk, causal != 0, np, clusters, [&](int rank) {
          return static_cast<long long>(ktiles_q(2 * (np - 1 - rank) + 1)) + 1;
        });
        timing_begin(stream);
        e = launch_pair_grid(kpair, sched.G, kThreads, LP::kAlloc, stream, tmQ, *tmKhalf, tmV,
                             static_cast<uint16_t *>(o), lse, N, Nk, sched, scale, scale_log2, causal, drop, status);
        timing_end(stream);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
      }
    }
  }
  using L = FwdSmem<D, DROP>;
  auto kern = fwd_kernel<D, F16, DROP, false>;
  static SmemOnce smem_set;
  e = set_smem_once(reinterpret_cast<const void *>(kern), L::kAlloc, &smem_set);
  if (e != cudaSuccess) return e;
  // persistent grid: at most one CTA per SM, each walking its static list of
  // query tiles; a tile costs its key tiles plus about one for its epilogue
  const TileSched sched = sched_cached(0, BH, N, Nk, causal != 0, nt, num_sms, [&](int rank) {
    return static_cast<long long>(ktiles_q(nt - 1 - rank)) + 1;
  });
  timing_begin(stream);
  kern<<<sched.G, fwd_threads<DROP, false>(), L::kAlloc, stream>>>(tmQ, tmK, tmV, static_cast<uint16_t *>(o), lse,
                                                  N, Nk, sched, scale, scale_log2, causal, drop, status);
  timing_end(stream);
  return cudaGetLastError();
}

template <bool DROP>
cudaError_t dispatch(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap *tmKhalf,
                     const CUtensorMap &tmV, void *o, float *lse, int B, int H, int N, int Nk, int d, float scale,
                     int causal, bool f16, const Dropout &drop, int *status, int num_sms, cudaStream_t stream) {
#define FA_FWD_LAUNCH(DD, FF)                                                                                  \
  return launch<DD, FF, DROP>(tmQ, tmK, tmKhalf, tmV, o, lse, B, H, N, Nk, scale, causal, drop, status, num_sms, \
                              stream)
  if (f16) {
    if (d == 64) FA_FWD_LAUNCH(64, true);
    if (d == 96) FA_FWD_LAUNCH(96, true);
    if (d == 256) FA_FWD_LAUNCH(256, true);
    FA_FWD_LAUNCH(128, true);
  }
  if (d == 64) FA_FWD_LAUNCH(64, false);
  if (d == 96) FA_FWD_LAUNCH(96, false);
  if (d == 256) FA_FWD_LAUNCH(256, false);
  FA_FWD_LAUNCH(128, false);
#undef FA_FWD_LAUNCH
}

}  // namespace

cudaError_t launch_fwd_16(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap *tmKhalf,
                          const CUtensorMap &tmV, void *o, float *lse, int B, int H, int N, int Nk, int d,
                          float scale, int causal, bool f16, const Dropout *drop, int *status, int num_sms,
                          cudaStream_t stream, int *launches) {
  *launches += 1;
  if (drop)
    return dispatch<true>(tmQ, tmK, tmKhalf, tmV, o, lse, B, H, N, Nk, d, scale, causal, f16, *drop, status,
                          num_sms, stream);
  return dispatch<false>(tmQ, tmK, tmKhalf, tmV, o, lse, B, H, N, Nk, d, scale, causal, f16, Dropout{}, status,
                         num_sms, stream);
}

}  // namespace fa
