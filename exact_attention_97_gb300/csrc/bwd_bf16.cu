// bwd_bf16.cu -- exact attention backward on the sm_103a tensor cores.
//
// What it computes (pages): backward by recomputation, "Flash Attention
// 原理与实现", section "Backward 的 Tiling 策略": the probabilities are rebuilt
// from Q, K and the saved statistic, p = exp(s - L) ("research-attention"
// tutorial, section 04), then
//     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D)  with D_i = sum_c dO_ic O_ic,
//     dQ = scale dS K,  dK = scale dS^T Q,
// and dQ, which every key block touches, is summed across blocks with fp32
// atomic adds (same blog, pitfalls item 3).
//
// Three kernels on one stream:
//   1. bwd_prep   D_i = dO_i . O_i (fp32), L_i in log2 units, both padded to
//                 whole 128-row tiles, and zeroing of the fp32 dQ
//                 accumulator; HBM-bound, 16-byte vector loads.
//   2. bwd_main   one CTA per (batch*head, 128-key block). K_j and V_j stay in
//                 shared memory; query tiles of 128 rows stream through a
//                 two-stage TMA ring (Q_i, dO_i). Per tile, five tcgen05 MMAs
//                 with fp32 accumulators in tensor memory (TMEM), keys on the
//                 TMEM lanes:
//                   S^T  = K Q_i^T        (TMEM)       -> P^T = 2^(s c - L_i log2 e)
//                   dP^T = V dO_i^T       (TMEM)       -> dS^T = P^T o (dP^T - D_i)
//                   dV  += P^T dO_i       (A = P^T read from TMEM as bf16)
//                   dK  += dS^T Q_i       (A = dS^T in shared memory)
//                   dQ_i = dS K           (d = 128: as dQ_i^T = K^T dS^T so a
//                                          warp's atomics hit 32 consecutive
//                                          floats; d = 64: rows of dQ_i)
//                 Warp roles: 0 TMA, 1 MMA issue, 2 TMEM allocation,
//                 4-7 P and dS (thread = key row), 8-11 dQ atomics and, at
//                 the end, the dK store; 4-7 also store dV.
//                 For d = 128 shared memory is short, so dS^T is written over
//                 the dO_i buffer once the dV MMA (its last reader) is done.
//   3. bwd_dq     dQ = scale * accumulator, rounded to bf16.
//
// TMEM columns (d = 128): S^T [0,128) with P^T over [0,64); dP^T [128,256),
//   reused by dQ^T after dS is built; dV [256,384); dK [384,512).
// TMEM columns (d = 64):  S^T [0,128); dP^T [128,256); dV [256,320);
//   dK [320,384); dQ [384,448).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kBlk = 128;       // keys per CTA and query rows per tile
constexpr int kThreads = 384;   // 12 warps
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kStages = (D == 128) ? 2 : 3;
  static constexpr int kTileBytes = kBlk * D * 2;
  static constexpr int kSubBytes = kBlk * 128;  // 128 rows x 64 bf16
  static constexpr bool kDsInDo = (D == 128);
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;
  static constexpr int kDO = kQ + kStages * kTileBytes;
  static constexpr int kDS = kDO + kStages * kTileBytes;  // only used when !kDsInDo
  static constexpr int kStage = kDS + (kDsInDo ? 0 : kBlk * kBlk * 2);  // dQ staging (d = 128)
  static constexpr int kStageRows = 32;                                 // query rows per chunk
  static constexpr int kBytes = kStage + (kDsInDo ? kStageRows * D * 4 : 0);
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns
  static constexpr uint32_t tS = 0, tDP = 128, tDV = 256, tDK = 256 + D, tDQ = (D == 128) ? 128 : 384;
};


__device__ __forceinline__ void load_rows(uint8_t *dst, const CUtensorMap *map, uint64_t *bar,
                                          int D, int row, int bh) {
  for (int x = 0; x < D; x += 64) tma_load_3d(dst + (x / 64) * (kBlk * 128), map, bar, x, row, bh);
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ------------------------------------------------------------------ kernel 1
// Per query row of a head padded to Np = 128*ceil(N/128) rows:
//   Lp = -L * log2(e) (so the main kernel forms p = 2^(s*c + Lp)), -inf past N;
//   Dp = sum_c dO_ic O_ic, 0 past N;
// and zeroing of the fp32 dQ accumulator rows. One group of D/8 threads per
// row, 16-byte loads.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o,
                                                       const __nv_bfloat16 *__restrict__ dO,
                                                       const float *__restrict__ lse,
                                                       float *__restrict__ Lp, float *__restrict__ Dp,
                                                       float *__restrict__ dq_acc, int N, int Np,
                                                       int64_t prow_total) {
  constexpr int kTpr = D / 8;  // threads per row
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t pr = gid / kTpr;  // padded row index
  const int part = static_cast<int>(gid % kTpr);
  const int64_t bh = pr / Np;
  const int i = static_cast<int>(pr % Np);
  const bool real = pr < prow_total && i < N;
  const int64_t r = bh * N + i;  // unpadded row
  float s = 0.f;
  if (real) {
    const uint4 a = *reinterpret_cast<const uint4 *>(o + r * D + part * 8);
    const uint4 b = *reinterpret_cast<const uint4 *>(dO + r * D + part * 8);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      s = fmaf(bf16lo(av[t]), bf16lo(bv[t]), s);
      s = fmaf(bf16hi(av[t]), bf16hi(bv[t]), s);
    }
    float4 *z = reinterpret_cast<float4 *>(dq_acc + r * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (pr < prow_total && part == 0) {
    Dp[pr] = real ? s : 0.f;
    Lp[pr] = real ? -lse[r] * kLog2e : -INFINITY;
  }
}

// ------------------------------------------------------------------ kernel 3
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float *__restrict__ dq_acc,
                                                     __nv_bfloat16 *__restrict__ dq, float scale,
                                                     int64_t n8) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4 *>(dq_acc)[2 * i];
  const float4 b = reinterpret_cast<const float4 *>(dq_acc)[2 * i + 1];
  uint4 r;
  r.x = pack_bf16x2(a.x * scale, a.y * scale);
  r.y = pack_bf16x2(a.z * scale, a.w * scale);
  r.z = pack_bf16x2(b.x * scale, b.y * scale);
  r.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4 *>(dq)[i] = r;
}

// ------------------------------------------------------------------ kernel 2
#ifndef FA_BWD_POLY_PAIRS
#define FA_BWD_POLY_PAIRS 0
#endif
constexpr int kBwdPolyPairs = FA_BWD_POLY_PAIRS;  // of every 8 exp pairs, this many on the FMA pipe

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmdO, const float *__restrict__ Lp,
                    const float *__restrict__ Dp, float *__restrict__ dq_acc,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, int N,
                    float scale, float scale_log2, int causal, int *status) {
  using C = BwdCfg<D>;
  constexpr int NST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t kv_full, qd_full[NST], qd_empty[NST], s_full, dp_full, p_ready, ds_ready,
      ds_free, dq_full, dq_free, dkdv_done, drain, stage_full, stage_free;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ __align__(16) float Lst[NST][kBlk], Dst[NST][kBlk];  // per stage, filled by bulk copy

  const int warp = warp_id(), lane = lane_id();
  const int n_tiles_all = (N + kBlk - 1) / kBlk;
  const int kb = blockIdx.x;  // low blocks see the most query tiles under the causal mask
  const int Np = n_tiles_all * kBlk;
  const int bh = blockIdx.y;
  const int i_first = causal ? kb : 0;
  const int n_tiles = n_tiles_all - i_first;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&kv_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&qd_full[s], 1);
      mbar_init(&qd_empty[s], 1);
    }
    mbar_init(&s_full, 1);
    mbar_init(&dp_full, 1);
    mbar_init(&p_ready, 128);
    mbar_init(&ds_ready, 128);
    mbar_init(&ds_free, 1);
    mbar_init(&dq_full, 1);
    mbar_init(&dq_free, 128);
    mbar_init(&dkdv_done, 1);
    mbar_init(&drain, 1);
    mbar_init(&stage_full, 128);
    mbar_init(&stage_free, 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(&kv_full, 2 * C::kTileBytes);
      load_rows(smem + C::kK, &tmK, &kv_full, D, kb * kBlk, bh);
      load_rows(smem + C::kV, &tmV, &kv_full, D, kb * kBlk, bh);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % NST;
        if (t >= NST && !mbar_wait(&qd_empty[st], ((t / NST) & 1) ^ 1, &abort_flag)) break;
        const int row = (i_first + t) * kBlk;
        mbar_arrive_expect_tx(&qd_full[st], 2 * C::kTileBytes + 2 * kBlk * 4);
        load_rows(smem + C::kQ + st * C::kTileBytes, &tmQ, &qd_full[st], D, row, bh);
        load_rows(smem + C::kDO + st * C::kTileBytes, &tmdO, &qd_full[st], D, row, bh);
        const size_t prow = static_cast<size_t>(bh) * Np + row;
        bulk_load(Lst[st], Lp + prow, kBlk * 4, &qd_full[st]);
        bulk_load(Dst[st], Dp + prow, kBlk * 4, &qd_full[st]);
        ++issued;
      }
      mbar_wait_drain(&kv_full, 0);
      for (int t = max(0, issued - NST); t < issued; ++t)
        mbar_wait_drain(&qd_full[t % NST], (t / NST) & 1);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // Order per tile t: dP_t, dV_t, S_{t+1}, dK_t, dQ_t. S_{t+1} goes ahead of
    // dK_t and dQ_t so that P_{t+1} is built while those two run.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(kBlk, kBlk, false, false);   // S^T, dP^T
      constexpr uint32_t id_kv = idesc_bf16(kBlk, D, false, true);      // dV, dK
      constexpr uint32_t id_dq =
          (D == 128) ? idesc_bf16(D, kBlk, true, true) : idesc_bf16(kBlk, D, true, true);
      const uint32_t k_addr = smem_u32(smem + C::kK), v_addr = smem_u32(smem + C::kV);
      auto issue_s = [&](int t) -> bool {  // S^T_t = K Q_t^T into the S columns
        const int st = t % NST;
        if (!mbar_wait(&qd_full[st], (t / NST) & 1, &abort_flag)) return false;
        tc_fence_after();
        const uint32_t q_addr = smem_u32(smem + C::kQ + st * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::kSubBytes + (kk % 4) * 32;
          mma_ss(tmem + C::tS, sdesc_sw128(k_addr + off, 16, 1024),
                 sdesc_sw128(q_addr + off, 16, 1024), id_s, kk > 0);
        }
        mma_commit(&s_full);
        return true;
      };
      bool ok = mbar_wait(&kv_full, 0, &abort_flag) && issue_s(0);
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int st = t % NST;
        const uint32_t ph = t & 1;
        const uint32_t q_addr = smem_u32(smem + C::kQ + st * C::kTileBytes);
        const uint32_t do_addr = smem_u32(smem + C::kDO + st * C::kTileBytes);
        const uint32_t ds_addr = C::kDsInDo ? do_addr : smem_u32(smem + C::kDS);
        // dP^T = V dO^T; with d = 128 its columns held dQ^T of the last tile
        if (C::kDsInDo && t > 0) {
          if (!mbar_wait(&dq_free, (t - 1) & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::kSubBytes + (kk % 4) * 32;
          mma_ss(tmem + C::tDP, sdesc_sw128(v_addr + off, 16, 1024),
                 sdesc_sw128(do_addr + off, 16, 1024), id_s, kk > 0);
        }
        mma_commit(&dp_full);
        // dV += P^T dO  (P^T as bf16 in TMEM columns [0,64))
        if (!mbar_wait(&p_ready, ph, &abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ts(tmem + C::tDV, tmem + C::tS + kk * 8, sdesc_sw128(do_addr + kk * 2048, C::kSubBytes, 1024),
                 id_kv, (t > 0 || kk > 0) ? 1u : 0u);
        if (C::kDsInDo) mma_commit(&ds_free);  // dO buffer may now take dS^T
        if (!mbar_wait(&ds_ready, ph, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        // the S columns are free again (P_t read by dV_t and by the dS pass)
        if (t + 1 < n_tiles && !issue_s(t + 1)) { ok = false; break; }
        // dK += dS^T Q
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::kSubBytes + (kk % 4) * 32;
          mma_ss(tmem + C::tDK, sdesc_sw128(ds_addr + off, 16, 1024),
                 sdesc_sw128(q_addr + kk * 2048, C::kSubBytes, 1024), id_kv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        // dQ
        if (!C::kDsInDo && t > 0) {
          if (!mbar_wait(&dq_free, (t - 1) & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk) {
          if (D == 128)  // dQ^T = K^T dS^T : A = K (MN-major), B = dS^T (MN-major)
            mma_ss(tmem + C::tDQ, sdesc_sw128(k_addr + kk * 2048, C::kSubBytes, 1024),
                   sdesc_sw128(ds_addr + kk * 2048, C::kSubBytes, 1024), id_dq, kk > 0);
          else  // dQ = dS K : A = dS (MN-major view of dS^T), B = K (MN-major)
            mma_ss(tmem + C::tDQ, sdesc_sw128(ds_addr + kk * 2048, C::kSubBytes, 1024),
                   sdesc_sw128(k_addr + kk * 2048, C::kSubBytes, 1024), id_dq, kk > 0);
        }
        mma_commit(&dq_full);
        mma_commit(&qd_empty[st]);
        if (!C::kDsInDo) mma_commit(&ds_free);
      }
      if (ok) mma_commit(&dkdv_done);
      mma_commit(&drain);
      mbar_wait_drain(&drain, 0);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ P, dS
    const int wq = warp - 4;
    const int kr = wq * 32 + lane;  // key row within the block (TMEM lane)
    const int key = kb * kBlk + kr;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint64_t cc = f2_pack(scale_log2, scale_log2);
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const uint32_t ph = t & 1;
      const int st = t % NST;
      const int q0 = (i_first + t) * kBlk;
      // -L log2(e) and D of this query tile arrive with Q and dO
      if (!mbar_wait_warp(&qd_full[st], (t / NST) & 1, &abort_flag)) { ok = false; break; }
      const float2 *L2 = reinterpret_cast<const float2 *>(Lst[st]);
      const float2 *D2 = reinterpret_cast<const float2 *>(Dst[st]);
      // queries below qmin see nothing of this key (causal); keys past N see nothing
      const int qmin = (key >= N) ? (q0 + kBlk) : (causal ? key : 0);
      if (!mbar_wait_warp(&s_full, ph, &abort_flag)) { ok = false; break; }
      tc_fence_after();
      // P^T = 2^(s c - L log2 e), in two halves of 64 query columns; half h is
      // written as 32 packed pairs into columns [32h, 32h+32), over scores
      // that have already been read
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[64];
        tmem_ld64(tmem + lane_addr + C::tS + h * 64, r);
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int c0 = h * 64 + 2 * u;
          const float2 nl = L2[c0 / 2];
          const uint64_t x2 =
              f2_fma(f2_pack(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])), cc, f2_pack(nl.x, nl.y));
          float p0, p1;
          if ((u & 7) < kBwdPolyPairs) {
            f2_unpack(ex2_poly2(x2), p0, p1);
          } else {
            float x0, x1;
            f2_unpack(x2, x0, x1);
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
          }
          if (q0 + c0 < qmin) p0 = 0.f;
          if (q0 + c0 + 1 < qmin) p1 = 0.f;
          pk[u] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tmem + lane_addr + C::tS + h * 32, pk);
      }
      tc_fence_before();
      mbar_arrive(&p_ready);
      // dS^T = P^T o (dP^T - D), in the same two halves
      if (!mbar_wait_warp(&dp_full, ph, &abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint8_t *dsb = C::kDsInDo ? (smem + C::kDO + st * C::kTileBytes) : (smem + C::kDS);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[64], pp[32];
        tmem_ld64(tmem + lane_addr + C::tDP + h * 64, r);
        tmem_ld32(tmem + lane_addr + C::tS + h * 32, pp);
        uint32_t ds[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const float2 dd = D2[h * 32 + u];
          const float d0 = bf16lo(pp[u]) * (__uint_as_float(r[2 * u]) - dd.x);
          const float d1 = bf16hi(pp[u]) * (__uint_as_float(r[2 * u + 1]) - dd.y);
          ds[u] = pack_bf16x2(d0, d1);
        }
        if (h == 0) {
          // the buffer dS^T goes to must be free of its last tensor-core reader
          const uint32_t fph = C::kDsInDo ? ph : ((t - 1) & 1);
          if ((C::kDsInDo || t > 0) && !mbar_wait_warp(&ds_free, fph, &abort_flag)) { ok = false; break; }
          tc_fence_after();
        }
        // row kr of dS^T, queries [64h, 64h+64): one 128-byte swizzled row of sub-tile h
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 *dst = reinterpret_cast<uint4 *>(dsb + h * C::kSubBytes + kr * 128 + ((c ^ (kr & 7)) << 4));
          *dst = make_uint4(ds[4 * c], ds[4 * c + 1], ds[4 * c + 2], ds[4 * c + 3]);
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();
      mbar_arrive(&ds_ready);
    }
    // epilogue: dV rows
    if (ok && mbar_wait_warp(&dkdv_done, 0, &abort_flag)) {
      tc_fence_after();
      __nv_bfloat16 *out = dv + (static_cast<size_t>(bh) * N + key) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + C::tDV + ch * 32, r);
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
        if (key < N) {
          uint4 *dst = reinterpret_cast<uint4 *>(out + ch * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------- dQ drain, dK
    const int wq = warp - 8;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const bool issuer = (warp == 8 && lane == 0);
    bool ok = true;
    int chunks = 0;  // staging chunks handed to the copy engine so far
    for (int t = 0; t < n_tiles; ++t) {
      const int q0 = (i_first + t) * kBlk;
      const int nq = min(kBlk, N - q0);
      if (!mbar_wait_warp(&dq_full, t & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after();
      if (D == 128) {
        // lane = head dimension c, columns = queries. Read the whole tile,
        // release the TMEM columns, then push it to the fp32 accumulator in
        // 32-row chunks through the staging buffer and bulk reduce-adds.
        uint32_t r[128];
        tmem_ld128(tmem + lane_addr + C::tDQ, r);
        tc_fence_before();
        mbar_arrive(&dq_free);
        const int c = wq * 32 + lane;
        float *stage = reinterpret_cast<float *>(smem + C::kStage);
#pragma unroll
        for (int ch = 0; ch < kBlk / C::kStageRows; ++ch) {
          const int rows = min(C::kStageRows, nq - ch * C::kStageRows);
          if (rows <= 0) break;
          if (chunks > 0 && !mbar_wait_warp(&stage_free, (chunks - 1) & 1, &abort_flag)) { ok = false; break; }
#pragma unroll
          for (int u = 0; u < C::kStageRows; ++u) stage[u * D + c] = __uint_as_float(r[ch * C::kStageRows + u]);
          fence_proxy_async_smem();
          mbar_arrive(&stage_full);
          if (issuer) {
            if (!mbar_wait(&stage_full, chunks & 1, &abort_flag)) { ok = false; break; }
            bulk_reduce_add_f32(dq_acc + (static_cast<size_t>(bh) * N + q0 + ch * C::kStageRows) * D, stage,
                                static_cast<uint32_t>(rows) * D * 4);
            bulk_commit();
            bulk_wait_read_all();
            mbar_arrive(&stage_free);
          }
          ++chunks;
        }
        if (!ok) break;
      } else {
        // lane = query row, columns = head dimension
        const int q = q0 + wq * 32 + lane;
        float4 *base = reinterpret_cast<float4 *>(dq_acc + (static_cast<size_t>(bh) * N + q) * D);
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_addr + C::tDQ + ch * 32, r);
          if (q < N) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              atomicAdd(base + ch * 8 + u, make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                                       __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])));
          }
        }
        tc_fence_before();
        mbar_arrive(&dq_free);
      }
    }
    if (issuer) bulk_wait_all();  // every reduce-add has landed before the CTA ends
    // epilogue: dK rows (times scale)
    if (ok && mbar_wait_warp(&dkdv_done, 0, &abort_flag)) {
      tc_fence_after();
      const int key = kb * kBlk + wq * 32 + lane;
      __nv_bfloat16 *out = dk + (static_cast<size_t>(bh) * N + key) * D;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + C::tDK + ch * 32, r);
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(__uint_as_float(r[2 * u]) * scale, __uint_as_float(r[2 * u + 1]) * scale);
        if (key < N) {
          uint4 *dst = reinterpret_cast<uint4 *>(out + ch * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && abort_flag) atomicExch(status, kErrTimeout);
}

template <int D>
cudaError_t launch(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                   const CUtensorMap &tmdO, const void *o, const void *dO, const float *lse,
                   void *dq, void *dk, void *dv, float *dq_acc, float *Lp, float *Dp, int B, int H,
                   int N, float scale, int causal, int *status, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int64_t rows = static_cast<int64_t>(B) * H * N;
  const int Np = (N + kBlk - 1) / kBlk * kBlk;
  {
    const int64_t prows = static_cast<int64_t>(B) * H * Np;
    const int64_t threads = prows * (D / 8);
    bwd_prep_kernel<D><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dO), lse, Lp, Dp,
        dq_acc, N, Np, prows);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = bwd_main_kernel<D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((N + kBlk - 1) / kBlk, B * H);
  timing_begin(stream);
  kern<<<grid, kThreads, C::kAlloc, stream>>>(tmQ, tmK, tmV, tmdO, Lp, Dp, dq_acc,
                                               static_cast<__nv_bfloat16 *>(dk),
                                               static_cast<__nv_bfloat16 *>(dv), N, scale,
                                               scale * kLog2e, causal, status);
  timing_end(stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n8 = rows * D / 8;
  bwd_dq_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16 *>(dq), scale, n8);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_bf16(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                            const CUtensorMap &tmdO, const void *o, const void *dO,
                            const float *lse, void *dq, void *dk, void *dv, float *dq_acc,
                            float *Lp, float *Dp, int B, int H, int N, int d, float scale,
                            int causal, int *status, int num_sms, cudaStream_t stream,
                            int *launches) {
  (void)num_sms;
  *launches += 3;
  if (d == 64)
    return launch<64>(tmQ, tmK, tmV, tmdO, o, dO, lse, dq, dk, dv, dq_acc, Lp, Dp, B, H, N, scale,
                      causal, status, stream);
  return launch<128>(tmQ, tmK, tmV, tmdO, o, dO, lse, dq, dk, dv, dq_acc, Lp, Dp, B, H, N, scale,
                     causal, status, stream);
}

}  // namespace fa
