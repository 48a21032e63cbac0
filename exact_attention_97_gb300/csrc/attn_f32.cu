// attn_f32.cu -- fp32 exact attention on the CUDA cores (FFMA), forward and
// backward. This is the path for float tensors and any head size 1..128; it
// exists because tensor-core TF32 (10-bit mantissa) cannot hold the 1e-4
// absolute error bound asked of fp32 inputs.
//
// Forward follows the tiled loop of "Flash Attention 原理与实现", section
// "Forward 的 Tiling 策略", with the running state (m, l, u) and rescale
// alpha = exp(m - m') of the "research-attention" tutorial, section 02: one
// warp owns one query row, keys arrive in chunks of 32 staged in shared memory,
// and the row is divided by l once at the end. L = m + ln l is saved
// (tutorial section 04).
//
// Backward recomputes p_ij = exp(s_ij - L_i) (tutorial section 04) and forms
// dV += p dO, dP = dO V^T, dS = p (dP - D_i), dQ = scale dS K,
// dK += scale dS^T Q (blog section "Backward 的 Tiling 策略"); the warp that
// owns query row i accumulates dQ_i in registers, and dK/dV rows, shared by
// all queries, are accumulated with fp32 atomic adds (blog, pitfalls item 3).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"

namespace fa {
namespace {

constexpr int kRowsPerBlock = 4;  // one warp per query row
constexpr int kChunk = 32;        // keys per shared-memory chunk

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Shared layout: Ks [kChunk][d+1] (padded: lanes read different rows),
// Vs [kChunk][d], per-warp rows [kRowsPerBlock][2][d] (q and dO).
__device__ __forceinline__ void load_chunk(float *Ks, float *Vs, const float *k, const float *v,
                                           int k0, int N, int d) {
  for (int idx = threadIdx.x; idx < kChunk * d; idx += blockDim.x) {
    const int j = idx / d, c = idx % d;
    const bool in = (k0 + j) < N;
    Ks[j * (d + 1) + c] = in ? k[(size_t)(k0 + j) * d + c] : 0.f;
    Vs[j * d + c] = in ? v[(size_t)(k0 + j) * d + c] : 0.f;
  }
}

__global__ void __launch_bounds__(kRowsPerBlock * 32)
    fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                   const float *__restrict__ v, float *__restrict__ o, float *__restrict__ lse,
                   int N, int d, float scale, int causal) {
  extern __shared__ float sm[];
  float *Ks = sm;
  float *Vs = Ks + kChunk * (d + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *qs = Vs + kChunk * d + warp * d;
  const size_t head = (size_t)blockIdx.y * N * d;
  const int row0 = blockIdx.x * kRowsPerBlock;
  const int i = row0 + warp;
  const bool active = i < N;
  if (active)
    for (int c = lane; c < d; c += 32) qs[c] = q[head + (size_t)i * d + c];

  float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int kend = causal ? min(N, row0 + kRowsPerBlock) : N;
  for (int k0 = 0; k0 < kend; k0 += kChunk) {
    __syncthreads();
    load_chunk(Ks, Vs, k + head, v + head, k0, N, d);
    __syncthreads();
    if (!active) continue;
    const int j = k0 + lane;
    const bool vis = j < N && (!causal || j <= i);
    float s = -INFINITY;
    if (vis) {
      float t = 0.f;
      const float *kr = Ks + lane * (d + 1);
      for (int c = 0; c < d; ++c) t = fmaf(qs[c], kr[c], t);
      s = t * scale;
    }
    const float m_new = fmaxf(m, warp_max(s));
    if (m_new == -INFINITY) continue;  // nothing visible yet: state unchanged
    const float alpha = expf(m - m_new);
    const float p = vis ? expf(s - m_new) : 0.f;
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[t] *= alpha;
    for (int jj = 0; jj < kChunk; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      if (pj == 0.f) continue;
      const float *vr = Vs + jj * d;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int c = lane + 32 * t;
        if (c < d) acc[t] = fmaf(pj, vr[c], acc[t]);
      }
    }
    m = m_new;
  }
  if (!active) return;
  const float inv_l = 1.f / l;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int c = lane + 32 * t;
    if (c < d) o[head + (size_t)i * d + c] = acc[t] * inv_l;
  }
  if (lane == 0) lse[(size_t)blockIdx.y * N + i] = m + logf(l);
}

// D_i = sum_c dO_ic O_ic, one warp per row.
__global__ void bwd_f32_rowdot_kernel(const float *__restrict__ o, const float *__restrict__ dO,
                                      float *__restrict__ D, int64_t rows, int d) {
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) s = fmaf(o[r * d + c], dO[r * d + c], s);
  s = warp_sum(s);
  if (lane == 0) D[r] = s;
}

__global__ void __launch_bounds__(kRowsPerBlock * 32)
    bwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                   const float *__restrict__ v, const float *__restrict__ lse,
                   const float *__restrict__ dO, const float *__restrict__ D,
                   float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dv, int N,
                   int d, float scale, int causal) {
  extern __shared__ float sm[];
  float *Ks = sm;
  float *Vs = Ks + kChunk * (d + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *qs = Vs + kChunk * d + warp * 2 * d;
  float *dos = qs + d;
  const size_t head = (size_t)blockIdx.y * N * d;
  const int row0 = blockIdx.x * kRowsPerBlock;
  const int i = row0 + warp;
  const bool active = i < N;
  float Li = 0.f, Di = 0.f;
  if (active) {
    for (int c = lane; c < d; c += 32) {
      qs[c] = q[head + (size_t)i * d + c];
      dos[c] = dO[head + (size_t)i * d + c];
    }
    Li = lse[(size_t)blockIdx.y * N + i];
    Di = D[(size_t)blockIdx.y * N + i];
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int kend = causal ? min(N, row0 + kRowsPerBlock) : N;
  for (int k0 = 0; k0 < kend; k0 += kChunk) {
    __syncthreads();
    load_chunk(Ks, Vs, k + head, v + head, k0, N, d);
    __syncthreads();
    if (!active) continue;
    const int j = k0 + lane;
    const bool vis = j < N && (!causal || j <= i);
    float p = 0.f, ds = 0.f;
    if (vis) {
      float s = 0.f, dp = 0.f;
      const float *kr = Ks + lane * (d + 1);
      const float *vr = v + head + (size_t)j * d;
      for (int c = 0; c < d; ++c) {
        s = fmaf(qs[c], kr[c], s);
        dp = fmaf(dos[c], vr[c], dp);
      }
      p = expf(s * scale - Li);
      ds = p * (dp - Di);
    }
    for (int jj = 0; jj < kChunk; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const float dsj = __shfl_sync(0xffffffffu, ds, jj);
      if (pj == 0.f && dsj == 0.f) continue;
      const float *kr = Ks + jj * (d + 1);
      float *dkr = dk + head + (size_t)(k0 + jj) * d;
      float *dvr = dv + head + (size_t)(k0 + jj) * d;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int c = lane + 32 * t;
        if (c < d) {
          acc[t] = fmaf(scale * dsj, kr[c], acc[t]);
          atomicAdd(dkr + c, scale * dsj * qs[c]);
          atomicAdd(dvr + c, pj * dos[c]);
        }
      }
    }
  }
  if (!active) return;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int c = lane + 32 * t;
    if (c < d) dq[head + (size_t)i * d + c] = acc[t];
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int B, int H, int N, int d, float scale, int causal,
                           cudaStream_t stream, int *launches) {
  const size_t smem = sizeof(float) * (kChunk * (d + 1) + kChunk * d + kRowsPerBlock * d);
  dim3 grid((N + kRowsPerBlock - 1) / kRowsPerBlock, B * H);
  fwd_f32_kernel<<<grid, kRowsPerBlock * 32, smem, stream>>>(q, k, v, o, lse, N, d, scale, causal);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *lse, const float *dO, float *dq, float *dk, float *dv,
                           int B, int H, int N, int d, float scale, int causal, float *D,
                           cudaStream_t stream, int *launches) {
  const int64_t rows = (int64_t)B * H * N;
  const size_t bytes = sizeof(float) * (size_t)rows * d;
  cudaError_t e = cudaMemsetAsync(dk, 0, bytes, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, bytes, stream);
  if (e != cudaSuccess) return e;
  bwd_f32_rowdot_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(o, dO, D, rows, d);
  const size_t smem =
      sizeof(float) * (kChunk * (d + 1) + kChunk * d + kRowsPerBlock * 2 * d);
  dim3 grid((N + kRowsPerBlock - 1) / kRowsPerBlock, B * H);
  bwd_f32_kernel<<<grid, kRowsPerBlock * 32, smem, stream>>>(q, k, v, lse, dO, D, dq, dk, dv, N,
                                                             d, scale, causal);
  *launches += 2;
  return cudaGetLastError();
}

}  // namespace fa
