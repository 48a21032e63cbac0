// kernels.h -- internal launchers behind the C ABI (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace fa {

// Dropout on the attention probabilities: element (i, j) of head h is kept
// iff byte j mod 4 of word i mod 4 of Philox4x32-10 with counter
// (j/4, i/4, head_base + h, offset) and key (k0, k1) is >= t; kept
// probabilities are scaled by inv_keep = 256 / (256 - t).
struct Dropout {
  uint32_t k0, k1;  // the 64-bit seed, low word first
  uint32_t offset;
  uint32_t head_base;  // index of the call's first head in a larger problem
  uint32_t t;       // byte threshold, 0..255
  float inv_keep;
};

// Error codes shared with include/fa.h (kept numerically identical).
enum : int {
  kOk = 0,
  kErrNull = 1,
  kErrShape = 2,
  kErrUnsupported = 3,
  kErrAlign = 4,
  kErrWorkspace = 5,
  kErrLaunch = 6,
  kErrTimeout = 7,
  kErrArch = 8,
  kErrArg = 9
};

// Benchmark timing hook: records the next free event pair (if any) around a
// main kernel. `begin` records the first event, `end` the second and advances.
void timing_begin(cudaStream_t stream);

void timing_end(cudaStream_t stream);

// A kernel instance's record of where its dynamic shared-memory limit has been
// raised: per device ordinal, the context epoch it was set in (0 = never).
// Function attributes belong to a context, so a device reset (a new primary
// context, hence a new epoch) makes the library set them again.
struct SmemOnce {
  std::atomic<uint32_t> epoch[64];
};

// Sets a kernel's dynamic shared-memory limit once per device and context
// (ordinals past 63 are set on every call). Call after the entry point has
// looked up its device (the epoch comes from that lookup).
cudaError_t set_smem_once(const void *kernel, int bytes, SmemOnce *done);

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int B, int H, int N, int d, float scale, int causal,
                           cudaStream_t stream, int *launches);

cudaError_t launch_bwd_f32(const float *q, const float *k, const float *v, const float *o,
                           const float *lse, const float *dO, float *dq, float *dk, float *dv,
                           int B, int H, int N, int d, float scale, int causal, float *D,
                           cudaStream_t stream, int *launches);

// N query rows and Nk key rows per head (causal: bottom-right aligned, Nk >= N).
// 16-bit tensor-core forward (bf16, or f16 when `f16`). tmQ/tmK/tmV are 3-D
// tensor maps {d, N, B*H} of that element type with a {64, 128, 1} box and
// 128-byte swizzle.
cudaError_t launch_fwd_16(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          void *o, float *lse, int B, int H, int N, int Nk, int d, float scale, int causal,
                          bool f16, const Dropout *drop, int *status, int num_sms, cudaStream_t stream,
                          int *launches);

// 16-bit tensor-core backward (three kernels: row terms, dK/dV pass, dQ
// pass). Lp and Dp are [B*H][Np] fp32 with Np = 128*ceil(N/128), in the
// caller's workspace. tmdK / tmdV are store maps {d, Nk, B*H} of dk / dv with
// a {16, 32, 1} box and 32-byte swizzle.
cudaError_t launch_bwd_16(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          const CUtensorMap &tmdO, const CUtensorMap &tmdK, const CUtensorMap &tmdV,
                          const void *o, const void *dO, const float *lse,
                          void *dq, void *dk, void *dv, float *Lp, float *Dp, int B, int H, int N, int Nk, int d,
                          float scale, int causal, bool f16, const Dropout *drop, int *status, int num_sms,
                          cudaStream_t stream, int *launches);

}  // namespace fa
