// kernels.h -- internal launchers behind the C ABI (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace fa {

// Dropout on the attention probabilities: element (i, j) of head h is kept
// iff byte j mod 4 of word i mod 4 of Philox4x32-10 with counter
// (j/4, i/4, head_base + h, offset) and key (k0, k1) is >= t; kept
// probabilities are scaled by inv_keep = 256 / (256 - t).
//
// Saved keep bits (mask != nullptr): the forward also writes every visited
// tile's bits there, and the backward passes read them instead of drawing
// them again. Layout: for head bh, query tile qt, key tile kt, a 2 KB block
// at ((bh * n_qt + qt) * n_kt + kt) * 2048 bytes of 512 words, word-major:
// bit 8 (b mod 4) + b / 4 (keep_bit(b), sm103.cuh) of word w * 128 + r is the
// keep bit of (query 128 qt + r, key 128 kt + 32 w + b). A row owner reads
// one word per 32 keys (coalesced across rows); the key owners of a warp
// take 32 consecutive words at once and transpose them.
struct Dropout {
  uint32_t k0, k1;  // the 64-bit seed, low word first
  uint32_t offset;
  uint32_t head_base;  // index of the call's first head in a larger problem
  uint32_t t;       // byte threshold, 0..255
  float inv_keep;
  uint32_t *mask;   // saved keep bits, or nullptr (draw them)
  int n_qt, n_kt;   // query and key tiles per head of the saved layout
  // backward only: the dK/dV pass draws the bits and writes them to `mask`,
  // and the dQ pass reads them there (0: both passes read `mask` if given)
  int dkdv_writes_mask;
};

// Byte offset of the saved keep bits of tile (qt, kt) of head bh.
__host__ __device__ inline size_t dropout_block(const Dropout &d, size_t bh, int qt, int kt) {
  return ((bh * static_cast<size_t>(d.n_qt) + qt) * static_cast<size_t>(d.n_kt) + kt) * 2048;
}

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
  kErrArg = 9,
  kErrCheck = 10  // only with FA_CHECKED: a device-side argument check failed
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

// ----------------------------------------------------------- CTA-pair grids
// Largest number of two-CTA clusters of `kernel` (threads per CTA, dynamic
// shared memory per CTA) that fit on the current device at once; 0 if none.
// Looked up once per kernel and device (the kernel's shared-memory attribute
// must already be set).
int max_pair_clusters(const void *kernel, int smem_bytes, int threads);

// The two-CTA (pair) kernels of d = 128 -- the forward and both backward
// passes with M = 256 MMAs split over the two SMs of a cluster -- are built
// only with FA_PAIR_KERNELS=1. On GB300 they run at the per-SM rate of the
// one-CTA kernels (the products keep N = 128, and that instruction rate, not
// operand traffic, bounds these kernels), so the default build leaves them out.
#ifndef FA_PAIR_KERNELS
#define FA_PAIR_KERNELS 0
#endif

// Clusters of a persistent pair kernel's grid: one per two SMs, at most as
// many as fit at once.
inline int pair_grid(const void *kernel, int smem_bytes, int threads, int num_sms) {
  const int fit = max_pair_clusters(kernel, smem_bytes, threads);
  const int want = num_sms / 2;
  return fit < want ? fit : want;
}

// Launches `kern` on `clusters` two-CTA clusters (grid 2 * clusters).
template <class Kern, class... Args>
cudaError_t launch_pair_grid(Kern kern, int clusters, int threads, int smem_bytes, cudaStream_t stream,
                             Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

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
// 128-byte swizzle; tmKhalf (may be null) is K's map with a {64, 64, 1} box,
// which the two-CTA (pair) kernel of d = 128 needs.
cudaError_t launch_fwd_16(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap *tmKhalf,
                          const CUtensorMap &tmV, void *o, float *lse, int B, int H, int N, int Nk, int d,
                          float scale, int causal, bool f16, const Dropout *drop, int *status, int num_sms,
                          cudaStream_t stream, int *launches);

// Load maps with {64, 64, 1} boxes (half tiles) of the backward's inputs, for
// the two-CTA (pair) kernels of d = 128.
struct HalfMaps {
  CUtensorMap q, k, v, dO;
};

// 16-bit tensor-core backward (three kernels: row terms, dK/dV pass, dQ
// pass). Lp and Dp are [B*H][Np] fp32 with Np = 128*ceil(N/128), in the
// caller's workspace. tmdK / tmdV are store maps {d, Nk, B*H} of dk / dv with
// a {16, 32, 1} box and 32-byte swizzle. `half` may be null (no pair kernels).
// Optional second stream for the backward: when the dK/dV and dQ grids fit
// on the GPU together, the dQ pass runs on `stream` forked from the caller's
// stream after the row-term kernel (event `fork`) and joins it back (`join`).
struct BwdSide {
  cudaStream_t stream;
  cudaEvent_t fork, join;
};

cudaError_t launch_bwd_16(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          const CUtensorMap &tmdO, const CUtensorMap &tmdK, const CUtensorMap &tmdV,
                          const HalfMaps *half, const void *o, const void *dO, const float *lse, void *dq, void *dk,
                          void *dv, float *Lp, float *Dp, int B, int H, int N, int Nk, int d, float scale, int causal,
                          bool f16, const Dropout *drop, int *status, int num_sms, cudaStream_t stream,
                          const BwdSide &side, int *launches);

}  // namespace fa
