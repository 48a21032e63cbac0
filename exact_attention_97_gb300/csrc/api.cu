// api.cu -- the exported C ABI (include/fa.h): argument checks, tensor-map
// construction and kernel launches. Nothing here allocates device memory or
// synchronises, except fa_device_status, which is documented to.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/fa.h"
#include "kernels.h"

namespace {

using namespace fa;

// Kernels record FA_ERR_TIMEOUT here when they give up on a wait.
__device__ int g_fa_status = 0;

thread_local int t_last_cuda_error = 0;
thread_local int t_last_launches = 0;
thread_local void **t_events = nullptr;
thread_local int t_event_pairs = 0;
thread_local int t_event_next = 0;

constexpr int kMaxDevices = 64;
// Per-device state, valid for one CUDA context: the status word's and the
// static scratch's device addresses belong to the context that loaded this
// library's module, so a new primary context (after cudaDeviceReset) makes
// every entry look them up again (the epoch also re-arms set_smem_once).
struct DeviceInfo {
  bool ready = false;
  CUcontext ctx = nullptr;
  int ok_arch = 0;
  int num_sms = 0;
  int *status = nullptr;
  unsigned char *scratch = nullptr;  // fa_bwd_static_scratch's array, looked up on first use
};
DeviceInfo g_dev[kMaxDevices];
std::atomic<uint32_t> g_epoch[kMaxDevices];  // context epoch per device (0 = none yet)
uint32_t g_epoch_next = 0;                   // under g_dev_mutex
std::mutex g_dev_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn g_ctx_get = nullptr;
std::once_flag g_ctx_once;

// The calling thread's current CUDA context (nullptr if none yet, or if the
// driver entry point is unavailable).
CUcontext current_context() {
  std::call_once(g_ctx_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
  });
  CUcontext c = nullptr;
  if (g_ctx_get && g_ctx_get(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

int record(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return e == cudaSuccess ? kOk : kErrLaunch;
}

// Looks up whether the current device is sm_103, its SM count and the address
// of the status word: once per device and context.
int current_device(DeviceInfo **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record(e);
  if (dev < 0 || dev >= kMaxDevices) return kErrArch;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo &d = g_dev[dev];
  if (d.ready && d.ok_arch && current_context() != d.ctx) d.ready = false;  // the context was replaced
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return record(e);
    d.ok_arch = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.status = nullptr;
    d.scratch = nullptr;
    if (d.ok_arch) {
      void *p = nullptr;  // also brings up the context and this library's module
      if ((e = cudaGetSymbolAddress(&p, g_fa_status)) != cudaSuccess) return record(e);
      d.status = static_cast<int *>(p);
      d.ctx = current_context();
    }
    g_epoch[dev].store(++g_epoch_next, std::memory_order_release);
    d.ready = true;
  }
  if (!d.ok_arch) return kErrArch;
  *out = &d;
  return kOk;
}

// A side stream and a fork / join event pair per host thread and device
// (and context): the backward runs its two passes concurrently on the
// caller's stream and this one when both grids fit on the GPU together.
// Per thread, so that concurrent callers never share the events.
struct SideStream {
  CUcontext ctx = nullptr;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream t_side[kMaxDevices];

// This thread's side stream on the current device, created on first use
// (nullptr members if creation fails: the passes then run one after the other).
const SideStream *side_stream(int dev, CUcontext ctx) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream &s = t_side[dev];
  if (s.stream && s.ctx == ctx) return &s;
  s = SideStream{};  // a replaced context took the old handles with it
  if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    s = SideStream{};
    return nullptr;
  }
  s.ctx = ctx;
  return &s;
}

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode ? kOk : kErrLaunch;
}

// 3-D map over a contiguous [BH][N][d] 16-bit tensor (bf16, or f16 when
// `f16`): dims {d, N, BH}, box {64, box_rows, 1}, 128-byte swizzle; rows past
// N (inside a head) read as zero.
int encode_map(CUtensorMap *map, const void *ptr, int BH, int N, int d, bool f16, int box_rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return kErrLaunch;
  }
  return kOk;
}

// Map for the backward's dK / dV stores: 32-row x 16-column boxes with a
// 32-byte swizzle, written from per-warp staging buffers. Rows past `N` in a
// box are not written.
int encode_store_map(CUtensorMap *map, void *ptr, int BH, int N, int d, bool f16) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {16, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr,
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return kErrLaunch;
  }
  return kOk;
}

// Tensor maps depend only on the address, the shape, the element type and
// the box / swizzle kind, so repeated calls on the same buffers (a training
// loop, a benchmark) reuse them: a small cache, first in first out, shared by
// all threads. Encoding costs a driver call per map otherwise.
struct MapKey {
  const void *ptr;
  int BH, N, d, f16, store;  // store: 0 load map (128-row box), 1 store map, 2 load map with 64-row box
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && BH == o.BH && N == o.N && d == o.d && f16 == o.f16 && store == o.store;
  }
};
constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
CUtensorMap g_map_val[kMapCache];
int g_map_used = 0, g_map_next = 0;

int cached_map(CUtensorMap *map, const void *ptr, int BH, int N, int d, bool f16, int kind) {
  const MapKey key{ptr, BH, N, d, f16 ? 1 : 0, kind};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_map_used; ++i)
      if (g_map_key[i] == key) {
        *map = g_map_val[i];
        return kOk;
      }
  }
  const int st = kind == 1 ? encode_store_map(map, const_cast<void *>(ptr), BH, N, d, f16)
                           : encode_map(map, ptr, BH, N, d, f16, kind == 2 ? 64 : 128);
  if (st != kOk) return st;
  std::lock_guard<std::mutex> lock(g_map_mu);
  g_map_key[g_map_next] = key;
  g_map_val[g_map_next] = *map;
  g_map_next = (g_map_next + 1) % kMapCache;
  if (g_map_used < kMapCache) ++g_map_used;
  return kOk;
}
int make_map(CUtensorMap *map, const void *ptr, int BH, int N, int d, bool f16) {
  return cached_map(map, ptr, BH, N, d, f16, 0);
}
int make_store_map(CUtensorMap *map, void *ptr, int BH, int N, int d, bool f16) {
  return cached_map(map, ptr, BH, N, d, f16, 1);
}
// 64-row boxes: the half tiles a CTA of a two-CTA (pair) kernel loads.
int make_half_map(CUtensorMap *map, const void *ptr, int BH, int N, int d, bool f16) {
  return cached_map(map, ptr, BH, N, d, f16, 2);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int B, int H, int N, int d, int dmax) {
  if (B < 1 || H < 1 || N < 1 || d < 1 || d > dmax) return kErrShape;
  const double elems = static_cast<double>(B) * H * N * d;
  if (elems >= 1099511627776.0) return kErrShape;  // 2^40
  if (static_cast<long long>(B) * H > 65535) return kErrUnsupported;  // grid.y limit
  return kOk;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout.
//   f32:  D [B*H*N] fp32.
//   bf16: -L*log2(e) and D, each [B*H][Np] fp32 with Np = 128*ceil(N/128)
//         (padding rows hold -inf / 0).
struct BwdWorkspace {
  size_t lp = 0, dp = 0, total = 0;  // byte offsets and size
};

BwdWorkspace ws_layout(int B, int H, int N, int d, int dtype) {
  (void)d;
  BwdWorkspace w;
  const size_t rows = static_cast<size_t>(B) * H * N;
  if (dtype == FA_F32) {
    w.total = round_up(rows * sizeof(float), 256);
    return w;
  }
  const size_t prow = static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + 127) / 128 * 128);
  w.lp = 0;
  w.dp = round_up(prow * sizeof(float), 256);
  w.total = w.dp + round_up(prow * sizeof(float), 256);
  return w;
}

size_t ws_bytes(int B, int H, int N, int d, int dtype) {
  if (check_shape(B, H, N, d, 128) != kOk) return 0;
  return ws_layout(B, H, N, d, dtype).total;
}

}  // namespace

namespace fa {
void timing_begin(cudaStream_t stream) {
  if (t_events && t_event_next < t_event_pairs)
    cudaEventRecord(static_cast<cudaEvent_t>(t_events[2 * t_event_next]), stream);
}
void timing_end(cudaStream_t stream) {
  if (t_events && t_event_next < t_event_pairs) {
    cudaEventRecord(static_cast<cudaEvent_t>(t_events[2 * t_event_next + 1]), stream);
    ++t_event_next;
  }
}
int max_pair_clusters(const void *kernel, int smem_bytes, int threads) {
  struct Entry {
    const void *kernel;
    int dev, smem, threads, clusters;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].kernel == kernel && cache[i].dev == dev && cache[i].smem == smem_bytes &&
          cache[i].threads == threads)
        return cache[i].clusters;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();  // a failed query is not sticky: leave no error for the next launch check
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (used < 64) cache[used++] = Entry{kernel, dev, smem_bytes, threads, n};
  return n;
}

cudaError_t set_smem_once(const void *kernel, int bytes, SmemOnce *done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool known = dev >= 0 && dev < kMaxDevices;
  const uint32_t epoch = known ? g_epoch[dev].load(std::memory_order_acquire) : 0u;
  if (epoch != 0 && done->epoch[dev].load(std::memory_order_acquire) == epoch) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && epoch != 0) done->epoch[dev].store(epoch, std::memory_order_release);
  return e;
}
}  // namespace fa

extern "C" {

int fa_set_kernel_timing(void **events, int n_pairs) {
  if (n_pairs == -1) return t_event_next;
  if (n_pairs < -1) return FA_ERR_ARG;
  t_events = (events && n_pairs > 0) ? events : nullptr;
  t_event_pairs = t_events ? n_pairs : 0;
  t_event_next = 0;
  return FA_OK;
}

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "B, H, N or d out of range";
    case FA_ERR_UNSUPPORTED: return "shape not supported by this build";
    case FA_ERR_ALIGN: return "pointer not aligned as required";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_LAUNCH: return "CUDA launch or tensor-map call failed";
    case FA_ERR_TIMEOUT: return "a kernel gave up waiting on a pipeline barrier";
    case FA_ERR_ARCH: return "current device is not sm_103";
    case FA_ERR_ARG: return "invalid argument";
    case FA_ERR_CHECK: return "a device-side check of the checked build failed";
    default: return "unknown status";
  }
}

int fa_last_cuda_error(void) { return t_last_cuda_error; }
int fa_last_launch_count(void) { return t_last_launches; }

size_t fa_bwd_workspace_size(int B, int H, int N, int d, int dtype) {
  if (dtype != FA_BF16 && dtype != FA_F32 && dtype != FA_F16) return 0;
  if (dtype == FA_F16) dtype = FA_BF16;  // same layout
  return ws_bytes(B, H, N, d, dtype);
}

int fa_status_async(int *dst, fa_stream_t stream) {
  if (!dst) return FA_ERR_NULL;
  if (!aligned(dst, 4)) return FA_ERR_ALIGN;
  DeviceInfo *dev = nullptr;
  int st = current_device(&dev);
  if (st != kOk) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(dst, dev->status, sizeof(int), cudaMemcpyDefault, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev->status, 0, sizeof(int), s);
  return e == cudaSuccess ? FA_OK : record(e);
}

int fa_status_word(int **dev_ptr) {
  if (!dev_ptr) return FA_ERR_NULL;
  DeviceInfo *dev = nullptr;
  int st = current_device(&dev);
  if (st != kOk) return st;
  *dev_ptr = dev->status;
  return FA_OK;
}

int fa_device_status(void) {
  DeviceInfo *dev = nullptr;
  int st = current_device(&dev);
  if (st != kOk) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return record(e);
  int v = 0;
  if ((e = cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return record(e);
  const int zero = 0;
  if ((e = cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
    return record(e);
  return v;
}

}  // extern "C"

namespace {

// Shared body of fa_fwd / fa_fwd_f16 / fa_fwd_kv: N query rows, Nk key rows.
int fwd16(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int Nk,
          int d, float scale, int causal, fa_stream_t stream, bool f16, const Dropout *drop = nullptr) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d, 256);
  if (st == kOk) st = check_shape(B, H, Nk, d, 256);
  if (st != kOk) return st;
  if (causal && Nk < N) return FA_ERR_SHAPE;  // leading queries would see no key
  if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (!isfinite(scale)) return FA_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_ALIGN;
  DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != kOk) return st;
  if ((st = get_encoder()) != kOk) return st;
  CUtensorMap tq, tk, tv, tkh;
  const int BH = B * H;
  if ((st = make_map(&tq, q, BH, N, d, f16)) != kOk || (st = make_map(&tk, k, BH, Nk, d, f16)) != kOk ||
      (st = make_map(&tv, v, BH, Nk, d, f16)) != kOk)
    return st;
  const bool pair = FA_PAIR_KERNELS && d == 128 && !drop;  // the two-CTA kernel's K map has 64-row boxes
  if (pair && (st = make_half_map(&tkh, k, BH, Nk, d, f16)) != kOk) return st;
  int launches = 0;
  cudaError_t e = launch_fwd_16(tq, tk, pair ? &tkh : nullptr, tv, o, lse, B, H, N, Nk, d, scale, causal ? 1 : 0,
                                f16, drop, dev->status, dev->num_sms, reinterpret_cast<cudaStream_t>(stream),
                                &launches);
  if (e != cudaSuccess) return record(e);
  t_last_launches = launches;
  return FA_OK;
}

// Shared body of fa_bwd / fa_bwd_f16 / fa_bwd_kv: N query rows, Nk key rows.
int bwd16(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
          void *dq, void *dk, void *dv, int B, int H, int N, int Nk, int d, float scale, int causal,
          void *workspace, size_t workspace_bytes, fa_stream_t stream, bool f16, const Dropout *drop = nullptr) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d, 256);
  if (st == kOk) st = check_shape(B, H, Nk, d, 256);
  if (st != kOk) return st;
  if (causal && Nk < N) return FA_ERR_SHAPE;
  if (d != 64 && d != 96 && d != 128) return FA_ERR_UNSUPPORTED;  // no d = 256 backward
  if (!isfinite(scale)) return FA_ERR_ARG;
  const void *ptrs[] = {q, k, v, o, dO, dq, dk, dv};
  for (const void *p : ptrs)
    if (!aligned(p, 16)) return FA_ERR_ALIGN;
  if (!aligned(lse, 4)) return FA_ERR_ALIGN;
  const size_t need = ws_bytes(B, H, N, d, FA_BF16);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return FA_ERR_ALIGN;
  DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != kOk) return st;
  if ((st = get_encoder()) != kOk) return st;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  const int BH = B * H;
  if ((st = make_map(&tq, q, BH, N, d, f16)) != kOk || (st = make_map(&tk, k, BH, Nk, d, f16)) != kOk ||
      (st = make_map(&tv, v, BH, Nk, d, f16)) != kOk || (st = make_map(&tdo, dO, BH, N, d, f16)) != kOk ||
      (st = make_store_map(&tdk, dk, BH, Nk, d, f16)) != kOk ||
      (st = make_store_map(&tdv, dv, BH, Nk, d, f16)) != kOk)
    return st;
  // the two-CTA kernels of d = 128 load half tiles (64-row boxes)
  HalfMaps half;
  const bool pair = FA_PAIR_KERNELS && d == 128 && !drop;
  if (pair && ((st = make_half_map(&half.q, q, BH, N, d, f16)) != kOk ||
               (st = make_half_map(&half.k, k, BH, Nk, d, f16)) != kOk ||
               (st = make_half_map(&half.v, v, BH, Nk, d, f16)) != kOk ||
               (st = make_half_map(&half.dO, dO, BH, N, d, f16)) != kOk))
    return st;
  const BwdWorkspace w = ws_layout(B, H, N, d, FA_BF16);
  char *ws = static_cast<char *>(workspace);
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return record(cudaGetLastError());
  const SideStream *side = side_stream(cur, dev->ctx);
  const BwdSide bs{side ? side->stream : nullptr, side ? side->fork : nullptr, side ? side->join : nullptr};
  int launches = 0;
  cudaError_t e = launch_bwd_16(tq, tk, tv, tdo, tdk, tdv, pair ? &half : nullptr, o, dO, lse, dq, dk, dv,
                                reinterpret_cast<float *>(ws + w.lp), reinterpret_cast<float *>(ws + w.dp), B, H, N,
                                Nk, d, scale, causal ? 1 : 0, f16, drop, dev->status, dev->num_sms,
                                reinterpret_cast<cudaStream_t>(stream), bs, &launches);
  if (e != cudaSuccess) return record(e);
  t_last_launches = launches;
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int d,
           float scale, int causal, fa_stream_t stream) {
  return fwd16(q, k, v, o, lse, B, H, N, N, d, scale, causal, stream, false);
}

int fa_fwd_f16(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int d,
               float scale, int causal, fa_stream_t stream) {
  return fwd16(q, k, v, o, lse, B, H, N, N, d, scale, causal, stream, true);
}

int fa_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Nq, int Nk,
              int d, float scale, int causal, int dtype, fa_stream_t stream) {
  if (dtype != FA_BF16 && dtype != FA_F16) return dtype == FA_F32 ? FA_ERR_UNSUPPORTED : FA_ERR_ARG;
  return fwd16(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream, dtype == FA_F16);
}

int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
           void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal, void *workspace,
           size_t workspace_bytes, fa_stream_t stream) {
  return bwd16(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, scale, causal, workspace, workspace_bytes, stream,
               false);
}

int fa_bwd_f16(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
               void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal,
               void *workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd16(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, scale, causal, workspace, workspace_bytes, stream,
               true);
}

int fa_bwd_kv(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
              void *dq, void *dk, void *dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
              int dtype, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (dtype != FA_BF16 && dtype != FA_F16) return dtype == FA_F32 ? FA_ERR_UNSUPPORTED : FA_ERR_ARG;
  return bwd16(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace, workspace_bytes,
               stream, dtype == FA_F16);
}

// Dropout parameters: p in [0, 1) to a byte threshold t = round(256 p).
static int make_dropout(float p, unsigned long long seed, unsigned int offset, unsigned int head_base,
                        Dropout *dr) {
  if (!(p >= 0.f && p < 1.f)) return FA_ERR_ARG;
  int t = static_cast<int>(lrint(256.0 * static_cast<double>(p)));
  if (t > 255) t = 255;
  dr->k0 = static_cast<uint32_t>(seed);
  dr->k1 = static_cast<uint32_t>(seed >> 32);
  dr->offset = offset;
  dr->head_base = head_base;
  dr->t = static_cast<uint32_t>(t);
  dr->inv_keep = static_cast<float>(256.0 / (256.0 - t));
  dr->mask = nullptr;
  dr->n_qt = dr->n_kt = 0;
  dr->dkdv_writes_mask = 0;
  return FA_OK;
}

// Bytes of saved keep bits for the shape (0 if a size is not positive): a 2 KB
// block per (head, query tile, key tile).
static size_t mask_bytes_for(int B, int H, int Nq, int Nk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return 0;
  return static_cast<size_t>(B) * H * ((static_cast<size_t>(Nq) + 127) / 128) * ((static_cast<size_t>(Nk) + 127) / 128) *
         2048;
}

// Attaches the caller's saved-bits buffer to the dropout parameters.
static int attach_mask(Dropout *dr, const void *mask, size_t mask_bytes, int B, int H, int Nq, int Nk) {
  const size_t need = mask_bytes_for(B, H, Nq, Nk);
  if (need == 0) return FA_ERR_SHAPE;
  if (!mask) return FA_ERR_NULL;
  if (!aligned(mask, 16)) return FA_ERR_ALIGN;
  if (mask_bytes < need) return FA_ERR_WORKSPACE;
  dr->mask = static_cast<uint32_t *>(const_cast<void *>(mask));
  dr->n_qt = (Nq + 127) / 128;
  dr->n_kt = (Nk + 127) / 128;
  return FA_OK;
}

size_t fa_dropout_mask_size(int B, int H, int Nq, int Nk) { return mask_bytes_for(B, H, Nq, Nk); }

// fa_bwd_dropout's workspace with room for the keep bits its dK/dV pass hands
// to its dQ pass: the plain workspace (a multiple of 256 bytes), then the
// saved-bits layout at *bits_at. 0 for a shape or dtype the call rejects.
static size_t bwd_dropout_ws_bytes(int B, int H, int Nq, int Nk, int d, int dtype, size_t *bits_at) {
  if (dtype != FA_BF16 && dtype != FA_F16) return 0;
  if (d != 64 && d != 96 && d != 128) return 0;
  const size_t base = ws_bytes(B, H, Nq, d, FA_BF16);
  const size_t bits = mask_bytes_for(B, H, Nq, Nk);
  if (base == 0 || bits == 0) return 0;
  if (bits_at) *bits_at = round_up(base, 256);
  return round_up(base, 256) + bits;
}

size_t fa_bwd_dropout_workspace_size(int B, int H, int Nq, int Nk, int d, int dtype) {
  return bwd_dropout_ws_bytes(B, H, Nq, Nk, d, dtype, nullptr);
}

int fa_fwd_dropout_mask(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Nq,
                        int Nk, int d, float scale, int causal, int dtype, float p_drop, unsigned long long seed,
                        unsigned int offset, unsigned int head_base, void *mask, size_t mask_bytes,
                        fa_stream_t stream) {
  if (dtype != FA_BF16 && dtype != FA_F16) return dtype == FA_F32 ? FA_ERR_UNSUPPORTED : FA_ERR_ARG;
  Dropout dr;
  int st = make_dropout(p_drop, seed, offset, head_base, &dr);
  if (st == FA_OK) st = attach_mask(&dr, mask, mask_bytes, B, H, Nq, Nk);
  if (st != FA_OK) return st;
  return fwd16(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream, dtype == FA_F16, &dr);
}

int fa_bwd_dropout_mask(const void *q, const void *k, const void *v, const void *o, const float *lse,
                        const void *dO, void *dq, void *dk, void *dv, int B, int H, int Nq, int Nk, int d,
                        float scale, int causal, int dtype, float p_drop, const void *mask, size_t mask_bytes,
                        void *workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (dtype != FA_BF16 && dtype != FA_F16) return dtype == FA_F32 ? FA_ERR_UNSUPPORTED : FA_ERR_ARG;
  Dropout dr;
  int st = make_dropout(p_drop, 0, 0, 0, &dr);  // the bits come from `mask`, not the generator
  if (st == FA_OK) st = attach_mask(&dr, mask, mask_bytes, B, H, Nq, Nk);
  if (st != FA_OK) return st;
  return bwd16(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace, workspace_bytes,
               stream, dtype == FA_F16, &dr);
}

int fa_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Nq,
                   int Nk, int d, float scale, int causal, int dtype, float p_drop, unsigned long long seed,
                   unsigned int offset, unsigned int head_base, fa_stream_t stream) {
  if (dtype != FA_BF16 && dtype != FA_F16) return dtype == FA_F32 ? FA_ERR_UNSUPPORTED : FA_ERR_ARG;
  Dropout dr;
  const int st = make_dropout(p_drop, seed, offset, head_base, &dr);
  if (st != FA_OK) return st;
  return fwd16(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream, dtype == FA_F16, &dr);
}

int fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dO,
                   void *dq, void *dk, void *dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   int dtype, float p_drop, unsigned long long seed, unsigned int offset, unsigned int head_base,
                   void *workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (dtype != FA_BF16 && dtype != FA_F16) return dtype == FA_F32 ? FA_ERR_UNSUPPORTED : FA_ERR_ARG;
  Dropout dr;
  const int st = make_dropout(p_drop, seed, offset, head_base, &dr);
  if (st != FA_OK) return st;
  // room for the keep bits: the dK/dV pass writes what it draws, the dQ pass reads it
  size_t bits_at = 0;
  const size_t with_bits = bwd_dropout_ws_bytes(B, H, Nq, Nk, d, dtype, &bits_at);
  if (with_bits != 0 && workspace && aligned(workspace, 256) && workspace_bytes >= with_bits) {
    dr.mask = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + bits_at);
    dr.n_qt = (Nq + 127) / 128;
    dr.n_kt = (Nk + 127) / 128;
    dr.dkdv_writes_mask = 1;
  }
  return bwd16(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace, workspace_bytes,
               stream, dtype == FA_F16, &dr);
}

int fa_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse, int B, int H,
               int N, int d, float scale, int causal, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d, 128);
  if (st != kOk) return st;
  if (!isfinite(scale)) return FA_ERR_ARG;
  const void *ptrs[] = {q, k, v, o, lse};
  for (const void *p : ptrs)
    if (!aligned(p, 4)) return FA_ERR_ALIGN;
  DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != kOk) return st;
  int launches = 0;
  cudaError_t e = launch_fwd_f32(q, k, v, o, lse, B, H, N, d, scale, causal ? 1 : 0,
                                 reinterpret_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return record(e);
  t_last_launches = launches;
  return FA_OK;
}

int fa_bwd_f32(const float *q, const float *k, const float *v, const float *o, const float *lse,
               const float *dO, float *dq, float *dk, float *dv, int B, int H, int N, int d,
               float scale, int causal, void *workspace, size_t workspace_bytes,
               fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d, 128);
  if (st != kOk) return st;
  if (!isfinite(scale)) return FA_ERR_ARG;
  const void *ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void *p : ptrs)
    if (!aligned(p, 4)) return FA_ERR_ALIGN;
  const size_t need = ws_bytes(B, H, N, d, FA_F32);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return FA_ERR_ALIGN;
  DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != kOk) return st;
  int launches = 0;
  cudaError_t e = launch_bwd_f32(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale,
                                 causal ? 1 : 0, static_cast<float *>(workspace),
                                 reinterpret_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return record(e);
  t_last_launches = launches;
  return FA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// fa_bwd_static_scratch: fa_bwd without a caller-supplied workspace.
//
// Some callers cannot allocate device memory when they call the backward
// pass: a host framework that reserves the GPU's memory up front in its own
// pool and lets nothing else call cudaMalloc, a plug-in whose fixed calling
// convention has no slot for a workspace pointer, or a latency-bound path that
// may not allocate after start-up (cudaMalloc can synchronise the device).
// For them the scratch lives in the file-scope array below, which every GPU
// that loads this library holds until the process exits.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[FA_STATIC_SCRATCH_BYTES];

// Device address of the static scratch on the current device, looked up once
// per device and context (the host-side name is only a stand-in for the
// device array).
int static_scratch(unsigned char **out) {
  DeviceInfo *dev = nullptr;
  int st = current_device(&dev);
  if (st != kOk) return st;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!dev->scratch) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return record(e);
    dev->scratch = static_cast<unsigned char *>(p);
  }
  *out = dev->scratch;
  return kOk;
}

}  // namespace

extern "C" int fa_bwd_static_scratch(const void *q, const void *k, const void *v, const void *o,
                                     const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                     int B, int H, int N, int d, float scale, int causal,
                                     fa_stream_t stream) {
  // What differs from fa_bwd: the size limit, checked before any device work
  // (an invalid shape falls through to fa_bwd's own checks), and the array.
  const size_t need = ws_bytes(B, H, N, d, FA_BF16);
  if (need > static_cast<size_t>(FA_STATIC_SCRATCH_BYTES)) return FA_ERR_WORKSPACE;
  unsigned char *ws = nullptr;
  if (need != 0) {
    const int st = static_scratch(&ws);
    if (st != kOk) return st;
  }
  // The first kernel of the pass rewrites every scratch byte it later reads
  // (the L and D rows, padding included), so the previous call's contents
  // never leak into this one.
  return bwd16(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, scale, causal, ws, FA_STATIC_SCRATCH_BYTES,
               stream, false);
}
