// Test-only kernel: exercises the library's bounded mbarrier wait with a
// short limit on a barrier that nothing ever arrives on. The wait must give
// up, raise the CTA abort flag, and let every other thread's wait return at
// once; nothing traps and the CUDA context stays usable.
#define FA_WAIT_LIMIT_CYCLES (20ll * 1000 * 1000)  // ~10 ms
#include "../../exact_attention_97_gb300/csrc/sm103.cuh"

#include <cuda_runtime.h>

__global__ void wait_timeout_kernel(int *out) {
  __shared__ uint64_t never, done;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(&never, 1);
    fa::mbar_init(&done, 1);
    fa::fence_mbar_init();
  }
  __syncthreads();
  const long long t0 = clock64();
  // every warp waits on the barrier nobody arrives on
  const bool ok = fa::mbar_wait_warp(&never, 0, &abort_flag);
  const long long waited = clock64() - t0;
  // a barrier that did complete is still observed by the teardown (drain) wait
  if (threadIdx.x == 0) fa::mbar_arrive(&done);
  __syncthreads();
  const bool drained = fa::mbar_wait_drain(&done, 0);
  if (threadIdx.x == 0) {
    out[0] = ok ? 1 : 0;
    out[1] = abort_flag;
    out[2] = drained ? 1 : 0;
    out[3] = static_cast<int>(waited / 1000);  // kilo-cycles waited by thread 0
  }
}

extern "C" int run_wait_timeout(int *host_out) {
  int *d = nullptr;
  if (cudaMalloc(&d, 4 * sizeof(int)) != cudaSuccess) return -1;
  cudaMemset(d, 0xff, 4 * sizeof(int));
  wait_timeout_kernel<<<4, 128>>>(d);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_out, d, 4 * sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return static_cast<int>(e);
}

// The same never-completed wait, and on giving up the kernel records the
// library's timeout code (7, FA_ERR_TIMEOUT) in `status`, the library's
// device status word passed in by address, as the attention kernels do when
// they abort. Lets a test check that the status reaches the Python caller.
__global__ void wait_timeout_status_kernel(int *status) {
  __shared__ uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(&never, 1);
    fa::fence_mbar_init();
  }
  __syncthreads();
  fa::mbar_wait_warp(&never, 0, &abort_flag);
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) atomicExch(status, 7);
}

extern "C" int run_wait_timeout_status(int *status_word) {
  wait_timeout_status_kernel<<<2, 64>>>(status_word);
  return static_cast<int>(cudaDeviceSynchronize());
}
