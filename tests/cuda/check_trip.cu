// Test-only kernel for the checked build's reporting path. FA_CHECK rejects a
// stand-in call that has no instruction behind it (so nothing is skipped that
// could matter), and report_checks turns the recorded bit into the library's
// check status, 10 (FA_ERR_CHECK), in `status` at the end of the kernel.
#define FA_CHECKED 1
#include "../../exact_attention_97_gb300/csrc/sm103.cuh"

#include <cuda_runtime.h>

namespace {
__device__ void stand_in(bool ok) { FA_CHECK(ok, fa::kCheckTmem); }
}  // namespace

__global__ void check_trip_kernel(int trip, int *status, unsigned *word) {
  // one thread of the second block breaks the rule when asked to
  stand_in(!(trip && blockIdx.x == 1 && threadIdx.x == 37));
  __syncthreads();
  fa::report_checks(status);
  if (blockIdx.x == 1 && threadIdx.x == 0) *word = fa::g_check_word;
}

// Runs the kernel once; host_out = {status word, check word}. The check word
// is sticky for the life of the module, so a clean run must come first.
extern "C" int run_check_trip(int trip, int *host_out) {
  int *d = nullptr;
  if (cudaMalloc(&d, 2 * sizeof(int)) != cudaSuccess) return -1;
  cudaMemset(d, 0, 2 * sizeof(int));
  check_trip_kernel<<<2, 64>>>(trip, d, reinterpret_cast<unsigned *>(d + 1));
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_out, d, 2 * sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return static_cast<int>(e);
}
