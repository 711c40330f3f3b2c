// Test helper: runs librpa's bounded mbarrier wait (sm100_ptx.cuh, mbar_wait)
// on a barrier that nothing arrives on, so a test can check that the wait
// gives up after its limit (or as soon as another warp raises the abort
// flag), that the kernel ends, and that the failure reaches the workspace
// error word.  Every wait here is bounded by the global timer.  Built by the
// test suite only; not part of the library.
#include <cuda_runtime.h>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace {
__global__ void wait_kernel(int* out, unsigned char* ws, unsigned long long limit_ns,
                            unsigned long long peer_abort_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    rpa::sm100::mbar_init(&bar, 1);
    abort_flag = 0;
    rpa::sm100::fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (threadIdx.x == 0) {
    const uint64_t t0 = rpa::sm100::global_timer_ns();
    const bool ok = rpa::sm100::mbar_wait(&bar, 0, abort, limit_ns);
    const uint64_t t1 = rpa::sm100::global_timer_ns();
    out[0] = ok ? 1 : 0;
    out[1] = *abort;
    out[2] = static_cast<int>((t1 - t0) / 1000);   // microseconds
    if (!ok) rpa::report_error(ws, RPA_DEVERR_TIMEOUT, 7);
  } else if (threadIdx.x == 32 && peer_abort_ns > 0) {
    // Another warp gives up on the CTA's behalf after peer_abort_ns.
    const uint64_t t0 = rpa::sm100::global_timer_ns();
    while (rpa::sm100::global_timer_ns() - t0 < peer_abort_ns) {
    }
    *abort = 1;
  }
}
}  // namespace

extern "C" int wait_timeout_check(void* ws, unsigned long long limit_ns,
                                  unsigned long long peer_abort_ns, int* out_host) {
  int* out = nullptr;
  if (cudaMalloc(&out, 3 * sizeof(int)) != cudaSuccess) return 1;
  wait_kernel<<<1, 64>>>(out, static_cast<unsigned char*>(ws), limit_ns, peer_abort_ns);
  const cudaError_t e = cudaDeviceSynchronize();
  cudaMemcpy(out_host, out, 3 * sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(out);
  return e == cudaSuccess ? 0 : 2;
}
