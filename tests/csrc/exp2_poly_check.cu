// Test helper: evaluates librpa's FMA-pipe 2^x (exp2_poly2) and CUDA's exp2f
// on the same arguments, so a test can compare them.  Built by the test suite
// only; not part of the library.
#include <cuda_runtime.h>

#include "sm100_ptx.cuh"

namespace {
__global__ void check_kernel(const float* x, float* poly, float* ref, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i + 1 >= n) return;
  const uint64_t p2 = rpa::sm100::exp2_poly2(rpa::sm100::f2_pack(x[i], x[i + 1]));
  float a, b;
  rpa::sm100::f2_unpack(p2, a, b);
  poly[i] = a;
  poly[i + 1] = b;
  ref[i] = exp2f(x[i]);
  ref[i + 1] = exp2f(x[i + 1]);
}
}  // namespace

extern "C" int exp2_poly_check(const float* x_host, float* poly_host, float* ref_host, int n) {
  float *x = nullptr, *poly = nullptr, *ref = nullptr;
  const size_t bytes = static_cast<size_t>(n) * sizeof(float);
  if (cudaMalloc(&x, bytes) != cudaSuccess || cudaMalloc(&poly, bytes) != cudaSuccess ||
      cudaMalloc(&ref, bytes) != cudaSuccess)
    return 1;
  cudaMemcpy(x, x_host, bytes, cudaMemcpyHostToDevice);
  const int pairs = n / 2;
  check_kernel<<<(pairs + 255) / 256, 256>>>(x, poly, ref, n);
  cudaError_t e = cudaDeviceSynchronize();
  cudaMemcpy(poly_host, poly, bytes, cudaMemcpyDeviceToHost);
  cudaMemcpy(ref_host, ref, bytes, cudaMemcpyDeviceToHost);
  cudaFree(x);
  cudaFree(poly);
  cudaFree(ref);
  return e == cudaSuccess ? 0 : 2;
}
