// Device helpers shared by the librpa kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rpa.h"

namespace rpa {

// Record the first device-side problem in the workspace error word; later
// ones keep the first.  Never traps: the caller skips the bad access.
__device__ __forceinline__ void report_error(unsigned char* ws, int32_t code, int32_t info) {
  int32_t* w = reinterpret_cast<int32_t*>(ws);
  if (atomicCAS(w, 0, code) == 0) w[1] = info;
}

// 2^x with the hardware's approximate exponential (relative error ~2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Pack two floats as bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// First visible key of the query at position pos: keys [first, pos].
__device__ __forceinline__ int32_t first_visible(int32_t pos, int32_t w) {
  return (w > 0 && pos - (w - 1) > 0) ? pos - (w - 1) : 0;
}

// Sequence holding flattened token t: largest s with cu[s] <= t (cu sorted).
__device__ __forceinline__ int32_t find_seq(const int32_t* cu, int32_t num_seqs, int32_t t) {
  int32_t lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Per-sequence metadata of the new-token kernels (KV write, prologue): the
// CTA copies cu_q_lens [num_seqs + 1] and kv_lens [num_seqs] into shared
// memory in one round of loads when they fit (kMaxStagedSeqs), so that each
// row's sequence search costs shared-memory reads instead of a chain of
// dependent global loads.
constexpr int kMaxStagedSeqs = 4096;

__host__ __device__ constexpr size_t staged_meta_bytes(int32_t num_seqs) {
  return num_seqs <= kMaxStagedSeqs ? static_cast<size_t>(2 * num_seqs + 1) * 4 : 0;
}

struct SeqMeta {
  const int32_t* cu;   // shared or global
  const int32_t* kl;
  int32_t n;

  // Sequence s of token t, its first token and its q_len.
  __device__ __forceinline__ int32_t seq(int32_t t) const {
    int32_t lo = 0, hi = n - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
  }
};

// Stage the metadata (all threads of the CTA take part; ends with a barrier
// when staged).  `smem` holds staged_meta_bytes(num_seqs) bytes.
__device__ __forceinline__ SeqMeta stage_seq_meta(int32_t* smem, const int32_t* cu,
                                                 const int32_t* kl, int32_t num_seqs) {
  if (num_seqs > kMaxStagedSeqs) return SeqMeta{cu, kl, num_seqs};
  for (int i = threadIdx.x; i < 2 * num_seqs + 1; i += blockDim.x)
    smem[i] = i <= num_seqs ? __ldg(cu + i) : __ldg(kl + (i - num_seqs - 1));
  __syncthreads();
  return SeqMeta{smem, smem + num_seqs + 1, num_seqs};
}

}  // namespace rpa
