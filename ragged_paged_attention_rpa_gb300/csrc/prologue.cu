// q/k/v prologue: the step right before attention, fused with the KV-cache
// write.  "Chasing speed of light on TPU v6e" (section "The Long Tail") folds
// the q/k/v RMS norms and the rotary embedding into the kernel before
// attention and emits q, k and v as separate arrays; here one kernel reads the
// projection's q, k and v rows once and writes
//   q_out[t][h]                         = rope(rmsnorm(q[t][h], w_q), pos)
//   k_pages[page][pos % P][g]           = rope(rmsnorm(k[t][g], w_k), pos)
//   v_pages[page][pos % P][g]           = rmsnorm(v[t][g], w_v)   (or v as given)
// with pos = kv_len - q_len + i for the i-th new token of its sequence and
// page = page_table[s][pos / P].
//
// rmsnorm(x, w)_d = x_d / sqrt(mean(x^2) + eps) * w_d, in fp32.
// rope (halves convention): dimension i < D/2 pairs with i + D/2 and the pair
// turns by a = pos * theta^(-2i/D).  The angle is formed as a double-float
// product (the frequencies are split on the host into hi + lo floats; the
// product's rounding error is recovered with an FMA) and reduced modulo 2 pi
// by Cody and Waite's method with 2 pi in three float parts, so cos/sin stay
// accurate for positions up to about 2^21 at frequency 1.
//
// One warp per (token, head) row, D/32 elements per lane: lane l holds
// dimensions [l E, l E + E), so the rotation partner of lane l is lane l ^ 16.
// HBM-bound: every input row is read once and every output row written once.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "rpa_internal.h"

namespace rpa {
namespace {

constexpr int kMaxHalf = 128;  // D / 2 for D <= 256

struct PrologueParams {
  const void* q;
  const void* k;
  const void* v;
  const float* wq;
  const float* wk;
  const float* wv;
  void* q_out;
  void* k_pages;
  void* v_pages;
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  unsigned char* ws;
  int32_t num_seqs, total_q, hq, hkv, page_size, page_shift, mpps, num_pages;
  float eps;
  int32_t rope;
  float c1, c2, c3;  // 2 pi = c1 + c2 + c3
  float inv_2pi;
  float freq_hi[kMaxHalf], freq_lo[kMaxHalf];  // theta^(-2i/D) = hi + lo
};

template <int E, typename T>
struct Row;

// E consecutive elements of a row as fp32 (16-byte aligned rows).
template <int E>
struct Row<E, __nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* src, float (&x)[E]) {
    static_assert(E == 2 || E == 4 || E == 8, "E");
    uint32_t w[E / 2];
    if constexpr (E == 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(src);
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else if constexpr (E == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(src);
      w[0] = u.x; w[1] = u.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(src);
    }
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* dst, const float (&x)[E]) {
    uint32_t w[E / 2];
#pragma unroll
    for (int i = 0; i < E / 2; ++i) w[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
    if constexpr (E == 8) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (E == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = w[0];
    }
  }
};

template <int E>
struct Row<E, float> {
  static __device__ __forceinline__ void load(const float* src, float (&x)[E]) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float2 u = *reinterpret_cast<const float2*>(src + i);
      x[i] = u.x;
      x[i + 1] = u.y;
    }
  }
  static __device__ __forceinline__ void store(float* dst, const float (&x)[E]) {
#pragma unroll
    for (int i = 0; i < E; i += 2) *reinterpret_cast<float2*>(dst + i) = make_float2(x[i], x[i + 1]);
  }
};

template <int D>
__device__ __forceinline__ void rms_norm(float (&x)[D / 32], const float* w, float eps, int lane) {
  constexpr int E = D / 32;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float r = 1.0f / sqrtf(ss * (1.0f / D) + eps);
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = x[e] * r * __ldg(w + lane * E + e);
}

template <int D>
__device__ __forceinline__ void rope(float (&x)[D / 32], const PrologueParams& p, int32_t pos,
                                     int lane) {
  constexpr int E = D / 32;
  const float P = static_cast<float>(pos);  // exact below 2^24
  const bool hi_half = lane >= 16;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = (lane & 15) * E + e;
    // a = pos * (hi + lo): a_hi + a_lo with the product's rounding error kept.
    const float fh = p.freq_hi[j], fl = p.freq_lo[j];
    const float a_hi = P * fh;
    const float a_lo = fmaf(P, fl, fmaf(P, fh, -a_hi));
    // r = a - k 2 pi; the first step is exact for |a| < 2^21.
    const float kq = rintf(a_hi * p.inv_2pi);
    float r = fmaf(-kq, p.c1, a_hi);
    r = fmaf(-kq, p.c2, r);
    r = fmaf(-kq, p.c3, r);
    r += a_lo;
    float s, c;
    sincosf(r, &s, &c);
    const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
    x[e] = hi_half ? fmaf(x[e], c, other * s) : fmaf(x[e], c, -other * s);
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(256) prologue_kernel(const __grid_constant__ PrologueParams p) {
  constexpr int E = D / 32;
  extern __shared__ int32_t s_meta[];
  const SeqMeta meta = stage_seq_meta(s_meta, p.cu_q_lens, p.kv_lens, p.num_seqs);
  const int lane = threadIdx.x & 31;
  const int heads = p.hq + p.hkv;
  const int64_t rows = static_cast<int64_t>(p.total_q) * heads;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    const int32_t t = static_cast<int32_t>(row / heads);
    const int32_t h = static_cast<int32_t>(row % heads);
    const bool is_q = h < p.hq;
    const int32_t g = h - p.hq;
    // The row's data first (it does not depend on the sequence lookup).
    const int64_t src = is_q ? (static_cast<int64_t>(t) * p.hq + h) * D + lane * E
                             : (static_cast<int64_t>(t) * p.hkv + g) * D + lane * E;
    float x[E], y[E];
    Row<E, T>::load(static_cast<const T*>(is_q ? p.q : p.k) + src, x);
    if (!is_q) Row<E, T>::load(static_cast<const T*>(p.v) + src, y);
    const int32_t s = meta.seq(t);
    const int32_t q0 = meta.cu[s];
    const int32_t ql = meta.cu[s + 1] - q0;
    const int32_t pos = meta.kl[s] - ql + (t - q0);
    if (pos < 0 || t - q0 >= ql) {
      if (lane == 0 && p.ws) report_error(p.ws, RPA_DEVERR_LENGTHS, s);
      continue;
    }
    if (is_q) {
      if (p.wq) rms_norm<D>(x, p.wq, p.eps, lane);
      if (p.rope) rope<D>(x, p, pos, lane);
      Row<E, T>::store(static_cast<T*>(p.q_out) + src, x);
      continue;
    }
    const int32_t slot = pos >> p.page_shift;
    const int32_t page = slot < p.mpps ? __ldg(p.page_table + static_cast<int64_t>(s) * p.mpps + slot)
                                       : -1;
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0 && p.ws)
        report_error(p.ws, slot < p.mpps ? RPA_DEVERR_PAGE_ID : RPA_DEVERR_LENGTHS, s);
      continue;
    }
    const int64_t dst = ((static_cast<int64_t>(page) * p.page_size + (pos & (p.page_size - 1))) *
                             p.hkv + g) * D + lane * E;
    if (p.wk) rms_norm<D>(x, p.wk, p.eps, lane);
    if (p.rope) rope<D>(x, p, pos, lane);
    Row<E, T>::store(static_cast<T*>(p.k_pages) + dst, x);
    if (p.wv) rms_norm<D>(y, p.wv, p.eps, lane);
    Row<E, T>::store(static_cast<T*>(p.v_pages) + dst, y);
  }
}

template <int D, typename T>
int launch_t(const PrologueParams& p, int64_t rows, cudaStream_t s) {
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, 152 * 8);
  prologue_kernel<D, T><<<static_cast<int>(blocks), 256, staged_meta_bytes(p.num_seqs), s>>>(p);
  return 0;
}

}  // namespace

bool prologue_supported(int32_t head_dim) {
  return head_dim == 64 || head_dim == 128 || head_dim == 256;
}

int launch_prologue(const PrologueArgs& a, void* stream) {
  if (a.total_q == 0) return 0;
  PrologueParams p;
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.wq = a.q_weight;
  p.wk = a.k_weight;
  p.wv = a.v_weight;
  p.q_out = a.q_out;
  p.k_pages = a.k_pages;
  p.v_pages = a.v_pages;
  p.page_table = a.page_table;
  p.cu_q_lens = a.cu_q_lens;
  p.kv_lens = a.kv_lens;
  p.ws = a.workspace;
  p.num_seqs = a.num_seqs;
  p.total_q = a.total_q;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.page_size = a.page_size;
  int shift = 0;
  while ((1 << shift) < a.page_size) ++shift;
  p.page_shift = shift;
  p.mpps = a.mpps;
  p.num_pages = a.num_pages;
  p.eps = a.eps;
  p.rope = a.rope_theta > 0.f ? 1 : 0;
  // 2 pi in three float parts, and the frequencies as float pairs (double
  // precision on the host).
  const double two_pi = 6.283185307179586476925286766559;
  p.c1 = static_cast<float>(two_pi);
  p.c2 = static_cast<float>(two_pi - static_cast<double>(p.c1));
  p.c3 = static_cast<float>(two_pi - static_cast<double>(p.c1) - static_cast<double>(p.c2));
  p.inv_2pi = static_cast<float>(1.0 / two_pi);
  const int half = a.head_dim / 2;
  for (int i = 0; i < kMaxHalf; ++i) {
    const double f = i < half && p.rope
                         ? std::pow(static_cast<double>(a.rope_theta), -2.0 * i / a.head_dim)
                         : 0.0;
    p.freq_hi[i] = static_cast<float>(f);
    p.freq_lo[i] = static_cast<float>(f - static_cast<double>(p.freq_hi[i]));
  }
  const int64_t rows = static_cast<int64_t>(a.total_q) * (a.hq + a.hkv);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f32 = a.elem_bytes == 4;
  switch (a.head_dim) {
    case 64: f32 ? launch_t<64, float>(p, rows, s) : launch_t<64, __nv_bfloat16>(p, rows, s); break;
    case 128: f32 ? launch_t<128, float>(p, rows, s) : launch_t<128, __nv_bfloat16>(p, rows, s); break;
    case 256: f32 ? launch_t<256, float>(p, rows, s) : launch_t<256, __nv_bfloat16>(p, rows, s); break;
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  trace_mark(RPA_KERNEL_PROLOGUE, stream);
  return 0;
}

}  // namespace rpa
