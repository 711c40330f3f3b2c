// The CUDA-core path: fp32 arithmetic on every sequence of the batch.
//
// It is the fp32 debug build (q/k/v/out in float32, checked to 1e-5
// normwise against the oracle) and the path for shapes the tensor-core kernels
// do not take.  It computes the attention of "Chasing speed of light on TPU
// v6e", section "Attention", footnotes 5 and 6 (exact softmax attention, fp32
// accumulators), over the paged cache of "TPU Deep Dive", chapter 8.
//
// Mapping: CTA (x, y) owns flattened query tokens [x*BQ, (x+1)*BQ) and KV head
// y, i.e. up to 32 rows (token, query head of that KV head).  A token chunk
// may straddle sequences; each piece is handled in turn.  The keys visible to
// any row of a piece are streamed through shared memory 32 at a time and
// shared by all its rows; each warp keeps an online softmax for 4 rows.
#include "common.cuh"
#include "rpa_internal.h"

namespace rpa {
namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;  // 32
constexpr int kKeys = 32;                     // keys per shared-memory chunk

struct SimtParams {
  int32_t num_seqs, hq, hkv, group, page_size, mpps, num_pages;
  int32_t total_q, tokens_per_cta;
  int32_t do_decode, do_prefill;
};

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
simt_attention_kernel(Args a, SimtParams p) {
  extern __shared__ float smem[];
  float* qs = smem;                           // [kRows][D]
  float* ks = qs + kRows * D;                 // [kKeys][D + 1]
  float* vs = ks + kKeys * (D + 1);           // [kKeys][D + 1]
  constexpr int DL = D / 32;                  // dims per lane

  const T* q = static_cast<const T*>(a.q);
  const T* kp = static_cast<const T*>(a.k_pages);
  const T* vp = static_cast<const T*>(a.v_pages);
  T* out = static_cast<T*>(a.out);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int G = p.group;

  int32_t t = blockIdx.x * p.tokens_per_cta;
  const int32_t t_end = min(p.total_q, t + p.tokens_per_cta);
  while (t < t_end) {
    const int32_t s = find_seq(a.cu_q_lens, p.num_seqs, t);
    const int32_t q0 = __ldg(a.cu_q_lens + s);
    const int32_t q1 = __ldg(a.cu_q_lens + s + 1);
    const int32_t seg_end = min(t_end, q1);
    const int32_t ql = q1 - q0;
    const bool take = (ql == 1) ? p.do_decode : p.do_prefill;
    if (take) {
      const int32_t L = __ldg(a.kv_lens + s);
      const int32_t W = a.window ? __ldg(a.window + s) : 0;
      const int32_t n_rows = (seg_end - t) * G;
      const int32_t pos_first = L - ql + (t - q0);
      const int32_t pos_last = L - ql + (seg_end - 1 - q0);
      const int32_t klo = first_visible(pos_first, W);
      const int32_t* pt = a.page_table + static_cast<int64_t>(s) * p.mpps;

      // Queries of this piece into shared memory.
      __syncthreads();
      for (int e = threadIdx.x; e < n_rows * D; e += blockDim.x) {
        const int r = e / D, dd = e % D;
        const int64_t tok = t + r / G;
        const int h = g * G + r % G;
        qs[r * D + dd] = to_float(q[(tok * p.hq + h) * D + dd]);
      }
      float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][DL];
      int32_t pos[kRowsPerWarp], lo[kRowsPerWarp];
#pragma unroll
      for (int k = 0; k < kRowsPerWarp; ++k) {
        m[k] = -INFINITY;
        l[k] = 0.f;
#pragma unroll
        for (int j = 0; j < DL; ++j) o[k][j] = 0.f;
        const int r = warp + kWarps * k;
        pos[k] = L - ql + (t + r / G - q0);
        lo[k] = first_visible(pos[k], W);
      }

      for (int32_t kc = klo; kc <= pos_last; kc += kKeys) {
        __syncthreads();
        for (int e = threadIdx.x; e < kKeys * D; e += blockDim.x) {
          const int kk = e / D, dd = e % D;
          const int32_t j = kc + kk;
          float kv = 0.f, vv = 0.f;
          if (j <= pos_last) {
            const int32_t slot = j / p.page_size;
            const int32_t page = slot < p.mpps ? __ldg(pt + slot) : -1;
            if (slot >= p.mpps) {
              report_error(a.workspace, RPA_DEVERR_LENGTHS, s);
            } else if (page < 0 || page >= p.num_pages) {
              report_error(a.workspace, RPA_DEVERR_PAGE_ID, s);
            } else {
              const int64_t idx =
                  ((static_cast<int64_t>(page) * p.page_size + j % p.page_size) * p.hkv + g) * D + dd;
              kv = to_float(kp[idx]);
              vv = to_float(vp[idx]);
            }
          }
          ks[kk * (D + 1) + dd] = kv;
          vs[kk * (D + 1) + dd] = vv;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kRowsPerWarp; ++k) {
          const int r = warp + kWarps * k;
          if (r >= n_rows) continue;
          const int32_t j = kc + lane;
          const bool vis = j <= pos[k] && j >= lo[k];
          float x = -INFINITY;
          if (vis) {
            float dot = 0.f;
            const float* qr = qs + r * D;
            const float* kr = ks + lane * (D + 1);
            for (int dd = 0; dd < D; ++dd) dot = fmaf(qr[dd], kr[dd], dot);
            x = a.sm_scale * dot;
          }
          float mc = x;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
          if (mc == -INFINITY) continue;  // no visible key in this chunk
          const float mn = fmaxf(m[k], mc);
          const float alpha = expf(m[k] - mn);
          const float pj = vis ? expf(x - mn) : 0.f;
          float ps = pj;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
          l[k] = l[k] * alpha + ps;
          m[k] = mn;
#pragma unroll
          for (int jd = 0; jd < DL; ++jd) o[k][jd] *= alpha;
          for (int jj = 0; jj < kKeys; ++jj) {
            const float pb = __shfl_sync(0xffffffffu, pj, jj);
            const float* vr = vs + jj * (D + 1);
#pragma unroll
            for (int jd = 0; jd < DL; ++jd) o[k][jd] = fmaf(pb, vr[lane + 32 * jd], o[k][jd]);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kRowsPerWarp; ++k) {
        const int r = warp + kWarps * k;
        if (r >= n_rows) continue;
        const int64_t tok = t + r / G;
        const int h = g * G + r % G;
        const float inv = 1.f / l[k];
#pragma unroll
        for (int jd = 0; jd < DL; ++jd)
          out[(tok * p.hq + h) * D + lane + 32 * jd] = from_float<T>(o[k][jd] * inv);
      }
    }
    t = seg_end;
  }
}

template <typename T, int D>
int launch_simt_t(const Plan& plan, const Args& a, cudaStream_t stream) {
  const size_t smem = (kRows * D + 2 * kKeys * (D + 1)) * sizeof(float);
  if (int e = ensure_dynamic_smem(reinterpret_cast<const void*>(simt_attention_kernel<T, D>),
                                  static_cast<int>(smem)))
    return e;
  SimtParams p;
  p.num_seqs = plan.num_seqs;
  p.hq = plan.hq;
  p.hkv = plan.hkv;
  p.group = plan.hq / plan.hkv;
  p.page_size = plan.p;
  p.mpps = plan.mpps;
  p.num_pages = plan.num_pages;
  p.total_q = static_cast<int32_t>(plan.total_q);
  p.tokens_per_cta = max(1, kRows / p.group);
  p.do_decode = plan.simt_decode;
  p.do_prefill = plan.simt_prefill;
  dim3 grid((p.total_q + p.tokens_per_cta - 1) / p.tokens_per_cta, plan.hkv);
  simt_attention_kernel<T, D><<<grid, kWarps * 32, smem, stream>>>(a, p);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) trace_mark(RPA_KERNEL_SIMT, stream);
  return static_cast<int>(e);
}

}  // namespace

int launch_simt(const Plan& plan, const Args& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f32 = plan.dtype == RPA_DTYPE_F32;
  switch (plan.d) {
    case 64: return f32 ? launch_simt_t<float, 64>(plan, a, s) : launch_simt_t<__nv_bfloat16, 64>(plan, a, s);
    case 128: return f32 ? launch_simt_t<float, 128>(plan, a, s) : launch_simt_t<__nv_bfloat16, 128>(plan, a, s);
    case 256: return f32 ? launch_simt_t<float, 256>(plan, a, s) : launch_simt_t<__nv_bfloat16, 256>(plan, a, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace rpa
