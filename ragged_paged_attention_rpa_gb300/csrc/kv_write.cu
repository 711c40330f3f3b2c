// KV-cache write: scatter the K and V rows of a step's new tokens into their
// pages, the cache update that "TPU Deep Dive" (chapter 8, "Continuous
// batching with static shapes") lists as fused into ragged paged attention.
//
// Token t of sequence s is the i-th of its q_len new tokens, at position
// pos = kv_len - q_len + i (the query positions the attention kernels use);
// its row for KV head g goes to page page_table[s][pos / P], slot pos % P:
//   k_pages[page][pos % P][g][:] = k_new[t][g][:]   (and V alike).
// One warp per (token, KV head) row, 16-byte vector copies; a data-movement
// kernel bound by HBM (each new row read once and written once).  The
// sequence lookups read cu_q_lens and kv_lens staged in shared memory.
#include <algorithm>

#include "common.cuh"
#include "rpa_internal.h"

namespace rpa {
namespace {

struct KvWriteParams {
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_pages;
  uint4* v_pages;
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  unsigned char* ws;  // error word (may be null)
  int32_t num_seqs, total_q, hkv, vec_per_row, page_size, page_shift, mpps, num_pages;
};

__global__ void __launch_bounds__(256) kv_write_kernel(const KvWriteParams p) {
  extern __shared__ int32_t s_meta[];
  const SeqMeta meta = stage_seq_meta(s_meta, p.cu_q_lens, p.kv_lens, p.num_seqs);
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(p.total_q) * p.hkv;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    const int32_t t = static_cast<int32_t>(row / p.hkv);
    const int32_t g = static_cast<int32_t>(row % p.hkv);
    const int64_t src = row * p.vec_per_row;
    // Rows of up to 32 vectors (D * element size <= 512 B): load them before
    // the lookups, which they do not depend on.
    const bool one = p.vec_per_row <= 32;
    uint4 kk = make_uint4(0, 0, 0, 0), vv = kk;
    if (one && lane < p.vec_per_row) {
      kk = __ldg(p.k_new + src + lane);
      vv = __ldg(p.v_new + src + lane);
    }
    const int32_t s = meta.seq(t);
    const int32_t q0 = meta.cu[s];
    const int32_t ql = meta.cu[s + 1] - q0;
    const int32_t pos = meta.kl[s] - ql + (t - q0);
    if (pos < 0 || t - q0 >= ql) {
      if (lane == 0 && p.ws) report_error(p.ws, RPA_DEVERR_LENGTHS, s);
      continue;
    }
    const int32_t slot = pos >> p.page_shift;
    if (slot >= p.mpps) {
      if (lane == 0 && p.ws) report_error(p.ws, RPA_DEVERR_LENGTHS, s);
      continue;
    }
    const int32_t page = __ldg(p.page_table + static_cast<int64_t>(s) * p.mpps + slot);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0 && p.ws) report_error(p.ws, RPA_DEVERR_PAGE_ID, s);
      continue;
    }
    const int64_t dst = ((static_cast<int64_t>(page) * p.page_size + (pos & (p.page_size - 1))) *
                             p.hkv + g) * p.vec_per_row;
    if (one) {
      if (lane < p.vec_per_row) {
        p.k_pages[dst + lane] = kk;
        p.v_pages[dst + lane] = vv;
      }
      continue;
    }
    for (int v = lane; v < p.vec_per_row; v += 32) {
      p.k_pages[dst + v] = __ldg(p.k_new + src + v);
      p.v_pages[dst + v] = __ldg(p.v_new + src + v);
    }
  }
}

}  // namespace

int launch_kv_write(const KvWriteArgs& a, void* stream) {
  if (a.total_q == 0) return 0;
  KvWriteParams p;
  p.k_new = static_cast<const uint4*>(a.k_new);
  p.v_new = static_cast<const uint4*>(a.v_new);
  p.k_pages = static_cast<uint4*>(a.k_pages);
  p.v_pages = static_cast<uint4*>(a.v_pages);
  p.page_table = a.page_table;
  p.cu_q_lens = a.cu_q_lens;
  p.kv_lens = a.kv_lens;
  p.ws = a.workspace;
  p.num_seqs = a.num_seqs;
  p.total_q = a.total_q;
  p.hkv = a.hkv;
  p.vec_per_row = a.head_dim * a.elem_bytes / 16;
  p.page_size = a.page_size;
  int shift = 0;
  while ((1 << shift) < a.page_size) ++shift;
  p.page_shift = shift;
  p.mpps = a.mpps;
  p.num_pages = a.num_pages;
  const int64_t rows = static_cast<int64_t>(a.total_q) * a.hkv;
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, 152 * 8);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kv_write_kernel<<<static_cast<int>(blocks), 256, staged_meta_bytes(p.num_seqs), s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  trace_mark(RPA_KERNEL_KV_WRITE, stream);
  return 0;
}

}  // namespace rpa
