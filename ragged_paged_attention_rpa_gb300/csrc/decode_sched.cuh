// The decode schedule as the split-KV decode kernels receive it (one
// launch's segments and CTA ranges, from the plan's host copies of the
// metadata), and the prologue that turns a CTA's range into its segment
// table and page list in shared memory.  Shared by the CUDA-core-MMA decode
// kernel (decode.cu) and the tensor-core decode kernel (decode_tc.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "rpa_internal.h"

namespace rpa {

constexpr int kDecBlk = 16;  // keys per block of the decode schedule

struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  const int32_t* window;
  __nv_bfloat16* out;
  unsigned char* ws;
  float* part_o;      // [2 * total CTAs][G][D]
  float* part_lse;    // [2 * total CTAs][G]
  int32_t hq, hkv, group, page_shift, mpps, num_pages;
  float scale_log2;   // sm_scale * log2(e)
  const float* k_scale;  // fp8 pages: per-KV-head scales (else unused)
  const float* v_scale;
};

// One launch's share of the block stream.  seqhead[i] = (sequence << 8) | kv
// head of segment i; blk0[i] = first block of segment i (blk0[n_seg] = total).
// CTA c takes blocks [c * bpc, (c + 1) * bpc) where bpc > 0, else
// [cta0[c], cta0[c + 1]).
template <int NSEG>
struct DecodeSched {
  int32_t n_seg, bpc, n_blocks, slot_base, seg_base, n_ctas;
  int32_t cta0[kMaxDecodeGrid + 1];
  int32_t cta_seg[kMaxDecodeGrid];   // first segment | last segment << 16
  int32_t seqhead[NSEG];
  int32_t blk0[NSEG + 1];
  // From the plan's host metadata (validated there): query token, first
  // visible key and length of each segment's sequence.
  int32_t q0[NSEG], lo[NSEG], len[NSEG];
};

template <int NSEG>
__device__ __forceinline__ int32_t range_start(const DecodeSched<NSEG>& sc, int c) {
  return sc.bpc > 0 ? min(c * sc.bpc, sc.n_blocks) : sc.cta0[c];
}

// The CTA whose range holds block x.
template <int NSEG>
__device__ __forceinline__ int cta_of(const DecodeSched<NSEG>& sc, int32_t x) {
  if (sc.bpc > 0) return x / sc.bpc;
  int lo = 0, hi = sc.n_ctas - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sc.cta0[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct SegInfo {
  int32_t s, g, q0;      // sequence, kv head, its query token
  int32_t kb, ke;        // keys [kb, ke) of this CTA's part (kb on a 16-key boundary)
  int32_t lo;            // first visible key of the sequence
  int32_t nb;            // 16-key blocks in this CTA's part
  int32_t slot0, pg_off; // first page-table slot; offset in the shared page list
  int32_t npg;           // pages of this part
  int32_t whole;         // the segment lies entirely in this CTA's range
  int32_t gseg;          // segment index in the launch
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Largest i in [0, n) with a[i] <= x (a sorted ascending, a[0] <= x).
template <int NSEG>
__device__ __forceinline__ int seg_of(const DecodeSched<NSEG>& sc, int32_t x) {
  int lo = 0, hi = sc.n_seg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sc.blk0[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Segment table of CTA c's range [cb0, cb1) (segments kfirst ..
// kfirst + nseg - 1 of the launch) and the page ids of the range, in one
// round of loads; every thread of the CTA takes part (two __syncthreads).
// A page id outside the pool, or a position past the page table, becomes -1
// and sets the error word.
template <int NSEG>
__device__ __forceinline__ void load_range_tables(const DecodeSched<NSEG>& sc,
                                                  const DecodeParams& p, int c, int32_t cb0,
                                                  int32_t cb1, int kfirst, int nseg,
                                                  SegInfo* s_seg, int32_t* s_pages,
                                                  int* s_npages) {
  // Segment t's entry (and, from the page counts of the segments before it,
  // its offset in the page list) comes from the launch parameters alone, so
  // one barrier publishes it.
  auto seg_info = [&](int t) {
    const int k = kfirst + t;
    const int32_t sh = sc.seqhead[k];
    SegInfo si;
    si.s = sh >> 8;
    si.g = sh & 255;
    si.gseg = k;
    si.q0 = sc.q0[k];
    const int32_t Lk = sc.len[k];
    const int32_t lo = sc.lo[k];
    const int32_t nb_plan = sc.blk0[k + 1] - sc.blk0[k];
    const int32_t jb = max(cb0, sc.blk0[k]) - sc.blk0[k];
    const int32_t je = min(cb1, sc.blk0[k + 1]) - sc.blk0[k];
    si.lo = lo;
    si.kb = (lo / kDecBlk + jb) * kDecBlk;
    si.ke = min(Lk, (lo / kDecBlk + je) * kDecBlk);
    if (si.ke < si.kb) si.ke = si.kb;
    si.nb = je - jb;
    si.whole = (jb == 0 && je == nb_plan) ? 1 : 0;
    si.slot0 = si.kb >> p.page_shift;
    si.npg = (si.ke > si.kb) ? ((si.ke - 1) >> p.page_shift) - si.slot0 + 1 : 0;
    si.pg_off = 0;
    return si;
  };
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int t = tid; t <= nseg; t += nthr) {
    int off = 0;
    for (int u = 0; u < t; ++u) off += seg_info(u).npg;
    if (t < nseg) {
      SegInfo si = seg_info(t);
      si.pg_off = off;
      s_seg[t] = si;
    } else {
      // One past the last segment: the length of the page list.
      *s_npages = min(off, kMaxCtaPages);
      if (off > kMaxCtaPages) report_error(p.ws, RPA_DEVERR_LENGTHS, c);
    }
  }
  __syncthreads();
  // Page ids of the range, read once (all loads in one round).
  for (int i = tid; i < *s_npages; i += nthr) {
    int t = 0;
    while (t + 1 < nseg && s_seg[t + 1].pg_off <= i) ++t;
    const SegInfo& si = s_seg[t];
    const int32_t slot = si.slot0 + (i - si.pg_off);
    int32_t page = -1;
    if (slot >= p.mpps) {
      report_error(p.ws, RPA_DEVERR_LENGTHS, si.s);
    } else {
      page = __ldg(p.page_table + static_cast<int64_t>(si.s) * p.mpps + slot);
      if (page < 0 || page >= p.num_pages) {
        report_error(p.ws, RPA_DEVERR_PAGE_ID, si.s);
        page = -1;
      }
    }
    s_pages[i] = page;
  }
  __syncthreads();
}

// Launch the log-sum-exp combine of launch dl's cut segments (decode.cu).
int launch_decode_combine(const Plan& plan, const DecodeParams& p, const Plan::DecodeLaunch& dl,
                          int head_dim, void* stream);

// Host: the decode kernels' parameters for a call's arguments.
inline DecodeParams make_decode_params(const Plan& plan, const Args& a) {
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k_pages);
  p.v = static_cast<const __nv_bfloat16*>(a.v_pages);
  p.page_table = a.page_table;
  p.cu_q_lens = a.cu_q_lens;
  p.kv_lens = a.kv_lens;
  p.window = a.window;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.ws = a.workspace;
  p.part_o = reinterpret_cast<float*>(a.workspace + plan.off_partial_o);
  p.part_lse = reinterpret_cast<float*>(a.workspace + plan.off_partial_lse);
  p.hq = plan.hq;
  p.hkv = plan.hkv;
  p.group = plan.hq / plan.hkv;
  int shift = 0;
  while ((1 << shift) < plan.p) ++shift;
  p.page_shift = shift;
  p.mpps = plan.mpps;
  p.num_pages = plan.num_pages;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  return p;
}

// Host: launch dl's schedule from the plan's host copies (segments relative
// to the launch, the per-CTA range table and each range's first and last
// segment).  Returns a cudaError_t.
template <int NSEG>
int fill_decode_sched(const Plan& plan, const Plan::DecodeLaunch& dl, DecodeSched<NSEG>& sc) {
  const int n = dl.seg_end - dl.seg_begin;
  if (n > NSEG) return static_cast<int>(cudaErrorInvalidValue);
  sc.n_seg = n;
  sc.bpc = dl.bpc;
  sc.n_ctas = dl.n_ctas;
  if (dl.bpc == 0) {
    if (dl.n_ctas > kMaxDecodeGrid) return static_cast<int>(cudaErrorInvalidValue);
    for (int i = 0; i <= dl.n_ctas; ++i) sc.cta0[i] = plan.dcta_blk0[dl.cta_begin + i];
  }
  sc.slot_base = dl.slot_base;
  sc.seg_base = dl.seg_begin;
  const int32_t base = plan.dseg_blk0[dl.seg_begin];
  for (int i = 0; i < n; ++i) {
    const int k = dl.seg_begin + i;
    sc.seqhead[i] = plan.dseg_seqhead[k];
    sc.blk0[i] = plan.dseg_blk0[k] - base;
    sc.q0[i] = plan.dseg_q0[k];
    sc.lo[i] = plan.dseg_lo[k];
    sc.len[i] = plan.dseg_len[k];
  }
  sc.blk0[n] = plan.dseg_blk0[dl.seg_end] - base;
  sc.n_blocks = sc.blk0[n];
  if (dl.bpc == 0) {
    // Segment of a block: last k with blk0[k] <= x (segments may be empty).
    auto seg_at = [&](int32_t x) {
      return static_cast<int32_t>(std::upper_bound(sc.blk0, sc.blk0 + n, x) - sc.blk0) - 1;
    };
    for (int i = 0; i < dl.n_ctas; ++i) {
      const int32_t b0 = sc.cta0[i], b1 = sc.cta0[i + 1];
      sc.cta_seg[i] = b0 < b1 ? (seg_at(b0) | (seg_at(b1 - 1) << 16)) : 0;
    }
  }
  return 0;
}

}  // namespace rpa
