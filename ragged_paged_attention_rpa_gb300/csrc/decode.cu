// Split-KV decode for sequences with one query token, and the log-sum-exp
// combine of the splits.
//
// Sources (page titles and sections):
//  * "TPU Deep Dive" slides, chapter 4, "Attention: small share, wrong
//    intensity": decode attention does about G = Hq/Hkv FLOPs per byte of KV
//    at any batch, so it is bound by HBM bandwidth; every byte of a sequence's
//    visible KV is read exactly once here.
//  * "Pallas kernel / vLLM on TPU ... 19,511 tokens per second", section
//    "Strategy 7": a KV block sized for long contexts wasted ~93% of its loads
//    on short ones.  Here no load goes past a sequence's last key (or before
//    its window), and the split length comes from the batch's real lengths.
//  * "Chasing speed of light on TPU v6e", footnote 6: fp32 softmax
//    accumulators (m, l and O stay fp32; only P is rounded to bf16 for the
//    tensor-core product, as any bf16 flash kernel does).
//
// CTA (s, c, g) streams keys [kb, ke) of split c of sequence s for KV head g.
// Its four warps are independent: warp w takes blocks of 16 keys w, w+4, ...,
// copies each block's K and V rows into its own shared-memory ring with
// coalesced 16-byte cp.async loads through the page table, and runs
//     S^T[16 keys x 8 heads] = K . Q^T     (mma.m16n8k16, bf16 -> fp32)
//     O^T[D x 8 heads]     += V^T . P^T   (P^T rebuilt in registers by a
//                                          warp-level 8x8 transpose)
// keeping an online softmax per head.  The warps merge through shared memory
// at the end.  One split writes the output; several write fp32 partials
// (O / l and log2-sum-exp), and the split that finishes last for a sequence
// (a per-sequence arrival counter in the workspace, reset by that split)
// merges them: out = sum_c 2^(lse_c - M) O_c / sum_c 2^(lse_c - M).
// The page ids of a split are read into shared memory once, before the copy
// pipeline starts, so no copy waits on a page-table load.
#include "common.cuh"
#include "rpa_internal.h"

namespace rpa {

namespace {

constexpr int kWarps = 4;
constexpr int kBlk = 16;  // keys per warp block (the MMA's M)
constexpr int kMaxMergeSplits = 64;

constexpr int stages_for(int D) { return D >= 256 ? 3 : 4; }

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
  float* part_o;
  float* part_lse;
  int32_t* arrivals;  // [num_seqs * hkv], zero between calls
  int32_t num_seqs, hq, hkv, group, page_shift, mpps, num_pages;
  int32_t kv_split, max_splits;
  float scale_log2;  // sm_scale * log2(e)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: zero-fill, nothing read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Element offset of 16-byte chunk `chunk` of row `row` in a [rows][D] bf16
// tile whose chunks are XOR-swizzled by row (conflict-free ldmatrix).
template <int D>
__device__ __forceinline__ int swz(int row, int chunk) {
  return row * D + ((chunk ^ (row & 7)) << 3);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32, 1) decode_split_kernel(DecodeParams p) {
  constexpr int S = stages_for(D);
  constexpr int KT = D / 16;        // k-steps of the score MMA, m-tiles of the PV MMA
  constexpr int CPR = D / 8;        // 16-byte chunks per row
  constexpr int RPI = 32 / CPR > 0 ? 32 / CPR : 1;  // rows per copy instruction
  constexpr int TILE = kBlk * D;    // elements of one K (or V) block
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __nv_bfloat16* smem = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __shared__ uint32_t valid_mask[kWarps][S];
  __shared__ float wm[kWarps][8], wl[kWarps][8];

  const int s = blockIdx.x, c = blockIdx.y, g = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t q0 = __ldg(p.cu_q_lens + s);
  if (__ldg(p.cu_q_lens + s + 1) - q0 != 1) return;
  const int32_t L = __ldg(p.kv_lens + s);
  const int32_t W = p.window ? __ldg(p.window + s) : 0;
  const int32_t lo = (W > 0 && L - W > 0) ? L - W : 0;
  const int32_t n = L - lo;
  const int32_t nsplit = (n + p.kv_split - 1) / p.kv_split;
  if (nsplit > p.max_splits && c == 0 && g == 0 && threadIdx.x == 0)
    report_error(p.ws, RPA_DEVERR_LENGTHS, s);
  if (c >= nsplit) return;
  const int32_t kb = lo + c * p.kv_split;
  const int32_t ke = min(L, kb + p.kv_split);
  const int32_t nblk = (ke - kb + kBlk - 1) / kBlk;
  const int32_t my_blocks = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;
  const int G = p.group;
  const int32_t* pt = p.page_table + static_cast<int64_t>(s) * p.mpps;
  const int32_t psize = 1 << p.page_shift;

  // Page ids of this split, read once (coalesced) into shared memory.
  __shared__ int32_t s_pages[kMaxSplitPages];
  const int32_t slot0 = kb >> p.page_shift;
  const int32_t npg = ((ke - 1) >> p.page_shift) - slot0 + 1;
  for (int i = threadIdx.x; i < npg && i < kMaxSplitPages; i += kWarps * 32) {
    const int32_t slot = slot0 + i;
    int32_t page = -1;
    if (slot >= p.mpps) {
      report_error(p.ws, RPA_DEVERR_LENGTHS, s);
    } else {
      page = __ldg(pt + slot);
      if (page < 0 || page >= p.num_pages) {
        report_error(p.ws, RPA_DEVERR_PAGE_ID, s);
        page = -1;
      }
    }
    s_pages[i] = page;
  }
  if (npg > kMaxSplitPages && threadIdx.x == 0) report_error(p.ws, RPA_DEVERR_LENGTHS, s);
  __syncthreads();

  __nv_bfloat16* ring = smem + warp * S * 2 * TILE;  // this warp's S stages of K then V
  // Issue the copies of this warp's i-th block into stage st (always commits).
  auto issue = [&](int i, int st) {
    if (i < my_blocks) {
      const int32_t key0 = kb + (warp + i * kWarps) * kBlk;
      // Lanes 0..15 look up the page of one key each.
      int32_t page = 0;
      bool ok = false;
      if (lane < kBlk) {
        const int32_t key = key0 + lane;
        const int32_t idx = (key >> p.page_shift) - slot0;
        if (key < ke && idx < kMaxSplitPages) {
          page = s_pages[idx];
          ok = page >= 0;
        }
      }
      const uint32_t vmask = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) valid_mask[warp][st] = vmask;
      __nv_bfloat16* kt = ring + st * 2 * TILE;
      __nv_bfloat16* vt = kt + TILE;
#pragma unroll
      for (int r0 = 0; r0 < kBlk; r0 += RPI) {
        const int r = r0 + lane / CPR;
        const int ch = lane % CPR;
        const int32_t pg = __shfl_sync(0xffffffffu, page, r & 31);
        const bool v = (vmask >> r) & 1u;
        const int32_t key = key0 + r;
        const int64_t off =
            ((static_cast<int64_t>(pg) * psize + (key & (psize - 1))) * p.hkv + g) * D + ch * 8;
        cp_async16(smem_u32(kt + swz<D>(r, ch)), v ? p.k + off : p.k, v);
        cp_async16(smem_u32(vt + swz<D>(r, ch)), v ? p.v + off : p.v, v);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < S - 1; ++i) issue(i, i);

  // Q^T as the B operand: lane holds head lane/4, dims 2(lane%4)+{0,1} (+8).
  // Loaded after the first copies are in flight.
  uint32_t qf[KT][2];
  {
    const int h = lane >> 2;
    const bool hv = h < G;
    const __nv_bfloat16* qr = p.q + (static_cast<int64_t>(q0) * p.hq + g * G + (hv ? h : 0)) * D;
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      const int d0 = kt * 16 + 2 * (lane & 3);
      qf[kt][0] = hv ? *reinterpret_cast<const uint32_t*>(qr + d0) : 0u;
      qf[kt][1] = hv ? *reinterpret_cast<const uint32_t*>(qr + d0 + 8) : 0u;
    }
  }

  float m[2] = {-INFINITY, -INFINITY};  // running max (log2 domain), heads 2(lane%4)+j
  float l[2] = {0.f, 0.f};              // this lane's share of the running sum
  float o[KT][4];
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int i = 0; i < my_blocks; ++i) {
    issue(i + S - 1, (i + S - 1) % S);
    cp_async_wait<S - 1>();
    __syncwarp();
    const int st = i % S;
    const __nv_bfloat16* kt = ring + st * 2 * TILE;
    const __nv_bfloat16* vt = kt + TILE;
    const uint32_t vmask = valid_mask[warp][st];

    // Scores S^T = K Q^T for 16 keys x 8 heads (two chains for latency).
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int row = lane & 15;
      const int hi = lane >> 4;
#pragma unroll
      for (int kt2 = 0; kt2 < KT; ++kt2) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(smem_u32(kt + swz<D>(row, 2 * kt2 + hi)), a0, a1, a2, a3);
        if (kt2 & 1) mma_bf16(sb, a0, a1, a2, a3, qf[kt2][0], qf[kt2][1]);
        else mma_bf16(sa, a0, a1, a2, a3, qf[kt2][0], qf[kt2][1]);
      }
    }
    // Row (key) validity: rows lane/4 and lane/4 + 8.
    const int r_top = lane >> 2, r_bot = r_top + 8;
    const bool v_top = (vmask >> r_top) & 1u, v_bot = (vmask >> r_bot) & 1u;
    float x[4];
    x[0] = v_top ? (sa[0] + sb[0]) * p.scale_log2 : -INFINITY;
    x[1] = v_top ? (sa[1] + sb[1]) * p.scale_log2 : -INFINITY;
    x[2] = v_bot ? (sa[2] + sb[2]) * p.scale_log2 : -INFINITY;
    x[3] = v_bot ? (sa[3] + sb[3]) * p.scale_log2 : -INFINITY;
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    // Every block holds at least one valid key, so the new max is finite.
    const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
    const float al0 = fast_exp2(m[0] - mn0), al1 = fast_exp2(m[1] - mn1);
    m[0] = mn0;
    m[1] = mn1;
    const float p0 = fast_exp2(x[0] - mn0), p1 = fast_exp2(x[1] - mn1);
    const float p2 = fast_exp2(x[2] - mn0), p3 = fast_exp2(x[3] - mn1);
    l[0] = l[0] * al0 + p0 + p2;
    l[1] = l[1] * al1 + p1 + p3;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }
    // P^T as the B operand of O^T += V^T P^T.
    const uint32_t b0 = transpose8x8(pack_bf16x2(p0, p1));
    const uint32_t b1 = transpose8x8(pack_bf16x2(p2, p3));
    {
      const int row = (lane & 7) + ((lane >> 4) << 3);
      const int hi = (lane >> 3) & 1;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(smem_u32(vt + swz<D>(row, 2 * mt + hi)), a0, a1, a2, a3);
        mma_bf16(o[mt], a0, a1, a2, a3, b0, b1);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // Reduce l over the lanes holding the same heads.
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
  }
  if (lane < 4) {
    wm[warp][2 * lane] = m[0];
    wm[warp][2 * lane + 1] = m[1];
    wl[warp][2 * lane] = l[0];
    wl[warp][2 * lane + 1] = l[1];
  }
  __syncthreads();  // every warp is done with its ring: reuse it for the merge
  float* so = reinterpret_cast<float*>(smem_raw);  // [kWarps][8][D]
  {
    // Scale this warp's O^T by exp2(m_w - M) before summing over warps.
    const int h0 = 2 * (lane & 3);
    float f[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][h0 + j]);
      f[j] = (m[j] == -INFINITY) ? 0.f : fast_exp2(m[j] - M);
    }
    float* base = so + warp * 8 * D;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int d = mt * 16 + (lane >> 2);
      base[h0 * D + d] = o[mt][0] * f[0];
      base[(h0 + 1) * D + d] = o[mt][1] * f[1];
      base[h0 * D + d + 8] = o[mt][2] * f[0];
      base[(h0 + 1) * D + d + 8] = o[mt][3] * f[1];
    }
  }
  __syncthreads();
  // Final values for G heads x D dims: 8 consecutive dims per thread step.
  for (int e = threadIdx.x * 8; e < G * D; e += kWarps * 32 * 8) {
    const int h = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][h]);
    float Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      Lsum += (wm[w][h] == -INFINITY) ? 0.f : wl[w][h] * fast_exp2(wm[w][h] - M);
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float4* src = reinterpret_cast<const float4*>(so + (w * 8 + h) * D + d);
      const float4 u = src[0], v = src[1];
      acc[0] += u.x; acc[1] += u.y; acc[2] += u.z; acc[3] += u.w;
      acc[4] += v.x; acc[5] += v.y; acc[6] += v.z; acc[7] += v.w;
    }
    const float inv = 1.f / Lsum;
    const int hq_idx = g * G + h;
    if (nsplit == 1) {
      uint4 pk;
      pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(q0) * p.hq + hq_idx) * D + d) = pk;
    } else {
      const int64_t row = (static_cast<int64_t>(s) * p.max_splits + c) * p.hq + hq_idx;
      float4* dst = reinterpret_cast<float4*>(p.part_o + row * D + d);
      dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
      if (d == 0) p.part_lse[row] = M + __log2f(Lsum);
    }
  }
  if (nsplit == 1) return;

  // Arrival: the last split of (sequence, KV head) to finish merges them all.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(p.arrivals + s * p.hkv + g, 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int ns = min(nsplit, kMaxMergeSplits);
  float* s_lse = reinterpret_cast<float*>(smem_raw);  // [ns][G], ring is free
  const int64_t row0 = static_cast<int64_t>(s) * p.max_splits * p.hq + g * G;
  for (int i = threadIdx.x; i < ns * G; i += kWarps * 32)
    s_lse[i] = __ldcg(p.part_lse + row0 + static_cast<int64_t>(i / G) * p.hq + i % G);
  __syncthreads();
  for (int e = threadIdx.x * 4; e < G * D; e += kWarps * 32 * 4) {
    const int h = e / D, d = e % D;
    float M = -INFINITY;
    for (int k = 0; k < ns; ++k) M = fmaxf(M, s_lse[k * G + h]);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < ns; ++k) {
      const float w = fast_exp2(s_lse[k * G + h] - M);
      const float4 u = __ldcg(reinterpret_cast<const float4*>(
          p.part_o + (row0 + static_cast<int64_t>(k) * p.hq + h) * D + d));
      wsum += w;
      acc.x += w * u.x; acc.y += w * u.y; acc.z += w * u.z; acc.w += w * u.w;
    }
    const float inv = 1.f / wsum;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(q0) * p.hq + g * G + h) * D + d) = pk;
  }
  if (threadIdx.x == 0) p.arrivals[s * p.hkv + g] = 0;  // ready for the next call
}

template <int D>
constexpr size_t decode_smem() {
  return static_cast<size_t>(kWarps) * stages_for(D) * 2 * kBlk * D * sizeof(__nv_bfloat16);
}

template <int D>
int launch_decode_t(const Plan& plan, const Args& a, cudaStream_t stream) {
  static_assert(decode_smem<D>() >= kWarps * 8 * D * sizeof(float), "merge buffer fits");
  static_assert(decode_smem<D>() >= kMaxMergeSplits * 8 * sizeof(float), "lse buffer fits");
  constexpr size_t smem = decode_smem<D>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return static_cast<int>(e);
    configured = true;
  }
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
  p.part_o = plan.max_splits > 1 ? reinterpret_cast<float*>(a.workspace + plan.off_partial_o) : nullptr;
  p.part_lse = plan.max_splits > 1 ? reinterpret_cast<float*>(a.workspace + plan.off_partial_lse) : nullptr;
  p.arrivals = plan.max_splits > 1 ? reinterpret_cast<int32_t*>(a.workspace + plan.off_arrivals) : nullptr;
  p.num_seqs = plan.num_seqs;
  p.hq = plan.hq;
  p.hkv = plan.hkv;
  p.group = plan.hq / plan.hkv;
  int shift = 0;
  while ((1 << shift) < plan.p) ++shift;
  p.page_shift = shift;
  p.mpps = plan.mpps;
  p.num_pages = plan.num_pages;
  p.kv_split = plan.kv_split;
  p.max_splits = plan.max_splits;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  dim3 grid(plan.num_seqs, plan.max_splits, plan.hkv);
  decode_split_kernel<D><<<grid, kWarps * 32, smem, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  trace_mark(RPA_KERNEL_DECODE_SPLIT, stream);
  return 0;
}

}  // namespace

// ---------------------------------------------------------------------------
// Fixed scratch for rpa_forward_decode_noalloc: the decode kernel's workspace
// (error word, split partials, arrival counters) in a file-scope device array,
// so that callers who cannot allocate device memory can still run decode.
// Every GPU that loads this library holds the array until the process exits.
// In host code `g_noalloc_scratch` names a host-side stand-in, never a device
// address; the device address comes from cudaGetSymbolAddress, resolved once
// per device (with that device current) on the first call on that device.

static __device__ __align__(256) unsigned char g_noalloc_scratch[RPA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

int noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return 0;
}

bool decode_supported(int32_t head_dim, int32_t group) {
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) && group >= 1 && group <= 8;
}

int decode_ctas_per_sm(int32_t head_dim) {
  switch (head_dim) {
    case 64: return static_cast<int>(220 * 1024 / decode_smem<64>());
    case 128: return static_cast<int>(220 * 1024 / decode_smem<128>());
    default: return static_cast<int>(220 * 1024 / decode_smem<256>());
  }
}

int launch_decode(const Plan& plan, const Args& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (plan.d) {
    case 64: return launch_decode_t<64>(plan, a, s);
    case 128: return launch_decode_t<128>(plan, a, s);
    case 256: return launch_decode_t<256>(plan, a, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace rpa
