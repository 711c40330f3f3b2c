// Split-KV decode for sequences with one query token, on one balanced wave.
//
// Sources (page titles and sections):
//  * "TPU Deep Dive" slides, chapter 4, "Attention: small share, wrong
//    intensity": decode attention does about G = Hq/Hkv FLOPs per byte of KV
//    at any batch, so it is bound by HBM bandwidth; every byte of a sequence's
//    visible KV is read exactly once here.
//  * "Pallas kernel / vLLM on TPU ... 19,511 tokens per second", section
//    "Strategy 7": a KV block sized for long contexts wasted ~93% of its loads
//    on short ones, and block size changes scheduling, not arithmetic.  Here no
//    load goes past a sequence's last key (or before its window), and the work
//    is cut by the batch's real lengths.
//  * "Chasing speed of light on TPU v6e", footnote 6: fp32 softmax
//    accumulators (m, l and O stay fp32; only P is rounded to bf16 for the
//    tensor-core product, as any bf16 flash kernel does).
//
// Schedule.  The visible keys of every (decode sequence, KV head) pair form a
// "segment" of 16-key blocks; the segments are laid end to end and the block
// stream is cut into contiguous ranges of equal cost (blocks plus a fixed
// charge per segment touched), one per CTA (one CTA per SM, a single wave),
// so every CTA finishes at about the same time whatever the length mix.  A
// CTA's range may start or end inside a segment.
//
// CTA.  Four independent compute warps take the range's blocks round-robin
// (warp w: blocks w, w+4, ... of each segment).  Blocks sit on absolute
// 16-key boundaries, so with pages of 16 tokens or more a block is 16
// consecutive rows of one page.  A fifth warp does all the copying: its lane
// w fetches warp w's blocks with TMA (one 4-D box over the pool per K or V
// block: every 128-byte chunk of the block's 16 rows, 128-byte swizzled) into
// w's own shared-memory ring, completion on the stage's full mbarrier, and
// refills a stage once w has released it on its empty mbarrier, so the
// compute warps only wait and compute.  The page ids of the CTA's whole range
// are read into shared memory once, first, in one round of loads (the
// range's first and last segment come from the plan).  Per block a compute
// warp runs
//     S^T[16 keys x 8 heads] = K . Q^T     (mma.m16n8k16, bf16 -> fp32)
//     O^T[D x 8 heads]     += V^T . P^T   (P^T rebuilt in registers by a
//                                          warp-level 8x8 transpose)
// with an online softmax per head.  The copy pipeline runs on across segment
// boundaries.  At the end of each segment the warps merge in shared memory,
// each scaling its state by its share of the normalised result first; a
// segment wholly inside the range writes the output, a cut one writes an fp32
// partial (O / l and log2-sum-exp).  A second kernel, launched as a
// programmatic dependent, combines the partials of every cut segment:
// out = sum_c 2^(lse_c - M) O_c / sum_c 2^(lse_c - M).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "decode_sched.cuh"
#include "rpa_internal.h"
#include "sm100_ptx.cuh"

namespace rpa {

namespace {

constexpr int kWarps = 4;  // compute warps; one more warp issues their copies
constexpr int kBlk = 16;  // keys per warp block (the MMA's M)

constexpr int stages_for(int D) { return D >= 256 ? 3 : 4; }

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
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two e4m3 values (low byte first) -> f16x2 (exact: e4m3 is a subset of f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
      : "=r"(r) : "r"(two));
  return r;
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <bool FP8>
__device__ __forceinline__ void mma_t(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                      uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (FP8) mma_f16(c, a0, a1, a2, a3, b0, b1);
  else mma_bf16(c, a0, a1, a2, a3, b0, b1);
}
template <bool FP8>
__device__ __forceinline__ uint32_t pack_t(float lo, float hi) {
  if constexpr (FP8) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}


// Element offset of 16-byte chunk `chunk` of row `row` in a 16-row bf16 tile
// as TMA writes it: D/64 boxes of [16 rows][64 dims], 128-byte swizzle (the
// 16-byte chunk index XORed with the row's low three bits).
__device__ __forceinline__ int swz(int row, int chunk) {
  return (chunk >> 3) * (16 * 64) + row * 64 + (((chunk & 7) ^ (row & 7)) << 3);
}

// Shared memory of a decode CTA: per warp a ring of S K slots and S V slots
// (one 16-key block of K or of V each, as TMA writes them: 128-byte swizzled
// rows; K slot s, then V slot s at S slots further), for fp8 pages a per-warp
// f16 copy of the V block being consumed, two Q tiles and the merge buffers.
// K and V have slots of their own so that a block's K slot is refilled as
// soon as its scores are out, before its V is used (fp8 pages: V is copied
// out first, and both slots go back after the scores).
template <int D, bool FP8>
struct DecodeSmem {
  static constexpr int S = FP8 ? 4 : stages_for(D);
  static constexpr int TILE = kBlk * D;                         // elements of a K (or V) tile
  static constexpr int ESZ = FP8 ? 1 : 2;                       // bytes per element as stored
  static constexpr size_t kSlotBytes = size_t(TILE) * ESZ;     // one K or V block
  static constexpr size_t kStageBytes = 2 * kSlotBytes;
  static constexpr size_t kRing = size_t(kWarps) * S * kStageBytes;
  static constexpr size_t kConv = FP8 ? size_t(kWarps) * TILE * 2 : 0;
  static constexpr size_t kQ = 2 * 8 * D * 2;                   // two Q tiles (G <= 8)
  static constexpr int kORow = D + 4;                           // padded row of the merge buffer
  static constexpr size_t kO = 2 * 8 * kORow * 4;               // two merge buffers
  static constexpr size_t kBytes = kRing + kConv + kQ + kO + 1024;  // + 1024-byte alignment
};

// An fp8 block (16 rows x D bytes, 128-byte swizzled rows of 128 bytes as TMA
// writes them) -> f16 in the layout swz() reads (16-byte chunks of 8).
template <int D>
__device__ __forceinline__ void fp8_tile_to_f16(const unsigned char* src, __nv_bfloat16* dst,
                                                int lane) {
  constexpr int kGroups = D / 8;   // 8-element groups per row
#pragma unroll
  for (int k = 0; k < (kBlk * kGroups) / 32; ++k) {
    const int gi = lane + 32 * k;
    const int r = gi / kGroups, d0 = (gi % kGroups) * 8;
    const int b = d0 & 127;
    const uint2 w = *reinterpret_cast<const uint2*>(
        src + (d0 >> 7) * (kBlk * 128) + r * 128 + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15)));
    uint4 o;
    o.x = e4m3x2_to_f16x2(w.x & 0xffffu);
    o.y = e4m3x2_to_f16x2(w.x >> 16);
    o.z = e4m3x2_to_f16x2(w.y & 0xffffu);
    o.w = e4m3x2_to_f16x2(w.y >> 16);
    *reinterpret_cast<uint4*>(dst + swz(r, d0 >> 3)) = o;
  }
}

template <int D, int NSEG, bool FP8>
__global__ void __launch_bounds__((kWarps + 1) * 32, 1)
decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const DecodeParams p, const __grid_constant__ DecodeSched<NSEG> sc) {
  using L = DecodeSmem<D, FP8>;
  constexpr int S = L::S;
  constexpr int KT = D / 16;        // k-steps of the score MMA, m-tiles of the PV MMA
  constexpr int TILE = L::TILE;
  extern __shared__ __align__(128) unsigned char smem_dyn[];
  unsigned char* smem_raw = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  __nv_bfloat16* conv = reinterpret_cast<__nv_bfloat16*>(smem_raw + L::kRing);
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem_raw + L::kRing + L::kConv);
  float* so = reinterpret_cast<float*>(smem_raw + L::kRing + L::kConv + L::kQ);
  __shared__ int32_t s_pages[kMaxCtaPages];
  __shared__ SegInfo s_seg[kMaxCtaSegs];
  __shared__ uint32_t valid_mask[kWarps][S];
  __shared__ float wm[kWarps][8], wl[kWarps][8];
  __shared__ int s_npages, s_abort;
  __shared__ __align__(8) uint64_t kfull_bar[kWarps][S], vfull_bar[kWarps][S];    // slot landed
  __shared__ __align__(8) uint64_t kempty_bar[kWarps][S], vempty_bar[kWarps][S];  // slot consumed
  __shared__ __align__(8) uint64_t q_bar[2];   // Q buffer t & 1 holds segment t's queries

  // The combine kernel may be scheduled now; it waits for this grid's end.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int G = p.group;
  const int c = blockIdx.x;
  const int32_t cb0 = range_start(sc, c);
  const int32_t cb1 = range_start(sc, c + 1);
  if (cb0 >= cb1) return;
  // First and last segment of the range: from the plan's per-CTA table, or
  // by search for ranges of a fixed block count.
  const int kfirst = sc.bpc > 0 ? seg_of(sc, cb0) : (sc.cta_seg[c] & 0xffff);
  const int klast = sc.bpc > 0 ? seg_of(sc, cb1 - 1) : (sc.cta_seg[c] >> 16);
  int nseg = klast - kfirst + 1;
  if (nseg > kMaxCtaSegs) {
    if (tid == 0) report_error(p.ws, RPA_DEVERR_LENGTHS, c);
    nseg = kMaxCtaSegs;
  }

  if (tid == 0) {
    for (int i = 0; i < kWarps * S; ++i) {
      sm100::mbar_init(&kfull_bar[i / S][i % S], 1);
      sm100::mbar_init(&vfull_bar[i / S][i % S], 1);
      sm100::mbar_init(&kempty_bar[i / S][i % S], 1);
      sm100::mbar_init(&vempty_bar[i / S][i % S], 1);
    }
    sm100::mbar_init(&q_bar[0], 1);
    sm100::mbar_init(&q_bar[1], 1);
    s_abort = 0;
    sm100::fence_barrier_init();
    sm100::prefetch_tmap(&tm_k);
    sm100::prefetch_tmap(&tm_v);
  }
  load_range_tables(sc, p, c, cb0, cb1, kfirst, nseg, s_seg, s_pages, &s_npages);

  volatile int* abort = &s_abort;
  auto page_of = [&](const SegInfo& si, int32_t key0) {
    const int32_t idx = si.pg_off + (key0 >> p.page_shift) - si.slot0;
    return idx < kMaxCtaPages ? s_pages[idx] : -1;
  };
  // Q of segment t: G x D contiguous bf16 (the G heads of KV head g are
  // adjacent), one bulk copy into buffer t & 1 on q_bar[t & 1].
  int q_last0 = -1, q_last1 = -1;   // (thread 0) last segment copied into buffer 0 / 1
  auto load_q = [&](int t) {
    const SegInfo& si = s_seg[t];
    if (t & 1) q_last1 = t; else q_last0 = t;
    const __nv_bfloat16* src = p.q + (static_cast<int64_t>(si.q0) * p.hq + si.g * G) * D;
    sm100::mbar_arrive_expect_tx(&q_bar[t & 1], G * D * 2);
    sm100::bulk_load(qs + (t & 1) * 8 * D, src, G * D * 2, &q_bar[t & 1]);
  };
  if (tid == 0)
    for (int t = 0; t < 2 && t < nseg; ++t) load_q(t);
  __syncthreads();

  if (warp == kWarps) {
    // ---- Copy warp: lane w (< 4) streams compute warp w's blocks (segment
    // t, local blocks w, w + 4, ...) through w's K and V slots, each as w
    // releases it.  Per block: its keys' validity mask (visible and on a good
    // page) into shared memory, then one 4-D TMA box each for K and V (a bad
    // page reads zeros), completion on the slot's full barrier.
    if (lane < kWarps) {
      const int w = lane;
      unsigned char* ring = smem_raw + w * S * L::kStageBytes;
      int ist = 0, isj = w;
      while (ist < nseg && isj >= s_seg[ist].nb) { ++ist; isj = w; }
      int i = 0, nk = 0, nv = 0;   // blocks taken; K and V copies issued
      for (; ist < nseg; ++i) {
        const int st = i % S;
        if (i >= S && !sm100::mbar_wait(&kempty_bar[w][st], ((i / S) - 1) & 1, abort, 2000000000ull)) {
          report_error(p.ws, RPA_DEVERR_TIMEOUT, c);
          break;
        }
        const SegInfo& si = s_seg[ist];
        const int32_t key0 = si.kb + isj * kBlk;
        const int32_t page = page_of(si, key0);
        uint32_t vmask = 0;
        if (page >= 0) {
          const int32_t a = max(si.lo - key0, 0), b = min(si.ke - key0, kBlk);
          if (b > a) vmask = ((1u << b) - 1u) & ~((1u << a) - 1u);
        }
        valid_mask[w][st] = vmask;
        // Rows of the block: page * P + (key0 % P); a bad page reads zeros.
        const int32_t row = page >= 0 ? page * (1 << p.page_shift) + (key0 & ((1 << p.page_shift) - 1))
                                      : -kBlk;
        // One box per K and per V block: every 128-byte chunk of the block's
        // 16 rows ([chunk][row][128 B] in the slot).
        unsigned char* kt = ring + st * L::kSlotBytes;
        unsigned char* vt = ring + (S + st) * L::kSlotBytes;
        if constexpr (FP8) {
          // fp8 pages: the compute warp copies V out (widened) before its
          // score MMAs, so K and V share the K slot's barriers.
          sm100::mbar_arrive_expect_tx(&kfull_bar[w][st], static_cast<uint32_t>(2 * L::kSlotBytes));
          sm100::tma_load_4d(kt, &tm_k, &kfull_bar[w][st], 0, si.g, row, 0);
          sm100::tma_load_4d(vt, &tm_v, &kfull_bar[w][st], 0, si.g, row, 0);
          ++nk;
        } else {
          sm100::mbar_arrive_expect_tx(&kfull_bar[w][st], static_cast<uint32_t>(L::kSlotBytes));
          sm100::tma_load_4d(kt, &tm_k, &kfull_bar[w][st], 0, si.g, row, 0);
          ++nk;
          if (i >= S && !sm100::mbar_wait(&vempty_bar[w][st], ((i / S) - 1) & 1, abort, 2000000000ull)) {
            report_error(p.ws, RPA_DEVERR_TIMEOUT, c);
            break;
          }
          sm100::mbar_arrive_expect_tx(&vfull_bar[w][st], static_cast<uint32_t>(L::kSlotBytes));
          sm100::tma_load_4d(vt, &tm_v, &vfull_bar[w][st], 0, si.g, row, 0);
          ++nv;
        }
        isj += kWarps;
        while (ist < nseg && isj >= s_seg[ist].nb) { ++ist; isj = w; }
      }
      if (*abort) {
        // Let every copy still in flight land before the CTA exits: the last
        // S K and V copies issued (one per slot).
        for (int k = max(nk - S, 0); k < nk; ++k) {
          int dummy = 0;
          sm100::mbar_wait(&kfull_bar[w][k % S], (k / S) & 1, &dummy, 200000000ull);
        }
        for (int k = max(nv - S, 0); k < nv; ++k) {
          int dummy = 0;
          sm100::mbar_wait(&vfull_bar[w][k % S], (k / S) & 1, &dummy, 200000000ull);
        }
      }
    }
    return;
  }
  // The compute warps synchronise among themselves (named barrier 1).
  auto compute_sync = []() { asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory"); };
  unsigned char* ring = smem_raw + warp * S * L::kStageBytes;

  int count = 0;  // blocks consumed by this warp
  // Whether block `count` has landed, as tested (mbar_test) during the
  // previous block's math; false: wait for it.  A wait whose result is
  // branched on costs its full latency even when the block is there.
  bool next_ready = false;
  for (int t = 0; t < nseg; ++t) {
    const SegInfo si = s_seg[t];
    if (!sm100::mbar_wait(&q_bar[t & 1], (t >> 1) & 1, abort, 2000000000ull)) {
      if (lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, c);
      break;
    }
    // Q^T as the B operand: lane holds head lane/4, dims 2(lane%4)+{0,1} (+8).
    uint32_t qf[KT][2];
    {
      const int h = lane >> 2;
      const bool hv = h < G;
      const __nv_bfloat16* qr = qs + (t & 1) * 8 * D + (hv ? h : 0) * D;
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        if constexpr (FP8) {
          // The K fragments of fp8 pages are read four bytes at a time (see
          // below): fragment dimensions {2c, 2c + 1} and {2c + 8, 2c + 9} of
          // each 16 (c = lane % 4) hold dimensions 4c .. 4c + 3; q's take the
          // same order, which leaves every score unchanged.  bf16 pairs ->
          // f16 pairs for the f16 products with the fp8 pages.
          const int d0 = kt * 16 + 4 * (lane & 3);
          const uint2 q4 = hv ? *reinterpret_cast<const uint2*>(qr + d0) : make_uint2(0u, 0u);
          qf[kt][0] = pack_f16x2(__uint_as_float(q4.x << 16), __uint_as_float(q4.x & 0xffff0000u));
          qf[kt][1] = pack_f16x2(__uint_as_float(q4.y << 16), __uint_as_float(q4.y & 0xffff0000u));
        } else {
          const int d0 = kt * 16 + 2 * (lane & 3);
          qf[kt][0] = hv ? *reinterpret_cast<const uint32_t*>(qr + d0) : 0u;
          qf[kt][1] = hv ? *reinterpret_cast<const uint32_t*>(qr + d0 + 8) : 0u;
        }
      }
    }
    // fp8 pages: the K scale joins the logit scale, the V scale the output.
    const float sl2 = FP8 ? p.scale_log2 * __ldg(p.k_scale + si.g) : p.scale_log2;
    const float vsc = FP8 ? __ldg(p.v_scale + si.g) : 1.f;
    float m[2] = {-INFINITY, -INFINITY};  // running max (log2 domain), heads 2(lane%4)+j
    float l[2] = {0.f, 0.f};              // this lane's share of the running sum
    float o[KT][4];
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    for (int j = warp; j < si.nb; j += kWarps, ++count) {
      const int st = count % S;
      const uint32_t par = (count / S) & 1;
      if (!next_ready && !sm100::mbar_wait(&kfull_bar[warp][st], par, abort, 2000000000ull)) {
        if (lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, c);
        break;
      }
      const __nv_bfloat16* kt = reinterpret_cast<const __nv_bfloat16*>(ring + st * L::kSlotBytes);
      const unsigned char* vraw = ring + (S + st) * L::kSlotBytes;
      const uint32_t vmask = valid_mask[warp][st];
      const __nv_bfloat16* vt;
      if constexpr (FP8) {
        // V as f16 in this warp's copy (its fragments need a transpose,
        // which ldmatrix does on 16-bit data), made first (K and V landed
        // together); both slots go back to the copy warp after the scores.
        __nv_bfloat16* cv = conv + warp * TILE;
        fp8_tile_to_f16<D>(vraw, cv, lane);
        __syncwarp();
        vt = cv;
      } else {
        vt = reinterpret_cast<const __nv_bfloat16*>(vraw);
      }
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (FP8) {
        // K fragments straight from the e4m3 stage ([128-dimension chunk]
        // [16 rows][128 B], 128-byte swizzled): lane (g = lane / 4, c =
        // lane % 4) reads dimensions 16 kt + 4c .. + 3 of rows g and g + 8
        // as one word each and widens them in registers (exact), in the
        // dimension order q's fragments were built in.
        const unsigned char* kraw = ring + st * L::kSlotBytes;
        const int g = lane >> 2, c4 = 4 * (lane & 3);
#pragma unroll
        for (int kt2 = 0; kt2 < KT; ++kt2) {
          const int d = kt2 * 16;
          const unsigned char* base = kraw + (d >> 7) * (kBlk * 128) + g * 128 +
                                      ((((d & 127) >> 4) ^ (g & 7)) << 4) + c4;
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(base);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(base + 8 * 128);
          const uint32_t a0 = e4m3x2_to_f16x2(w0 & 0xffffu), a2 = e4m3x2_to_f16x2(w0 >> 16);
          const uint32_t a1 = e4m3x2_to_f16x2(w1 & 0xffffu), a3 = e4m3x2_to_f16x2(w1 >> 16);
          if (kt2 & 1) mma_t<FP8>(sb, a0, a1, a2, a3, qf[kt2][0], qf[kt2][1]);
          else mma_t<FP8>(sa, a0, a1, a2, a3, qf[kt2][0], qf[kt2][1]);
        }
      } else {
        const int row = lane & 15;
        const int hi = lane >> 4;
#pragma unroll
        for (int kt2 = 0; kt2 < KT; ++kt2) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(smem_u32(kt + swz(row, 2 * kt2 + hi)), a0, a1, a2, a3);
          if (kt2 & 1) mma_t<FP8>(sb, a0, a1, a2, a3, qf[kt2][0], qf[kt2][1]);
          else mma_t<FP8>(sa, a0, a1, a2, a3, qf[kt2][0], qf[kt2][1]);
        }
      }
      // The scores are out: the K slot (fp8: and the V slot) goes back to
      // the copy warp.  Then a look at this block's V and the next block's K
      // (this warp's blocks run on across segments).
      __syncwarp();
      if (lane == 0) sm100::mbar_arrive(&kempty_bar[warp][st]);
      const bool v_ready = FP8 || sm100::mbar_test(&vfull_bar[warp][st], par);
      next_ready = sm100::mbar_test(&kfull_bar[warp][(count + 1) % S], ((count + 1) / S) & 1);
      const int r_top = lane >> 2, r_bot = r_top + 8;
      const bool v_top = (vmask >> r_top) & 1u, v_bot = (vmask >> r_bot) & 1u;
      float x[4];
      x[0] = v_top ? (sa[0] + sb[0]) * sl2 : -INFINITY;
      x[1] = v_top ? (sa[1] + sb[1]) * sl2 : -INFINITY;
      x[2] = v_bot ? (sa[2] + sb[2]) * sl2 : -INFINITY;
      x[3] = v_bot ? (sa[3] + sb[3]) * sl2 : -INFINITY;
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
      const uint32_t b0 = transpose8x8(pack_t<FP8>(p0, p1));
      const uint32_t b1 = transpose8x8(pack_t<FP8>(p2, p3));
      if (!v_ready && !sm100::mbar_wait(&vfull_bar[warp][st], par, abort, 2000000000ull)) {
        if (lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, c);
        break;
      }
      {
        const int row = (lane & 7) + ((lane >> 4) << 3);
        const int hi = (lane >> 3) & 1;
        if ((vmask & 0xffffu) == 0xffffu) {
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(smem_u32(vt + swz(row, 2 * mt + hi)), a0, a1, a2, a3);
            mma_t<FP8>(o[mt], a0, a1, a2, a3, b0, b1);
          }
        } else {
          // A block at a segment's edge: its masked keys have P = 0, but
          // their V rows (free slots past the last key, keys before the
          // window) may hold anything and 0 x NaN is NaN, so those keys'
          // columns of the V^T fragments are zeroed.  In the m16n8k16 A
          // fragment, a0 / a1 hold keys 2(lane % 4) + {0, 1}, a2 / a3 the
          // same keys + 8 (the lower key in the lower half).
          const int k0 = 2 * (lane & 3);
          const uint32_t mlo = (((vmask >> k0) & 1u) ? 0x0000ffffu : 0u) |
                               (((vmask >> (k0 + 1)) & 1u) ? 0xffff0000u : 0u);
          const uint32_t mhi = (((vmask >> (k0 + 8)) & 1u) ? 0x0000ffffu : 0u) |
                               (((vmask >> (k0 + 9)) & 1u) ? 0xffff0000u : 0u);
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(smem_u32(vt + swz(row, 2 * mt + hi)), a0, a1, a2, a3);
            mma_t<FP8>(o[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, b0, b1);
          }
        }
      }
      // Every lane's reads of the V slot are done: hand it back to the copy warp.
      __syncwarp();
      if (!FP8 && lane == 0) sm100::mbar_arrive(&vempty_bar[warp][st]);
    }

    // ---- Merge the four warps' states for segment t.
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
    compute_sync();
    // Every warp holds segment t's queries in registers now: buffer t & 1
    // takes segment t + 2's (the async copy is ordered after those reads).
    if (tid == 0 && t + 2 < nseg) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      load_q(t + 2);
    }
    // Each warp scales its state by its share of the normalised result,
    // 2^(m_w - M) / L (times the V scale), with M the segment's max and L
    // = sum_w l_w 2^(m_w - M) its sum; the scaled states are then summed in a
    // fixed order: warps 0 and 1 store into buffers 0 and 1, warps 2 and 3
    // add into them, and the two buffers are added while storing.
    const int slot = sc.slot_base + 2 * c + (t == 0 ? 0 : 1);
    {
      const int h0 = 2 * (lane & 3);
      float f[2];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][h0 + jj]);
        float Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
          Lsum += (wm[w][h0 + jj] == -INFINITY) ? 0.f
                                                 : wl[w][h0 + jj] * fast_exp2(wm[w][h0 + jj] - M);
        f[jj] = (m[jj] == -INFINITY) ? 0.f : fast_exp2(m[jj] - M) * (vsc / Lsum);
        // A cut segment's partial carries its log2-sum-exp.
        if (!si.whole && warp == 0 && lane < 4 && h0 + jj < G)
          p.part_lse[static_cast<int64_t>(slot) * G + h0 + jj] = M + __log2f(Lsum);
      }
      float* buf = so + (warp & 1) * 8 * L::kORow;
      for (int round = 0; round < 2; ++round) {
        if ((warp >> 1) == round) {
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            const int d = mt * 16 + (lane >> 2);
            float* r0 = buf + h0 * L::kORow + d;
            float* r1 = buf + (h0 + 1) * L::kORow + d;
            if (round == 0) {
              r0[0] = o[mt][0] * f[0];
              r0[8] = o[mt][2] * f[0];
              r1[0] = o[mt][1] * f[1];
              r1[8] = o[mt][3] * f[1];
            } else {
              r0[0] += o[mt][0] * f[0];
              r0[8] += o[mt][2] * f[0];
              r1[0] += o[mt][1] * f[1];
              r1[8] += o[mt][3] * f[1];
            }
          }
        }
        if (round == 0) compute_sync();
      }
    }
    compute_sync();
    // Write the output (whole segment) or this CTA's partial (O / L).
    for (int e = tid * 4; e < G * D; e += kWarps * 32 * 4) {
      const int h = e / D, d = e % D;
      const float* s0 = so + h * L::kORow + d;
      const float* s1 = s0 + 8 * L::kORow;
      const float4 u = make_float4(s0[0] + s1[0], s0[1] + s1[1], s0[2] + s1[2], s0[3] + s1[3]);
      if (si.whole) {
        uint2 pk;
        pk.x = pack_bf16x2(u.x, u.y);
        pk.y = pack_bf16x2(u.z, u.w);
        *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(si.q0) * p.hq + si.g * G + h) * D + d) = pk;
      } else {
        *reinterpret_cast<float4*>(p.part_o + (static_cast<int64_t>(slot) * G + h) * D + d) = u;
      }
    }
    compute_sync();
  }
  if (*abort) {
    // (The copy warp drains its own K / V copies.)
    if (tid == 0)
      for (int b = 0; b < 2; ++b) {
        const int last = b ? q_last1 : q_last0;
        if (last >= 0) {
          int dummy = 0;
          sm100::mbar_wait(&q_bar[b], (last >> 1) & 1, &dummy, 200000000ull);
        }
      }
    return;
  }
}

// Combine of the segments cut across CTAs: one CTA per cut segment,
//   out = sum_c 2^(lse_c - M) O_c / sum_c 2^(lse_c - M),  M = max_c lse_c,
// over the fp32 partials (O_c = O / l of part c, lse_c its log2-sum-exp).
// Launched as a programmatic dependent of the decode kernel: its CTAs start
// early and wait for every decode CTA's partials to be visible, so the merge
// runs against an idle memory system, in one round of loads.
struct CombineList {
  int32_t n, slot_base;
  Plan::DecodeCut cut[kMaxDecodeCtas];
};

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
decode_combine_kernel(const DecodeParams p, const __grid_constant__ CombineList cl) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (static_cast<int>(blockIdx.x) >= cl.n) return;
  const Plan::DecodeCut cut = cl.cut[blockIdx.x];
  const int G = p.group, tid = threadIdx.x;
  auto slot_of = [&](int i) { return cl.slot_base + 2 * (cut.ca + i) + (i == 0 ? cut.first : 0); };
  // Each thread owns kPer groups of 4 output values (one head each) and reads
  // every part's log2-sum-exp and partial for them in one round of loads
  // (four parts at a time), rescaling its running sum as the maximum grows.
  constexpr int kPer = (8 * D) / (kWarps * 32 * 4);          // float4 groups per thread (G <= 8)
  float4 acc[kPer];
  float M[kPer], wsum[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    M[u] = -INFINITY;
    wsum[u] = 0.f;
  }
  for (int i0 = 0; i0 < cut.nparts; i0 += 4) {
    float4 v[4][kPer];
    float lse[4][kPer];
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = tid * 4 + u * kWarps * 32 * 4;
        const bool ok = i0 + ii < cut.nparts && e < G * D;
        const int64_t sl = ok ? slot_of(i0 + ii) : 0;
        v[ii][u] = ok ? __ldcg(reinterpret_cast<const float4*>(p.part_o + sl * G * D + e))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        lse[ii][u] = ok ? __ldcg(p.part_lse + sl * G + e / D) : -INFINITY;
      }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      float mn = M[u];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) mn = fmaxf(mn, lse[ii][u]);
      if (mn == -INFINITY) continue;
      const float f = fast_exp2(M[u] - mn);   // 0 while nothing is accumulated
      acc[u].x *= f; acc[u].y *= f; acc[u].z *= f; acc[u].w *= f;
      wsum[u] *= f;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const float wt = fast_exp2(lse[ii][u] - mn);
        wsum[u] += wt;
        acc[u].x += wt * v[ii][u].x;
        acc[u].y += wt * v[ii][u].y;
        acc[u].z += wt * v[ii][u].z;
        acc[u].w += wt * v[ii][u].w;
      }
      M[u] = mn;
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid * 4 + u * kWarps * 32 * 4;
    if (e >= G * D) continue;
    const int h = e / D, d = e % D;
    const float inv = 1.f / wsum[u];
    uint2 pk;
    pk.x = pack_bf16x2(acc[u].x * inv, acc[u].y * inv);
    pk.y = pack_bf16x2(acc[u].z * inv, acc[u].w * inv);
    *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(cut.q0) * p.hq + cut.g * G + h) * D + d) = pk;
  }
}

template <int D>
int launch_combine(const Plan& plan, const DecodeParams& p, const Plan::DecodeLaunch& dl,
                   cudaStream_t stream) {
  CombineList& cl = thread_staging<CombineList>();  // copied into the launch parameters
  for (int off = 0; off < dl.n_cut; off += kMaxDecodeCtas) {
    cl.n = std::min(kMaxDecodeCtas, dl.n_cut - off);
    cl.slot_base = dl.slot_base;
    for (int i = 0; i < cl.n; ++i) cl.cut[i] = plan.dcut[dl.cut_begin + off + i];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl.n);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, p, cl);
    if (e != cudaSuccess) return static_cast<int>(e);
    trace_mark(RPA_KERNEL_DECODE_COMBINE, stream);
  }
  return 0;
}

template <int D, int NSEG, bool FP8>
int launch_one(const Plan& plan, const DecodeParams& p, const CUtensorMap& tk,
               const CUtensorMap& tv, const Plan::DecodeLaunch& dl, cudaStream_t stream) {
  constexpr size_t smem = DecodeSmem<D, FP8>::kBytes;
  if (int e = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_kernel<D, NSEG, FP8>),
                                  static_cast<int>(smem)))
    return e;
  // Host staging, copied into the launch parameters.
  DecodeSched<NSEG>& sc = thread_staging<DecodeSched<NSEG>>();
  if (int e = fill_decode_sched(plan, dl, sc)) return e;
  decode_kernel<D, NSEG, FP8><<<dl.n_ctas, (kWarps + 1) * 32, smem, stream>>>(tk, tv, p, sc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  trace_mark(RPA_KERNEL_DECODE_SPLIT, stream);
  return 0;
}

template <int D>
int launch_decode_t(const Plan& plan, const Args& a, cudaStream_t stream) {
  const DecodeParams p = make_decode_params(plan, a);
  CUtensorMap tk, tv;
  const uint64_t rows = static_cast<uint64_t>(plan.num_pages) * plan.p;
  const bool fp8 = plan.kv_fp8;
  if (!make_tmap_4d_chunks(&tk, a.k_pages, D, plan.hkv, rows, 1, kBlk, fp8) ||
      !make_tmap_4d_chunks(&tv, a.v_pages, D, plan.hkv, rows, 1, kBlk, fp8))
    return static_cast<int>(cudaErrorInvalidValue);
  for (const Plan::DecodeLaunch& dl : plan.dlaunch) {
    const int n = dl.seg_end - dl.seg_begin;
    int err;
    if (fp8)
      err = n <= kDecodeSegSmall
                ? launch_one<D, kDecodeSegSmall, true>(plan, p, tk, tv, dl, stream)
                : launch_one<D, kDecodeSegLarge, true>(plan, p, tk, tv, dl, stream);
    else
      err = n <= kDecodeSegSmall
                ? launch_one<D, kDecodeSegSmall, false>(plan, p, tk, tv, dl, stream)
                : launch_one<D, kDecodeSegLarge, false>(plan, p, tk, tv, dl, stream);
    if (!err) err = launch_combine<D>(plan, p, dl, stream);
    if (err) return err;
  }
  return 0;
}

}  // namespace

// ---------------------------------------------------------------------------
// Fixed scratch for rpa_forward_decode_noalloc: the decode kernel's workspace
// (error word and detail word, then the split partials) in a file-scope device
// array, so that callers who cannot allocate device memory can still run
// decode.  Every GPU that loads this library holds the array until the process
// exits.  The array starts zeroed (a static device variable), so its error
// word starts at zero and stays sticky until rpa_get_device_error reads it;
// the partials are written before they are read within each call.  In host
// code `g_noalloc_scratch` names a host-side stand-in, never a device address;
// the device address comes from cudaGetSymbolAddress, looked up once per
// device (with that device current, under a lock) by the first call on it.

static __device__ __align__(256) unsigned char g_noalloc_scratch[RPA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

int noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return 0;
}

int launch_decode_combine(const Plan& plan, const DecodeParams& p, const Plan::DecodeLaunch& dl,
                          int head_dim, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (head_dim) {
    case 64: return launch_combine<64>(plan, p, dl, s);
    case 128: return launch_combine<128>(plan, p, dl, s);
    case 256: return launch_combine<256>(plan, p, dl, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

bool decode_supported(int32_t head_dim, int32_t group, int32_t page_size) {
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) && group >= 1 && group <= 8 &&
         page_size >= kBlk;
}

int decode_ctas_per_sm(int32_t) { return 1; }

int launch_decode(const Plan& plan, const Args& a, void* stream) {
  if (plan.decode_tc) return launch_decode_tc(plan, a, stream);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (plan.d) {
    case 64: return launch_decode_t<64>(plan, a, s);
    case 128: return launch_decode_t<128>(plan, a, s);
    case 256: return launch_decode_t<256>(plan, a, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace rpa
