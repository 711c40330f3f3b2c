// Tensor-core prefill (tcgen05 + TMA) for sequences with more than one query.
//
// Sources (page titles and sections):
//  * "Chasing speed of light on TPU v6e", section "Attention": the kernel
//    works through the prompt in query blocks; each block keeps its queries
//    on chip and streams every key it attends to, so each key is read once per
//    block that wants it.  Footnote 6: vLLM-TPU scales the query block with
//    the head-group ratio.  Here a block is 128 MMA rows = (128 / G) query
//    tokens x the G query heads of one KV head, so every K/V tile read from
//    memory feeds all G heads at once.
//  * Same page, footnote 5: flash attention reads Q, K, V and O once and the
//    score matrix never leaves on-chip memory: here S and P live in tensor
//    memory (TMEM), O accumulates in TMEM.  Footnote 6: fp32 accumulators.
//  * Same page, section "Attention": sliding-window layers let a key be seen
//    by the W queries that follow it, so whole KV tiles outside a block's
//    causal window are never loaded.
//
// One CTA (persistent, one per SM) walks a longest-first list of work items
// (sequence, query block, KV head).  Warp roles:
//   warp 0     TMA producer of the Q block (once per item) and of 64-key K
//              tiles gathered page by page through the page table (3-deep ring);
//   warp 1     TMA producer of the V tiles (2-deep ring), so K runs ahead of V;
//   warp 2     MMA issuer: copies each item's Q block from shared memory into
//              tensor memory once (tcgen05.cp), then S = Q K^T (Q from TMEM,
//              K from SMEM: the score MMAs no longer re-read Q through shared
//              memory, whose bandwidth bounded them) and O += P V (P from
//              TMEM, V from SMEM); tcgen05.commit onto mbarriers.  The score
//              tile runs one ahead of the PV product (two S buffers; P is
//              written over its own S);
//   warps 3-6  softmax: one thread per row (TMEM lane), 64 keys per tile;
//              reads S from TMEM, masks causal and window edges (interior
//              tiles skip the mask), keeps the running max / sum in fp32,
//              exponentiates with the MUFU unit and, for one pair in four,
//              with a polynomial on the FMA pipe (paired fp32 instructions),
//              writes P (bf16) to TMEM, rescales O in TMEM only when the max
//              grew by more than 2^8 (the result is the same; it bounds P by
//              256); epilogue O / l -> bf16 -> global.
// Every wait is bounded; on a timeout the CTA records RPA_DEVERR_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "rpa_internal.h"
#include "sm100_ptx.cuh"

namespace rpa {
namespace {

using namespace sm100;

constexpr int kBM = 128;        // MMA rows per block
constexpr int kBN = 64;         // keys per KV tile
constexpr int kKS = 3;          // K ring depth
constexpr int kVS = 2;          // V ring depth
constexpr int kThreads = 224;   // K producer, V producer, MMA, 4 softmax warps
constexpr int kPolyEvery = 4;   // one pair of exponentials in four on the FMA pipe
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait, then give up
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s per drain wait

struct ItemList {
  int32_t n;
  PrefillItem items[kMaxItemsPerLaunch];
};

struct PrefillParams {
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  const int32_t* window;
  __nv_bfloat16* out;
  unsigned char* ws;
  int32_t hq, group, qb_tokens, page_size, page_shift, box_rows, mpps, num_pages;
  float scale_log2;
};

template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms per row
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kKVBytes = kBN * D * 2;           // one K (or V) tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kKS * kKVBytes;
  static constexpr int kBarOff = kVOff + kVS * kKVBytes;
  static constexpr int kUsed = kBarOff + 256 + 1024;    // barriers + alignment slack
  // Ask for more than half an SM's shared memory so that exactly one CTA
  // (which owns the SM's tensor memory) is resident per SM.
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  // TMEM columns.
  // O: D columns; Q: D/2 (bf16 pairs); two S buffers of 64, P (bf16 pairs)
  // written over the first 32 columns of its own S buffer.
  static constexpr int kOCol = 0;
  static constexpr int kQCol = D;
  static constexpr int kSCol = D + D / 2;
  static constexpr int kCols = (D + D / 2 + 2 * kBN) <= 256 ? 256 : 512;
};

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[kKS], k_empty[kKS], v_full[kVS], v_empty[kVS];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free;
  uint64_t fin;          // all MMAs of this CTA complete (teardown)
  uint32_t tmem_base;
  int abort;
};

struct Geom {
  int32_t seq, g, t0, ntok, pos_first, kt0, ntiles, W;
  bool ok;
};

__device__ __forceinline__ Geom item_geom(const PrefillParams& p, const PrefillItem& it) {
  Geom r;
  r.seq = it.seq;
  r.g = it.qb_head & 255;
  const int32_t qb = it.qb_head >> 8;
  const int32_t q0 = __ldg(p.cu_q_lens + r.seq);
  const int32_t ql = __ldg(p.cu_q_lens + r.seq + 1) - q0;
  const int32_t L = __ldg(p.kv_lens + r.seq);
  r.W = p.window ? __ldg(p.window + r.seq) : 0;
  r.t0 = q0 + qb * p.qb_tokens;
  r.ntok = min(p.qb_tokens, ql - qb * p.qb_tokens);
  r.pos_first = L - ql + qb * p.qb_tokens;
  const int32_t pos_last = r.pos_first + r.ntok - 1;
  r.ok = r.ntok > 0 && r.pos_first >= 0 && pos_last < L &&
         (pos_last >> p.page_shift) < p.mpps;
  const int32_t klo = first_visible(r.pos_first, r.W);
  r.kt0 = klo / kBN;
  r.ntiles = r.ok ? pos_last / kBN - r.kt0 + 1 : 0;
  return r;
}

// TMA source row of box `b` of KV tile j of an item (-box_rows: a box wholly
// out of bounds, which the TMA fills with zeros).
__device__ __forceinline__ int32_t box_row(const PrefillParams& p, const Geom& gm, int j, int b) {
  const int32_t key = (gm.kt0 + j) * kBN + b * p.box_rows;
  const int32_t pos_last = gm.pos_first + gm.ntok - 1;
  if (key > pos_last) return -p.box_rows;
  const int32_t page = __ldg(p.page_table + static_cast<int64_t>(gm.seq) * p.mpps +
                             (key >> p.page_shift));
  if (page < 0 || page >= p.num_pages) {
    report_error(p.ws, RPA_DEVERR_PAGE_ID, gm.seq);
    return -p.box_rows;
  }
  return page * p.page_size + (key & (p.page_size - 1));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const PrefillParams p,
                  const __grid_constant__ ItemList items) {
  using Lay = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem + Lay::kQOff);
  __nv_bfloat16* k_s = reinterpret_cast<__nv_bfloat16*>(smem + Lay::kKOff);
  __nv_bfloat16* v_s = reinterpret_cast<__nv_bfloat16*>(smem + Lay::kVOff);
  Barriers& B = *reinterpret_cast<Barriers*>(smem + Lay::kBarOff);
  volatile int* abort = &B.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&B.q_full, 1);
    mbar_init(&B.q_empty, 1);
    for (int i = 0; i < kKS; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.k_empty[i], 1);
    }
    for (int i = 0; i < kVS; ++i) {
      mbar_init(&B.v_full[i], 1);
      mbar_init(&B.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.p_full[i], 128);
      mbar_init(&B.o_done[i], 1);
    }
    mbar_init(&B.o_free, 128);
    mbar_init(&B.fin, 1);
    B.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 2) {
    tmem_alloc(&B.tmem_base, Lay::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const int G = p.group;

  if (warp <= 1) {
    // ------------------------------------------------------------ producers
    // Warp 0 loads Q and K, warp 1 loads V; each keeps its own ring.
    const bool is_k = warp == 0;
    const int depth = is_k ? kKS : kVS;
    uint64_t* full = is_k ? B.k_full : B.v_full;
    uint64_t* empty = is_k ? B.k_empty : B.v_empty;
    __nv_bfloat16* ring = is_k ? k_s : v_s;
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    uint32_t T = 0, I = 0, issued_q = 0;
    const int nbox = kBN / p.box_rows;
    const uint32_t q_box_bytes = static_cast<uint32_t>(G * p.qb_tokens) * 128u;
    bool alive = true;
    for (int it = blockIdx.x; it < items.n && alive; it += gridDim.x) {
      const Geom gm = item_geom(p, items.items[it]);
      if (!gm.ok) {
        if (lane == 0 && is_k) report_error(p.ws, RPA_DEVERR_LENGTHS, gm.seq);
        continue;
      }
      const uint32_t Icur = I++;
      if (is_k && lane == 0) {
        alive = mbar_wait(&B.q_empty, (Icur & 1) ^ 1, abort, kWaitNs);
        if (alive) {
          mbar_arrive_expect_tx(&B.q_full, q_box_bytes * Lay::kChunks);
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d(q_s + c * kBM * 64, &tm_q, &B.q_full, c * 64, gm.g * G, gm.t0);
          ++issued_q;
        }
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      for (int j = 0; j < gm.ntiles && alive; ++j, ++T) {
        const int st = T % depth;
        const uint32_t ph = (T / depth) & 1;
        const int32_t row = lane < nbox ? box_row(p, gm, j, lane) : 0;
        if (lane == 0) alive = mbar_wait(&empty[st], ph ^ 1, abort, kWaitNs);
        alive = __shfl_sync(0xffffffffu, alive, 0);
        if (!alive) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], Lay::kKVBytes);
        __syncwarp();
        if (lane < nbox)
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d(ring + st * kBN * D + c * kBN * 64 + lane * p.box_rows * 64, tm, &full[st],
                        c * 64, gm.g, row);
      }
    }
    if (!alive && lane == 0) {
      // Let every copy this warp started land before its shared memory goes.
      report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
      for (uint32_t t = (T > static_cast<uint32_t>(depth) ? T - depth : 0); t < T; ++t) {
        int dummy = 0;
        mbar_wait(&full[t % depth], (t / depth) & 1, &dummy, kDrainNs);
      }
      if (is_k && issued_q > 0) {
        int dummy = 0;
        mbar_wait(&B.q_full, (issued_q - 1) & 1, &dummy, kDrainNs);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kBN, 0);
      constexpr uint32_t kIdPV = idesc_bf16(D, 1);
      const uint32_t q_base = smem_addr(q_s), k_base = smem_addr(k_s), v_base = smem_addr(v_s);
      uint32_t T = 0, I = 0;
      bool alive = true;
      auto issue_pv = [&](uint32_t Tp, int jp) -> bool {
        const int sb = Tp & 1;
        const int vs = Tp % kVS;
        if (!mbar_wait(&B.p_full[sb], (Tp >> 1) & 1, abort, kWaitNs)) return false;
        if (!mbar_wait(&B.v_full[vs], (Tp / kVS) & 1, abort, kWaitNs)) return false;
        if (jp == 0 && !mbar_wait(&B.o_free, (I & 1) ^ 1, abort, kWaitNs)) return false;
        tc_fence_after();
        const uint32_t vb = v_base + vs * Lay::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // V as MN-major B: 8-key groups 1024 B apart (SBO), 64-dim chunks
          // one tile-chunk apart (LBO); 16 keys per MMA = 2048 B.  P (A) sits
          // in the first 32 columns of its S buffer, 8 columns per 16 keys.
          const uint64_t bdesc = smem_desc(vb + kk * 2048, kBN * 128, 1024);
          mma_ts(tmem + Lay::kOCol, tmem + Lay::kSCol + sb * kBN + kk * 8, bdesc, kIdPV,
                 (jp > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&B.o_done[sb]);
        mma_commit(&B.v_empty[vs]);
        return true;
      };
      // S(j) into S buffer (T & 1): A = Q from TMEM (8 columns per 16 dims),
      // B = K, K-major 128-byte swizzle (16 elements = 32 B inside a 64-wide
      // chunk; chunks 8 KB apart).
      auto issue_s = [&](uint32_t Ts) -> bool {
        const int ks = Ts % kKS;
        if (!mbar_wait(&B.k_full[ks], (Ts / kKS) & 1, abort, kWaitNs)) return false;
        tc_fence_after();
        const uint32_t kb = k_base + ks * Lay::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t c = kk >> 2, w = (kk & 3) * 32;
          const uint64_t bdesc = smem_desc(kb + c * (kBN * 128) + w, 16, 1024);
          mma_ts(tmem + Lay::kSCol + (Ts & 1) * kBN, tmem + Lay::kQCol + kk * 8, bdesc, kIdS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&B.s_full[Ts & 1]);
        mma_commit(&B.k_empty[ks]);
        return true;
      };
      for (int it = blockIdx.x; it < items.n && alive; it += gridDim.x) {
        const Geom gm = item_geom(p, items.items[it]);
        if (!gm.ok) continue;
        alive = mbar_wait(&B.q_full, I & 1, abort, kWaitNs);
        if (!alive) break;
        // Q: shared memory -> tensor memory, one 16-dim slice per copy (the
        // same K-major swizzled slices an MMA would read).  In order with the
        // MMAs, so it lands after the previous item's last score tile; the
        // shared-memory buffer is free for the next item once the copies are
        // done.
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t c = kk >> 2, w = (kk & 3) * 32;
          tmem_cp_128x256b(tmem + Lay::kQCol + kk * 8,
                           smem_desc(q_base + c * (kBM * 128) + w, 16, 1024));
        }
        mma_commit(&B.q_empty);
        // Order: S(0), then for each j: S(j + 1), PV(j).  S(j + 1) overwrites
        // the buffer holding P(j - 1), which PV(j - 1) (issued before it) read.
        const int n = gm.ntiles;
        if (n > 0) alive = issue_s(T);
        for (int j = 0; j < n && alive; ++j) {
          if (j + 1 < n) {
            alive = issue_s(T + j + 1);
            if (!alive) break;
          }
          alive = issue_pv(T + j, j);
        }
        T += n;
        ++I;
      }
      // Every MMA issued must finish before TMEM is released.
      mma_commit(&B.fin);
      int dummy = 0;
      mbar_wait(&B.fin, 0, &dummy, kDrainNs);
      if (!alive) report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;                            // TMEM lane quarter of this warp
    const int r = 32 * q4 + lane;                       // TMEM lane = row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const int tok = r / G, head = r % G;
    const float c = p.scale_log2;
    uint32_t T = 0;
    bool alive = true;
    for (int it = blockIdx.x; it < items.n && alive; it += gridDim.x) {
      const Geom gm = item_geom(p, items.items[it]);
      if (!gm.ok) continue;
      const bool valid = tok < gm.ntok && r < G * p.qb_tokens;
      const int32_t pos = gm.pos_first + tok;
      const int32_t lo = first_visible(pos, gm.W);
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < gm.ntiles; ++j, ++T) {
        const int sb = T & 1;          // S buffer (P is written over it)
        if (!mbar_wait(&B.s_full[sb], (T >> 1) & 1, abort, kWaitNs)) {
          alive = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        {
          uint32_t (&lo32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
          uint32_t (&hi32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
          tmem_ld32(lane_addr + Lay::kSCol + sb * kBN, lo32);
          tmem_ld32(lane_addr + Lay::kSCol + sb * kBN + 32, hi32);
        }
        tmem_wait_ld();
        const int32_t key0 = (gm.kt0 + j) * kBN;
        // Interior tiles (every key visible to every row of the warp) skip
        // the per-element mask; elsewhere masked scores become -inf.
        const bool full = __all_sync(0xffffffffu, valid && key0 >= lo && key0 + kBN - 1 <= pos);
        float mx;
        if (full) {
          float m3[22];
#pragma unroll
          for (int i = 0; i < 21; ++i)
            m3[i] = fmax3(__uint_as_float(sr[3 * i]), __uint_as_float(sr[3 * i + 1]),
                          __uint_as_float(sr[3 * i + 2]));
          m3[21] = __uint_as_float(sr[63]);
#pragma unroll
          for (int i = 0; i < 7; ++i) m3[i] = fmax3(m3[3 * i], m3[3 * i + 1], m3[3 * i + 2]);
          m3[7] = m3[21];
          mx = fmax3(fmax3(m3[0], m3[1], m3[2]), fmax3(m3[3], m3[4], m3[5]), fmaxf(m3[6], m3[7]));
        } else {
          mx = -INFINITY;
#pragma unroll
          for (int cc = 0; cc < 64; ++cc) {
            const int32_t key = key0 + cc;
            const bool vis = valid && key >= lo && key <= pos;
            if (!vis) sr[cc] = 0xff800000u;   // -inf
            mx = fmaxf(mx, __uint_as_float(sr[cc]));
          }
        }
        // Scaling after the max keeps the order (c >= 0).
        mx = (mx == -INFINITY) ? -INFINITY : mx * c;
        const float m_new = fmaxf(m_ref, mx);
        const bool grow = m_new > m_ref + 8.f;           // also true for the first visible key
        const bool rescale_o = grow && l > 0.f;
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O holds earlier tiles: wait for the last PV, then scale in TMEM.
          const uint32_t Tp = T - 1;
          if (!mbar_wait(&B.o_done[Tp & 1], (Tp >> 1) & 1, abort, kWaitNs)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const float f = rescale_o ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(lane_addr + Lay::kOCol + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) o[cc] = __float_as_uint(__uint_as_float(o[cc]) * f);
            tmem_st32(lane_addr + Lay::kOCol + c0, o);
          }
          tmem_wait_st();
        }
        if (grow) {
          if (l > 0.f) l *= fast_exp2(m_ref - m_new);
          m_ref = m_new;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        uint32_t pk[32];
        float ls;
        if (full) {
          // Paired fp32 arithmetic; one pair in kPolyEvery takes its 2^x on
          // the FMA pipe instead of the MUFU unit.
          const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_use, -m_use);
          uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[2 * cc]),
                                               __uint_as_float(sr[2 * cc + 1])), c2, nm2);
            uint64_t p2;
            if (cc % kPolyEvery == kPolyEvery - 1) {
              p2 = exp2_poly2(x2);
            } else {
              float x0, x1;
              f2_unpack(x2, x0, x1);
              p2 = f2_pack(fast_exp2(x0), fast_exp2(x1));
            }
            acc = f2_add(acc, p2);
            float p0, p1;
            f2_unpack(p2, p0, p1);
            pk[cc] = pack_bf16x2(p0, p1);
          }
          float a0, a1;
          f2_unpack(acc, a0, a1);
          ls = a0 + a1;
        } else {
          ls = 0.f;
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const float p0 = sr[2 * cc] == 0xff800000u
                                 ? 0.f : fast_exp2(fmaf(__uint_as_float(sr[2 * cc]), c, -m_use));
            const float p1 = sr[2 * cc + 1] == 0xff800000u
                                 ? 0.f : fast_exp2(fmaf(__uint_as_float(sr[2 * cc + 1]), c, -m_use));
            ls += p0 + p1;
            pk[cc] = pack_bf16x2(p0, p1);
          }
        }
        l += ls;
        // P over the first 32 columns of this tile's S buffer (already read).
        tmem_st32(lane_addr + Lay::kSCol + sb * kBN, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&B.p_full[sb]);
      }
      if (!alive) break;
      if (gm.ntiles == 0) continue;
      // Epilogue: wait for the last PV, then O / l -> bf16 -> out.
      const uint32_t Tl = T - 1;
      if (!mbar_wait(&B.o_done[Tl & 1], (Tl >> 1) & 1, abort, kWaitNs)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow =
          p.out + (static_cast<int64_t>(gm.t0 + tok) * p.hq + gm.g * G + head) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(lane_addr + Lay::kOCol + c0, o);
        tmem_wait_ld();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
            dst[q] = v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&B.o_free);
    }
    if (!alive && lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
  }

  // Teardown: every MMA must be finished before TMEM is released.
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kCols);
  }
}

template <int D>
int launch_prefill_t(const Plan& plan, const Args& a, cudaStream_t stream) {
  using Lay = Layout<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kBytes);
    if (e != cudaSuccess) return static_cast<int>(e);
    configured = true;
  }
  const int G = plan.hq / plan.hkv;
  const int qb = plan.q_block;
  const int box_rows = plan.p < kBN ? plan.p : kBN;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d(&tq, a.q, D, plan.hq, static_cast<uint64_t>(plan.total_q), G, qb) ||
      !make_tmap_3d(&tk, a.k_pages, D, plan.hkv, static_cast<uint64_t>(plan.num_pages) * plan.p, 1,
                    box_rows) ||
      !make_tmap_3d(&tv, a.v_pages, D, plan.hkv, static_cast<uint64_t>(plan.num_pages) * plan.p, 1,
                    box_rows))
    return static_cast<int>(cudaErrorInvalidValue);
  PrefillParams p;
  p.page_table = a.page_table;
  p.cu_q_lens = a.cu_q_lens;
  p.kv_lens = a.kv_lens;
  p.window = a.window;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.ws = a.workspace;
  p.hq = plan.hq;
  p.group = G;
  p.qb_tokens = qb;
  p.page_size = plan.p;
  int shift = 0;
  while ((1 << shift) < plan.p) ++shift;
  p.page_shift = shift;
  p.box_rows = box_rows;
  p.mpps = plan.mpps;
  p.num_pages = plan.num_pages;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  static ItemList list;  // host staging; copied into the launch parameters
  const size_t n = plan.items.size();
  for (size_t off = 0; off < n; off += kMaxItemsPerLaunch) {
    const int cnt = static_cast<int>(std::min<size_t>(kMaxItemsPerLaunch, n - off));
    list.n = cnt;
    for (int i = 0; i < cnt; ++i) list.items[i] = plan.items[off + i];
    const int grid = std::min(cnt, plan.prefill_ctas);
    prefill_tc_kernel<D><<<grid, kThreads, Lay::kBytes, stream>>>(tq, tk, tv, p, list);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return static_cast<int>(e);
    trace_mark(RPA_KERNEL_PREFILL_TC, stream);
  }
  return 0;
}

}  // namespace

bool prefill_tc_supported(int32_t head_dim, int32_t page_size, int32_t group) {
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) && page_size >= 16 &&
         group >= 1 && group <= kBM;
}

int prefill_ctas_per_sm(int32_t) { return 1; }

int prefill_tokens_per_block(int32_t, int32_t group) { return group >= kBM ? 1 : kBM / group; }

int launch_prefill_tc(const Plan& plan, const Args& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (plan.d) {
    case 64: return launch_prefill_t<64>(plan, a, s);
    case 128: return launch_prefill_t<128>(plan, a, s);
    case 256: return launch_prefill_t<256>(plan, a, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace rpa
