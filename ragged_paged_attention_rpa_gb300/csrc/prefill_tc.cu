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
//   warp 0     TMA producer: Q block once per item, then 64-key K and V tiles
//              gathered page by page through the page table (2-stage ring);
//   warp 1     MMA issuer: S = Q K^T (SMEM x SMEM -> TMEM), O += P V (P read
//              from TMEM, V from SMEM), tcgen05.commit onto mbarriers;
//   warps 2-9  softmax: two warps per 32-row quarter, each taking 32 of a
//              tile's 64 keys; reads S from TMEM, masks causal and window edges
//              (interior half-tiles skip the mask), exchanges row maxima with
//              its partner through shared memory, keeps the running max / sum,
//              writes P (bf16) to TMEM, rescales its half of O in TMEM only
//              when the max grew by more than 2^8 (the result is the same; it
//              bounds P by 256); epilogue O / l -> bf16 -> global.
// Every wait is bounded; on a timeout the CTA records RPA_DEVERR_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "rpa_internal.h"
#include "sm100_ptx.cuh"

namespace rpa {
namespace {

using namespace sm100;

constexpr int kBM = 128;        // MMA rows per block
constexpr int kBN = 64;         // keys per KV tile
constexpr int kThreads = 320;   // producer, MMA, 8 softmax warps
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
  static constexpr int kKOff = kQOff + kQBytes;          // 2 stages
  static constexpr int kVOff = kKOff + 2 * kKVBytes;     // 2 stages
  static constexpr int kBarOff = kVOff + 2 * kKVBytes;
  static constexpr int kUsed = kBarOff + 4096 + 1024;   // barriers + exchange + alignment slack
  // Ask for more than half an SM's shared memory so that exactly one CTA
  // (which owns the SM's tensor memory) is resident per SM.
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  // TMEM columns.
  static constexpr int kOCol = 0;
  static constexpr int kSCol = D;                        // 2 x 64
  static constexpr int kPCol = D + 2 * kBN;              // 2 x 32
  static constexpr int kCols = (D + 2 * kBN + kBN) <= 256 ? 256 : 512;
};

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free;
  uint64_t fin;          // all MMAs of this CTA complete (teardown)
  uint32_t tmem_base;
  int abort;
  uint64_t xbar[4];         // per row quarter: both softmax warps have posted their values
  float xmax[2][2][4][32];  // row max of each half-tile, by tile parity / half / quarter / lane
  float xl[2][4][32];       // row sums of each half, for the epilogue
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.k_empty[i], 1);
      mbar_init(&B.v_full[i], 1);
      mbar_init(&B.v_empty[i], 1);
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.p_full[i], 256);
      mbar_init(&B.o_done[i], 1);
    }
    mbar_init(&B.o_free, 256);
    mbar_init(&B.fin, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&B.xbar[i], 64);
    B.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&B.tmem_base, Lay::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const int G = p.group;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t T = 0, I = 0;
    const int nbox = kBN / p.box_rows;
    const uint32_t q_box_bytes = static_cast<uint32_t>(G * p.qb_tokens) * 128u;
    bool alive = true;
    for (int it = blockIdx.x; it < items.n && alive; it += gridDim.x) {
      const Geom gm = item_geom(p, items.items[it]);
      if (!gm.ok) {
        if (lane == 0) report_error(p.ws, RPA_DEVERR_LENGTHS, gm.seq);
        continue;
      }
      const uint32_t Icur = I++;
      if (lane == 0) {
        alive = mbar_wait(&B.q_empty, (Icur & 1) ^ 1, abort, kWaitNs);
        if (alive) {
          mbar_arrive_expect_tx(&B.q_full, q_box_bytes * Lay::kChunks);
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d(q_s + c * kBM * 64, &tm_q, &B.q_full, c * 64, gm.g * G, gm.t0);
        }
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      const int32_t* pt = p.page_table + static_cast<int64_t>(gm.seq) * p.mpps;
      const int32_t pos_last = gm.pos_first + gm.ntok - 1;
      for (int j = 0; j < gm.ntiles && alive; ++j, ++T) {
        const int st = T & 1;
        const uint32_t ph = (T >> 1) & 1;
        const int32_t key0 = (gm.kt0 + j) * kBN;
        // Lane b < nbox resolves the page of box b (rows key0 + b * box_rows ...).
        int32_t row = -p.box_rows;  // out of bounds: the TMA fills zeros
        if (lane < nbox) {
          const int32_t key = key0 + lane * p.box_rows;
          const int32_t slot = key >> p.page_shift;
          if (key <= pos_last) {
            const int32_t page = __ldg(pt + slot);
            if (page >= 0 && page < p.num_pages)
              row = page * p.page_size + (key & (p.page_size - 1));
            else
              report_error(p.ws, RPA_DEVERR_PAGE_ID, gm.seq);
          }
        }
        if (lane == 0) alive = mbar_wait(&B.k_empty[st], ph ^ 1, abort, kWaitNs);
        alive = __shfl_sync(0xffffffffu, alive, 0);
        if (!alive) break;
        if (lane == 0) mbar_arrive_expect_tx(&B.k_full[st], Lay::kKVBytes);
        __syncwarp();
        if (lane < nbox)
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d(k_s + st * kBN * D + c * kBN * 64 + lane * p.box_rows * 64, &tm_k,
                        &B.k_full[st], c * 64, gm.g, row);
        if (lane == 0) alive = mbar_wait(&B.v_empty[st], ph ^ 1, abort, kWaitNs);
        alive = __shfl_sync(0xffffffffu, alive, 0);
        if (!alive) break;
        if (lane == 0) mbar_arrive_expect_tx(&B.v_full[st], Lay::kKVBytes);
        __syncwarp();
        if (lane < nbox)
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d(v_s + st * kBN * D + c * kBN * 64 + lane * p.box_rows * 64, &tm_v,
                        &B.v_full[st], c * 64, gm.g, row);
      }
    }
    if (!alive && lane == 0) {
      // Let every copy this CTA started land before its shared memory goes.
      report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
      for (int i = 0; i < 2; ++i) {
        for (uint32_t ph = 0; ph < 2; ++ph) {
          int dummy = 0;
          mbar_wait(&B.k_full[i], ph, &dummy, kDrainNs);
          dummy = 0;
          mbar_wait(&B.v_full[i], ph, &dummy, kDrainNs);
        }
      }
      int dummy = 0;
      mbar_wait(&B.q_full, 0, &dummy, kDrainNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kBN, 0);
      constexpr uint32_t kIdPV = idesc_bf16(D, 1);
      const uint32_t q_base = smem_addr(q_s), k_base = smem_addr(k_s), v_base = smem_addr(v_s);
      uint32_t T = 0, I = 0;
      bool alive = true;
      auto issue_pv = [&](uint32_t Tp, int jp) -> bool {
        const int st = Tp & 1;
        const uint32_t ph = (Tp >> 1) & 1;
        if (!mbar_wait(&B.p_full[st], ph, abort, kWaitNs)) return false;
        if (!mbar_wait(&B.v_full[st], ph, abort, kWaitNs)) return false;
        if (jp == 0 && !mbar_wait(&B.o_free, (I & 1) ^ 1, abort, kWaitNs)) return false;
        tc_fence_after();
        const uint32_t vb = v_base + st * Lay::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // V as MN-major B: 8-key groups 1024 B apart (SBO), 64-dim chunks
          // one tile-chunk apart (LBO); 16 keys per MMA = 2048 B.
          const uint64_t bdesc = smem_desc(vb + kk * 2048, kBN * 128, 1024);
          mma_ts(tmem + Lay::kOCol, tmem + Lay::kPCol + st * (kBN / 2) + kk * 8, bdesc, kIdPV,
                 (jp > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&B.o_done[st]);
        mma_commit(&B.v_empty[st]);
        return true;
      };
      for (int it = blockIdx.x; it < items.n && alive; it += gridDim.x) {
        const Geom gm = item_geom(p, items.items[it]);
        if (!gm.ok) continue;
        alive = mbar_wait(&B.q_full, I & 1, abort, kWaitNs);
        for (int j = 0; j < gm.ntiles && alive; ++j, ++T) {
          const int st = T & 1;
          const uint32_t ph = (T >> 1) & 1;
          if (!mbar_wait(&B.k_full[st], ph, abort, kWaitNs)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb = k_base + st * Lay::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // K-major, 128-byte swizzle: 16 elements = 32 B inside a 64-wide
            // chunk; chunks of Q are 16 KB apart, chunks of K 8 KB apart.
            const uint32_t c = kk >> 2, w = (kk & 3) * 32;
            const uint64_t adesc = smem_desc(q_base + c * (kBM * 128) + w, 16, 1024);
            const uint64_t bdesc = smem_desc(kb + c * (kBN * 128) + w, 16, 1024);
            mma_ss(tmem + Lay::kSCol + st * kBN, adesc, bdesc, kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&B.s_full[st]);
          mma_commit(&B.k_empty[st]);
          if (j >= 1 && !issue_pv(T - 1, j - 1)) {
            alive = false;
            break;
          }
        }
        if (alive && gm.ntiles > 0) alive = issue_pv(T - 1, gm.ntiles - 1);
        mma_commit(&B.q_empty);
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
    // Warps 2..9: quarter q = warp % 4 owns TMEM lanes (rows) 32q..32q+31;
    // half hf owns key columns 32hf..32hf+31 of every 64-key tile and O
    // columns [hf D/2, (hf+1) D/2).  The two warps of a quarter exchange row
    // maxima (and, at the end, row sums) through shared memory.
    const int q4 = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = 32 * q4 + lane;                       // TMEM lane = row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const int tok = r / G, head = r % G;
    const float c = p.scale_log2;
    uint32_t T = 0;
    uint32_t xph = 0;   // phase of this quarter's exchange barrier
    bool alive = true;
    for (int it = blockIdx.x; it < items.n && alive; it += gridDim.x) {
      const Geom gm = item_geom(p, items.items[it]);
      if (!gm.ok) continue;
      const bool valid = tok < gm.ntok && r < G * p.qb_tokens;
      const int32_t pos = gm.pos_first + tok;
      const int32_t lo = first_visible(pos, gm.W);
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < gm.ntiles; ++j, ++T) {
        const int st = T & 1;
        const uint32_t ph = (T >> 1) & 1;
        if (!mbar_wait(&B.s_full[st], ph, abort, kWaitNs)) {
          alive = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(lane_addr + Lay::kSCol + st * kBN + hf * 32, sr);
        tmem_wait_ld();
        const int32_t key0 = (gm.kt0 + j) * kBN + hf * 32;
        // Interior half-tiles (every key visible to every row of the warp)
        // skip the per-element mask; elsewhere masked scores become -inf.
        const bool full = __all_sync(0xffffffffu, valid && key0 >= lo && key0 + 31 <= pos);
        float mx = -INFINITY;
        if (full) {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) mx = fmaxf(mx, __uint_as_float(sr[cc]));
        } else {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int32_t key = key0 + cc;
            const bool vis = valid && key >= lo && key <= pos;
            if (!vis) sr[cc] = __float_as_uint(-INFINITY);
            mx = fmaxf(mx, __uint_as_float(sr[cc]));
          }
        }
        // Row max over both halves; scaling after the max keeps the order (c >= 0).
        B.xmax[T & 1][hf][q4][lane] = mx;
        mbar_arrive(&B.xbar[q4]);
        if (!mbar_wait(&B.xbar[q4], xph, abort, kWaitNs)) {
          alive = false;
          break;
        }
        xph ^= 1;
        mx = fmaxf(mx, B.xmax[T & 1][hf ^ 1][q4][lane]);
        mx = (mx == -INFINITY) ? -INFINITY : mx * c;
        const float m_new = fmaxf(m_ref, mx);
        const bool grow = m_new > m_ref + 8.f;           // also true for the first visible key
        const bool rescale_o = grow && m_ref != -INFINITY;
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O holds earlier tiles: wait for the last PV, then scale this
          // warp's half of the O columns in TMEM.
          const uint32_t Tp = T - 1;
          if (!mbar_wait(&B.o_done[Tp & 1], (Tp >> 1) & 1, abort, kWaitNs)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const float f = rescale_o ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll 1
          for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
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
        uint32_t pk[16];
        float ls = 0.f;
        if (full) {
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * cc]), c, -m_use));
            const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * cc + 1]), c, -m_use));
            ls += p0 + p1;
            pk[cc] = pack_bf16x2(p0, p1);
          }
        } else {
          constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const float p0 = sr[2 * cc] == kNegInf
                                 ? 0.f : fast_exp2(fmaf(__uint_as_float(sr[2 * cc]), c, -m_use));
            const float p1 = sr[2 * cc + 1] == kNegInf
                                 ? 0.f : fast_exp2(fmaf(__uint_as_float(sr[2 * cc + 1]), c, -m_use));
            ls += p0 + p1;
            pk[cc] = pack_bf16x2(p0, p1);
          }
        }
        l += ls;
        // The P buffer was last read by the PV two tiles back.
        if (T >= 2 && !mbar_wait(&B.o_done[st], ((T - 2) >> 1) & 1, abort, kWaitNs)) {
          alive = false;
          break;
        }
        tc_fence_after();
        tmem_st16(lane_addr + Lay::kPCol + st * (kBN / 2) + hf * 16, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&B.p_full[st]);
      }
      if (!alive) break;
      if (gm.ntiles == 0) continue;
      // Row sum over both halves.
      B.xl[hf][q4][lane] = l;
      mbar_arrive(&B.xbar[q4]);
      if (!mbar_wait(&B.xbar[q4], xph, abort, kWaitNs)) {
        alive = false;
        break;
      }
      xph ^= 1;
      l += B.xl[hf ^ 1][q4][lane];
      // Epilogue: wait for the last PV, then O / l -> bf16 -> out (this
      // warp's half of the columns).
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
      for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
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
      // xl is rewritten for the next item only after both warps of the
      // quarter have read it: they meet again at the next tile's exchange.
      tc_fence_before();
      mbar_arrive(&B.o_free);
    }
    if (!alive && lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
  }

  // Teardown: every MMA must be finished before TMEM is released.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kCols);
  }
}

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  }
  return fn;
}

// 3-D bf16 tensor map [outer][mid][D] with a 128-byte-swizzled box
// (64, box_mid, box_outer).
bool make_map(CUtensorMap* m, const void* base, uint64_t d, uint64_t mid, uint64_t outer,
              uint32_t box_mid, uint32_t box_outer) {
  EncodeFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d, mid, outer};
  cuuint64_t strides[2] = {d * 2, d * mid * 2};
  cuuint32_t box[3] = {64, box_mid, box_outer};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
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
  if (!make_map(&tq, a.q, D, plan.hq, static_cast<uint64_t>(plan.total_q), G, qb) ||
      !make_map(&tk, a.k_pages, D, plan.hkv, static_cast<uint64_t>(plan.num_pages) * plan.p, 1,
                box_rows) ||
      !make_map(&tv, a.v_pages, D, plan.hkv, static_cast<uint64_t>(plan.num_pages) * plan.p, 1,
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
         group >= 1 && group <= kBM && encode_fn() != nullptr;
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
