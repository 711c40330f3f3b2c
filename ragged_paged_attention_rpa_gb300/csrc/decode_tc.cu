// Split-KV decode on the tensor cores (tcgen05), bf16 pages.  Same schedule,
// same outputs (and the same split partials, merged by the same combine
// kernel) as the CUDA-core decode kernel in decode.cu; what changes is who
// does the arithmetic, so that an SM's time goes to keeping its copies in
// flight.
//
// Sources (page titles and sections):
//  * "TPU Deep Dive" slides, chapter 4, "Attention: small share, wrong
//    intensity": decode attention does about G = Hq/Hkv FLOPs per byte of KV,
//    so it is bound by HBM bandwidth; every visible KV byte is read once.
//  * "Chasing speed of light on TPU v6e", footnote 6: fp32 softmax
//    accumulators (m, l, O in fp32; P rounded to bf16 for the product).
//
// CTA (one per SM, 384 threads).  Its range's segment parts (sequence, KV
// head, keys [kb, ke)) are walked in 128-key tiles on absolute 128-key
// boundaries (so a tile lies in one page when pages hold >= 128 tokens):
//   warp 0    K producer: Q of each segment (one box per 64-dimension chunk
//             of the group's heads) and, per tile, one 16 KB stage per
//             64-dimension chunk ([128 keys][128 B], 128-byte swizzle)
//   warp 2    V producer: per tile D/64 stages of 8192/D keys x D dims
//   warp 1    score MMA issuer (one elected lane) and tensor-memory owner:
//               S^T[128 keys x 16]  = K . Q^T   (M = 128, N = 16, both
//                                                K-major)
//   warp 3    PV MMA issuer:
//               O^T[128 dims x 16] = V^T . P^T  (per 128-dimension half; V^T
//                                                is the MN-major view of the
//                                                V stage, P^T K-major bf16)
//             S and each tile's O^T land in double-buffered TMEM columns
//   warps 4-7 softmax (thread = TMEM lane = key of the tile): mask, per-head
//             tile maximum (a warp reduce-scatter and a four-warp exchange),
//             P = 2^(s - m) to shared memory, the running m and l, and each
//             tile's rescale factors 2^(m_old - m_new) for the O warps
//   warps 8-11 O and output (thread = TMEM lane = dimension): the running O
//             in fp32 registers, O = O * 2^(m_old - m_new) + O^T(tile), and
//             at the end of a segment part the output (whole segment) or the
//             part's fp32 partial and log2-sum-exp.
// Nothing waits on a ring it does not consume: the score MMAs of later tiles
// run as soon as their K lands, the softmax runs up to two tiles ahead of the
// PV MMAs, and a V stage is released as soon as its tile's P is ready, so the
// copies of both rings stay in flight.
// Boxes never cross a page: a tile's rows come in aligned runs of 16, 32, 64
// or 128 keys (the largest that fits, one tensor map per height), and a
// stage wholly inside the part and one page comes as one box.  Every wait is
// bounded; a wait that gives up sets the error word and the CTA winds down,
// letting its copies land and its MMAs finish before it frees TMEM.
#include <algorithm>

#include "common.cuh"
#include "decode_sched.cuh"
#include "rpa_internal.h"
#include "sm100_ptx.cuh"

namespace rpa {

namespace {

using namespace sm100;

constexpr int kTcThreads = 384;
constexpr int kTcSoftmaxWarp0 = 4;
constexpr int kTcOaccWarp0 = 8;
constexpr int kTileKeys = 128;    // keys per score tile (the MMA's M)
constexpr int kStage = 16384;     // bytes per ring stage
constexpr int kNH = 8;            // head columns the softmax keeps (G <= 8)
constexpr int kMaxStages = 8;     // per ring
constexpr int kTmemCols = 128;    // S: 2 x 16 columns; O^T: 2 x (D / 128) x 16
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait, then give up
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s per drain wait

template <int D>
struct TcLayout {
  static constexpr int kChunks = D / 64;           // 64-dimension chunks
  static constexpr int kVKeys = 8192 / D;          // keys per V stage
  static constexpr int kVUnits = kVKeys / 16;      // 16-key units per V stage
  static constexpr int kHalves = D / 128;          // 128-dimension halves (MMA M)
  static constexpr int kQBytes = kChunks * 2048;   // [chunk][16 head rows][128 B]
  static constexpr int kPBytes = 4096;             // [2 key chunks][16 head rows][128 B]
  static constexpr int kQOff = 0;
  static constexpr int kPOff = 2 * kQBytes;
  static constexpr int kRingOff = kPOff + 2 * kPBytes;
  // Shared memory left after the static tables (< 8 KB) and the alignment
  // slack, in whole stages, split between the two rings.
  static constexpr int kStages = (227 * 1024 - 8192 - 1024 - kRingOff) / kStage;
  static constexpr int kKS = kStages / 2 < kMaxStages ? kStages / 2 : kMaxStages;
  static constexpr int kVS = kStages - kKS < kMaxStages ? kStages - kKS : kMaxStages;
  static constexpr int kKOff = kRingOff;
  static constexpr int kVOff = kKOff + kKS * kStage;
  static constexpr int kBytes = kVOff + kVS * kStage;
  static constexpr int kDynBytes = kBytes + 1024;  // + alignment to 1024 bytes
  static_assert(kKS >= kChunks && kVS >= kChunks, "a ring must hold one tile");
  static_assert(2 * 16 + 2 * kHalves * 16 <= kTmemCols, "tensor memory columns");
};

struct TcBarriers {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kMaxStages], k_empty[kMaxStages];
  uint64_t v_full[kMaxStages], v_empty[kMaxStages];
  uint64_t s_full[2], s_empty[2];   // S buffer written by the MMAs / read out
  uint64_t p_full[2], p_free[2];    // P^T buffer written / read by the MMAs
  uint64_t o_full[2], o_empty[2];   // O^T buffer written / read out
  uint64_t red_full[2], l_full[2];  // softmax warps' exchanges
  uint64_t a_full[2], a_empty[2];   // a tile's rescale factors handed over / taken
  uint64_t f_full[2], f_empty[2];   // a segment's row sums and maxima
  uint64_t fin[2];                  // every MMA of each issuer complete
  uint32_t tmem_base;
  int abort;
};

// Tensor maps of one launch.  Heights of the K / V boxes: 16 << i rows.
struct TcMaps {
  CUtensorMap q;      // q as (D, hq, tokens), box (64, min(16, hq), 1)
  CUtensorMap k[4];   // K pool as (D, hkv, pages * P), box (64, 1, 16 << i)
  CUtensorMap v[4];   // V pool, the same
  CUtensorMap v4;     // V pool as (64, hkv, pages * P, D / 64), box (64, 1, kVKeys, D / 64)
};

// Key tile jt of a segment part: its first key (a multiple of 128) and the
// 16-key units [u0, u1) of the tile that hold keys of the part.
struct TileGeo {
  int32_t key0;
  int u0, u1;
};

__device__ __forceinline__ int part_tiles(const SegInfo& si) {
  return si.ke > si.kb ? ((si.ke - 1) >> 7) - (si.kb >> 7) + 1 : 0;
}

__device__ __forceinline__ TileGeo tile_geo(const SegInfo& si, int jt) {
  TileGeo t;
  t.key0 = ((si.kb >> 7) + jt) << 7;
  t.u0 = (max(si.kb, t.key0) - t.key0) >> 4;
  t.u1 = (min(si.ke, t.key0 + kTileKeys) - t.key0 + 15) >> 4;
  return t;
}

// Page id of `key` of a segment part (-1: a bad page id or past the list).
__device__ __forceinline__ int32_t page_at(const SegInfo& si, const int32_t* s_pages, int npages,
                                           int shift, int32_t key) {
  const int idx = si.pg_off + (key >> shift) - si.slot0;
  return (idx >= 0 && idx < npages) ? s_pages[idx] : -1;
}

// Units [x0, x1) cut into aligned power-of-two runs of at most hmax units
// (hmax a power of two no larger than a page): box(x, h) for each run.
template <typename F>
__device__ __forceinline__ void for_runs(int x0, int x1, int hmax, F&& box) {
  for (int x = x0; x < x1;) {
    int h = hmax;
    while (h > 1 && ((x & (h - 1)) != 0 || x + h > x1)) h >>= 1;
    box(x, h);
    x += h;
  }
}

// Warp maximum (or sum) of 8 per-lane values, scattered: lane l ends with
// the reduction of value (l >> 2) & 7 over the warp.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter8(const float (&v)[kNH], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
  float r4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float send = u16 ? v[k] : v[k + 4];
    const float keep = u16 ? v[k + 4] : v[k];
    r4[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  float r2[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float send = u8 ? r4[k] : r4[k + 2];
    const float keep = u8 ? r4[k + 2] : r4[k];
    r2[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  float r1 = op(u4 ? r2[1] : r2[0], __shfl_xor_sync(0xffffffffu, u4 ? r2[0] : r2[1], 4));
  r1 = op(r1, __shfl_xor_sync(0xffffffffu, r1, 2));
  r1 = op(r1, __shfl_xor_sync(0xffffffffu, r1, 1));
  return r1;
}

template <int D, int NSEG>
__global__ void __launch_bounds__(kTcThreads, 1)
decode_tc_kernel(const __grid_constant__ TcMaps maps, const DecodeParams p,
                 const __grid_constant__ DecodeSched<NSEG> sc) {
  using L = TcLayout<D>;
  extern __shared__ __align__(128) unsigned char smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ int32_t s_pages[kMaxCtaPages];
  __shared__ SegInfo s_seg[kMaxCtaSegs];
  __shared__ __align__(16) float s_red[2][4][kNH];
  __shared__ __align__(16) float s_lsum[2][4][kNH];
  __shared__ __align__(16) float s_alpha[2][kNH];
  __shared__ float s_fin_l[2][kNH], s_fin_m[2][kNH];
  __shared__ __align__(8) TcBarriers B;
  __shared__ int s_npages;

  // The combine kernel may be scheduled now; it waits for this grid's end.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int G = p.group;
  const int P = 1 << p.page_shift;
  const int c = blockIdx.x;
  const int32_t cb0 = range_start(sc, c);
  const int32_t cb1 = range_start(sc, c + 1);
  if (cb0 >= cb1) return;   // the whole CTA, before any barrier
  const int kfirst = sc.bpc > 0 ? seg_of(sc, cb0) : (sc.cta_seg[c] & 0xffff);
  const int klast = sc.bpc > 0 ? seg_of(sc, cb1 - 1) : (sc.cta_seg[c] >> 16);
  int nseg = klast - kfirst + 1;
  if (nseg > kMaxCtaSegs) {
    if (tid == 0) report_error(p.ws, RPA_DEVERR_LENGTHS, c);
    nseg = kMaxCtaSegs;
  }
  volatile int* abort = &B.abort;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.q_full[i], 1);
      mbar_init(&B.q_empty[i], 1);
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_empty[i], 128);
      mbar_init(&B.p_full[i], 128);
      mbar_init(&B.p_free[i], 1);
      mbar_init(&B.o_full[i], 1);
      mbar_init(&B.o_empty[i], 128);
      mbar_init(&B.red_full[i], 128);
      mbar_init(&B.l_full[i], 128);
      mbar_init(&B.a_full[i], kNH);
      mbar_init(&B.a_empty[i], 128);
      mbar_init(&B.f_full[i], kNH);
      mbar_init(&B.f_empty[i], 128);
    }
    for (int i = 0; i < L::kKS; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.k_empty[i], 1);
    }
    for (int i = 0; i < L::kVS; ++i) {
      mbar_init(&B.v_full[i], 1);
      mbar_init(&B.v_empty[i], 1);
    }
    mbar_init(&B.fin[0], 1);
    mbar_init(&B.fin[1], 1);
    B.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.k[0]);
    prefetch_tmap(&maps.v[0]);
  }
  if (warp == 1) {
    tmem_alloc(&B.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Q buffers (rows past the group's heads are never written), P buffers and
  // the V ring start zeroed: a V row no copy has written yet meets P = 0 in
  // the product, and 0 x NaN would be NaN.  Later, a V row holds either a
  // visible key's value or zeros (rows outside the visible keys that a copy
  // brings in are cleared before the MMAs read them).
  {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int o = tid * 16; o < L::kRingOff; o += kTcThreads * 16)
      *reinterpret_cast<uint4*>(smem + o) = z;
    for (int o = tid * 16; o < L::kVS * kStage; o += kTcThreads * 16)
      *reinterpret_cast<uint4*>(smem + L::kVOff + o) = z;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  load_range_tables(sc, p, c, cb0, cb1, kfirst, nseg, s_seg, s_pages, &s_npages);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const int npages = s_npages;

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == 0;
    if (lane == 0) {
      const int depth = is_k ? L::kKS : L::kVS;
      uint64_t* full = is_k ? B.k_full : B.v_full;
      uint64_t* empty = is_k ? B.k_empty : B.v_empty;
      uint8_t* ring = smem + (is_k ? L::kKOff : L::kVOff);
      const int hq_box = p.hq < 16 ? p.hq : 16;
      // Largest run of 16-key units one box may take (within a page).
      const int hk = min(8, P >> 4);
      const int hv = min(L::kVUnits, P >> 4);
      uint32_t C = 0;
      int u = 0;
      bool alive = true;
      for (int t = 0; t < nseg && alive; ++t) {
        const SegInfo si = s_seg[t];
        const int nt = part_tiles(si);
        if (nt == 0) continue;
        if (is_k) {
          // The segment's queries: the group's heads (and up to 16 - G more,
          // or zeros past the last head), one box per 64-dimension chunk.
          alive = mbar_wait(&B.q_empty[u & 1], ((u >> 1) & 1) ^ 1, abort, kWaitNs);
          if (!alive) break;
          uint8_t* qd = smem + L::kQOff + (u & 1) * L::kQBytes;
          mbar_arrive_expect_tx(&B.q_full[u & 1],
                                static_cast<uint32_t>(hq_box * 128 * L::kChunks));
          for (int ch = 0; ch < L::kChunks; ++ch)
            tma_load_3d(qd + ch * 2048, &maps.q, &B.q_full[u & 1], ch * 64, si.g * G, si.q0);
        }
        ++u;
        auto row_of = [&](int32_t key, int32_t page) { return page * P + (key & (P - 1)); };
        for (int jt = 0; jt < nt && alive; ++jt) {
          const TileGeo tg = tile_geo(si, jt);
          if (is_k) {
            uint32_t bytes = 0;
            for_runs(tg.u0, tg.u1, hk, [&](int x, int h) {
              if (page_at(si, s_pages, npages, p.page_shift, tg.key0 + 16 * x) >= 0)
                bytes += h * 2048;
            });
            for (int ch = 0; ch < L::kChunks; ++ch, ++C) {
              const int st = C % depth;
              alive = mbar_wait(&empty[st], ((C / depth) & 1) ^ 1, abort, kWaitNs);
              if (!alive) break;
              uint8_t* dst = ring + st * kStage;
              mbar_arrive_expect_tx(&full[st], bytes);
              for_runs(tg.u0, tg.u1, hk, [&](int x, int h) {
                const int32_t key = tg.key0 + 16 * x;
                const int32_t page = page_at(si, s_pages, npages, p.page_shift, key);
                if (page >= 0)
                  tma_load_3d(dst + x * 2048, &maps.k[__ffs(h) - 1], &full[st], ch * 64, si.g,
                              row_of(key, page));
              });
            }
          } else {
            for (int sv = 0; sv < L::kChunks; ++sv) {
              const int a = max(tg.u0, sv * L::kVUnits);
              const int b = min(tg.u1, (sv + 1) * L::kVUnits);
              if (a >= b) continue;   // no key of the part: the MMAs skip it too
              const int st = C % depth;
              alive = mbar_wait(&empty[st], ((C / depth) & 1) ^ 1, abort, kWaitNs);
              if (!alive) break;
              ++C;
              uint8_t* dst = ring + st * kStage;
              const int32_t kst = tg.key0 + sv * L::kVKeys;
              const int32_t page0 = page_at(si, s_pages, npages, p.page_shift, kst);
              if (a == sv * L::kVUnits && b == (sv + 1) * L::kVUnits && L::kVKeys <= P &&
                  page0 >= 0) {
                // The whole stage: every chunk of kVKeys rows of one page.
                mbar_arrive_expect_tx(&full[st], kStage);
                tma_load_4d(dst, &maps.v4, &full[st], 0, si.g, row_of(kst, page0), 0);
              } else {
                uint32_t bytes = 0;
                for_runs(a, b, hv, [&](int x, int h) {
                  if (page_at(si, s_pages, npages, p.page_shift, tg.key0 + 16 * x) >= 0)
                    bytes += h * 2048 * L::kChunks;
                });
                mbar_arrive_expect_tx(&full[st], bytes);
                for_runs(a, b, hv, [&](int x, int h) {
                  const int32_t key = tg.key0 + 16 * x;
                  const int32_t page = page_at(si, s_pages, npages, p.page_shift, key);
                  if (page < 0) return;
                  for (int ch = 0; ch < L::kChunks; ++ch)
                    tma_load_3d(dst + ch * (L::kVKeys * 128) + (x - sv * L::kVUnits) * 2048,
                                &maps.v[__ffs(h) - 1], &full[st], ch * 64, si.g,
                                row_of(key, page));
                });
              }
            }
          }
        }
      }
      if (!alive) {
        // Let every copy this warp started land before the CTA exits.
        report_error(p.ws, RPA_DEVERR_TIMEOUT, c);
        int dummy = 0;
        for (uint32_t t = (C > static_cast<uint32_t>(depth) ? C - depth : 0); t < C; ++t)
          mbar_wait(&full[t % depth], (t / depth) & 1, &dummy, kDrainNs);
        if (is_k)
          for (int w = (u > 2 ? u - 2 : 0); w < u; ++w)
            mbar_wait(&B.q_full[w & 1], (w >> 1) & 1, &dummy, kDrainNs);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the score MMAs, warp 3 the PV MMAs (one elected lane
    // each; a commit tracks its own lane's MMAs), so that neither ring waits
    // on the other's copies.
    constexpr uint32_t kIdS = idesc_bf16_ab(128, 16, 0, 0);
    constexpr uint32_t kIdPV = idesc_bf16_ab(128, 16, 1, 0);
    const bool is_s = warp == 1;
    const uint32_t q_base = smem_u32(smem + L::kQOff), p_base = smem_u32(smem + L::kPOff);
    const uint32_t k_base = smem_u32(smem + L::kKOff), v_base = smem_u32(smem + L::kVOff);
    // Descriptors as base + byte offset / 16 (the start-address field;
    // every operand lies below 256 KB), built once rather than per MMA.
    const uint64_t q_d0 = smem_desc(q_base, 16, 1024), p_d0 = smem_desc(p_base, 16, 1024);
    const uint64_t k_d0 = smem_desc(k_base, 16, 1024);
    const uint64_t v_d0 = smem_desc(v_base, L::kVKeys * 128, 1024);
    uint32_t j = 0;
    int ks = 0, vs = 0;          // ring slot and phase of the next K / V stage
    uint32_t kph = 0, vph = 0;
    // Whether the next K / V stage has landed, tested (mbar_test) while the
    // current stage's MMAs were issued; false: wait for it.
    bool k_ready = false, v_ready = false;
    int u = 0;
    bool alive = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool ok = mbar_wait(bar, parity, abort, kWaitNs);
      return __all_sync(0xffffffffu, ok);
    };
    // V rows of keys the query does not see that a copy brought in (before
    // the window's first key, past the sequence's last) may hold anything;
    // they meet P = 0, so they are zeroed before the MMAs read the stage.
    auto clear_v_edges = [&](const SegInfo& si, int32_t kst, int vs) {
      const int a0 = max(0, si.kb - kst), a1 = min(L::kVKeys, si.lo - kst);
      const int32_t e16 = (si.ke + 15) & ~15;
      const int b0 = max(0, si.ke - kst), b1 = min(L::kVKeys, e16 - kst);
      const int na = max(0, a1 - a0), nb = max(0, b1 - b0);
      if (na + nb == 0) return;
      uint8_t* st = smem + L::kVOff + vs * kStage;
      for (int x = lane; x < (na + nb) * L::kChunks * 8; x += 32) {
        const int rr = x / (L::kChunks * 8), rem = x % (L::kChunks * 8);
        const int row = rr < na ? a0 + rr : b0 + (rr - na);
        *reinterpret_cast<uint4*>(st + (rem >> 3) * (L::kVKeys * 128) + row * 128 +
                                  (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    };
    // O^T(jp) = V^T . P^T(jp), one V stage at a time.  The V stage is the
    // MN-major A operand: 64-dimension chunks kVKeys x 128 B apart (LBO),
    // 8-key groups 1024 B apart (SBO), 16 keys per MMA = 2048 B.  P^T (B) is
    // K-major: 16 keys = 32 B inside a 64-key chunk of 2048 B.
    auto issue_pv = [&](uint32_t jp, const SegInfo& si, const TileGeo& tg) -> bool {
      const int b = jp & 1;
      if (!wait(&B.p_full[b], (jp >> 1) & 1)) return false;
      if (!wait(&B.o_empty[b], ((jp >> 1) & 1) ^ 1)) return false;
      uint32_t acc = 0;
#pragma unroll 1
      for (int sv = 0; sv < L::kChunks; ++sv) {
        const int a = max(tg.u0, sv * L::kVUnits);
        const int e = min(tg.u1, (sv + 1) * L::kVUnits);
        if (a >= e) continue;
        if (!v_ready && !wait(&B.v_full[vs], vph)) return false;
        clear_v_edges(si, tg.key0 + sv * L::kVKeys, vs);
        tc_fence_after();
        const int vcur = vs;
        const uint64_t vd = v_d0 + static_cast<uint64_t>(vs * (kStage >> 4));
        if (++vs == L::kVS) {
          vs = 0;
          vph ^= 1;
        }
        v_ready = __all_sync(0xffffffffu, mbar_test(&B.v_full[vs], vph));
        const uint64_t pd = p_d0 + static_cast<uint64_t>((b * L::kPBytes) >> 4);
#pragma unroll
        for (int dh = 0; dh < L::kHalves; ++dh) {
#pragma unroll
          for (int kk = 0; kk < L::kVUnits; ++kk) {
            const int kg = sv * L::kVUnits + kk;   // 16-key group of the tile
            mma_ss(tmem + 32 + 32 * b + 16 * dh,
                   vd + static_cast<uint64_t>((dh * 2 * (L::kVKeys * 128) + kk * 2048) >> 4),
                   pd + static_cast<uint64_t>(((kg >> 2) * 2048 + (kg & 3) * 32) >> 4), kIdPV,
                   (acc >> dh) & 1u);
            acc |= 1u << dh;
          }
        }
        mma_commit(&B.v_empty[vcur]);
      }
      mma_commit(&B.o_full[b]);
      mma_commit(&B.p_free[b]);
      return true;
    };
    for (int t = 0; t < nseg && alive; ++t) {
      const SegInfo si = s_seg[t];
      const int nt = part_tiles(si);
      if (nt == 0) continue;
      if (!is_s) {
        for (int jt = 0; jt < nt && alive; ++jt, ++j) alive = issue_pv(j, si, tile_geo(si, jt));
        continue;
      }
      if (!(alive = wait(&B.q_full[u & 1], (u >> 1) & 1))) break;
      tc_fence_after();
      const uint32_t qb = q_base + (u & 1) * L::kQBytes;
      for (int jt = 0; jt < nt; ++jt, ++j) {
        const int b = j & 1;
        // S(j): one K stage (a 64-dimension chunk of the tile's keys) at a
        // time; K (A) and Q (B) K-major, 16 dimensions = 32 B per MMA.
        if (!(alive = wait(&B.s_empty[b], ((j >> 1) & 1) ^ 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < L::kChunks; ++ch) {
          if (!k_ready && !(alive = wait(&B.k_full[ks], kph))) break;
          tc_fence_after();
          const int kcur = ks;
          const uint64_t kd = k_d0 + static_cast<uint64_t>(ks * (kStage >> 4));
          const uint64_t qd = q_d0 + static_cast<uint64_t>(((qb - q_base) + ch * 2048) >> 4);
          if (++ks == L::kKS) {
            ks = 0;
            kph ^= 1;
          }
          k_ready = __all_sync(0xffffffffu, mbar_test(&B.k_full[ks], kph));
          mma_ss4_commit(tmem + 16 * b, kd, kd + 2, kd + 4, kd + 6, qd, qd + 2, qd + 4, qd + 6,
                         kIdS, ch > 0 ? 1u : 0u, &B.k_empty[kcur]);
        }
        if (!alive) break;
        mma_commit(&B.s_full[b]);
        if (jt == nt - 1) mma_commit(&B.q_empty[u & 1]);
      }
      ++u;
    }
    // Every MMA this warp issued must finish before TMEM is released.
    uint64_t* fin = &B.fin[is_s ? 0 : 1];
    mma_commit(fin);
    int dummy = 0;
    mbar_wait(fin, 0, &dummy, kDrainNs);
    __syncwarp();
    if (!alive && lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, c);
  } else if (warp < kTcOaccWarp0) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp - kTcSoftmaxWarp0;     // TMEM lane quarter
    const int i = q4 * 32 + lane;              // key row of S
    const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const float sl2 = p.scale_log2;
    uint32_t j = 0;
    int u = 0;
    bool alive = true;
    // Waits the warp agrees on (the TMEM loads after them are warp-wide).
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool ok = mbar_wait(bar, parity, abort, kWaitNs);
      return __all_sync(0xffffffffu, ok);
    };
    for (int t = 0; t < nseg && alive; ++t) {
      const SegInfo si = s_seg[t];
      const int nt = part_tiles(si);
      if (nt == 0) continue;
      float m[kNH], lth[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        m[h] = -INFINITY;
        lth[h] = 0.f;
      }
      for (int jt = 0; jt < nt; ++jt, ++j) {
        const int b = j & 1;
        if (!(alive = wait(&B.s_full[b], (j >> 1) & 1))) break;
        tc_fence_after();
        uint32_t sr[kNH];
        tmem_ld8(tl + 16 * b, sr);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&B.s_empty[b]);
        const TileGeo tg = tile_geo(si, jt);
        const int32_t key = tg.key0 + i;
        bool valid = key >= si.lo && key >= si.kb && key < si.ke;
        if (valid) valid = page_at(si, s_pages, npages, p.page_shift, key) >= 0;
        float x[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h)
          x[h] = (valid && h < G) ? __uint_as_float(sr[h]) * sl2 : -INFINITY;
        // Tile maximum per head: warp reduce-scatter, then the four warps.
        const float wmax = reduce_scatter8<true>(x, lane);
        if ((lane & 3) == 0) s_red[b][q4][lane >> 2] = wmax;
        mbar_arrive(&B.red_full[b]);
        if (!(alive = wait(&B.red_full[b], (j >> 1) & 1))) break;
        float tmax[kNH];
#pragma unroll
        for (int h4 = 0; h4 < kNH; h4 += 4) {
          float4 r0 = *reinterpret_cast<const float4*>(&s_red[b][0][h4]);
#pragma unroll
          for (int w = 1; w < 4; ++w) {
            const float4 rw = *reinterpret_cast<const float4*>(&s_red[b][w][h4]);
            r0.x = fmaxf(r0.x, rw.x);
            r0.y = fmaxf(r0.y, rw.y);
            r0.z = fmaxf(r0.z, rw.z);
            r0.w = fmaxf(r0.w, rw.w);
          }
          tmax[h4] = r0.x;
          tmax[h4 + 1] = r0.y;
          tmax[h4 + 2] = r0.z;
          tmax[h4 + 3] = r0.w;
        }
        float al[kNH], pv[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          const float mn = fmaxf(m[h], tmax[h]);
          // Nothing visible yet (mn = -inf): no rescale, P = 0.
          al[h] = mn == -INFINITY ? 1.f : fast_exp2(m[h] - mn);
          pv[h] = fast_exp2(x[h] - (mn == -INFINITY ? 0.f : mn));
          lth[h] = fmaf(lth[h], al[h], pv[h]);
          m[h] = mn;
        }
        // P^T (K-major, 128-byte swizzle): head row h, key i at byte
        // 2 (i % 64) of key chunk i / 64, the 16-byte unit XOR h.
        if (!(alive = wait(&B.p_free[b], ((j >> 1) & 1) ^ 1))) break;
        {
          const uint32_t pb = smem_u32(smem + L::kPOff + b * L::kPBytes) + (i >> 6) * 2048 +
                              ((i & 7) << 1);
          const int g16 = (i & 63) >> 3;
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const __nv_bfloat16 v = __float2bfloat16_rn(pv[h]);
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(pb + h * 128 + ((g16 ^ h) << 4)),
                         "h"(*reinterpret_cast<const unsigned short*>(&v))
                         : "memory");
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&B.p_full[b]);
        }
        // The tile's rescale factors for the O accumulation: thread h < 8
        // hands over head h's.
        if (i < kNH) {
          float a = al[0];
#pragma unroll
          for (int h = 1; h < kNH; ++h) a = i == h ? al[h] : a;
          if (!mbar_wait(&B.a_empty[b], ((j >> 1) & 1) ^ 1, abort, kWaitNs)) alive = false;
          s_alpha[b][i] = a;
          mbar_arrive(&B.a_full[b]);
        }
        if (!(alive = __all_sync(0xffffffffu, alive))) break;
      }
      if (!alive) break;
      // Row sums: warp reduce-scatter, then the four warps; thread h < 8
      // hands head h's sum and maximum to the output warps.
      const float wsum = reduce_scatter8<false>(lth, lane);
      const int lb = u & 1;
      if ((lane & 3) == 0) s_lsum[lb][q4][lane >> 2] = wsum;
      mbar_arrive(&B.l_full[lb]);
      if (!(alive = wait(&B.l_full[lb], (u >> 1) & 1))) break;
      if (i < kNH) {
        float mi = m[0];
#pragma unroll
        for (int h = 1; h < kNH; ++h) mi = i == h ? m[h] : mi;
        const float li = s_lsum[lb][0][i] + s_lsum[lb][1][i] + s_lsum[lb][2][i] + s_lsum[lb][3][i];
        if (!mbar_wait(&B.f_empty[lb], ((u >> 1) & 1) ^ 1, abort, kWaitNs)) alive = false;
        s_fin_l[lb][i] = li;
        s_fin_m[lb][i] = mi;
        mbar_arrive(&B.f_full[lb]);
      }
      if (!(alive = __all_sync(0xffffffffu, alive))) break;
      ++u;
    }
  } else {
    // ------------------------------------------------------------ O and output
    // Thread = TMEM lane = dimension row of O^T (of each 128-dimension half).
    const int q4 = warp - kTcOaccWarp0;
    const int i = q4 * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    uint32_t j = 0;
    int u = 0;
    bool alive = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool ok = mbar_wait(bar, parity, abort, kWaitNs);
      return __all_sync(0xffffffffu, ok);
    };
    for (int t = 0; t < nseg && alive; ++t) {
      const SegInfo si = s_seg[t];
      const int nt = part_tiles(si);
      if (nt == 0) continue;
      float o[L::kHalves][kNH];
#pragma unroll
      for (int dh = 0; dh < L::kHalves; ++dh)
#pragma unroll
        for (int h = 0; h < kNH; ++h) o[dh][h] = 0.f;
      for (int jt = 0; jt < nt; ++jt, ++j) {
        const int b = j & 1;
        // O = O * 2^(m_old - m_new) + O^T(j).
        if (!(alive = wait(&B.a_full[b], (j >> 1) & 1))) break;
        float al[kNH];
        {
          const float4 a0 = *reinterpret_cast<const float4*>(&s_alpha[b][0]);
          const float4 a1 = *reinterpret_cast<const float4*>(&s_alpha[b][4]);
          al[0] = a0.x; al[1] = a0.y; al[2] = a0.z; al[3] = a0.w;
          al[4] = a1.x; al[5] = a1.y; al[6] = a1.z; al[7] = a1.w;
        }
        mbar_arrive(&B.a_empty[b]);
        if (!(alive = wait(&B.o_full[b], (j >> 1) & 1))) break;
        tc_fence_after();
        uint32_t r[L::kHalves][kNH];
#pragma unroll
        for (int dh = 0; dh < L::kHalves; ++dh) tmem_ld8(tl + 32 + 32 * b + 16 * dh, r[dh]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&B.o_empty[b]);
#pragma unroll
        for (int dh = 0; dh < L::kHalves; ++dh)
#pragma unroll
          for (int h = 0; h < kNH; ++h) o[dh][h] = fmaf(o[dh][h], al[h], __uint_as_float(r[dh][h]));
      }
      if (!alive) break;
      const int lb = u & 1;
      if (!(alive = wait(&B.f_full[lb], (u >> 1) & 1))) break;
      float lsum[kNH], mfin[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        lsum[h] = s_fin_l[lb][h];
        mfin[h] = s_fin_m[lb][h];
      }
      mbar_arrive(&B.f_empty[lb]);
      ++u;
      const int slot = sc.slot_base + 2 * c + (t == 0 ? 0 : 1);
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        if (h >= G) break;
        const float inv = lsum[h] > 0.f ? 1.f / lsum[h] : 0.f;
        if (si.whole) {
          __nv_bfloat16* orow = p.out + (static_cast<int64_t>(si.q0) * p.hq + si.g * G + h) * D;
#pragma unroll
          for (int dh = 0; dh < L::kHalves; ++dh)
            orow[dh * 128 + i] = __float2bfloat16_rn(o[dh][h] * inv);
        } else {
          float* orow = p.part_o + (static_cast<int64_t>(slot) * G + h) * D;
#pragma unroll
          for (int dh = 0; dh < L::kHalves; ++dh) orow[dh * 128 + i] = o[dh][h] * inv;
          if (i == 0)
            p.part_lse[static_cast<int64_t>(slot) * G + h] =
                lsum[h] > 0.f ? mfin[h] + __log2f(lsum[h]) : -INFINITY;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int NSEG>
int launch_tc_one(const Plan& plan, const DecodeParams& p, const TcMaps& maps,
                  const Plan::DecodeLaunch& dl, cudaStream_t stream) {
  constexpr int smem = TcLayout<D>::kDynBytes;
  if (int e = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_tc_kernel<D, NSEG>), smem))
    return e;
  DecodeSched<NSEG>& sc = thread_staging<DecodeSched<NSEG>>();
  if (int e = fill_decode_sched(plan, dl, sc)) return e;
  decode_tc_kernel<D, NSEG><<<dl.n_ctas, kTcThreads, smem, stream>>>(maps, p, sc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  trace_mark(RPA_KERNEL_DECODE_SPLIT, stream);
  return 0;
}

template <int D>
int launch_decode_tc_t(const Plan& plan, const Args& a, cudaStream_t stream) {
  using L = TcLayout<D>;
  const DecodeParams p = make_decode_params(plan, a);
  TcMaps& maps = thread_staging<TcMaps>();
  const uint64_t rows = static_cast<uint64_t>(plan.num_pages) * plan.p;
  const uint32_t hq_box = plan.hq < 16 ? static_cast<uint32_t>(plan.hq) : 16u;
  bool ok = make_tmap_3d(&maps.q, a.q, D, plan.hq, static_cast<uint64_t>(plan.total_q), hq_box, 1);
  // Only boxes no taller than a page are ever used.
  for (int i = 0; i < 4 && ok; ++i)
    if ((16 << i) <= plan.p)
      ok = make_tmap_3d(&maps.k[i], a.k_pages, D, plan.hkv, rows, 1, 16u << i) &&
           make_tmap_3d(&maps.v[i], a.v_pages, D, plan.hkv, rows, 1, 16u << i);
  if (ok && L::kVKeys <= plan.p)
    ok = make_tmap_4d_chunks(&maps.v4, a.v_pages, D, plan.hkv, rows, 1, L::kVKeys, false);
  if (!ok) return static_cast<int>(cudaErrorInvalidValue);
  for (const Plan::DecodeLaunch& dl : plan.dlaunch) {
    const int n = dl.seg_end - dl.seg_begin;
    int err = n <= kDecodeSegSmall ? launch_tc_one<D, kDecodeSegSmall>(plan, p, maps, dl, stream)
                                   : launch_tc_one<D, kDecodeSegLarge>(plan, p, maps, dl, stream);
    if (!err) err = launch_decode_combine(plan, p, dl, D, stream);
    if (err) return err;
  }
  return 0;
}

}  // namespace

bool decode_tc_supported(int32_t head_dim, int32_t group, int32_t page_size, bool kv_fp8) {
  return (head_dim == 128 || head_dim == 256) && group >= 1 && group <= kNH &&
         page_size >= 16 && !kv_fp8;
}

int launch_decode_tc(const Plan& plan, const Args& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (plan.d) {
    case 128: return launch_decode_tc_t<128>(plan, a, s);
    case 256: return launch_decode_tc_t<256>(plan, a, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace rpa
