// Tensor-core prefill on pairs of SMs (tcgen05 .cta_group::2).
//
// Sources (page titles and sections): as the single-SM prefill kernel
// ("Chasing speed of light on TPU v6e", section "Attention" and footnotes 5
// and 6: query blocks kept on chip, every key streamed once per block that
// wants it, fp32 accumulators; sliding windows skip whole KV tiles).
//
// A cluster of two CTAs on two SMs takes work items of two adjacent query
// blocks of one (sequence, KV head): CTA rank r holds block 2p + r, 128 MMA
// rows ((128 / G) tokens x the G query heads).  One M = 256 MMA covers both:
//   S = Q K^T   A = each CTA's Q block (its shared memory), B = the 128-key
//               tile split by key: keys [64r, 64r + 64) in CTA r's shared
//               memory; each CTA's TMEM receives its 128 rows x 128 keys;
//   O += P V    A = P from each CTA's TMEM, B = V split by dimension:
//               dimensions [rD/2, (r+1)D/2) in CTA r; each TMEM receives its
//               128 rows x D.
// So each SM stages half of every K and V tile.  Against the single-SM
// kernel this halves the copy traffic into each SM's shared memory and the
// B-operand reads out of it, which together with the A reads bound that
// kernel, and doubles the tiles its copy ring covers.
//
// Roles per CTA: warp 0 loads Q and its half of K, warp 1 its half of V;
// warp 2 of rank 0 issues every MMA of the pair (elect.sync) and commits to
// the mbarriers of both CTAs at once (multicast); warps 3-10 run the softmax
// of the CTA's rows (two warps per TMEM lane quarter, as the single-SM
// kernel) and the epilogue.  Copies of both CTAs complete on rank 0's
// "full" barriers, softmax warps of both arrive on rank 0's "P ready" and
// "O free" barriers; rank 0's MMA commits arrive on both CTAs' "empty",
// "S ready" and "O done" barriers.  Every wait is bounded.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "rpa_internal.h"
#include "sm100_ptx.cuh"

namespace rpa {
namespace {

using namespace sm100;

constexpr int kBM = 128;        // MMA rows per CTA (256 per pair)
constexpr int kBN = 128;        // keys per score tile
constexpr int kHalfN = 64;      // keys of a score tile staged by each CTA
constexpr int kTileAlign = 64;  // score tiles start on multiples of this many keys
constexpr int kStage = 8192;    // bytes per K or V ring stage
constexpr int kKS = 10;         // K ring depth (stages)
constexpr int kVS = 10;         // V ring depth (stages)
constexpr int kThreads = 352;   // K producer, V producer, MMA, 8 softmax warps
constexpr int kSoftmaxWarps = 8;
constexpr int kPolyEvery = 32;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;

struct ItemList {
  int32_t n;
  PrefillItem items[kMaxItemsPerLaunch];  // qb_head = (pair << 8) | kv head
};

struct PairParams {
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  const int32_t* window;
  __nv_bfloat16* out;
  unsigned char* ws;
  int32_t hq, group, qb_tokens, page_size, page_shift, box_rows_k, box_rows_v, mpps, num_pages;
  float scale_log2;
};

// Per CTA: Q block, K ring (a stage: 64 keys x one 64-dimension chunk), V
// ring (a stage: kVKeys keys x the CTA's D / 2 dimensions).
template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;
  static constexpr int kVDims = D / 2;                   // V dimensions per CTA
  static constexpr int kVChunks = kVDims / 64;
  static constexpr int kVKeys = kStage / (kVDims * 2);   // keys per V stage
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kKS * kStage;
  static constexpr int kBarOff = kVOff + kVS * kStage;
  static constexpr int kXchOff = kBarOff + 512;
  static constexpr int kUsed = kXchOff + 2 * 2 * kBM * 4;
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  static constexpr int kOCol = 0;                        // O: D columns
  static constexpr int kSCol = D;                        // two S buffers of 128
  static constexpr int kCols = 512;
};

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[kKS], k_empty[kKS], v_full[kVS], v_empty[kVS];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free;
  uint64_t fin;
  uint64_t xbar[4];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Barriers) <= 512, "barrier block");

// Geometry of this CTA's query block inside a pair item, and the pair's
// key tiles (the same for both CTAs).
struct Geom {
  int32_t seq, g, t0, ntok, pos_first;  // this CTA's block
  int32_t key_first, ntiles, pos_last;  // the pair: tiles and its last query
  int32_t lo;                           // the pair: first key any query sees
  int32_t W;
  bool ok;
};

__device__ __forceinline__ Geom pair_geom(const PairParams& p, const PrefillItem& it,
                                          uint32_t rank) {
  Geom r;
  r.seq = it.seq;
  r.g = it.qb_head & 255;
  const int32_t pair = it.qb_head >> 8;
  const int32_t q0 = __ldg(p.cu_q_lens + r.seq);
  const int32_t ql = __ldg(p.cu_q_lens + r.seq + 1) - q0;
  const int32_t L = __ldg(p.kv_lens + r.seq);
  r.W = p.window ? __ldg(p.window + r.seq) : 0;
  const int32_t qbt = p.qb_tokens;
  const int32_t b0 = 2 * pair;
  const int32_t n0 = min(qbt, ql - b0 * qbt);
  const int32_t n1 = max(0, min(qbt, ql - (b0 + 1) * qbt));
  const int32_t first0 = L - ql + b0 * qbt;
  r.pos_last = n1 > 0 ? first0 + qbt + n1 - 1 : first0 + n0 - 1;
  const int32_t qb = b0 + static_cast<int32_t>(rank);
  r.t0 = q0 + qb * qbt;
  r.ntok = rank == 0 ? n0 : n1;
  r.pos_first = L - ql + qb * qbt;
  r.ok = n0 > 0 && first0 >= 0 && r.pos_last < L && (r.pos_last >> p.page_shift) < p.mpps;
  r.lo = first_visible(first0, r.W);
  r.key_first = r.lo / kTileAlign * kTileAlign;
  r.ntiles = r.ok ? (r.pos_last - r.key_first) / kBN + 1 : 0;
  return r;
}

template <int N>
__device__ __forceinline__ float max_tree(const uint32_t* v) {
  if constexpr (N == 1) {
    return __uint_as_float(v[0]);
  } else if constexpr (N == 2) {
    return fmaxf(__uint_as_float(v[0]), __uint_as_float(v[1]));
  } else {
    constexpr int M = (N + 2) / 3;
    uint32_t t[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const float a = __uint_as_float(v[3 * i]);
      float m = a;
      if (3 * i + 2 < N)
        m = fmax3(a, __uint_as_float(v[3 * i + 1]), __uint_as_float(v[3 * i + 2]));
      else if (3 * i + 1 < N)
        m = fmaxf(a, __uint_as_float(v[3 * i + 1]));
      t[i] = __float_as_uint(m);
    }
    return max_tree<M>(t);
  }
}

// TMA source row of the box of `rows` keys starting at `key` (-rows: wholly
// outside the keys the pair's queries see, past its last query or before its
// first visible key; the TMA fills it with zeros and the page table is not
// read).
__device__ __forceinline__ int32_t box_row(const PairParams& p, const Geom& gm, int32_t key,
                                           int32_t rows) {
  if (key > gm.pos_last || key + rows <= gm.lo) return -rows;
  const int32_t page = __ldg(p.page_table + static_cast<int64_t>(gm.seq) * p.mpps +
                             (key >> p.page_shift));
  if (page < 0 || page >= p.num_pages) {
    report_error(p.ws, RPA_DEVERR_PAGE_ID, gm.seq);
    return -rows;
  }
  return page * p.page_size + (key & (p.page_size - 1));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const PairParams p,
                    const __grid_constant__ ItemList items) {
  using Lay = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Both CTAs of the pair take the same branch here (same launch, same
  // shared-memory layout), so neither is left waiting for the other.
  if (smem_addr(smem_raw) & 1023u) {
    if (threadIdx.x == 0) report_error(p.ws, RPA_DEVERR_LAUNCH, blockIdx.x);
    return;
  }
  uint8_t* smem = smem_raw;
  __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem + Lay::kQOff);
  Barriers& B = *reinterpret_cast<Barriers*>(smem + Lay::kBarOff);
  volatile int* abort = &B.abort;
  const uint32_t rank = cluster_rank();
  const int pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

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
      mbar_init(&B.p_full[i], 2 * kSoftmaxWarps);
      mbar_init(&B.o_done[i], 1);
    }
    mbar_init(&B.o_free, 2 * kSoftmaxWarps);
    mbar_init(&B.fin, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&B.xbar[i], 64);
    B.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 2) {
    tmem_alloc_pair(&B.tmem_base, Lay::kCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before either touches the other's
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const int G = p.group;

  if (warp <= 1) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == 0;
    const int depth = is_k ? kKS : kVS;
    uint64_t* full = is_k ? B.k_full : B.v_full;
    uint64_t* empty = is_k ? B.k_empty : B.v_empty;
    uint8_t* ring = smem + (is_k ? Lay::kKOff : Lay::kVOff);
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    const int rows = is_k ? p.box_rows_k : p.box_rows_v;
    const int stage_keys = is_k ? kHalfN : Lay::kVKeys;
    const int nbox = stage_keys / rows;                            // <= 8
    const int stages = is_k ? Lay::kChunks : kBN / Lay::kVKeys;    // per tile
    const uint32_t q_box_bytes = static_cast<uint32_t>(G * p.qb_tokens) * 128u;
    uint32_t C = 0, I = 0, issued_q = 0;
    bool alive = true;
    for (int it = pair_id; it < items.n && alive; it += n_pairs) {
      const Geom gm = pair_geom(p, items.items[it], rank);
      if (!gm.ok) {
        if (lane == 0 && is_k) report_error(p.ws, RPA_DEVERR_LENGTHS, gm.seq);
        continue;
      }
      const uint32_t Icur = I++;
      if (is_k && lane == 0) {
        alive = mbar_wait_cluster(&B.q_empty, (Icur & 1) ^ 1, abort, kWaitNs);
        if (alive) {
          if (rank == 0) mbar_arrive_expect_tx(&B.q_full, 2 * q_box_bytes * Lay::kChunks);
          const uint32_t qbar = cluster_addr(&B.q_full, 0);
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d_pair(q_s + c * kBM * 64, &tm_q, qbar, c * 64, gm.g * G, gm.t0);
          ++issued_q;
        }
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      for (int j = 0; j < gm.ntiles && alive; ++j) {
        const int32_t key0 = gm.key_first + j * kBN;
        // This CTA's half: keys [64 rank, 64 rank + 64) of the tile for K,
        // every key of the tile (kVKeys per stage) for V.
        const int32_t krow = (is_k && lane < nbox)
                                 ? box_row(p, gm, key0 + kHalfN * rank + lane * rows, rows)
                                 : 0;
        for (int sgi = 0; sgi < stages; ++sgi, ++C) {
          const int st = C % depth;
          const uint32_t ph = (C / depth) & 1;
          const int32_t row = is_k ? krow
                              : (lane < nbox ? box_row(p, gm, key0 + sgi * Lay::kVKeys + lane * rows, rows)
                                             : 0);
          if (lane == 0) alive = mbar_wait_cluster(&empty[st], ph ^ 1, abort, kWaitNs);
          alive = __shfl_sync(0xffffffffu, alive, 0);
          if (!alive) break;
          if (lane == 0 && rank == 0) mbar_arrive_expect_tx(&full[st], 2 * kStage);
          __syncwarp();
          if (lane < nbox) {
            const uint32_t bar = cluster_addr(&full[st], 0);
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(ring + st * kStage) + lane * rows * 64;
            if (is_k) {
              tma_load_3d_pair(dst, tm, bar, sgi * 64, gm.g, row);
            } else {
              for (int c = 0; c < Lay::kVChunks; ++c)
                tma_load_3d_pair(dst + c * Lay::kVKeys * 64, tm, bar,
                                 static_cast<int32_t>(rank) * Lay::kVDims + c * 64, gm.g, row);
            }
          }
        }
      }
    }
    if (!alive && lane == 0) {
      report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
      // Rank 0's full barriers count both CTAs' copies: let them land.
      if (rank == 0) {
        for (uint32_t t = (C > static_cast<uint32_t>(depth) ? C - depth : 0); t < C; ++t) {
          int dummy = 0;
          mbar_wait_cluster(&full[t % depth], (t / depth) & 1, &dummy, kDrainNs);
        }
        if (is_k && issued_q > 0) {
          int dummy = 0;
          mbar_wait_cluster(&B.q_full, (issued_q - 1) & 1, &dummy, kDrainNs);
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (rank == 0) {
      constexpr uint32_t kIdS = idesc_bf16_m(2 * kBM, kBN, 0);
      constexpr uint32_t kIdPV = idesc_bf16_m(2 * kBM, D, 1);
      const uint32_t q_base = smem_addr(q_s);
      const uint32_t k_base = smem_addr(smem + Lay::kKOff), v_base = smem_addr(smem + Lay::kVOff);
      uint32_t T = 0, I = 0;
      // Ring slot and phase of the next K / V stage.
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      // Descriptors as base + byte offset / 16 (the start-address field;
      // every operand lies below 256 KB), built once rather than per MMA.
      const uint64_t q_d0 = smem_desc(q_base, 16, 1024);
      const uint64_t k_d0 = smem_desc(k_base, 16, 1024);
      const uint64_t v_d0 = smem_desc(v_base, Lay::kVKeys * 128, 1024);
      bool alive = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait_cluster(bar, parity, abort, kWaitNs);
        return __all_sync(0xffffffffu, ok);
      };
      // O += P V: per V stage (kVKeys keys), B = the pair's V split by
      // dimension (MN-major: 8-key groups 1024 B apart, 64-dimension chunks
      // kVKeys x 128 B apart); A = P from the S buffer's first 64 columns.
      //
      // A masked key has P = 0, but 0 x NaN is NaN: the V rows of keys no
      // query of the pair sees (before its first visible key, past its last
      // query) may hold anything, so they are zeroed in both CTAs' stages
      // (the partner's through its cluster address) before the MMA reads
      // them.  Boxes wholly outside those keys arrive as zeros already.
      auto clear_v_edges = [&](const Geom& gm, int32_t kst, int vs) {
        const int a = max(0, min(Lay::kVKeys, gm.lo - kst));              // rows [0, a)
        const int b = max(0, min(Lay::kVKeys, gm.pos_last + 1 - kst));    // rows [b, kVKeys)
        if ((a == 0 && b == Lay::kVKeys) || a == Lay::kVKeys || b == 0) return;
        const uint32_t st0 = cluster_addr(smem + Lay::kVOff + vs * kStage, 0);
        const uint32_t st1 = cluster_addr(smem + Lay::kVOff + vs * kStage, 1);
        const int nrows = a + (Lay::kVKeys - b);
        for (int u = lane; u < 2 * nrows * Lay::kVChunks * 8; u += 32) {
          const int cta = u & 1, v = u >> 1;
          const int rr = v / (Lay::kVChunks * 8), rem = v % (Lay::kVChunks * 8);
          const int row = rr < a ? rr : b + (rr - a);
          const uint32_t addr = (cta ? st1 : st0) + (rem >> 3) * (Lay::kVKeys * 128) + row * 128 +
                                (rem & 7) * 16;
          asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u)
                       : "memory");
        }
        // The pair's MMA reads both stages through the async proxy.
        asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
        __syncwarp();
      };
      auto issue_pv = [&](const Geom& gm, uint32_t Tp, int jp) -> bool {
        const int sb = Tp & 1;
        if (!wait(&B.p_full[sb], (Tp >> 1) & 1)) return false;
        if (jp == 0 && !wait(&B.o_free, (I & 1) ^ 1)) return false;
        const uint32_t p_col = tmem + Lay::kSCol + sb * kBN;
#pragma unroll 1
        for (int sgi = 0; sgi < kBN / Lay::kVKeys; ++sgi) {
          if (!wait(&B.v_full[vs], vph)) return false;
          clear_v_edges(gm, gm.key_first + jp * kBN + sgi * Lay::kVKeys, vs);
          tc_fence_after();
          const uint64_t vd = v_d0 + static_cast<uint64_t>(vs * (kStage >> 4));
#pragma unroll
          for (int kk = 0; kk < Lay::kVKeys / 16; ++kk) {
            const int kg = sgi * (Lay::kVKeys / 16) + kk;
            mma_ts_pair(tmem + Lay::kOCol, p_col + kg * 8, vd + ((kk * 2048) >> 4), kIdPV,
                        (jp > 0 || kg > 0) ? 1u : 0u);
          }
          mma_commit_pair(&B.v_empty[vs]);
          if (++vs == kVS) {
            vs = 0;
            vph ^= 1;
          }
        }
        mma_commit_pair(&B.o_done[sb]);
        return true;
      };
      // S = Q K^T: per K stage (one 64-dimension chunk), A = each CTA's Q
      // (K-major, chunks 16 KB apart), B = its 64 keys of the tile.
      auto issue_s = [&](uint32_t Ts) -> bool {
        const uint32_t sc = tmem + Lay::kSCol + (Ts & 1) * kBN;
#pragma unroll 1
        for (int c = 0; c < Lay::kChunks; ++c) {
          if (!wait(&B.k_full[ks], kph)) return false;
          tc_fence_after();
          const uint64_t kd = k_d0 + static_cast<uint64_t>(ks * (kStage >> 4));
#pragma unroll
          for (int w = 0; w < 4; ++w)
            mma_ss_pair(sc, q_d0 + ((c * (kBM * 128) + w * 32) >> 4), kd + ((w * 32) >> 4), kIdS,
                        (c > 0 || w > 0) ? 1u : 0u);
          mma_commit_pair(&B.k_empty[ks]);
          if (++ks == kKS) {
            ks = 0;
            kph ^= 1;
          }
        }
        mma_commit_pair(&B.s_full[Ts & 1]);
        return true;
      };
      for (int it = pair_id; it < items.n && alive; it += n_pairs) {
        const Geom gm = pair_geom(p, items.items[it], 0);
        if (!gm.ok) continue;
        alive = wait(&B.q_full, I & 1);
        if (!alive) break;
        const int n = gm.ntiles;
        if (n > 0) alive = issue_s(T);
        if (n <= 1) mma_commit_pair(&B.q_empty);
        for (int j = 0; j < n && alive; ++j) {
          if (j + 1 < n) {
            alive = issue_s(T + j + 1);
            if (!alive) break;
            if (j + 2 == n) mma_commit_pair(&B.q_empty);
          }
          alive = issue_pv(gm, T + j, j);
        }
        T += n;
        ++I;
      }
      if (!alive && lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
      // Every MMA of the pair must finish before either CTA frees its TMEM
      // or shared memory (the teardown's cluster barrier orders rank 1
      // after this wait).
      mma_commit_pair(&B.fin);
      int dummy = 0;
      mbar_wait_cluster(&B.fin, 0, &dummy, kDrainNs);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;
    const int h = (warp - 3) >> 2;
    const int r = 32 * q4 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const int tok = r / G, head = r % G;
    const float c = p.scale_log2;
    float* xch = reinterpret_cast<float*>(smem + Lay::kXchOff);
    uint64_t* xbar = &B.xbar[q4];
    const uint32_t p_full0 = cluster_addr(&B.p_full[0], 0);
    const uint32_t p_full1 = cluster_addr(&B.p_full[1], 0);
    const uint32_t o_free0 = cluster_addr(&B.o_free, 0);
    uint32_t T = 0, X = 0;
    bool alive = true;
    // One arrival per warp on rank 0's barrier: local in rank 0; relaxed and
    // remote in rank 1 (what it signals, TMEM stores or loads, has already
    // completed: tcgen05.wait::st / ::ld).
    auto arrive_rank0 = [&](uint64_t* bar, uint32_t bar_cluster) {
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(bar); else mbar_arrive_remote_relaxed(bar_cluster);
      }
    };
    auto swap = [&](float v) -> float {
      xch[((X & 1) * 2 + h) * kBM + r] = v;
      tc_fence_before();
      mbar_arrive(xbar);
      const bool ok = mbar_wait(xbar, X & 1, abort, kWaitNs);
      tc_fence_after();
      const float o = xch[((X & 1) * 2 + (h ^ 1)) * kBM + r];
      ++X;
      if (!ok) alive = false;
      return o;
    };
    for (int it = pair_id; it < items.n && alive; it += n_pairs) {
      const Geom gm = pair_geom(p, items.items[it], rank);
      if (!gm.ok) continue;
      const bool valid = tok < gm.ntok && r < G * p.qb_tokens;
      const int32_t pos = gm.pos_first + tok;
      const int32_t lo = first_visible(pos, gm.W);
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < gm.ntiles; ++j, ++T) {
        const int sb = T & 1;
        if (!mbar_wait_cluster(&B.s_full[sb], (T >> 1) & 1, abort, kWaitNs)) {
          alive = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(lane_addr + Lay::kSCol + sb * kBN + 64 * h,
                  *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(lane_addr + Lay::kSCol + sb * kBN + 64 * h + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_ld();
        const int32_t key0 = gm.key_first + j * kBN + 64 * h;
        const bool full = __all_sync(0xffffffffu, valid && key0 >= lo && key0 + 63 <= pos);
        if (!full) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc) {
            const int32_t key = key0 + cc;
            const bool vis = valid && key >= lo && key <= pos;
            if (!vis) sr[cc] = 0xff800000u;
          }
        }
        float mx = max_tree<64>(sr);
        mx = fmaxf(mx, swap(mx));
        if (!alive) break;
        mx = (mx == -INFINITY) ? -INFINITY : mx * c;
        const float m_new = fmaxf(m_ref, mx);
        const bool grow = m_new > m_ref + 8.f;
        const bool rescale_o = grow && m_ref != -INFINITY;
        if (__any_sync(0xffffffffu, rescale_o)) {
          const uint32_t Tp = T - 1;
          if (!mbar_wait_cluster(&B.o_done[Tp & 1], (Tp >> 1) & 1, abort, kWaitNs)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const float f = rescale_o ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll 1
          for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
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
        // Paired fp32 arithmetic (masked scores are -inf: 2^-inf = +0).
        // One pair in kPolyEvery takes its 2^x on the FMA pipe.
        uint32_t pk[32];
        float ls;
        {
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
        }
        l += ls;
        tmem_st32(lane_addr + Lay::kSCol + sb * kBN + 32 * h, pk);
        tmem_wait_st();
        tc_fence_before();
        arrive_rank0(&B.p_full[sb], sb ? p_full1 : p_full0);
      }
      if (!alive) break;
      if (gm.ntiles == 0) continue;
      l += swap(l);
      if (!alive) break;
      const uint32_t Tl = T - 1;
      if (!mbar_wait_cluster(&B.o_done[Tl & 1], (Tl >> 1) & 1, abort, kWaitNs)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow =
          p.out + (static_cast<int64_t>(gm.t0 + tok) * p.hq + gm.g * G + head) * D;
#pragma unroll 1
      for (int c0 = h * (D / 2); c0 < (h + 1) * (D / 2); c0 += 32) {
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
      arrive_rank0(&B.o_free, o_free0);
    }
    if (!alive && lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
  }

  // Teardown: every pair MMA has finished (warp 2 waited on fin); neither
  // CTA leaves while the other may still reach into its shared memory.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, Lay::kCols);
  }
}

template <int D>
int launch_pair_t(const Plan& plan, const Args& a, cudaStream_t stream) {
  using Lay = Layout<D>;
  if (int e = ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_pair_kernel<D>), Lay::kBytes))
    return e;
  // Clusters of two that fit at once (per thread: the query is cheap and its
  // answer does not change for a device).
  static thread_local int max_pairs = 0;
  if (max_pairs == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * plan.num_sms / 2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay::kBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel<D>, &cfg);
    if (e != cudaSuccess || n <= 0) return static_cast<int>(e != cudaSuccess ? e : cudaErrorInvalidConfiguration);
    max_pairs = n;
  }
  const int G = plan.hq / plan.hkv;
  const int qb = plan.q_block;
  const int box_rows_k = std::min(plan.p, kHalfN);
  const int box_rows_v = std::min(std::min(plan.p, Lay::kVKeys), kTileAlign);
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d(&tq, a.q, D, plan.hq, static_cast<uint64_t>(plan.total_q), G, qb) ||
      !make_tmap_3d(&tk, a.k_pages, D, plan.hkv, static_cast<uint64_t>(plan.num_pages) * plan.p, 1,
                    box_rows_k) ||
      !make_tmap_3d(&tv, a.v_pages, D, plan.hkv, static_cast<uint64_t>(plan.num_pages) * plan.p, 1,
                    box_rows_v))
    return static_cast<int>(cudaErrorInvalidValue);
  PairParams p;
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
  p.box_rows_k = box_rows_k;
  p.box_rows_v = box_rows_v;
  p.mpps = plan.mpps;
  p.num_pages = plan.num_pages;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  ItemList& list = thread_staging<ItemList>();  // copied into the launch parameters
  const size_t n = plan.items.size();
  for (size_t off = 0; off < n; off += kMaxItemsPerLaunch) {
    const int cnt = static_cast<int>(std::min<size_t>(kMaxItemsPerLaunch, n - off));
    list.n = cnt;
    for (int i = 0; i < cnt; ++i) list.items[i] = plan.items[off + i];
    const int pairs = std::min(cnt, std::min(max_pairs, plan.prefill_ctas / 2));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay::kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_pair_kernel<D>, tq, tk, tv, p, list);
    if (e != cudaSuccess) return static_cast<int>(e);
    trace_mark(RPA_KERNEL_PREFILL_TC, stream);
  }
  return 0;
}

}  // namespace

bool prefill_pair_supported(int32_t head_dim, int32_t page_size, int32_t group) {
  return (head_dim == 128 || head_dim == 256) && page_size >= 16 && group >= 1 && group <= kBM;
}

int launch_prefill_pair(const Plan& plan, const Args& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (plan.d) {
    case 128: return launch_pair_t<128>(plan, a, s);
    case 256: return launch_pair_t<256>(plan, a, s);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace rpa
