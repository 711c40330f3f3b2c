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
// One CTA (persistent, one per SM) walks its own list of work items
// (sequence, query block, KV head), given by the plan: items, longest first,
// go to the CTA with the fewest key tiles so far.  On request an item's key
// tiles are split across CTAs; each part writes an fp32 partial (O / l and
// the log2-sum-exp per row) that prefill_combine_kernel merges.  Warp roles:
//   warp 0     TMA producer of the Q block (once per item) and of K, gathered
//              page by page through the page table into a ring of 16 KB
//              stages (one 64-dimension chunk of a 128-key tile each);
//   warp 1     TMA producer of V into its own ring of 16 KB stages (8192 / D
//              keys x all D dimensions each), so K runs ahead of V;
//   warp 2     MMA issuer: S = Q K^T over 128-key tiles (SMEM x SMEM -> TMEM,
//              N = 128: narrower score MMAs leave the tensor core partly
//              idle) and O += P V (P from TMEM, V from SMEM), one ring stage
//              at a time; tcgen05.commit onto mbarriers.  The score tile runs
//              one ahead of the PV product (two S buffers; P is written over
//              its own S);
//   warp 3     idle (completes the first warpgroup);
//   warps 4-11 softmax: two warps per 32 rows (a TMEM lane quarter), one
//              thread per row and 64 of the tile's 128 keys each; the pair
//              swaps row maxima through shared memory every tile;
//              reads S from TMEM, masks causal and window edges (interior
//              tiles skip the mask), keeps the running max / sum in fp32,
//              exponentiates with the MUFU unit and, for one pair in 32,
//              with a polynomial on the FMA pipe (paired fp32 instructions),
//              writes P (bf16) to TMEM, rescales O in TMEM only when the max
//              grew by more than 2^8 (the result is the same; it bounds P by
//              256); at an item's end hands its row sums to the epilogue
//              and goes straight on to the next item's first tile, the next
//              item's geometry read during the current item;
//   warps 12-15 epilogue: one thread per row; waits for the item's last PV,
//              O / l -> bf16 -> global (32-byte stores), then frees O for the
//              next item's first PV, so the softmax warps never wait for an
//              item's last PV nor drain O themselves.
// The warpgroups rebalance registers at the start (setmaxnreg): the
// producers and the epilogue give registers to the softmax warps.
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
constexpr int kBN = 128;        // keys per score tile (N of the score MMAs)
constexpr int kTileAlign = 64;  // score tiles start on multiples of this many keys
constexpr int kStage = 16384;   // bytes per K or V ring stage
constexpr int kKS = 5;          // K ring depth (stages)
constexpr int kVS = 5;          // V ring depth (stages)
constexpr int kThreads = 512;   // 4 warpgroups: producers + MMA, 2 x softmax, epilogue
constexpr int kSoftmaxWarp0 = 4;  // warps 4-11: softmax (two warpgroups)
constexpr int kEpiWarp0 = 12;     // warps 12-15: epilogue (one warpgroup)
// Register split (setmaxnreg) against the launch's 512 x 128: the producer /
// MMA warpgroup and the epilogue warpgroup give back to 80 per thread, the
// two softmax warpgroups grow to 176: 128 x 80 + 128 x 80 + 256 x 176 =
// 65536.
constexpr int kRegsLaunch = 128, kRegsCtl = 80, kRegsEpi = 80, kRegsSoftmax = 176;
static_assert(128 * kRegsCtl + 128 * kRegsEpi + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch's registers");
constexpr int kPolyEvery = 32;  // one pair of exponentials in 32 on the FMA pipe
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait, then give up
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s per drain wait

// The launch's items.  n_ctas > 0: CTA c runs items [cta0[c], cta0[c + 1])
// in order (the plan's per-CTA lists); else CTA c runs c, c + grid, ...
struct ItemList {
  int32_t n;
  int32_t n_ctas;
  // 1: items in longest-first order, taken as CTAs get free: CTA c starts on
  // item c, then takes item gridDim.x + (a work counter in the workspace
  // header, incremented atomically); the last CTA to finish resets it.
  int32_t dyn;
  int32_t cta0[kMaxPrefillGrid + 1];
  PrefillItem items[kMaxItemsPerLaunch];
};

struct ItemRange {
  int32_t begin, end, step;
};

__device__ __forceinline__ ItemRange my_items(const ItemList& items) {
  if (items.n_ctas > 0)
    return ItemRange{items.cta0[blockIdx.x], items.cta0[blockIdx.x + 1], 1};
  return ItemRange{static_cast<int32_t>(blockIdx.x), items.n, static_cast<int32_t>(gridDim.x)};
}

struct PrefillParams {
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  const int32_t* window;
  __nv_bfloat16* out;
  unsigned char* ws;
  int32_t hq, group, qb_tokens, page_size, page_shift, box_rows_k, box_rows_v, mpps, num_pages;
  float scale_log2;
  // Parts of split items (PrefillItem::split != 0): partial O / l and
  // log2-sum-exp per row, in the part's slot.
  float* ppart_o;      // [slot][kBM][D]
  float* ppart_lse;    // [slot][kBM]
  int32_t out_v8;      // `out` is 32-byte aligned: the epilogue stores 32 bytes at once
  int32_t v_4d;        // tm_v is 4-D (chunks outermost): one box per V stage
};

// One 32-byte store (eight 32-bit words) to a 32-byte aligned address.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst),
               "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
               "r"(w[7])
               : "memory");
}

// A score tile's K streams through the K ring one 64-dimension chunk at a
// time (128 keys x 128 B = one stage); its V streams through the V ring
// kVKeys keys at a time (all D dimensions, kVKeys x D x 2 B = one stage).
// Either way a tile is D / 64 stages, and one stage feeds whole MMAs, so the
// tensor core starts on a tile before all of it has landed.
template <int D>
struct Layout {
  static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms per row
  static constexpr int kVKeys = 8192 / D;                // keys per V stage
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kKS * kStage;
  static constexpr int kBarOff = kVOff + kVS * kStage;
  static constexpr int kXchOff = kBarOff + 512;         // softmax pair exchange
  static constexpr int kLOff = kXchOff + 2 * 2 * kBM * 4;   // row sums, softmax -> epilogue
  static constexpr int kUsed = kLOff + kBM * 4;
  // Ask for more than half an SM's shared memory so that exactly one CTA
  // (which owns the SM's tensor memory) is resident per SM.
  static constexpr int kBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  static_assert(kUsed <= 227 * 1024, "more shared memory than one CTA may have");
  // TMEM columns: O (D), then two S buffers of 128; P (bf16 pairs) is
  // written over the first 64 columns of its own S buffer.
  static constexpr int kOCol = 0;
  static constexpr int kSCol = D;
  static constexpr int kCols = 512;                      // D + 256 <= 512
};

struct Geom {
  int32_t seq, g, t0, ntok, pos_first, key_first, ntiles, W;
  int32_t lo;   // first key visible to any query of the item
  bool ok;
};

// An item as the K producer hands it to the other warps: its geometry, its
// split code and whether the stream of items has ended.
struct ItemSlot {
  Geom gm;
  int32_t split;
  int32_t end;
};
constexpr int kItemRing = 3;
// Warps that take each item from the ring: V producer, MMA issuer, eight
// softmax warps, four epilogue warps.
constexpr int kItemReaders = 14;

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[kKS], k_empty[kKS], v_full[kVS], v_empty[kVS];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free;       // the epilogue has read O out of TMEM
  uint64_t l_full, l_empty;  // an item's row sums handed over / taken
  uint64_t fin;          // all MMAs of this CTA complete (teardown)
  uint64_t xbar[4];      // softmax pair exchange, one per TMEM lane quarter
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  ItemSlot item[kItemRing];
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(Barriers) <= 512, "barrier block");


__device__ __forceinline__ Geom item_geom(const PrefillParams& p, const PrefillItem& it) {
  Geom r;
  if (it.seq < 0) {   // padding of an interleaved range list
    r.ok = false;
    r.ntiles = 0;
    return r;
  }
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
  r.lo = klo;
  // Tiles start on a 64-key boundary at or below the first visible key (a
  // 128-key boundary would mask up to 127 keys of a window's first tile).
  r.key_first = klo / kTileAlign * kTileAlign;
  r.ntiles = r.ok ? (pos_last - r.key_first) / kBN + 1 : 0;
  if (it.split != 0) {
    // One part of a split item: tiles [j0, j0 + n) of the item's range.
    const int32_t j0 = split_first(it.split), n = split_tiles(it.split);
    r.key_first += j0 * kBN;
    r.ntiles = max(0, min(n, r.ntiles - j0));
  }
  return r;
}

// Maximum of N floats (stored as bits) as a tree of three-input maxima.
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

// TMA source row of the box of `rows` keys starting at `key` (a box never
// crosses a page; -rows: a box wholly outside the keys the item's queries
// see, past its last query or before its first visible key, which the TMA
// fills with zeros without reading the page table).
__device__ __forceinline__ int32_t box_row(const PrefillParams& p, const Geom& gm, int32_t key,
                                           int32_t rows) {
  const int32_t pos_last = gm.pos_first + gm.ntok - 1;
  if (key > pos_last || key + rows <= gm.lo) return -rows;
  const int32_t page = __ldg(p.page_table + static_cast<int64_t>(gm.seq) * p.mpps +
                             (key >> p.page_shift));
  if (page < 0 || page >= p.num_pages) {
    report_error(p.ws, RPA_DEVERR_PAGE_ID, gm.seq);
    return -rows;
  }
  return page * p.page_size + (key & (p.page_size - 1));
}

// The workspace header's work counter of a dynamic item list: [0] items
// taken beyond the first wave, [1] CTAs finished.  The last CTA to finish
// sets both back to zero for the next launch (every CTA's last take comes
// before its own finish).
__device__ __forceinline__ void leave_item_counter(unsigned char* ws) {
  int32_t* ctr = reinterpret_cast<int32_t*>(ws + kPrefillCounterOff);
  __threadfence();
  if (atomicAdd(&ctr[1], 1) == static_cast<int32_t>(gridDim.x) - 1) {
    atomicExch(&ctr[0], 0);
    atomicExch(&ctr[1], 0);
  }
}

// Zero rows [0, a) and [b, kVKeys) of a V stage ([chunk][kVKeys rows][128 B]),
// then order the stores before the tensor core's reads (whole warp).  Out of
// line: inlined into the MMA warp's stage loop, this rarely taken code cost
// ~3% of the prefill's time.  A key row is D / 64 chunks of 128 bytes,
// kVKeys x 128 B apart; the swizzle permutes 16-byte units inside a row, so
// whole rows are cleared whatever it is.
template <int kVKeys, int kChunks>
__device__ __noinline__ void zero_v_rows(uint8_t* st, int a, int b, int lane) {
  const int nrows = a + (kVKeys - b);
  for (int u = lane; u < nrows * kChunks * 8; u += 32) {
    const int rr = u / (kChunks * 8), rem = u % (kChunks * 8);
    const int row = rr < a ? rr : b + (rr - a);
    *reinterpret_cast<uint4*>(st + (rem >> 3) * (kVKeys * 128) + row * 128 + (rem & 7) * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  // The tensor core reads the stage through the async proxy.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// A warp takes item number R from the ring (every lane waits and reads;
// lane 0 releases the slot).  False when the wait gave up.
__device__ __forceinline__ bool take_item(Barriers& B, uint32_t& R, ItemSlot& e,
                                          volatile int* abort, int lane) {
  const int sl = R % kItemRing;
  const bool ok = mbar_wait(&B.item_full[sl], (R / kItemRing) & 1, abort, kWaitNs);
  if (!__all_sync(0xffffffffu, ok)) return false;
  e = B.item[sl];
  __syncwarp();
  if (lane == 0) mbar_arrive(&B.item_empty[sl]);
  ++R;
  return true;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const PrefillParams p,
                  const __grid_constant__ ItemList items) {
  using Lay = Layout<D>;
  // The 128-byte swizzle needs 1024-byte aligned tiles; the layout fills
  // the shared memory with no slack, so a misaligned base ends the launch.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {
    if (threadIdx.x == 0) {
      report_error(p.ws, RPA_DEVERR_LAUNCH, blockIdx.x);
      if (items.dyn) leave_item_counter(p.ws);
    }
    return;
  }
  // A combine of split items may be scheduled now; it waits for this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint8_t* smem = smem_raw;
  const ItemRange mine = my_items(items);
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
      mbar_init(&B.p_full[i], 256);
      mbar_init(&B.o_done[i], 1);
    }
    mbar_init(&B.o_free, 128);
    mbar_init(&B.l_full, 128);
    mbar_init(&B.l_empty, 128);
    for (int i = 0; i < 4; ++i) mbar_init(&B.xbar[i], 64);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&B.item_full[i], 1);
      mbar_init(&B.item_empty[i], kItemReaders);
    }
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
  // Each warpgroup rebalances its registers at the start of its branch (all
  // four of its warps at the same instruction).
  if (warp < kSoftmaxWarp0) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
  if (warp <= 1) {
    // ------------------------------------------------------------ producers
    // Warp 0 loads Q and K, warp 1 loads V; each keeps its own ring of
    // 16 KB stages, counted by C across tiles and items.
    const bool is_k = warp == 0;
    const int depth = is_k ? kKS : kVS;
    uint64_t* full = is_k ? B.k_full : B.v_full;
    uint64_t* empty = is_k ? B.k_empty : B.v_empty;
    uint8_t* ring = smem + (is_k ? Lay::kKOff : Lay::kVOff);
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    const int rows = is_k ? p.box_rows_k : p.box_rows_v;
    const int nbox = (is_k ? kBN : Lay::kVKeys) / rows;    // boxes per stage (<= 8)
    uint32_t C = 0, I = 0, issued_q = 0, R = 0;
    const uint32_t q_box_bytes = static_cast<uint32_t>(G * p.qb_tokens) * 128u;
    bool alive = true;
    int32_t* ctr = reinterpret_cast<int32_t*>(p.ws + kPrefillCounterOff);
    // K producer: the item after `it` (lane 0).
    auto next_item = [&](int32_t it) -> int32_t {
      if (!items.dyn) return it + mine.step;
      return static_cast<int32_t>(gridDim.x) + atomicAdd(&ctr[0], 1);
    };
    int32_t it = items.dyn ? static_cast<int32_t>(blockIdx.x) : mine.begin;
    const int32_t it_end = items.dyn ? items.n : mine.end;
    for (;;) {
      Geom gm;
      bool end = false;
      if (is_k) {
        // Lane 0 takes the next item with work in it and hands it to the
        // other warps through the ring.
        if (lane == 0) {
          int32_t split = 0;
          for (;;) {
            if (it >= it_end) {
              end = true;
              break;
            }
            gm = item_geom(p, items.items[it]);
            split = items.items[it].split;
            if (gm.ok) break;
            if (items.items[it].seq >= 0) report_error(p.ws, RPA_DEVERR_LENGTHS, gm.seq);
            it = next_item(it);
          }
          const int sl = R % kItemRing;
          alive = mbar_wait(&B.item_empty[sl], ((R / kItemRing) & 1) ^ 1, abort, kWaitNs);
          if (alive) {
            B.item[sl].gm = gm;
            B.item[sl].split = split;
            B.item[sl].end = end ? 1 : 0;
            mbar_arrive(&B.item_full[sl]);
            if (!end) it = next_item(it);
          }
        }
        ++R;
        alive = __shfl_sync(0xffffffffu, alive, 0);
        if (!alive) break;
        __syncwarp();
        // Every lane reads the item back (the copies below need it).
        const ItemSlot e = B.item[(R - 1) % kItemRing];
        gm = e.gm;
        end = e.end != 0;
      } else {
        ItemSlot e;
        if (!(alive = take_item(B, R, e, abort, lane))) break;
        gm = e.gm;
        end = e.end != 0;
      }
      if (end) break;
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
      // Source rows of a tile's boxes (lane < nbox: one box per stage), each
      // a page-table load.  They are read a tile ahead, all at once: read
      // one by one just before their stage, their latency (~600 cycles
      // each) paced the ring at more than the tile's MMA time.
      auto tile_rows = [&](int j, int32_t (&rw)[Lay::kChunks]) {
        const int32_t key0 = gm.key_first + j * kBN;
        if (is_k) {
          // K: the same 128 keys for every chunk of the tile.
          const int32_t kr = lane < nbox ? box_row(p, gm, key0 + lane * rows, rows) : 0;
#pragma unroll
          for (int sgi = 0; sgi < Lay::kChunks; ++sgi) rw[sgi] = kr;
        } else {
#pragma unroll
          for (int sgi = 0; sgi < Lay::kChunks; ++sgi)
            rw[sgi] = lane < nbox ? box_row(p, gm, key0 + sgi * Lay::kVKeys + lane * rows, rows) : 0;
        }
      };
      int32_t rcur[Lay::kChunks], rnext[Lay::kChunks];
      if (gm.ntiles > 0) tile_rows(0, rcur);
      for (int j = 0; j < gm.ntiles && alive; ++j) {
        if (j + 1 < gm.ntiles) tile_rows(j + 1, rnext);
        // Rolled: unrolled, this loop's copies of the three TMA paths made
        // the kernel's code large enough to cost ~4% of its time.
#pragma unroll 1
        for (int sgi = 0; sgi < Lay::kChunks; ++sgi, ++C) {
          const int st = C % depth;
          const uint32_t ph = (C / depth) & 1;
          const int32_t row = rcur[sgi];
          if (lane == 0) alive = mbar_wait(&empty[st], ph ^ 1, abort, kWaitNs);
          alive = __shfl_sync(0xffffffffu, alive, 0);
          if (!alive) break;
          if (lane == 0) mbar_arrive_expect_tx(&full[st], kStage);
          __syncwarp();
          if (lane < nbox) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(ring + st * kStage) + lane * rows * 64;
            if (is_k) {
              tma_load_3d(dst, tm, &full[st], sgi * 64, gm.g, row);
            } else if (p.v_4d) {
              // The stage's keys in one box of every 64-dimension chunk.
              tma_load_4d(dst, tm, &full[st], 0, gm.g, row, 0);
            } else {
              for (int c = 0; c < Lay::kChunks; ++c)
                tma_load_3d(dst + c * Lay::kVKeys * 64, tm, &full[st], c * 64, gm.g, row);
            }
          }
        }
#pragma unroll
        for (int sgi = 0; sgi < Lay::kChunks; ++sgi) rcur[sgi] = rnext[sgi];
      }
      if (!alive) break;
    }
    if (!alive && lane == 0) {
      // Let every copy this warp started land before its shared memory goes.
      report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
      for (uint32_t t = (C > static_cast<uint32_t>(depth) ? C - depth : 0); t < C; ++t) {
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
    // The whole warp walks the schedule and waits; one elected lane issues
    // every MMA and commit (see mma_ss).
    constexpr uint32_t kIdS = idesc_bf16(kBN, 0);
    constexpr uint32_t kIdPV = idesc_bf16(D, 1);
    const uint32_t q_base = smem_addr(q_s), k_base = smem_addr(k_s), v_base = smem_addr(v_s);
    uint32_t T = 0, I = 0, IO = 0;    // tiles, items (with PV)
    // Ring slot and phase of the next K / V stage.
    int ks = 0, vs = 0;
    uint32_t kph = 0, vph = 0;
    // Whether the next K / V stage has landed, as tested (mbar_test) while
    // the current stage's MMAs were issued; false: wait for it.
    bool k_ready = false, v_ready = false;
    // Shared-memory descriptors differ between operands of one kind only in
    // the start-address field (bits 0-13: the byte address / 16), and every
    // operand lies below 256 KB, so the operand at byte offset `off` from a
    // base has the base's descriptor + off / 16.  Built once here: rebuilt
    // for every MMA, their 64-bit arithmetic made this warp's issue, not the
    // tensor core, set the pace of a tile.  (The chunk and stage loops stay
    // rolled: unrolled, the larger code ran the kernel ~20% slower.)
    const uint64_t q_d0 = smem_desc(q_base, 16, 1024);
    const uint64_t k_d0 = smem_desc(k_base, 16, 1024);
    const uint64_t v_d0 = smem_desc(v_base, Lay::kVKeys * 128, 1024);
    bool alive = true;
    // A wait the whole warp agrees on.
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool ok = mbar_wait(bar, parity, abort, kWaitNs);
      return __all_sync(0xffffffffu, ok);
    };
    // O += P(Tp) V(Tp): one V stage (kVKeys keys x D) at a time.  V is the
    // MN-major B operand: 8-key groups 1024 B apart (SBO), 64-dimension
    // chunks kVKeys x 128 B apart (LBO); 16 keys per MMA = 2048 B.  P (A)
    // sits in the first 64 columns of its S buffer, 8 columns per 16 keys.
    //
    // A masked key has P = 0, but 0 x NaN is NaN: the V rows of keys no query
    // of the item sees (before its first visible key, past its last query)
    // may hold anything (free slots of the last page, pages a sliding-window
    // cache has let go), so they are zeroed in the stage before the MMA reads
    // it.  Boxes wholly outside those keys arrive as zeros already; only the
    // stages at the two ends of an item need this.
    auto clear_v_edges = [&](const Geom& gm, int32_t kst, int vs) {
      const int32_t last = gm.pos_first + gm.ntok - 1;
      // Interior stages (every key visible to some query of the item): nothing.
      if (kst >= gm.lo && kst + Lay::kVKeys <= last + 1) return;
      const int a = max(0, min(Lay::kVKeys, gm.lo - kst));        // rows [0, a): before
      const int b = max(0, min(Lay::kVKeys, last + 1 - kst));     // rows [b, kVKeys): past
      if (a == Lay::kVKeys || b == 0) return;   // the whole stage arrived as zeros
      zero_v_rows<Lay::kVKeys, Lay::kChunks>(reinterpret_cast<uint8_t*>(v_s) + vs * kStage, a, b,
                                             lane);
    };
    auto issue_pv = [&](const Geom& gm, uint32_t Tp, int jp) -> bool {
      const int sb = Tp & 1;
      if (!wait(&B.p_full[sb], (Tp >> 1) & 1)) return false;
      if (jp == 0 && !wait(&B.o_free, (IO & 1) ^ 1)) return false;
      const uint32_t p_col = tmem + Lay::kSCol + sb * kBN;
#pragma unroll 1
      for (int sgi = 0; sgi < Lay::kChunks; ++sgi) {
        if (!v_ready && !wait(&B.v_full[vs], vph)) return false;
        clear_v_edges(gm, gm.key_first + jp * kBN + sgi * Lay::kVKeys, vs);
        tc_fence_after();
        const int vcur = vs;
        const uint64_t vd = v_d0 + static_cast<uint64_t>(vs * (kStage >> 4));
        if (++vs == kVS) {
          vs = 0;
          vph ^= 1;
        }
        v_ready = __all_sync(0xffffffffu, mbar_test(&B.v_full[vs], vph));
        // kVKeys / 16 MMAs of 16 keys (P: 8 columns, V: 2048 B = 128
        // descriptor units apart), in pairs; the stage's commit with the last.
        constexpr int kPairs = Lay::kVKeys / 32;
        const uint32_t pc = p_col + sgi * (Lay::kVKeys / 2);
#pragma unroll
        for (int q = 0; q < kPairs - 1; ++q)
          mma_ts2(tmem + Lay::kOCol, pc + 16 * q, pc + 16 * q + 8, vd + 256 * q, vd + 256 * q + 128,
                  kIdPV, (jp > 0 || sgi > 0 || q > 0) ? 1u : 0u);
        mma_ts2_commit(tmem + Lay::kOCol, pc + 16 * (kPairs - 1), pc + 16 * (kPairs - 1) + 8,
                       vd + 256 * (kPairs - 1), vd + 256 * (kPairs - 1) + 128, kIdPV,
                       (jp > 0 || sgi > 0 || kPairs > 1) ? 1u : 0u, &B.v_empty[vcur]);
      }
      mma_commit(&B.o_done[sb]);
      return true;
    };
    // S(Ts) into S buffer (Ts & 1): one K stage (a 64-dimension chunk of 128
    // keys) at a time.  Q and K are K-major with the 128-byte swizzle: 16
    // elements = 32 B inside a chunk; Q's chunks are 16 KB apart.
    auto issue_s = [&](uint32_t Ts) -> bool {
      const uint32_t sc = tmem + Lay::kSCol + (Ts & 1) * kBN;
#pragma unroll 1
      for (int c = 0; c < Lay::kChunks; ++c) {
        if (!k_ready && !wait(&B.k_full[ks], kph)) return false;
        tc_fence_after();
        const int kcur = ks;
        const uint64_t kd = k_d0 + static_cast<uint64_t>(ks * (kStage >> 4));
        if (++ks == kKS) {
          ks = 0;
          kph ^= 1;
        }
        k_ready = __all_sync(0xffffffffu, mbar_test(&B.k_full[ks], kph));
        // Four MMAs of 16 dimensions (32 B = 2 descriptor units apart).
        const uint64_t qd = q_d0 + static_cast<uint64_t>((c * (kBM * 128)) >> 4);
        mma_ss4_commit(sc, qd, qd + 2, qd + 4, qd + 6, kd, kd + 2, kd + 4, kd + 6, kIdS,
                       c > 0 ? 1u : 0u, &B.k_empty[kcur]);
      }
      mma_commit(&B.s_full[Ts & 1]);
      return true;
    };
    uint32_t R = 0;
    for (;;) {
      ItemSlot e;
      if (!(alive = take_item(B, R, e, abort, lane))) break;
      if (e.end) break;
      const Geom gm = e.gm;
      alive = wait(&B.q_full, I & 1);
      if (!alive) break;
      // Order: S(0), then for each j: S(j + 1), PV(j).  S(j + 1) overwrites
      // the buffer holding P(j - 1), which PV(j - 1) (issued before it) read.
      // Q is released once the item's last score tile is issued.
      const int n = gm.ntiles;
      if (n > 0) alive = issue_s(T);
      if (n <= 1) mma_commit(&B.q_empty);
      for (int j = 0; j < n && alive; ++j) {
        if (j + 1 < n) {
          alive = issue_s(T + j + 1);
          if (!alive) break;
          if (j + 2 == n) mma_commit(&B.q_empty);
        }
        alive = issue_pv(gm, T + j, j);
      }
      T += n;
      ++I;
      if (n > 0) ++IO;
      if (!alive) break;
    }
    // Every MMA issued must finish before TMEM is released.
    mma_commit(&B.fin);
    int dummy = 0;
    mbar_wait(&B.fin, 0, &dummy, kDrainNs);
    __syncwarp();
    if (!alive && lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
  }
  // (warp 3: nothing to do)
  } else if (warp < kEpiWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax
    // Two warps per TMEM lane quarter (32 rows): half h takes keys
    // [64h, 64h + 64) of every tile and columns [hD/2, (h+1)D/2) of O.  The
    // pair swaps row maxima every tile (and row sums once per item) through
    // shared memory, paced by the quarter's mbarrier; both then take the
    // same decisions, so O and P stay consistent.
    const int q4 = warp & 3;                            // TMEM lane quarter of this warp
    const int h = (warp - kSoftmaxWarp0) >> 2;          // key / column half
    const int r = 32 * q4 + lane;                       // TMEM lane = row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const int tok = r / G;
    const float c = p.scale_log2;
    float* xch = reinterpret_cast<float*>(smem + Lay::kXchOff);   // [2][2][kBM]
    uint64_t* xbar = &B.xbar[q4];
    uint32_t T = 0, X = 0, L = 0;                       // tiles, exchanges, items handed over
    bool alive = true;
    // Publish v for this row, wait for the partner's, return it.
    auto swap = [&](float v) -> float {
      xch[((X & 1) * 2 + h) * kBM + r] = v;
      tc_fence_before();                // this warp's TMEM reads come first
      mbar_arrive(xbar);
      const bool ok = mbar_wait(xbar, X & 1, abort, kWaitNs);
      tc_fence_after();
      const float o = xch[((X & 1) * 2 + (h ^ 1)) * kBM + r];
      ++X;
      if (!ok) alive = false;
      return o;
    };
    uint32_t R = 0;
    while (alive) {
      ItemSlot e;
      if (!take_item(B, R, e, abort, lane)) {
        alive = false;
        break;
      }
      if (e.end) break;
      const Geom gm = e.gm;
      const bool valid = tok < gm.ntok && r < G * p.qb_tokens;
      const int32_t pos = gm.pos_first + tok;
      const int32_t lo = first_visible(pos, gm.W);
      float m_ref = -INFINITY, l = 0.f;                 // l: this half's sum
      for (int j = 0; j < gm.ntiles; ++j, ++T) {
        const int sb = T & 1;          // S buffer (P is written over it)
        if (!mbar_wait(&B.s_full[sb], (T >> 1) & 1, abort, kWaitNs)) {
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
        // Interior halves (every key visible to every row of the warp) skip
        // the per-element mask; elsewhere masked scores become -inf.
        const bool full = __all_sync(0xffffffffu, valid && key0 >= lo && key0 + 63 <= pos);
        if (!full) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc) {
            const int32_t key = key0 + cc;
            const bool vis = valid && key >= lo && key <= pos;
            if (!vis) sr[cc] = 0xff800000u;   // -inf
          }
        }
        float mx = max_tree<64>(sr);
        mx = fmaxf(mx, swap(mx));
        if (!alive) break;
        // Scaling after the max keeps the order (c >= 0).
        mx = (mx == -INFINITY) ? -INFINITY : mx * c;
        const float m_new = fmaxf(m_ref, mx);
        const bool grow = m_new > m_ref + 8.f;           // also true for the first visible key
        const bool rescale_o = grow && m_ref != -INFINITY;
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O holds earlier tiles: wait for the last PV, then scale this
          // half's columns in TMEM.
          const uint32_t Tp = T - 1;
          if (!mbar_wait(&B.o_done[Tp & 1], (Tp >> 1) & 1, abort, kWaitNs)) {
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
        // P for this half's 64 keys: 32 packed columns over the S buffer's
        // columns [32h, 32h + 32), scores of half 0 that both halves have
        // read before the exchange above.
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
        mbar_arrive(&B.p_full[sb]);
      }
      if (!alive) break;
      if (gm.ntiles == 0) {
        // An empty part still tells the combine that it holds nothing.
        if (e.split != 0 && h == 0 && valid)
          p.ppart_lse[static_cast<int64_t>(split_slot(e.split)) * kBM + r] = -INFINITY;
        continue;
      }
      // The row sum over both halves; then the first half hands it to the
      // epilogue warps (one slot, taken before the next item's sums come)
      // and writes a split part's log2-sum-exp.
      l += swap(l);
      if (!alive) break;
      if (h == 0) {
        if (e.split != 0 && valid)
          p.ppart_lse[static_cast<int64_t>(split_slot(e.split)) * kBM + r] =
              (l > 0.f) ? m_ref + __log2f(l) : -INFINITY;
        if (!mbar_wait(&B.l_empty, (L & 1) ^ 1, abort, kWaitNs)) {
          alive = false;
          break;
        }
        reinterpret_cast<float*>(smem + Lay::kLOff)[r] = l;
        mbar_arrive(&B.l_full);
      }
      ++L;
    }
    if (!alive && lane == 0) report_error(p.ws, RPA_DEVERR_TIMEOUT, blockIdx.x);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    // ------------------------------------------------------------ epilogue
    // One thread per row (TMEM lane).  Per item with key tiles: take the row
    // sums from the softmax warps, wait for the item's last PV, then O / l
    // -> bf16 -> out (or fp32 O / l into a split part's slot) and free O for
    // the next item's first PV.  Meanwhile the softmax warps already work on
    // the next item's first score tile.
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const int tok = r / G, head = r % G;
    const float* l_s = reinterpret_cast<const float*>(smem + Lay::kLOff);
    uint32_t T = 0, L = 0;                              // tiles, items taken over
    bool alive = true;
    uint32_t R = 0;
    while (alive) {
      ItemSlot e;
      if (!take_item(B, R, e, abort, lane)) {
        alive = false;
        break;
      }
      if (e.end) break;
      const Geom gm = e.gm;
      if (gm.ntiles == 0) continue;
      T += gm.ntiles;
      const uint32_t Tl = T - 1;
      const bool valid = tok < gm.ntok && r < G * p.qb_tokens;
      if (!mbar_wait(&B.l_full, L & 1, abort, kWaitNs)) {
        alive = false;
        break;
      }
      const float l = l_s[r];
      mbar_arrive(&B.l_empty);
      ++L;
      if (!mbar_wait(&B.o_done[Tl & 1], (Tl >> 1) & 1, abort, kWaitNs)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      if (e.split != 0) {
        // A part of a split item: fp32 O / l (a row with no visible key
        // here: zeros; its log2-sum-exp, -inf, came from the softmax warps).
        float* prow = p.ppart_o + (static_cast<int64_t>(split_slot(e.split)) * kBM + r) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_addr + Lay::kOCol + c0, o);
          tmem_wait_ld();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(prow + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                                   __uint_as_float(o[4 * q + 2]) * inv,
                                   __uint_as_float(o[4 * q + 3]) * inv);
          }
        }
      } else {
        __nv_bfloat16* orow =
            p.out + (static_cast<int64_t>(gm.t0 + tok) * p.hq + gm.g * G + head) * D;
        // Each thread writes 32 bytes of its own row per 16 columns (one
        // store when `out` is 32-byte aligned, else two), while the next 16
        // columns load from TMEM.
        auto store16 = [&](const uint32_t (&o)[16], int col) {
          if (!valid) return;
          uint32_t w[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            w[q] = pack_bf16x2(__uint_as_float(o[2 * q]) * inv, __uint_as_float(o[2 * q + 1]) * inv);
          if (p.out_v8) {
            st_global_v8(orow + col, w);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + col);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        };
        uint32_t oa[16], ob[16];
        tmem_ld16(lane_addr + Lay::kOCol, oa);
        tmem_wait_ld();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          tmem_ld16(lane_addr + Lay::kOCol + c0 + 16, ob);
          store16(oa, c0);
          tmem_wait_ld();
          if (c0 + 32 < D) tmem_ld16(lane_addr + Lay::kOCol + c0 + 32, oa);
          store16(ob, c0 + 16);
          tmem_wait_ld();
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
  if (threadIdx.x == 0 && items.dyn) leave_item_counter(p.ws);
}

struct SplitList {
  int32_t n;
  PrefillSplit g[kMaxSplitGroupsPerLaunch];
};

// Merge the parts of each split item: for every row of the item's query
// block, out = sum_k 2^(lse_k - M) O_k / sum_k 2^(lse_k - M) with M the
// largest lse_k, rounded to bf16.  Grid (items, rows / 8), one warp per row:
// the lanes read the parts' log2-sum-exps together, then every part's row
// loads are issued before they are summed.
template <int D>
__global__ void __launch_bounds__(256)
prefill_combine_kernel(const PrefillParams p, const __grid_constant__ SplitList gl) {
  constexpr int E = D / 32;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (static_cast<int>(blockIdx.x) >= gl.n) return;
  const PrefillSplit g = gl.g[blockIdx.x];
  const int G = p.group;
  const int32_t kvh = g.qb_head & 255, qb = g.qb_head >> 8;
  const int32_t q0 = __ldg(p.cu_q_lens + g.seq);
  const int32_t ql = __ldg(p.cu_q_lens + g.seq + 1) - q0;
  const int32_t ntok = min(p.qb_tokens, ql - qb * p.qb_tokens);
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= ntok * G) return;
  // Largest log2-sum-exp over the parts (lane k reads parts k, k + 32, ...).
  float M = -INFINITY;
  for (int k = lane; k < g.nparts; k += 32)
    M = fmaxf(M, p.ppart_lse[static_cast<int64_t>(g.slot0 + k) * kBM + r]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[E], wsum = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int k0 = 0; k0 < g.nparts; k0 += 32) {
    const int nk = min(32, g.nparts - k0);
    const float lse_l = lane < nk ? p.ppart_lse[static_cast<int64_t>(g.slot0 + k0 + lane) * kBM + r]
                                  : -INFINITY;
    const float w_l = lse_l == -INFINITY ? 0.f : fast_exp2(lse_l - M);
    for (int k = 0; k < nk; ++k) {
      const float w = __shfl_sync(0xffffffffu, w_l, k);
      wsum += w;
      const float* src = p.ppart_o + (static_cast<int64_t>(g.slot0 + k0 + k) * kBM + r) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + e);
        acc[e] = fmaf(w, v.x, acc[e]);
        acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
        acc[e + 2] = fmaf(w, v.z, acc[e + 2]);
        acc[e + 3] = fmaf(w, v.w, acc[e + 3]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int tok = r / G, head = r % G;
  __nv_bfloat16* dst = p.out +
      (static_cast<int64_t>(q0 + qb * p.qb_tokens + tok) * p.hq + kvh * G + head) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
}

template <int D>
int launch_prefill_combine(const Plan& plan, const PrefillParams& p, cudaStream_t stream) {
  SplitList& gl = thread_staging<SplitList>();  // copied into the launch parameters
  const int n = static_cast<int>(plan.psplit.size());
  for (int off = 0; off < n; off += kMaxSplitGroupsPerLaunch) {
    gl.n = std::min(kMaxSplitGroupsPerLaunch, n - off);
    for (int i = 0; i < gl.n; ++i) gl.g[i] = plan.psplit[off + i];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gl.n, kBM / 8);   // 8 rows (warps) per CTA
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_combine_kernel<D>, p, gl);
    if (e != cudaSuccess) return static_cast<int>(e);
    trace_mark(RPA_KERNEL_PREFILL_COMBINE, stream);
  }
  return 0;
}

template <int D>
int launch_prefill_t(const Plan& plan, const Args& a, cudaStream_t stream) {
  using Lay = Layout<D>;
  if (int e = ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_tc_kernel<D>), Lay::kBytes))
    return e;
  const int G = plan.hq / plan.hkv;
  const int qb = plan.q_block;
  const int box_rows_k = std::min(plan.p, kTileAlign);   // boxes never cross a page
  const int box_rows_v = std::min(std::min(plan.p, Lay::kVKeys), kTileAlign);
  CUtensorMap tq, tk, tv;
  // A V stage that is one box high (its kVKeys keys in one page) takes all
  // its 64-dimension chunks in one 4-D box ([chunk][key][128 B], the stage's
  // layout); otherwise one 3-D box per chunk and per page.
  const uint64_t pool_rows = static_cast<uint64_t>(plan.num_pages) * plan.p;
  const bool v_4d = Lay::kChunks > 1 && box_rows_v == Lay::kVKeys;
  if (!make_tmap_3d(&tq, a.q, D, plan.hq, static_cast<uint64_t>(plan.total_q), G, qb) ||
      !make_tmap_3d(&tk, a.k_pages, D, plan.hkv, pool_rows, 1, box_rows_k) ||
      !(v_4d ? make_tmap_4d_chunks(&tv, a.v_pages, D, plan.hkv, pool_rows, 1, box_rows_v, false)
             : make_tmap_3d(&tv, a.v_pages, D, plan.hkv, pool_rows, 1, box_rows_v)))
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
  p.box_rows_k = box_rows_k;
  p.box_rows_v = box_rows_v;
  p.v_4d = v_4d ? 1 : 0;
  p.mpps = plan.mpps;
  p.num_pages = plan.num_pages;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0 ? 1 : 0;
  p.ppart_o = reinterpret_cast<float*>(a.workspace + plan.off_ppart_o);
  p.ppart_lse = reinterpret_cast<float*>(a.workspace + plan.off_ppart_lse);
  ItemList& list = thread_staging<ItemList>();  // copied into the launch parameters
  const size_t n = plan.items.size();
  for (size_t off = 0; off < n; off += kMaxItemsPerLaunch) {
    const int cnt = static_cast<int>(std::min<size_t>(kMaxItemsPerLaunch, n - off));
    list.n = cnt;
    for (int i = 0; i < cnt; ++i) list.items[i] = plan.items[off + i];
    int grid = std::min(cnt, plan.prefill_ctas);
    list.n_ctas = 0;
    list.dyn = plan.prefill_dynamic ? 1 : 0;
    if (plan.prefill_dynamic && (off != 0 || cnt != static_cast<int>(n)))
      return static_cast<int>(cudaErrorInvalidValue);
    if (!plan.pcta0.empty()) {
      // Per-CTA lists (the plan keeps them to one launch).
      if (off != 0 || plan.pcta0.back() != cnt ||
          static_cast<int>(plan.pcta0.size()) - 1 > kMaxPrefillGrid)
        return static_cast<int>(cudaErrorInvalidValue);
      grid = static_cast<int>(plan.pcta0.size()) - 1;
      list.n_ctas = grid;
      for (int c = 0; c <= grid; ++c) list.cta0[c] = plan.pcta0[c];
    }
    prefill_tc_kernel<D><<<grid, kThreads, Lay::kBytes, stream>>>(tq, tk, tv, p, list);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return static_cast<int>(e);
    trace_mark(RPA_KERNEL_PREFILL_TC, stream);
  }
  if (!plan.psplit.empty()) return launch_prefill_combine<D>(plan, p, stream);
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
