// Internal declarations shared by the host API, the scheduler and the kernel
// launchers of librpa.  Not part of the public interface (include/rpa.h).
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>
#include <memory>
#include <vector>

#include "rpa.h"

#ifdef __CUDACC__
#define RPA_HD __host__ __device__
#else
#define RPA_HD
#endif

namespace rpa {

// Workspace layout: a 256-byte header (error word first), then the decode
// split partials.  Offsets are multiples of 256 bytes.
constexpr size_t kHeaderBytes = 256;
// Offset in the header of the dynamic prefill item counter (two int32: items
// taken, CTAs finished), zero between launches.
constexpr size_t kPrefillCounterOff = 64;

// One prefill work item: query block `qb` (of plan.q_block tokens) of
// sequence `seq`, for KV head `head`.  Ordered longest first in the plan.
struct PrefillItem {
  int32_t seq;
  int32_t qb_head;  // (query block index << 8) | kv head
  // 0: every key tile of the item.  Else one part of an item whose key
  // tiles the plan split across CTAs: (slot << 21) | (first tile << 10) |
  // tile count, as unsigned bits; the part leaves an fp32 partial in `slot`
  // and a combine merges the parts.  seq < 0: padding, skipped.
  int32_t split;
};
constexpr int kSplitMaxSlots = 2048, kSplitMaxFirst = 2048, kSplitMaxTiles = 1023;
RPA_HD constexpr int32_t split_code(int32_t slot, int32_t j0, int32_t n) {
  return static_cast<int32_t>((static_cast<uint32_t>(slot) << 21) |
                              (static_cast<uint32_t>(j0) << 10) | static_cast<uint32_t>(n));
}
RPA_HD constexpr int32_t split_slot(int32_t c) {
  return static_cast<int32_t>(static_cast<uint32_t>(c) >> 21);
}
RPA_HD constexpr int32_t split_first(int32_t c) {
  return static_cast<int32_t>((static_cast<uint32_t>(c) >> 10) & 2047u);
}
RPA_HD constexpr int32_t split_tiles(int32_t c) {
  return static_cast<int32_t>(static_cast<uint32_t>(c) & 1023u);
}

// Most work items one tensor-core prefill launch carries in its parameters;
// longer lists are split over several launches.
constexpr int kMaxItemsPerLaunch = 2048;

// Score tiles of the tensor-core prefill: 128 keys, starting on multiples of
// 64 keys at or below the first visible key.
constexpr int kPrefillTileKeys = 128;
constexpr int kPrefillTileAlign = 64;

// An item split into parts: its partial slots are [slot0, slot0 + nparts).
struct PrefillSplit {
  int32_t seq, qb_head, slot0, nparts;
};
constexpr int kMaxSplitGroupsPerLaunch = 1024;
// Largest persistent prefill grid whose per-CTA item lists the launch
// parameters carry.
constexpr int kMaxPrefillGrid = 256;

// Decode schedule limits: segments one decode launch carries in its
// parameters (two sizes), and segments / pages one decode CTA's range may
// touch (their tables sit in shared memory).
constexpr int kDecodeSegSmall = 256;
constexpr int kDecodeSegLarge = 1024;
constexpr int kMaxCtaSegs = 64;
constexpr int kMaxCtaPages = 512;
// Most CTAs a cost-balanced decode launch lists (their range starts travel in
// the launch parameters), and the charge, in 16-key blocks, for each segment
// a CTA's range touches (its in-CTA merge and output).
constexpr int kMaxDecodeCtas = 1024;
// Largest decode grid the plan's per-CTA range table describes (one wave:
// at most one CTA per SM).
constexpr int kMaxDecodeGrid = 512;
constexpr int kDecodeSegCost = 7;

struct Plan {
  // Problem description (checked against every rpa_forward call).
  int32_t num_seqs = 0, hq = 0, hkv = 0, d = 0, p = 0, mpps = 0, num_pages = 0;
  int32_t dtype = RPA_DTYPE_BF16;
  bool kv_fp8 = false;               // K/V pages are e4m3 bytes (decode only)
  bool has_window = false;
  int64_t total_q = 0;

  int32_t path = RPA_PATH_SIMT;     // path actually used
  bool simt_decode = false;          // decode sequences handled by the SIMT kernel
  bool simt_prefill = false;         // prefill sequences handled by the SIMT kernel
  bool decode_tc = false;            // split-KV decode on the tensor-core kernel
  int32_t num_sms = 152;
  // Mixed batches (decode and tensor-core prefill work in one call): the two
  // persistent grids run side by side on disjoint SMs, decode on
  // decode_sms of them and prefill on prefill_sms (forked onto a second
  // stream and joined back); 0: each grid takes every SM, one after the other.
  bool overlap = false;
  int32_t decode_sms = 0, prefill_sms = 0;
  // The planner's cost estimates (microseconds) behind that choice.
  float est_decode_us = 0.f, est_prefill_us = 0.f;

  // Decode (q_len == 1) on the split-KV kernel.  Segments = (sequence, KV
  // head) pairs in stream order; blocks are 16 keys; each launch cuts its
  // segments' block stream into contiguous ranges, one per CTA: ranges of
  // equal cost (blocks plus a fixed charge per segment touched), listed in
  // dcta_blk0, or, where bpc > 0, ranges of bpc blocks each.
  struct DecodeLaunch {
    int32_t seg_begin, seg_end;  // segments [seg_begin, seg_end)
    int32_t bpc;                 // > 0: blocks per CTA (uniform ranges)
    int32_t n_ctas;
    int32_t slot_base;           // first partial slot (two per CTA)
    int32_t cta_begin;           // bpc == 0: ranges in dcta_blk0[cta_begin ...]
    int32_t cut_begin, n_cut;    // segments cut across CTAs: dcut[cut_begin ...]
  };
  // A segment cut across CTAs ca .. ca + nparts - 1 of its launch: CTA ca
  // holds its partial in slot 2 ca + first (first = 1 when the segment is
  // not the first of ca's range), every later CTA c in slot 2 c.
  struct DecodeCut {
    int32_t ca, first, nparts, q0, g;
  };
  int32_t num_decode = 0;
  int32_t kv_split = 0;   // tokens of the longest CTA range of the first launch
  int32_t max_splits = 0; // most CTAs any segment is cut across
  int64_t decode_ctas = 0;
  std::vector<int32_t> dseg_seqhead;  // (sequence << 8) | kv head
  std::vector<int32_t> dseg_blk0;     // block prefix, size segments + 1
  std::vector<int32_t> dseg_q0, dseg_lo, dseg_len;  // query token, first visible key, length
  std::vector<DecodeLaunch> dlaunch;
  std::vector<int32_t> dcta_blk0;     // per launch: n_ctas + 1 range starts (launch-relative)
  std::vector<DecodeCut> dcut;
  int32_t dec_slots = 0;              // partial slots over all launches

  // Prefill (q_len > 1).
  int32_t num_prefill = 0;
  int32_t q_block = 0;
  bool prefill_pairs = false;      // items are pairs of query blocks (SM-pair kernel)
  // Items in longest-first order, each taken by the next CTA to get free
  // (else CTA c runs its own list, pcta0).
  bool prefill_dynamic = false;
  int32_t prefill_groups = 0;         // groups of the dynamic prefill list
  std::vector<PrefillItem> items;  // longest first, or per-CTA lists (pcta0)
  // Per-CTA item lists: CTA c runs items [pcta0[c], pcta0[c + 1]) in order;
  // empty: CTA c runs items c, c + grid, ... (a list too long for one launch).
  std::vector<int32_t> pcta0;
  int32_t prefill_max_tiles = 0;    // key tiles of the busiest CTA
  std::vector<PrefillSplit> psplit; // items split across CTAs (combined afterwards)
  int32_t n_split_items = 0;        // partial slots (parts of split items)
  int32_t prefill_ctas = 0;

  // Workspace.
  size_t off_partial_o = 0, off_partial_lse = 0, ws_bytes = kHeaderBytes;
  size_t off_ppart_o = 0, off_ppart_lse = 0;   // prefill parts: [slot][128 rows][D], [slot][128]
};

// Scheduler (plan.cpp): fills everything but the problem description, which
// the caller has set and validated.
rpa_status_t build_schedule(Plan& plan, const int32_t* cu_q_lens, const int32_t* kv_lens,
                            const int32_t* window, const rpa_plan_options& opts);

// Host-side checks of the metadata (plan.cpp).
rpa_status_t validate_metadata(const int32_t* cu_q_lens, const int32_t* kv_lens,
                               int32_t num_seqs, int32_t page_size,
                               int32_t max_pages_per_seq);

// Arguments every kernel launcher receives.
struct Args {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  const int32_t* window;
  float sm_scale;
  void* out;
  unsigned char* workspace;
  const float* k_scale = nullptr;  // fp8 pages: per-KV-head scales of K and V
  const float* v_scale = nullptr;
};

// Kernel launchers; each returns cudaError_t as int (0 = success).
int launch_simt(const Plan& plan, const Args& a, void* stream);
int launch_decode(const Plan& plan, const Args& a, void* stream);
int launch_prefill_tc(const Plan& plan, const Args& a, void* stream);
int launch_prefill_pair(const Plan& plan, const Args& a, void* stream);

// KV-cache write of a step's new tokens (kv_write.cu).
struct KvWriteArgs {
  const void* k_new;
  const void* v_new;
  void* k_pages;
  void* v_pages;
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  unsigned char* workspace;  // error word, or null
  int32_t num_seqs, total_q, hkv, head_dim, elem_bytes, page_size, mpps, num_pages;
};
int launch_kv_write(const KvWriteArgs& a, void* stream);

// The q/k/v prologue (prologue.cu): q/k RMS norm + rotary embedding, v norm,
// q to q_out and k/v into their pages.
struct PrologueArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* q_weight;  // null: no norm
  const float* k_weight;
  const float* v_weight;
  float eps, rope_theta;  // rope_theta <= 0: no rotation
  void* q_out;
  void* k_pages;
  void* v_pages;
  const int32_t* page_table;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  unsigned char* workspace;  // error word, or null
  int32_t num_seqs, total_q, hq, hkv, head_dim, elem_bytes, page_size, mpps, num_pages;
};
bool prologue_supported(int32_t head_dim);
int launch_prologue(const PrologueArgs& a, void* stream);

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); thread-safe.  Returns a cudaError_t.
int ensure_dynamic_smem(const void* kernel, int bytes);

// Per-thread host staging for a launch's parameter block (large structs that
// are filled, then copied into the launch): one heap copy per thread, freed
// when the thread exits.
template <typename T>
T& thread_staging() {
  static thread_local std::unique_ptr<T> buf;
  if (!buf) buf.reset(new T());
  return *buf;
}

// Tracing hooks (trace.cpp): trace_start before a call's first launch,
// trace_mark after each launch (no-ops unless tracing is on).
void trace_start(void* stream);
void trace_mark(int kernel, void* stream);

// Whether the tensor-core prefill supports this shape (prefill_tc.cu).
bool prefill_tc_supported(int32_t head_dim, int32_t page_size, int32_t group);
// Whether the SM-pair prefill supports this shape (prefill_pair.cu).
bool prefill_pair_supported(int32_t head_dim, int32_t page_size, int32_t group);
// Device address of the fixed no-allocation scratch array on the current
// device (decode.cu); resolved on the first call per device.
int noalloc_scratch(void** ptr);

// Whether the split-KV decode supports this shape (decode.cu).
bool decode_supported(int32_t head_dim, int32_t group, int32_t page_size);
// Whether its tensor-core kernel does (decode_tc.cu), and that kernel's
// launcher (launch_decode hands over to it when plan.decode_tc is set).
bool decode_tc_supported(int32_t head_dim, int32_t group, int32_t page_size, bool kv_fp8);
int launch_decode_tc(const Plan& plan, const Args& a, void* stream);

// TMA tensor maps (tmap.cpp): a 3-D bf16 tensor [outer][mid][d] with a
// 128-byte-swizzled box of (64, box_mid, box_outer) elements.
bool tmap_available();
bool make_tmap_3d(CUtensorMap* m, const void* base, uint64_t d, uint64_t mid, uint64_t outer,
                  uint32_t box_mid, uint32_t box_outer);
// The same tensor as 4-D (64-element chunks outermost): one box brings every
// chunk of box_outer rows, landing as [chunk][row][128 B] (bytes for fp8).
bool make_tmap_4d_chunks(CUtensorMap* m, const void* base, uint64_t d, uint64_t mid,
                         uint64_t outer, uint32_t box_mid, uint32_t box_outer, bool fp8);
// The same over a byte tensor (fp8 pages), box (128, box_mid, box_outer).
bool make_tmap_3d_u8(CUtensorMap* m, const void* base, uint64_t d, uint64_t mid, uint64_t outer,
                     uint32_t box_mid, uint32_t box_outer);

}  // namespace rpa
