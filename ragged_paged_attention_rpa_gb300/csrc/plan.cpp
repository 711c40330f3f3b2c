// The scheduler: maps a ragged batch onto the GPU kernels.  Host only.
//
// Sources (page titles and sections):
//  * "TPU Deep Dive" slides, chapter 8, "Continuous batching with static
//    shapes": one step holds decoding and prefilling sequences together, and
//    ragged paged attention runs decode, prefill and mixed work from one
//    flattened batch.  Here every sequence with q_len == 1 is decode work for
//    the split-KV kernel, every sequence with q_len > 1 is prefill work.
//  * "Pallas kernel / vLLM on TPU ... 19,511 tokens per second", section
//    "Strategy 7": a fixed 2048-token KV block left ~93% of each decode block
//    as masked padding when contexts averaged ~140 tokens, and block size only
//    changes scheduling, never the result.  So the decode split length is
//    chosen per batch from the real lengths, never past a sequence's end.
//  * "Chasing speed of light on TPU v6e", section "Attention" and footnote 6:
//    each key is read once per query block that wants it, so the query block
//    grows with the head-group ratio (the MMA rows are q-block x group).
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdint>
#include <functional>
#include <numeric>
#include <queue>
#include <vector>

#include "rpa_internal.h"

namespace rpa {

int prefill_ctas_per_sm(int32_t head_dim);  // prefill_tc.cu
int prefill_tokens_per_block(int32_t head_dim, int32_t group);  // prefill_tc.cu

rpa_status_t validate_metadata(const int32_t* cu, const int32_t* kv, int32_t num_seqs,
                               int32_t page_size, int32_t max_pages_per_seq) {
  if (cu[0] != 0) return RPA_ERR_INVALID_ARG;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int64_t ql = static_cast<int64_t>(cu[s + 1]) - cu[s];
    if (ql < 0 || kv[s] < 0 || kv[s] < ql) return RPA_ERR_INVALID_ARG;
    int64_t pages = (static_cast<int64_t>(kv[s]) + page_size - 1) / page_size;
    if (pages > max_pages_per_seq) return RPA_ERR_INVALID_ARG;
  }
  return RPA_OK;
}

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Visible keys of the decode query of a sequence: [lo, L).
inline int64_t decode_visible(int32_t L, int32_t w) {
  int64_t lo = (w > 0 && L - w > 0) ? L - w : 0;
  return L - lo;
}

// Decode schedule: the visible keys of every (decode sequence, KV head) pair
// form a segment of 16-key blocks; the blocks of all segments are laid end to
// end and cut into contiguous ranges, one per CTA (at most one per SM: a
// single wave).  A range costs its blocks plus kDecodeSegCost for every
// segment it touches (each segment ends in a merge of the CTA's warps and a
// write); the cut makes the largest cost as small as the SM count allows, so
// CTAs that touch many short sequences get fewer blocks.  A range also ends
// where it would touch more segments or pages than the kernel's
// shared-memory tables hold.  A forced range size (options) gives ranges of
// equal block counts instead.
void plan_decode(Plan& plan, const int32_t* cu, const int32_t* kv, const int32_t* win,
                 int32_t forced_tokens) {
  plan.dseg_seqhead.clear();
  plan.dseg_blk0.assign(1, 0);
  plan.dseg_q0.clear();
  plan.dseg_lo.clear();
  plan.dseg_len.clear();
  plan.dlaunch.clear();
  plan.dcta_blk0.clear();
  plan.dcut.clear();
  std::vector<int32_t> seg_lo;  // first block's first key of each segment
  int32_t ndec = 0;
  for (int32_t s = 0; s < plan.num_seqs; ++s) {
    if (cu[s + 1] - cu[s] != 1) continue;
    ++ndec;
    const int32_t w = win ? win[s] : 0;
    const int32_t lo = (w > 0 && kv[s] - w > 0) ? kv[s] - w : 0;
    // Blocks sit on absolute 16-key boundaries (keys before lo are masked),
    // so with pages of 16 or more tokens a block never straddles two pages.
    const int32_t nb = static_cast<int32_t>(ceil_div(kv[s], 16) - lo / 16);
    for (int32_t g = 0; g < plan.hkv; ++g) {
      plan.dseg_seqhead.push_back((s << 8) | g);
      plan.dseg_blk0.push_back(plan.dseg_blk0.back() + nb);
      plan.dseg_q0.push_back(cu[s]);
      plan.dseg_lo.push_back(lo);
      plan.dseg_len.push_back(kv[s]);
      seg_lo.push_back(lo / 16 * 16);
    }
  }
  plan.num_decode = ndec;
  const int32_t nseg = static_cast<int32_t>(plan.dseg_seqhead.size());
  if (nseg == 0) return;
  const std::vector<int32_t>& blk0 = plan.dseg_blk0;
  const int32_t dec_sms = plan.decode_sms > 0 ? plan.decode_sms : plan.num_sms;
  const int32_t P = plan.p;
  int32_t pshift = 0;                      // page sizes are powers of two
  while ((1 << pshift) < P) ++pshift;
  // Pages holding local blocks [jb, jb + t) of segment k.
  auto pages_of = [&](int32_t k, int32_t jb, int32_t t) {
    const int64_t kb = seg_lo[k] + 16 * static_cast<int64_t>(jb);
    const int64_t ke = seg_lo[k] + 16 * static_cast<int64_t>(jb + t);
    return static_cast<int32_t>(((ke - 1) >> pshift) - (kb >> pshift) + 1);
  };
  // Segments and pages touched by CTA range [b0, b1) of launch segments [sb, se).
  auto fits = [&](int32_t sb, int32_t se, int32_t bpc) {
    const int32_t base = blk0[sb], total = blk0[se] - base;
    int32_t k = sb;
    for (int32_t b0 = 0; b0 < total; b0 += bpc) {
      const int32_t b1 = std::min(total, b0 + bpc);
      while (blk0[k + 1] - base <= b0) ++k;
      int32_t segs = 0, pages = 0;
      for (int32_t kk = k; kk < se && blk0[kk] - base < b1; ++kk) {
        ++segs;
        const int32_t jb = std::max(b0, blk0[kk] - base) - (blk0[kk] - base);
        const int32_t je = std::min(b1, blk0[kk + 1] - base) - (blk0[kk] - base);
        pages += pages_of(kk, jb, je - jb);
      }
      if (segs > kMaxCtaSegs || pages > kMaxCtaPages) return false;
    }
    return true;
  };
  // Greedy cut of launch segments [sb, se) into ranges of cost <= T (each
  // range takes at least one block); returns the range starts (launch-relative,
  // closing entry = total), or stops early once more than `cap` ranges.
  auto cut = [&](int32_t sb, int32_t se, int64_t T, int32_t cap, std::vector<int32_t>& starts) {
    const int32_t base = blk0[sb], total = blk0[se] - base;
    starts.assign(1, 0);
    int32_t b = 0, k = sb;
    while (b < total) {
      if (static_cast<int32_t>(starts.size()) > cap) return;
      int64_t cost = 0;
      int32_t segs = 0, pages = 0;
      bool first = true;
      while (b < total) {
        while (blk0[k + 1] - base <= b) ++k;
        const int32_t jb = b - (blk0[k] - base);
        const int32_t rem = blk0[k + 1] - base - b;
        if (segs == kMaxCtaSegs) break;
        int64_t t = std::min<int64_t>(rem, T - cost - kDecodeSegCost);
        if (t <= 0) {
          if (!first) break;
          t = 1;
        }
        // Largest t whose pages still fit.
        const int32_t room = kMaxCtaPages - pages;
        if (pages_of(k, jb, static_cast<int32_t>(t)) > room) {
          const int64_t kb = seg_lo[k] + 16 * static_cast<int64_t>(jb);
          const int64_t tmax = ((((kb >> pshift) + room) << pshift) - kb) / 16;
          if (tmax <= 0 && !first) break;
          t = std::max<int64_t>(1, std::min(t, tmax));
        }
        cost += kDecodeSegCost + t;
        ++segs;
        pages += pages_of(k, jb, static_cast<int32_t>(t));
        b += static_cast<int32_t>(t);
        first = false;
        if (t < rem) break;  // the range ends inside this segment
      }
      starts.push_back(b);
    }
  };
  int32_t slot_base = 0;
  int64_t max_splits = 1, ctas = 0;
  std::vector<int32_t> starts;
  for (int32_t sb = 0; sb < nseg; sb += kDecodeSegLarge) {
    const int32_t se = std::min(nseg, sb + kDecodeSegLarge);
    const int32_t total = blk0[se] - blk0[sb];
    const int32_t base = blk0[sb];
    Plan::DecodeLaunch dl{sb, se, 0, 0, slot_base, 0, 0, 0};
    bool uniform = forced_tokens > 0;
    if (!uniform) {
      const int32_t cap = std::min<int32_t>(dec_sms, kMaxDecodeGrid);
      const int64_t segs = se - sb;
      // Bounds on the smallest feasible cap T: every segment costs at least
      // once, so cap ranges need T >= (blocks + cost x segments) / cap; and a
      // range the greedy cut closes costs at least T - cost, while the ranges
      // together cost at most blocks + cost x (segments + cap), so T at that
      // sum / (cap - 1) + cost + 1 needs no more than cap ranges (the table
      // limits aside, which the check below covers).
      int64_t lo = std::max<int64_t>(kDecodeSegCost + 1,
                                     ceil_div(total + kDecodeSegCost * segs, static_cast<int64_t>(cap)));
      int64_t hi = total + static_cast<int64_t>(kDecodeSegCost) * (segs + 1);
      auto feasible = [&](int64_t T, std::vector<int32_t>& st) {
        cut(sb, se, T, cap, st);
        return static_cast<int32_t>(st.size()) - 1 <= cap && st.back() == total;
      };
      std::vector<int32_t> best;                 // the cut of the smallest feasible cap so far
      bool ok = false;
      if (cap > 1) {
        const int64_t hi2 =
            ceil_div(total + kDecodeSegCost * (segs + cap), static_cast<int64_t>(cap) - 1) +
            kDecodeSegCost + 1;
        if (hi2 < hi && feasible(hi2, best)) {
          hi = hi2;
          ok = true;
        }
      }
      if (!ok) ok = feasible(hi, best);
      if (!ok) {
        uniform = true;  // the tables' limits alone need more CTAs than listed
      } else {
        lo = std::min(lo, hi);
        while (lo < hi) {
          const int64_t mid = (lo + hi) / 2;
          if (feasible(mid, starts)) {
            hi = mid;
            best.swap(starts);
          } else {
            lo = mid + 1;
          }
        }
        starts.swap(best);
        dl.n_ctas = static_cast<int32_t>(starts.size()) - 1;
        dl.cta_begin = static_cast<int32_t>(plan.dcta_blk0.size());
        plan.dcta_blk0.insert(plan.dcta_blk0.end(), starts.begin(), starts.end());
      }
    }
    if (uniform) {
      int32_t bpc = forced_tokens > 0
                        ? static_cast<int32_t>(ceil_div(forced_tokens, 16))
                        : static_cast<int32_t>(ceil_div(total, static_cast<int64_t>(dec_sms)));
      bpc = std::max<int32_t>(1, bpc);
      while (bpc > 1 && !fits(sb, se, bpc)) bpc = std::max<int32_t>(1, bpc * 3 / 4);
      dl.bpc = bpc;
      dl.n_ctas = static_cast<int32_t>(ceil_div(total, bpc));
      starts.clear();
      for (int32_t c = 0; c <= dl.n_ctas; ++c) starts.push_back(std::min(total, c * bpc));
    }
    slot_base += 2 * dl.n_ctas;
    ctas += dl.n_ctas;
    // Longest range, the segments cut across CTAs (merged by the combine
    // kernel) and the most ranges any segment is cut across.
    int32_t longest = 0;
    for (int32_t c = 0; c < dl.n_ctas; ++c) longest = std::max(longest, starts[c + 1] - starts[c]);
    if (sb == 0) plan.kv_split = longest * 16;
    dl.cut_begin = static_cast<int32_t>(plan.dcut.size());
    for (int32_t k = sb; k < se; ++k) {
      const int32_t b0 = blk0[k] - base, b1 = blk0[k + 1] - base;
      if (b1 == b0) continue;
      const int64_t ca = std::upper_bound(starts.begin(), starts.end(), b0) - starts.begin() - 1;
      const int64_t cb = std::upper_bound(starts.begin(), starts.end(), b1 - 1) - starts.begin() - 1;
      max_splits = std::max<int64_t>(max_splits, cb - ca + 1);
      if (cb > ca)
        plan.dcut.push_back({static_cast<int32_t>(ca), starts[ca] != b0 ? 1 : 0,
                             static_cast<int32_t>(cb - ca + 1), plan.dseg_q0[k],
                             plan.dseg_seqhead[k] & 255});
    }
    dl.n_cut = static_cast<int32_t>(plan.dcut.size()) - dl.cut_begin;
    plan.dlaunch.push_back(dl);
  }
  plan.max_splits = static_cast<int32_t>(max_splits);
  plan.decode_ctas = ctas;
  plan.dec_slots = slot_base;
}

// Prefill work items, longest first for a persistent grid: (sequence, query
// block, KV head), or with SM pairs (sequence, pair of adjacent query blocks,
// KV head), costed by the keys the item streams.
// K and V bytes per group of (sequence, KV head) pairs in the dynamic
// prefill list: about a third of the 126 MB L2.
constexpr double kL2GroupBytes = 40.0 * 1024 * 1024;

void plan_prefill(Plan& plan, const int32_t* cu, const int32_t* kv, const int32_t* win,
                  int32_t forced_q_block, int32_t forced_split, bool dynamic, bool grouping) {
  const int32_t group = plan.hq / plan.hkv;
  const int32_t max_qb = prefill_tokens_per_block(plan.d, group);
  // Query tokens per CTA: a requested block larger than one 128-row tile
  // holds was refused or sent to SM pairs (half the block per SM) by the
  // caller.
  int32_t qb = max_qb;
  if (forced_q_block > 0) qb = plan.prefill_pairs ? forced_q_block / 2 : forced_q_block;
  plan.q_block = qb;
  struct Cost {
    int64_t cost;
    int64_t tiles;
    PrefillItem item;
    int32_t idx;   // position in (sequence, block, head) order
  };
  std::vector<Cost> all;
  for (int32_t s = 0; s < plan.num_seqs; ++s) {
    const int32_t ql = cu[s + 1] - cu[s];
    if (ql <= 1) continue;
    const int32_t L = kv[s];
    const int32_t w = win ? win[s] : 0;
    const int64_t span = plan.prefill_pairs ? 2 * qb : qb;   // query tokens per item
    const int64_t nb = ceil_div(ql, span);
    for (int64_t b = 0; b < nb; ++b) {
      // Keys streamed by this item: from the first visible key of its first
      // query to its last query's own position.
      int64_t pos0 = static_cast<int64_t>(L) - ql + b * span;
      int64_t pos1 = std::min<int64_t>(static_cast<int64_t>(L) - ql + (b + 1) * span, L) - 1;
      int64_t lo = (w > 0 && pos0 - (w - 1) > 0) ? pos0 - (w - 1) : 0;
      int64_t keys = pos1 - lo + 1;
      // Key tiles the kernel streams: from the 64-aligned tile start at or
      // below the first visible key to the last query's position.
      const int64_t key_first = lo / kPrefillTileAlign * kPrefillTileAlign;
      const int64_t tiles = (pos1 - key_first) / kPrefillTileKeys + 1;
      for (int32_t h = 0; h < plan.hkv; ++h)
        all.push_back({keys, tiles, PrefillItem{s, static_cast<int32_t>((b << 8) | h), 0},
                       static_cast<int32_t>(all.size())});
    }
  }
  // Longest first; ties keep (sequence, block, head) order, which keeps the
  // CTAs that share a KV head's pages close together in time.
  std::sort(all.begin(), all.end(), [](const Cost& a, const Cost& b) {
    return a.cost != b.cost ? a.cost > b.cost : a.idx < b.idx;
  });
  plan.items.clear();
  plan.psplit.clear();
  plan.pcta0.clear();
  plan.prefill_dynamic = false;
  plan.prefill_groups = 0;
  plan.n_split_items = 0;
  plan.prefill_max_tiles = 0;
  const int64_t slots = static_cast<int64_t>(plan.prefill_sms > 0 ? plan.prefill_sms : plan.num_sms) *
                       prefill_ctas_per_sm(plan.d);
  // A persistent grid takes the items round-robin, longest first; its time
  // is set by the CTA with the most tiles.  On request (prefill_split = n),
  // lay every item's key tiles end to end and cut them into ranges of n
  // tiles, one per CTA, as decode does: an item crossing a range boundary is
  // split into parts, each leaving an fp32 partial that a combine merges.
  // Not chosen automatically: on multi-token decode (one short item per
  // sequence, the longest setting the step) GB300 measured 48.3 us split
  // against 46.7 us whole, the kernel streaming each K tile in four column
  // chunks, not the item balance, being the limit there.
  const int64_t per = forced_split;
  bool split = !plan.prefill_pairs && forced_split > 0 && !all.empty();
  std::vector<std::vector<PrefillItem>> per_cta;
  if (split) {
    // Sequence order keeps an item's parts (and a sequence's items) adjacent.
    std::vector<Cost> order = all;
    std::sort(order.begin(), order.end(),
              [](const Cost& a, const Cost& b) { return a.idx < b.idx; });
    int64_t cta = 0, room = per, slot = 0;
    per_cta.assign(1, {});
    for (const Cost& c : order) {
      int64_t j0 = 0;
      PrefillSplit g{c.item.seq, c.item.qb_head, static_cast<int32_t>(slot), 0};
      std::vector<std::pair<int64_t, int64_t>> parts;   // (cta, j0 << 32 | n)
      while (j0 < c.tiles) {
        if (room == 0) {
          ++cta;
          room = per;
          per_cta.emplace_back();
        }
        const int64_t n = std::min(room, c.tiles - j0);
        parts.push_back({cta, (j0 << 32) | n});
        j0 += n;
        room -= n;
      }
      if (parts.size() == 1) {
        per_cta[static_cast<size_t>(parts[0].first)].push_back(c.item);
        continue;
      }
      for (const auto& pr : parts) {
        const int64_t pj0 = pr.second >> 32, pn = pr.second & 0xffffffff;
        if (slot >= kSplitMaxSlots || pj0 >= kSplitMaxFirst || pn > kSplitMaxTiles) {
          split = false;
          break;
        }
        per_cta[static_cast<size_t>(pr.first)].push_back(
            PrefillItem{c.item.seq, c.item.qb_head,
                        split_code(static_cast<int32_t>(slot), static_cast<int32_t>(pj0),
                                   static_cast<int32_t>(pn))});
        ++slot;
        ++g.nparts;
      }
      if (!split) break;
      plan.psplit.push_back(g);
    }
    // CTA c runs its range's parts in order (per-CTA lists, one launch).
    size_t count = 0;
    for (const auto& v : per_cta) count += v.size();
    const size_t grid = per_cta.size();
    if (split && count <= static_cast<size_t>(kMaxItemsPerLaunch) &&
        grid <= static_cast<size_t>(kMaxPrefillGrid)) {
      plan.prefill_max_tiles = static_cast<int32_t>(per);
      plan.pcta0.assign(1, 0);
      for (const auto& v : per_cta) {
        plan.items.insert(plan.items.end(), v.begin(), v.end());
        plan.pcta0.push_back(static_cast<int32_t>(plan.items.size()));
      }
      plan.n_split_items = static_cast<int32_t>(slot);
      plan.prefill_ctas = static_cast<int32_t>(grid);
      return;
    }
    plan.items.clear();
    plan.psplit.clear();
  }
  // Longest processing time first: each item, longest first, goes to the CTA
  // with the fewest tiles so far; CTA c then runs its list in that order.
  // (Striding over the longest-first list instead gives CTA 0 the largest
  // item of every round: +7% tiles on the busiest CTA for a causal 8k
  // prefill, +38% on the mixed batch's prefill part.)
  const int64_t grid = std::min<int64_t>(static_cast<int64_t>(all.size()), slots);
  if (!plan.prefill_pairs && static_cast<int64_t>(all.size()) <= kMaxItemsPerLaunch &&
      grid <= kMaxPrefillGrid && grid > 0) {
    // Min-heap of (tiles so far << 16 | CTA): ties go to the lowest CTA.
    std::vector<uint64_t> heap(static_cast<size_t>(grid));
    for (int32_t c = 0; c < grid; ++c) heap[static_cast<size_t>(c)] = static_cast<uint64_t>(c);
    std::vector<int32_t> owner(all.size());
    plan.pcta0.assign(static_cast<size_t>(grid) + 1, 0);
    for (size_t i = 0; i < all.size(); ++i) {
      const uint64_t top = heap[0];
      const int32_t c = static_cast<int32_t>(top & 0xffff);
      owner[i] = c;
      ++plan.pcta0[static_cast<size_t>(c) + 1];
      // Replace the root with its new load and sift it down.
      const uint64_t v = top + (static_cast<uint64_t>(all[i].tiles) << 16);
      size_t j = 0;
      const size_t n = heap.size();
      for (;;) {
        size_t k = 2 * j + 1;
        if (k >= n) break;
        if (k + 1 < n && heap[k + 1] < heap[k]) ++k;
        if (heap[k] >= v) break;
        heap[j] = heap[k];
        j = k;
      }
      heap[j] = v;
    }
    plan.prefill_ctas = static_cast<int32_t>(grid);
    if (dynamic) {
      // The same order, each item taken by whichever CTA gets free first:
      // on SMs of equal speed that is this assignment; where some SMs
      // stream faster than others (their share of HBM and L2 differs by
      // ~10% on GB300), the faster ones take more items instead of the
      // slowest setting the makespan.
      //
      // When the prefill's K and V outgrow L2 and each (sequence, KV head)
      // is read by several items, the list runs in groups of (sequence, KV
      // head) pairs of at most kL2GroupBytes of K and V, longest first within
      // each group: the items that share keys then run close together and
      // find them in L2, where longest first over the whole batch would
      // stream every head's keys at once and read each from HBM again and
      // again (2.7x the algorithmic bytes on the causal 8k prefill).
      const int64_t pairs = static_cast<int64_t>(plan.num_prefill) * plan.hkv;
      // Sliding windows reuse keys only between neighbouring query blocks,
      // which longest first keeps together already: only batches whose
      // prefill sequences all see their whole prefix are grouped.  Groups of
      // equal bytes (ceil(total / kL2GroupBytes) of them): a small last group
      // would start its longest items late and leave a tail.
      double total = 0;
      bool whole_prefix = true;
      for (int32_t sq = 0; sq < plan.num_seqs; ++sq) {
        if (cu[sq + 1] - cu[sq] <= 1) continue;
        total += static_cast<double>(kv[sq]) * plan.d * 2.0 * 2.0 * plan.hkv;
        const int32_t w = win ? win[sq] : 0;
        if (w > 0 && w < kv[sq]) whole_prefix = false;
      }
      const int32_t ngroups = std::max<int32_t>(1, static_cast<int32_t>(std::ceil(total / kL2GroupBytes)));
      std::vector<int32_t> gid(static_cast<size_t>(plan.num_seqs) * plan.hkv, 0);
      double acc = 0;
      for (int32_t sq = 0; sq < plan.num_seqs; ++sq) {
        if (cu[sq + 1] - cu[sq] <= 1) continue;
        for (int32_t h = 0; h < plan.hkv; ++h) {
          gid[static_cast<size_t>(sq) * plan.hkv + h] =
              std::min(ngroups - 1, static_cast<int32_t>(acc * ngroups / total));
          acc += static_cast<double>(kv[sq]) * plan.d * 2.0 * 2.0;
        }
      }
      std::vector<Cost> order = all;
      plan.prefill_groups = 1;
      if (grouping && whole_prefix && total > 1.5 * kL2GroupBytes &&
          static_cast<int64_t>(all.size()) >= 4 * pairs) {
        plan.prefill_groups = ngroups;
        auto g_of = [&](const Cost& c) {
          return gid[static_cast<size_t>(c.item.seq) * plan.hkv + (c.item.qb_head & 255)];
        };
        std::stable_sort(order.begin(), order.end(),
                         [&](const Cost& a, const Cost& b) { return g_of(a) < g_of(b); });
      }
      for (const Cost& c : order) plan.items.push_back(c.item);
      plan.pcta0.clear();
      plan.prefill_dynamic = true;
    } else {
      // CTA-major placement, each CTA's items in assignment (longest-first) order.
      for (size_t c = 0; c < static_cast<size_t>(grid); ++c) plan.pcta0[c + 1] += plan.pcta0[c];
      plan.items.resize(all.size());
      std::vector<int32_t> fill(plan.pcta0.begin(), plan.pcta0.end() - 1);
      for (size_t i = 0; i < all.size(); ++i)
        plan.items[static_cast<size_t>(fill[owner[i]]++)] = all[i].item;
    }
    uint64_t busiest = 0;
    for (const uint64_t v : heap) busiest = std::max(busiest, v >> 16);
    plan.prefill_max_tiles = static_cast<int32_t>(busiest);
    return;
  }
  for (const Cost& c : all) plan.items.push_back(c.item);
  {
    const int64_t g = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(all.size()),
                                                             slots / (plan.prefill_pairs ? 2 : 1)));
    std::vector<int64_t> load(static_cast<size_t>(g), 0);
    for (size_t i = 0; i < all.size(); ++i) load[i % static_cast<size_t>(g)] += all[i].tiles;
    plan.prefill_max_tiles = static_cast<int32_t>(*std::max_element(load.begin(), load.end()));
  }
  const int64_t per_item = plan.prefill_pairs ? 2 : 1;      // CTAs per item
  plan.prefill_ctas = static_cast<int32_t>(
      per_item * std::min<int64_t>(static_cast<int64_t>(plan.items.size()), slots / per_item));
}

// Key tiles of the prefill work items with `span` query tokens each (the
// same geometry as plan_prefill): their sum, the largest, and the count.
struct TileStats {
  int64_t total = 0, largest = 0, items = 0;
};
TileStats prefill_tile_stats(const Plan& plan, const int32_t* cu, const int32_t* kv,
                             const int32_t* win, int64_t span) {
  TileStats t;
  for (int32_t s = 0; s < plan.num_seqs; ++s) {
    const int32_t ql = cu[s + 1] - cu[s];
    if (ql <= 1) continue;
    const int32_t L = kv[s];
    const int32_t w = win ? win[s] : 0;
    for (int64_t b = 0; b < ceil_div(ql, span); ++b) {
      const int64_t pos0 = static_cast<int64_t>(L) - ql + b * span;
      const int64_t pos1 = std::min<int64_t>(pos0 + span, L) - 1;
      const int64_t lo = (w > 0 && pos0 - (w - 1) > 0) ? pos0 - (w - 1) : 0;
      const int64_t tiles =
          (pos1 - lo / kPrefillTileAlign * kPrefillTileAlign) / kPrefillTileKeys + 1;
      t.total += tiles * plan.hkv;
      t.largest = std::max(t.largest, tiles);
      t.items += plan.hkv;
    }
  }
  return t;
}

// Cost model of a mixed batch's two persistent grids (microseconds), fitted
// to GB300 timings of the mixed batch's decode part on 30-152 SMs and its
// prefill part on 40-152 SMs: the decode grid streams its KV bytes at ~78
// GB/s per SM (each CTA's copy ring, not HBM, sets the pace; the rate that
// puts the split where a sweep of it measured the shortest step) until ~5 TB/s,
// plus its ramp, merges and combine; the single-SM prefill kernel at D = 256
// takes ~1.6 us per 128-key tile and ~3.2 us per item epilogue (both scale
// with D), its makespan set by the busier of the average CTA and the longest
// item, plus its ramp and tail.
constexpr double kDecodeSmGBs = 78.0;
constexpr double kDecodeHbmGBs = 5000.0;
constexpr double kDecodeFixedUs = 8.0;
constexpr double kPrefillTileUs256 = 1.6;
constexpr double kPrefillItemUs256 = 3.2;
constexpr double kPrefillFixedUs = 20.0;

// RPA_DECODE_KERNEL_AUTO takes the tensor-core decode kernel where it applies.
constexpr bool kDecodeTcByDefault = false;

double decode_cost_us(double bytes, int32_t sms) {
  return bytes / std::min(sms * kDecodeSmGBs, kDecodeHbmGBs) * 1e-3 + kDecodeFixedUs;
}

double prefill_cost_us(const TileStats& t, int32_t head_dim, int32_t sms) {
  const double f = head_dim / 256.0;
  const double tiles = std::max(static_cast<double>(t.total) / sms, static_cast<double>(t.largest));
  return tiles * kPrefillTileUs256 * f + std::ceil(static_cast<double>(t.items) / sms) *
         kPrefillItemUs256 * f + kPrefillFixedUs;
}

}  // namespace

rpa_status_t build_schedule(Plan& plan, const int32_t* cu, const int32_t* kv,
                            const int32_t* win, const rpa_plan_options& opts) {
  const int32_t group = plan.hq / plan.hkv;
  plan.num_decode = plan.num_prefill = 0;
  for (int32_t s = 0; s < plan.num_seqs; ++s) {
    int32_t ql = cu[s + 1] - cu[s];
    if (ql > 1) ++plan.num_prefill;
  }
  const int32_t want = opts.path;
  if (want != RPA_PATH_AUTO && want != RPA_PATH_SIMT && want != RPA_PATH_TC)
    return RPA_ERR_INVALID_ARG;
  const bool f32 = plan.dtype == RPA_DTYPE_F32;
  if (want == RPA_PATH_TC && f32) return RPA_ERR_UNSUPPORTED;
  bool tc_decode = false, tc_prefill = false;
  if (want != RPA_PATH_SIMT && !f32) {
    tc_decode = decode_supported(plan.d, group, plan.p);
    tc_prefill = prefill_tc_supported(plan.d, plan.p, group);
  }
  int32_t ndec = 0;
  for (int32_t s = 0; s < plan.num_seqs; ++s) ndec += (cu[s + 1] - cu[s] == 1);
  // fp8 (e4m3) K/V pages: the split-KV decode kernel only.
  if (opts.kv_dtype != 0 && opts.kv_dtype != plan.dtype) {
    if (opts.kv_dtype != RPA_DTYPE_FP8_E4M3) return RPA_ERR_INVALID_ARG;
    // fp8 rows are fetched in 128-byte boxes: head_dim a multiple of 128.
    if (plan.dtype != RPA_DTYPE_BF16 || want == RPA_PATH_SIMT || plan.num_prefill > 0 ||
        !tc_decode || plan.d % 128 != 0)
      return RPA_ERR_UNSUPPORTED;
  }
  plan.kv_fp8 = opts.kv_dtype == RPA_DTYPE_FP8_E4M3;
  // Which split-KV decode kernel: the tensor-core one where it applies,
  // unless the CUDA-core one is asked for.
  if (opts.decode_kernel < RPA_DECODE_KERNEL_AUTO || opts.decode_kernel > RPA_DECODE_KERNEL_TC)
    return RPA_ERR_INVALID_ARG;
  const bool tcgen_decode =
      tc_decode && decode_tc_supported(plan.d, group, plan.p, plan.kv_fp8);
  if (opts.decode_kernel == RPA_DECODE_KERNEL_TC && ndec > 0 && !tcgen_decode)
    return RPA_ERR_UNSUPPORTED;
  plan.decode_tc = ndec > 0 && tcgen_decode &&
                   (opts.decode_kernel == RPA_DECODE_KERNEL_TC ||
                    (opts.decode_kernel == RPA_DECODE_KERNEL_AUTO && kDecodeTcByDefault));
  if (want == RPA_PATH_TC) {
    if ((ndec > 0 && !tc_decode) || (plan.num_prefill > 0 && !tc_prefill))
      return RPA_ERR_UNSUPPORTED;
  }
  if (f32 || want == RPA_PATH_SIMT) {
    // The fp32 debug build, and the explicit SIMT path, take the CUDA-core
    // kernel for everything.
    if (group > 32) return RPA_ERR_UNSUPPORTED;
  }
  plan.simt_decode = ndec > 0 && !tc_decode;
  plan.simt_prefill = plan.num_prefill > 0 && !tc_prefill;
  if ((plan.simt_decode || plan.simt_prefill) && group > 32) return RPA_ERR_UNSUPPORTED;
  plan.path = (tc_decode && ndec > 0) || (tc_prefill && plan.num_prefill > 0)
                  ? RPA_PATH_TC
                  : RPA_PATH_SIMT;

  plan.num_decode = ndec;
  plan.kv_split = plan.max_splits = plan.dec_slots = 0;
  plan.decode_ctas = 0;
  plan.dseg_seqhead.clear();
  plan.dseg_blk0.clear();
  plan.dlaunch.clear();

  plan.items.clear();
  plan.q_block = 0;
  plan.prefill_ctas = 0;
  const bool pairs_ok = tc_prefill && prefill_pair_supported(plan.d, plan.p, group);
  if (opts.prefill_pairs == 2 && plan.num_prefill > 0 && !pairs_ok) return RPA_ERR_UNSUPPORTED;
  // A requested query block is either one CTA's 128-row tile or less
  // (128 / G tokens), or, on SM pairs, two such halves (one M = 256 MMA over
  // both); anything larger would need several tiles per KV tile, which the
  // tensor memory at these head sizes cannot hold, and is refused rather
  // than silently shrunk.
  const int32_t max_qb = prefill_tokens_per_block(plan.d, group);
  bool want_pairs = opts.prefill_pairs == 2;
  if (tc_prefill && plan.num_prefill > 0 && opts.q_block > 0) {
    if (opts.q_block > 2 * max_qb) return RPA_ERR_UNSUPPORTED;
    if (opts.q_block > max_qb) {
      if (!pairs_ok) return RPA_ERR_UNSUPPORTED;
      want_pairs = true;
    }
    if (want_pairs && (opts.q_block % 2 != 0)) return RPA_ERR_UNSUPPORTED;
  }
  // Chosen only on request (prefill_pairs = 2, or a query block of two
  // tiles): on GB300 the pair kernel's cross-SM barrier round trips cost
  // more per tile than its halved copy traffic saves.
  plan.prefill_pairs = pairs_ok && plan.num_prefill > 0 && want_pairs;

  // A mixed batch ("TPU Deep Dive" slides, chapter 8, "Continuous batching
  // with static shapes": one step holds decoding and prefilling sequences)
  // puts HBM-bound decode and tensor-bound prefill work in one call.  One
  // after the other, each grid leaves the other's resource idle; side by
  // side on disjoint SMs, decode streams from HBM while prefill keeps the
  // tensor cores busy.  The split of the SMs evens the two grids' modelled
  // times; it is taken when that beats running them one after the other.
  plan.overlap = false;
  plan.decode_sms = plan.prefill_sms = 0;
  plan.est_decode_us = plan.est_prefill_us = 0.f;
  if (opts.decode_sms < -1) return RPA_ERR_INVALID_ARG;
  if (tc_decode && ndec > 0 && tc_prefill && plan.num_prefill > 0 && !plan.prefill_pairs &&
      opts.decode_sms >= 0 && plan.num_sms >= 2) {
    double dec_bytes = 0;
    for (int32_t s = 0; s < plan.num_seqs; ++s) {
      if (cu[s + 1] - cu[s] != 1) continue;
      const int32_t w = win ? win[s] : 0;
      const int32_t lo = (w > 0 && kv[s] - w > 0) ? kv[s] - w : 0;
      dec_bytes += static_cast<double>(ceil_div(kv[s], 16) - lo / 16) * 16.0 * plan.hkv *
                   plan.d * 2.0 * (plan.kv_fp8 ? 1.0 : 2.0);
    }
    const int32_t qb_cta = opts.q_block > 0 ? opts.q_block : max_qb;
    const TileStats ts = prefill_tile_stats(plan, cu, kv, win, qb_cta);
    const int32_t n = plan.num_sms;
    int32_t best = 0;
    double best_t = decode_cost_us(dec_bytes, n) + prefill_cost_us(ts, plan.d, n);
    if (opts.decode_sms > 0) {
      best = std::min(opts.decode_sms, n - 1);
      best_t = std::max(decode_cost_us(dec_bytes, best), prefill_cost_us(ts, plan.d, n - best));
    } else {
      for (int32_t x = 1; x < n; ++x) {
        const double t = std::max(decode_cost_us(dec_bytes, x), prefill_cost_us(ts, plan.d, n - x));
        if (t < best_t) {
          best_t = t;
          best = x;
        }
      }
    }
    if (best > 0) {
      plan.overlap = true;
      plan.decode_sms = best;
      plan.prefill_sms = n - best;
      plan.est_decode_us = static_cast<float>(decode_cost_us(dec_bytes, best));
      plan.est_prefill_us = static_cast<float>(prefill_cost_us(ts, plan.d, n - best));
    }
  }

  if (tc_decode && ndec > 0) plan_decode(plan, cu, kv, win, opts.kv_split);
  if (tc_prefill && plan.num_prefill > 0)
    plan_prefill(plan, cu, kv, win, opts.q_block, opts.prefill_split,
                 opts.prefill_dynamic == 0, opts.prefill_grouping == 0);

  // Workspace: header, then the decode partials (two slots per decode CTA,
  // G x D fp32 each, plus G log2-sum-exps).
  size_t off = kHeaderBytes;
  plan.off_partial_o = plan.off_partial_lse = 0;
  if (!plan.dlaunch.empty()) {
    const size_t rows = static_cast<size_t>(plan.dec_slots) * group;
    plan.off_partial_o = off;
    off += (rows * plan.d * sizeof(float) + 255) / 256 * 256;
    plan.off_partial_lse = off;
    off += (rows * sizeof(float) + 255) / 256 * 256;
  }
  plan.off_ppart_o = plan.off_ppart_lse = 0;
  if (plan.n_split_items > 0) {
    // Prefill parts: one 128-row fp32 partial and its log2-sum-exps each.
    const size_t rows = static_cast<size_t>(plan.n_split_items) * 128;
    plan.off_ppart_o = off;
    off += (rows * plan.d * sizeof(float) + 255) / 256 * 256;
    plan.off_ppart_lse = off;
    off += (rows * sizeof(float) + 255) / 256 * 256;
  }
  plan.ws_bytes = off;
  return RPA_OK;
}

}  // namespace rpa
