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
// end and cut into equal contiguous ranges, one per CTA (one per SM: a single
// balanced wave), so every CTA streams the same number of bytes whatever the
// length mix.  Ranges shrink (more CTAs) only when one would touch more
// segments or pages than the kernel's shared-memory tables hold.
void plan_decode(Plan& plan, const int32_t* cu, const int32_t* kv, const int32_t* win,
                 int32_t forced_tokens) {
  plan.dseg_seqhead.clear();
  plan.dseg_blk0.assign(1, 0);
  plan.dseg_q0.clear();
  plan.dseg_lo.clear();
  plan.dseg_len.clear();
  plan.dlaunch.clear();
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
  const int32_t P = plan.p;
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
        const int64_t kb = seg_lo[kk] + 16 * static_cast<int64_t>(jb);
        const int64_t ke = seg_lo[kk] + 16 * static_cast<int64_t>(je);  // upper bound
        pages += static_cast<int32_t>((ke - 1) / P - kb / P + 1);
      }
      if (segs > kMaxCtaSegs || pages > kMaxCtaPages) return false;
    }
    return true;
  };
  int32_t slot_base = 0;
  int64_t max_splits = 1, ctas = 0;
  for (int32_t sb = 0; sb < nseg; sb += kDecodeSegLarge) {
    const int32_t se = std::min(nseg, sb + kDecodeSegLarge);
    const int32_t total = blk0[se] - blk0[sb];
    int32_t bpc = forced_tokens > 0
                      ? static_cast<int32_t>(ceil_div(forced_tokens, 16))
                      : static_cast<int32_t>(ceil_div(total, static_cast<int64_t>(plan.num_sms)));
    bpc = std::max<int32_t>(1, bpc);
    while (bpc > 1 && !fits(sb, se, bpc)) bpc = std::max<int32_t>(1, bpc * 3 / 4);
    const int32_t n_ctas = static_cast<int32_t>(ceil_div(total, bpc));
    plan.dlaunch.push_back({sb, se, bpc, n_ctas, slot_base});
    slot_base += 2 * n_ctas;
    ctas += n_ctas;
    for (int32_t k = sb; k < se; ++k) {
      const int64_t ca = (blk0[k] - blk0[sb]) / bpc;
      const int64_t cb = (blk0[k + 1] - 1 - blk0[sb]) / bpc;
      max_splits = std::max<int64_t>(max_splits, cb - ca + 1);
    }
  }
  plan.kv_split = plan.dlaunch.front().bpc * 16;
  plan.max_splits = static_cast<int32_t>(max_splits);
  plan.decode_ctas = ctas;
  plan.dec_slots = slot_base;
}

void plan_prefill(Plan& plan, const int32_t* cu, const int32_t* kv, const int32_t* win,
                  int32_t forced_q_block) {
  const int32_t group = plan.hq / plan.hkv;
  const int32_t max_qb = prefill_tokens_per_block(plan.d, group);
  int32_t qb = max_qb;
  if (forced_q_block > 0) qb = std::min(forced_q_block, max_qb);
  plan.q_block = qb;
  struct Cost {
    int64_t cost;
    PrefillItem item;
  };
  std::vector<Cost> all;
  for (int32_t s = 0; s < plan.num_seqs; ++s) {
    const int32_t ql = cu[s + 1] - cu[s];
    if (ql <= 1) continue;
    const int32_t L = kv[s];
    const int32_t w = win ? win[s] : 0;
    const int64_t nb = ceil_div(ql, qb);
    for (int64_t b = 0; b < nb; ++b) {
      // Keys streamed by this block: from the first visible key of its first
      // query to its last query's own position.
      int64_t pos0 = static_cast<int64_t>(L) - ql + b * qb;
      int64_t pos1 = std::min<int64_t>(static_cast<int64_t>(L) - ql + (b + 1) * qb, L) - 1;
      int64_t lo = (w > 0 && pos0 - (w - 1) > 0) ? pos0 - (w - 1) : 0;
      int64_t keys = pos1 - lo + 1;
      for (int32_t h = 0; h < plan.hkv; ++h)
        all.push_back({keys, PrefillItem{s, static_cast<int32_t>((b << 8) | h)}});
    }
  }
  // Longest first; ties keep (sequence, block, head) order, which keeps the
  // CTAs that share a KV head's pages close together in time.
  std::stable_sort(all.begin(), all.end(),
                   [](const Cost& a, const Cost& b) { return a.cost > b.cost; });
  plan.items.clear();
  for (const Cost& c : all) plan.items.push_back(c.item);
  const int64_t slots = static_cast<int64_t>(plan.num_sms) * prefill_ctas_per_sm(plan.d);
  plan.prefill_ctas = static_cast<int32_t>(
      std::min<int64_t>(static_cast<int64_t>(plan.items.size()), slots));
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
  if (tc_decode && ndec > 0) plan_decode(plan, cu, kv, win, opts.kv_split);

  plan.items.clear();
  plan.q_block = 0;
  plan.prefill_ctas = 0;
  if (tc_prefill && plan.num_prefill > 0) plan_prefill(plan, cu, kv, win, opts.q_block);

  // Workspace: header, then the decode partials (two slots per decode CTA,
  // G x D fp32 each, plus G log2-sum-exps) and one arrival counter per
  // decode segment.
  size_t off = kHeaderBytes;
  plan.off_partial_o = plan.off_partial_lse = plan.off_arrivals = 0;
  if (!plan.dlaunch.empty()) {
    const size_t rows = static_cast<size_t>(plan.dec_slots) * group;
    plan.off_partial_o = off;
    off += (rows * plan.d * sizeof(float) + 255) / 256 * 256;
    plan.off_partial_lse = off;
    off += (rows * sizeof(float) + 255) / 256 * 256;
    plan.off_arrivals = off;
    off += (plan.dseg_seqhead.size() * sizeof(int32_t) + 255) / 256 * 256;
  }
  plan.ws_bytes = off;
  return RPA_OK;
}

}  // namespace rpa
