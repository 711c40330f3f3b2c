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

int decode_ctas_per_sm(int32_t head_dim);   // decode.cu
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

// Makespan, in token-equivalents per CTA slot, of greedy in-order dispatch of
// `costs` onto `slots` identical slots (what the block scheduler does with a
// one-CTA-per-slot grid).
double list_schedule(const std::vector<double>& costs, int slots) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int i = 0; i < slots; ++i) free_at.push(0.0);
  double end = 0.0;
  for (double c : costs) {
    double t = free_at.top();
    free_at.pop();
    t += c;
    end = std::max(end, t);
    free_at.push(t);
  }
  return end;
}

// Fixed cost of one decode CTA (launch, prologue, merge) and of the combine
// launch, in tokens streamed by one CTA slot in the same time.
constexpr double kCtaOverheadTokens = 96.0;
constexpr double kCombineLaunchTokens = 128.0;

void plan_decode(Plan& plan, const int32_t* cu, const int32_t* kv, const int32_t* win,
                 int32_t forced_split) {
  std::vector<int64_t> vis;
  std::vector<int32_t> seqs;
  for (int32_t s = 0; s < plan.num_seqs; ++s) {
    if (cu[s + 1] - cu[s] != 1) continue;
    seqs.push_back(s);
    vis.push_back(decode_visible(kv[s], win ? win[s] : 0));
  }
  plan.num_decode = static_cast<int32_t>(seqs.size());
  if (seqs.empty()) return;
  const int slots = plan.num_sms * decode_ctas_per_sm(plan.d);
  const int32_t group = plan.hq / plan.hkv;
  std::vector<int32_t> candidates;
  // A split's page ids must fit the kernel's shared-memory table, and a
  // sequence may have at most kMaxSplits splits.
  const int64_t max_split_len = std::max<int64_t>(64, (kMaxSplitPages - 2) / 64 * 64 * plan.p);
  int64_t max_vis0 = 1;
  for (int64_t n : vis) max_vis0 = std::max(max_vis0, n);
  const int64_t min_split_len = ceil_div(ceil_div(max_vis0, kMaxSplits), 64) * 64;
  auto clamp_split = [&](int64_t x) {
    x = std::max<int64_t>(x, min_split_len);
    x = std::min<int64_t>(x, max_split_len);
    return static_cast<int32_t>(std::max<int64_t>(64, x));
  };
  if (forced_split > 0) {
    candidates.push_back(clamp_split(ceil_div(forced_split, 64) * 64));
  } else {
    for (int32_t c : {64, 128, 192, 256, 320, 384, 512, 640, 768, 1024, 1536, 2048, 3072, 4096})
      candidates.push_back(clamp_split(c));
  }
  // Evaluate the candidate nearest to two waves first so that the lower bound
  // below prunes most of the others without simulating them.
  int64_t total_vis = 0, max_vis = 0;
  for (int64_t n : vis) {
    total_vis += n;
    max_vis = std::max(max_vis, n);
  }
  const double two_waves = static_cast<double>(total_vis) * plan.hkv / (2.0 * slots);
  std::stable_sort(candidates.begin(), candidates.end(), [&](int32_t a, int32_t b) {
    return std::abs(a - two_waves) < std::abs(b - two_waves);
  });
  double best = -1.0;
  int32_t best_split = candidates.front();
  std::vector<double> costs;
  for (int32_t split : candidates) {
    // Lower bound: total work over the slots, or the longest CTA.
    int64_t ctas = 0;
    for (int64_t n : vis) ctas += ceil_div(n, split);
    ctas *= plan.hkv;
    const double lb = std::max(
        (static_cast<double>(total_vis) * plan.hkv + kCtaOverheadTokens * ctas) / slots,
        kCtaOverheadTokens + static_cast<double>(std::min<int64_t>(split, max_vis)));
    if (best >= 0 && lb >= best) continue;
    // Grid order: x = sequence (fastest), y = split, z = kv head.
    int64_t max_n = 0;
    for (int64_t n : vis) max_n = std::max(max_n, ceil_div(n, split));
    costs.clear();
    costs.reserve(static_cast<size_t>(ctas));
    bool any_multi = false;
    for (int32_t h = 0; h < plan.hkv; ++h)
      for (int64_t c = 0; c < max_n; ++c)
        for (size_t i = 0; i < vis.size(); ++i) {
          int64_t n = ceil_div(vis[i], split);
          if (c >= n) continue;
          int64_t tok = std::min<int64_t>(split, vis[i] - c * split);
          any_multi |= n > 1;
          // A split writes and the combine reads G x D fp32 partials: 2G tokens.
          costs.push_back(kCtaOverheadTokens + tok + (n > 1 ? 2.0 * group : 0.0));
        }
    double t = list_schedule(costs, slots) + (any_multi ? kCombineLaunchTokens : 0.0);
    if (best < 0 || t < best - 1e-9 || (std::abs(t - best) <= 1e-9 && split > best_split)) {
      best = t;
      best_split = split;
    }
  }
  plan.kv_split = best_split;
  int64_t max_n = 0, ctas = 0;
  for (int64_t n : vis) {
    max_n = std::max(max_n, ceil_div(n, best_split));
    ctas += ceil_div(n, best_split);
  }
  plan.max_splits = static_cast<int32_t>(std::max<int64_t>(max_n, 1));
  plan.decode_ctas = ctas * plan.hkv;
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
    tc_decode = decode_supported(plan.d, group);
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
  plan.kv_split = plan.max_splits = 0;
  plan.decode_ctas = 0;
  if (tc_decode && ndec > 0) plan_decode(plan, cu, kv, win, opts.kv_split);

  plan.items.clear();
  plan.q_block = 0;
  plan.prefill_ctas = 0;
  if (tc_prefill && plan.num_prefill > 0) plan_prefill(plan, cu, kv, win, opts.q_block);

  // Workspace: header, then decode partials when some sequence splits.
  size_t off = kHeaderBytes;
  plan.off_partial_o = plan.off_partial_lse = 0;
  if (plan.max_splits > 1) {
    const size_t rows = static_cast<size_t>(plan.num_seqs) * plan.max_splits * plan.hq;
    plan.off_partial_o = off;
    off += (rows * plan.d * sizeof(float) + 255) / 256 * 256;
    plan.off_partial_lse = off;
    off += (rows * sizeof(float) + 255) / 256 * 256;
    plan.off_arrivals = off;
    off += (static_cast<size_t>(plan.num_seqs) * plan.hkv * sizeof(int32_t) + 255) / 256 * 256;
  }
  plan.ws_bytes = off;
  return RPA_OK;
}

}  // namespace rpa
