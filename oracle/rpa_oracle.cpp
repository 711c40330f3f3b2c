// Ragged paged attention: the CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow definition that the
// GPU kernels are checked against.  Only the test suite, the smoke check and
// the benchmark's CPU-baseline leg may load it; the product library never
// links, calls or includes it, and it includes nothing from the product.
//
// What it computes (sources, by page title and section):
//   * "TPU Deep Dive" slides, chapter 8, "Continuous batching with static
//     shapes": every query token of a step sits in one flattened array and
//     per-sequence metadata (here cu_q_lens, kv_lens) carries the ragged
//     structure; ragged paged attention reads the KV cache through a paged
//     layout ("KV cache layout", same chapter).
//   * "Chasing speed of light on TPU v6e", section "Attention" and footnote 5:
//     attention is exact softmax attention of every query over the keys it may
//     see; a flash kernel only reorders that computation.  So the oracle is the
//     definition itself: a straight loop, one output row at a time, no tiling
//     and no online softmax.
//   * Same page, footnote 6: the softmax accumulators are kept in fp32.  The
//     fp32 mode below accumulates every sum in float; the fp64 mode exists to
//     check the fp32 mode.
//   * Same page, section "Attention": in a sliding-window layer a key is wanted
//     by the W queries that follow it (itself included).  Reading adopted: key
//     j is visible to the query at position pos iff j <= pos and, when the
//     sequence has a window W > 0, pos - j < W.
//   * "Pallas kernel / vLLM on TPU ... 19,511 tokens per second", section
//     "Strategy 3": the query heads of a group share one key/value head
//     (Gemma 2B: eight query heads of dimension 256 share one KV head).
//     Reading adopted: query head h reads KV head h / (Hq / Hkv).
//   * Query positions: the q_len new tokens of a sequence are its last q_len
//     KV positions, so query i of sequence s sits at pos = L_s - q_len_s + i.
//
// Definition, for every sequence s, query i < q_len_s and query head h:
//   pos   = L_s - q_len_s + i
//   g     = h / (Hq / Hkv)
//   vis   = { j : 0 <= j <= pos, and (W_s <= 0 or pos - j < W_s) }
//   k_j   = k_pages[page_table[s][j / P]][j % P][g][:]    (v_j the same)
//   x_j   = sm_scale * sum_d q[t][h][d] * k_j[d]          t = cu_q_lens[s] + i
//   m     = max_j x_j,  p_j = exp(x_j - m),  l = sum_j p_j
//   out[t][h][:] = sum_j p_j * v_j[:] / l,   then rounded to bf16 (nearest even)
//
// Build: g++ -O2 -ffp-contract=off -fopenmp -shared -fPIC (see build.py).
// -ffp-contract=off keeps a*b+c as two roundings on every host, so x86 and Arm
// builds compute the same float operations.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_META = 2 };

// bf16 is the upper half of an IEEE float; widening is exact.
inline float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round a float to the nearest bf16, ties to even (NaN kept quiet).
inline uint16_t float_to_bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

struct Problem {
  int in_dtype;  // 0: bf16 bits (uint16), 1: float32
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int32_t* page_table;
  int32_t max_pages_per_seq;
  const int32_t* cu_q_lens;
  const int32_t* kv_lens;
  const int32_t* window;  // may be null: every sequence full causal
  int32_t num_seqs, hq, hkv, d, p, num_pages;
};

inline double load(const Problem& pr, const void* base, int64_t idx) {
  if (pr.in_dtype == 0)
    return bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx]);
  return static_cast<const float*>(base)[idx];
}

// Element (token slot `slot` of physical page `page`, kv head g, dim dd).
inline int64_t kv_index(const Problem& pr, int64_t page, int64_t slot, int64_t g,
                        int64_t dd) {
  return ((page * pr.p + slot) * pr.hkv + g) * pr.d + dd;
}

int validate(const Problem& pr) {
  if (pr.num_seqs < 0 || pr.hq <= 0 || pr.hkv <= 0 || pr.d <= 0 || pr.p <= 0 ||
      pr.num_pages < 0 || pr.max_pages_per_seq < 0)
    return ORACLE_BAD_ARG;
  if (pr.hq % pr.hkv != 0) return ORACLE_BAD_ARG;
  if (pr.in_dtype != 0 && pr.in_dtype != 1) return ORACLE_BAD_ARG;
  if (pr.cu_q_lens[0] != 0) return ORACLE_BAD_META;
  for (int32_t s = 0; s < pr.num_seqs; ++s) {
    int32_t ql = pr.cu_q_lens[s + 1] - pr.cu_q_lens[s];
    int32_t L = pr.kv_lens[s];
    if (ql < 0 || L < ql) return ORACLE_BAD_META;
    int64_t pages = (static_cast<int64_t>(L) + pr.p - 1) / pr.p;
    if (pages > pr.max_pages_per_seq) return ORACLE_BAD_META;
    if (ql == 0) continue;
    // Only the pages holding keys visible to some query are read.
    for (int64_t pg = 0; pg < pages; ++pg) {
      int32_t id = pr.page_table[static_cast<int64_t>(s) * pr.max_pages_per_seq + pg];
      if (id < 0 || id >= pr.num_pages) return ORACLE_BAD_META;
    }
  }
  return ORACLE_OK;
}

// Locate flattened row r = t * hq + h: its sequence s and query index i.
inline void locate(const Problem& pr, int64_t r, int32_t* s_out, int32_t* i_out,
                   int32_t* h_out) {
  int64_t t = r / pr.hq;
  *h_out = static_cast<int32_t>(r % pr.hq);
  // Linear search: the oracle favours obviousness over speed.
  int32_t s = 0;
  while (s + 1 <= pr.num_seqs && !(t < pr.cu_q_lens[s + 1])) ++s;
  *s_out = s;
  *i_out = static_cast<int32_t>(t - pr.cu_q_lens[s]);
}

inline void visible_range(const Problem& pr, int32_t s, int32_t i, int64_t* lo,
                          int64_t* pos_out) {
  int32_t ql = pr.cu_q_lens[s + 1] - pr.cu_q_lens[s];
  int64_t pos = static_cast<int64_t>(pr.kv_lens[s]) - ql + i;
  int32_t w = pr.window ? pr.window[s] : 0;
  int64_t first = 0;
  if (w > 0 && pos - (w - 1) > 0) first = pos - (w - 1);
  *lo = first;
  *pos_out = pos;
}

// One output row in precision T (float or double).  `x` is scratch of at least
// pos+1 elements.  Writes D values to `out_row` and, if `prow` is given, the
// normalised probabilities p_j / l for j in [lo, pos].
template <typename T>
void one_row(const Problem& pr, double sm_scale, int32_t s, int32_t i, int32_t h,
             T* x, double* out_row, double* prow) {
  const int64_t t = static_cast<int64_t>(pr.cu_q_lens[s]) + i;
  const int32_t group = pr.hq / pr.hkv;
  const int32_t g = h / group;
  int64_t lo, pos;
  visible_range(pr, s, i, &lo, &pos);
  const T scale = static_cast<T>(sm_scale);
  const int32_t* pt = pr.page_table + static_cast<int64_t>(s) * pr.max_pages_per_seq;
  const int64_t q_base = (t * pr.hq + h) * pr.d;

  // Scores.
  T m = -INFINITY;
  for (int64_t j = lo; j <= pos; ++j) {
    const int64_t page = pt[j / pr.p];
    const int64_t slot = j % pr.p;
    T dot = 0;
    for (int32_t dd = 0; dd < pr.d; ++dd) {
      T qv = static_cast<T>(load(pr, pr.q, q_base + dd));
      T kv = static_cast<T>(load(pr, pr.k_pages, kv_index(pr, page, slot, g, dd)));
      dot = dot + qv * kv;
    }
    T xj = scale * dot;
    x[j - lo] = xj;
    if (xj > m) m = xj;
  }
  // Probabilities (unnormalised) and their sum.
  T l = 0;
  for (int64_t j = lo; j <= pos; ++j) {
    T pj = std::exp(x[j - lo] - m);
    x[j - lo] = pj;
    l = l + pj;
  }
  // Weighted sum of values, then normalise.
  for (int32_t dd = 0; dd < pr.d; ++dd) {
    T acc = 0;
    for (int64_t j = lo; j <= pos; ++j) {
      const int64_t page = pt[j / pr.p];
      const int64_t slot = j % pr.p;
      T vv = static_cast<T>(load(pr, pr.v_pages, kv_index(pr, page, slot, g, dd)));
      acc = acc + x[j - lo] * vv;
    }
    out_row[dd] = static_cast<double>(acc / l);
  }
  if (prow) {
    for (int64_t j = lo; j <= pos; ++j) prow[j - lo] = static_cast<double>(x[j - lo] / l);
  }
}

}  // namespace

extern "C" {

// Compute output rows.  Row r is (token t = r / Hq, query head h = r % Hq).
//   precision : 32 (fp32 accumulation, the parity oracle) or 64 (checker)
//   in_dtype  : 0 = q/k/v hold bf16 bit patterns (uint16), 1 = float32
//   rows      : row indices to compute, or null for every row in order
//   out       : [n_rows, D] doubles (fp32 mode stores float values exactly)
//   out_bf16  : optional [n_rows, D] bf16 bit patterns of the rounded output
//   threads   : OpenMP threads (<= 0: library default)
// Returns 0 on success, 1 for a bad argument, 2 for inconsistent metadata.
int rpa_oracle_rows(int precision, int in_dtype, const void* q, const void* k_pages,
                    const void* v_pages, const int32_t* page_table,
                    int32_t max_pages_per_seq, const int32_t* cu_q_lens,
                    const int32_t* kv_lens, const int32_t* window, int32_t num_seqs,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, int32_t num_pages, double sm_scale,
                    const int64_t* rows, int64_t n_rows, double* out,
                    uint16_t* out_bf16, int threads) {
  if (precision != 32 && precision != 64) return ORACLE_BAD_ARG;
  Problem pr{in_dtype, q, k_pages, v_pages, page_table, max_pages_per_seq,
             cu_q_lens, kv_lens, window, num_seqs, num_q_heads, num_kv_heads,
             head_dim, page_size, num_pages};
  int rc = validate(pr);
  if (rc != ORACLE_OK) return rc;
  const int64_t total_rows = static_cast<int64_t>(cu_q_lens[num_seqs]) * num_q_heads;
  if (rows == nullptr) n_rows = total_rows;
  for (int64_t n = 0; rows && n < n_rows; ++n)
    if (rows[n] < 0 || rows[n] >= total_rows) return ORACLE_BAD_ARG;
  int32_t max_len = 0;
  for (int32_t s = 0; s < num_seqs; ++s) max_len = kv_lens[s] > max_len ? kv_lens[s] : max_len;

#ifdef _OPENMP
  int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
  {
    std::vector<float> xf(static_cast<size_t>(max_len) + 1);
    std::vector<double> xd(static_cast<size_t>(max_len) + 1);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
    for (int64_t n = 0; n < n_rows; ++n) {
      const int64_t r = rows ? rows[n] : n;
      int32_t s, i, h;
      locate(pr, r, &s, &i, &h);
      double* o = out + n * head_dim;
      if (precision == 32)
        one_row<float>(pr, sm_scale, s, i, h, xf.data(), o, nullptr);
      else
        one_row<double>(pr, sm_scale, s, i, h, xd.data(), o, nullptr);
      if (out_bf16) {
        for (int32_t dd = 0; dd < head_dim; ++dd)
          out_bf16[n * head_dim + dd] = float_to_bf16_bits(static_cast<float>(o[dd]));
      }
    }
  }
  return ORACLE_OK;
}

// The normalised softmax row of one output row: p[0 .. hi-lo] for keys
// lo..hi (the visible keys, inclusive).  `p` must hold kv_lens[s] doubles.
int rpa_oracle_prow(int precision, int in_dtype, const void* q, const void* k_pages,
                    const void* v_pages, const int32_t* page_table,
                    int32_t max_pages_per_seq, const int32_t* cu_q_lens,
                    const int32_t* kv_lens, const int32_t* window, int32_t num_seqs,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, int32_t num_pages, double sm_scale, int64_t row,
                    double* p, int64_t* lo_out, int64_t* hi_out) {
  if (precision != 32 && precision != 64) return ORACLE_BAD_ARG;
  Problem pr{in_dtype, q, k_pages, v_pages, page_table, max_pages_per_seq,
             cu_q_lens, kv_lens, window, num_seqs, num_q_heads, num_kv_heads,
             head_dim, page_size, num_pages};
  int rc = validate(pr);
  if (rc != ORACLE_OK) return rc;
  const int64_t total_rows = static_cast<int64_t>(cu_q_lens[num_seqs]) * num_q_heads;
  if (row < 0 || row >= total_rows) return ORACLE_BAD_ARG;
  int32_t s, i, h;
  locate(pr, row, &s, &i, &h);
  int64_t lo, pos;
  visible_range(pr, s, i, &lo, &pos);
  std::vector<double> o(head_dim);
  if (precision == 32) {
    std::vector<float> x(static_cast<size_t>(pos - lo) + 1);
    one_row<float>(pr, sm_scale, s, i, h, x.data(), o.data(), p);
  } else {
    std::vector<double> x(static_cast<size_t>(pos - lo) + 1);
    one_row<double>(pr, sm_scale, s, i, h, x.data(), o.data(), p);
  }
  *lo_out = lo;
  *hi_out = pos;
  return ORACLE_OK;
}

// Round float32 values to bf16 bit patterns, nearest even.
void rpa_oracle_round_bf16(const float* in, uint16_t* out, int64_t n) {
  for (int64_t k = 0; k < n; ++k) out[k] = float_to_bf16_bits(in[k]);
}

}  // extern "C"
