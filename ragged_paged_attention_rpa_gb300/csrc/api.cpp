// The C ABI of librpa (include/rpa.h): argument checks, plan objects and the
// launch sequence of rpa_forward.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <utility>

#include "rpa.h"
#include "rpa_internal.h"

struct rpa_plan {
  rpa::Plan p;
};

namespace {

bool is_pow2(int32_t x) { return x > 0 && (x & (x - 1)) == 0; }

// RPA_LOG=1 in the environment: every rpa_plan prints one line to stderr.
bool log_plans() {
  static const bool on = [] {
    const char* v = std::getenv("RPA_LOG");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

void log_plan(const rpa::Plan& p) {
  int64_t cuts = static_cast<int64_t>(p.dcut.size());
  std::fprintf(stderr,
               "librpa plan: %d seqs (%d decode, %d prefill), %s path; decode: %d launch(es), "
               "%lld CTAs, longest range %d tokens, %lld cut sequences; prefill: %zu items on "
               "%d CTAs, q_block %d, busiest CTA %d key tiles, %d split parts; workspace %zu "
               "bytes\n",
               p.num_seqs, p.num_decode, p.num_prefill,
               p.path == RPA_PATH_TC ? "tensor-core" : "CUDA-core",
               static_cast<int>(p.dlaunch.size()), static_cast<long long>(p.decode_ctas),
               p.kv_split, static_cast<long long>(cuts), p.items.size(), p.prefill_ctas,
               p.q_block, p.prefill_max_tiles, p.n_split_items, p.ws_bytes);
}

bool aligned(const void* ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0;
}

int32_t device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

extern "C" {

rpa_status_t rpa_plan(rpa_plan_t** plan, const int32_t* cu_q_lens_host,
                      const int32_t* kv_lens_host, const int32_t* window_host,
                      int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t page_size, int32_t max_pages_per_seq,
                      int32_t num_pages, int32_t dtype, const rpa_plan_options* opts,
                      size_t* workspace_bytes) {
  if (plan == nullptr) return RPA_ERR_INVALID_ARG;
  *plan = nullptr;
  if (cu_q_lens_host == nullptr || (num_seqs > 0 && kv_lens_host == nullptr))
    return RPA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      page_size <= 0 || max_pages_per_seq < 0 || num_pages < 0)
    return RPA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return RPA_ERR_INVALID_ARG;
  if (dtype != RPA_DTYPE_BF16 && dtype != RPA_DTYPE_F32) return RPA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return RPA_ERR_UNSUPPORTED;
  if (!is_pow2(page_size) || page_size > 256) return RPA_ERR_UNSUPPORTED;
  rpa_plan_options o{};
  o.struct_size = sizeof(rpa_plan_options);
  if (opts != nullptr) {
    if (opts->struct_size < static_cast<int32_t>(sizeof(int32_t)) ||
        opts->struct_size > static_cast<int32_t>(sizeof(rpa_plan_options)))
      return RPA_ERR_INVALID_ARG;
    std::memcpy(&o, opts, static_cast<size_t>(opts->struct_size));
  }
  if (o.q_block < 0 || o.kv_split < 0 || o.num_sms < 0 || o.prefill_pairs < 0 ||
      o.prefill_pairs > 2 || o.kv_dtype < 0 || o.kv_dtype > RPA_DTYPE_FP8_E4M3 ||
      o.prefill_split < -1 || o.prefill_split > 65535 || o.decode_sms < -1 ||
      o.decode_kernel < 0 || o.decode_kernel > RPA_DECODE_KERNEL_TC || o.prefill_dynamic < -1 ||
      o.prefill_dynamic > 0 || o.prefill_grouping < -1 || o.prefill_grouping > 0)
    return RPA_ERR_INVALID_ARG;
  rpa_status_t st = rpa::validate_metadata(cu_q_lens_host, kv_lens_host, num_seqs,
                                           page_size, max_pages_per_seq);
  if (st != RPA_OK) return st;

  struct rpa_plan* pl = new (std::nothrow) struct rpa_plan();
  if (pl == nullptr) return RPA_ERR_INVALID_ARG;
  rpa::Plan& p = pl->p;
  p.num_seqs = num_seqs;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.d = head_dim;
  p.p = page_size;
  p.mpps = max_pages_per_seq;
  p.num_pages = num_pages;
  p.dtype = dtype;
  p.has_window = window_host != nullptr;
  p.total_q = cu_q_lens_host[num_seqs];
  int32_t sms = o.num_sms;
  if (sms == 0) sms = device_sm_count();
  p.num_sms = sms > 0 ? sms : 152;
  st = rpa::build_schedule(p, cu_q_lens_host, kv_lens_host, window_host, o);
  if (st != RPA_OK) {
    delete pl;
    return st;
  }
  *plan = pl;
  if (workspace_bytes) *workspace_bytes = p.ws_bytes;
  if (log_plans()) log_plan(p);
  return RPA_OK;
}

rpa_status_t rpa_plan_destroy(rpa_plan_t* plan) {
  delete plan;
  return RPA_OK;
}

rpa_status_t rpa_plan_get_info(const rpa_plan_t* plan, rpa_plan_info* info) {
  if (plan == nullptr || info == nullptr) return RPA_ERR_INVALID_ARG;
  const rpa::Plan& p = plan->p;
  info->path = p.path;
  info->num_decode_seqs = p.num_decode;
  info->num_prefill_seqs = p.num_prefill;
  // Query tokens per work item: on SM pairs each CTA holds half of them.
  info->q_block = p.prefill_pairs ? 2 * p.q_block : p.q_block;
  info->kv_split = p.kv_split;
  info->max_splits = p.max_splits;
  info->num_prefill_items = static_cast<int32_t>(p.items.size());
  info->prefill_ctas = p.prefill_ctas;
  info->workspace_bytes = static_cast<int64_t>(p.ws_bytes);
  info->prefill_pairs = p.prefill_pairs ? 1 : 0;
  info->kv_dtype = p.kv_fp8 ? RPA_DTYPE_FP8_E4M3 : p.dtype;
  info->prefill_split_items = static_cast<int32_t>(p.psplit.size());
  info->prefill_split_parts = p.n_split_items;
  info->prefill_max_tiles = p.prefill_max_tiles;
  info->decode_sms = p.overlap ? p.decode_sms : 0;
  info->prefill_sms = p.overlap ? p.prefill_sms : 0;
  info->prefill_dynamic = p.prefill_dynamic ? 1 : 0;
  info->prefill_groups = p.prefill_groups;
  info->decode_kernel = (p.num_decode > 0 && !p.simt_decode)
                            ? (p.decode_tc ? RPA_DECODE_KERNEL_TC : RPA_DECODE_KERNEL_MMA)
                            : 0;
  return RPA_OK;
}

namespace {

// Launches the attention kernels of a validated call (after the optional
// KV-cache write).
// The CUDA error behind this thread's last RPA_ERR_CUDA from a launch.
thread_local int32_t g_last_cuda_error = 0;

rpa_status_t cuda_failed(int err) {
  g_last_cuda_error = err;
  return RPA_ERR_CUDA;
}

// The second stream of a mixed batch's side-by-side grids: one per host
// thread and device, created by the thread's first such call on the device
// (non-blocking, so it never waits on the legacy default stream by itself),
// with the two events that fork it from and join it back to the caller's
// stream.  Under stream capture the fork and the join become graph edges.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  ~SideStream() {
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    if (stream) cudaStreamDestroy(stream);
  }
};
constexpr int kMaxSideDevices = 64;

int side_stream(SideStream** out) {
  static thread_local SideStream side[kMaxSideDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxSideDevices) return static_cast<int>(cudaErrorInvalidDevice);
  SideStream& r = side[dev];
  if (r.stream == nullptr) {
    if ((e = cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&r.join, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&r.stream, cudaStreamNonBlocking)) != cudaSuccess)
      return static_cast<int>(e);
  }
  *out = &r;
  return 0;
}

rpa_status_t forward_launch(const rpa::Plan& p, const rpa::Args& a,
                            const rpa::KvWriteArgs* kvw, rpa_stream_t stream,
                            const rpa::PrologueArgs* pro = nullptr) {
  int err = 0;
  rpa::trace_start(stream);
  if (kvw != nullptr && (err = rpa::launch_kv_write(*kvw, stream)) != 0) return cuda_failed(err);
  if (pro != nullptr && (err = rpa::launch_prologue(*pro, stream)) != 0) return cuda_failed(err);
  const bool decode = p.num_decode > 0 && !p.simt_decode;
  const bool prefill = !p.items.empty();
  if (decode && prefill && p.overlap) {
    // Side by side: the prefill grid (prefill_sms CTAs) on the side stream,
    // forked after everything enqueued so far, the decode grid (decode_sms
    // CTAs) on the caller's stream; the caller's stream then waits for the
    // prefill.  Together the grids fill the SMs once.
    SideStream* side = nullptr;
    if ((err = side_stream(&side)) != 0) return cuda_failed(err);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaEventRecord(side->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
    if (e != cudaSuccess) return cuda_failed(static_cast<int>(e));
    rpa_stream_t ss = reinterpret_cast<rpa_stream_t>(side->stream);
    rpa::trace_start(ss);
    err = rpa::launch_prefill_tc(p, a, ss);
    if (err) return cuda_failed(err);
    if ((e = cudaEventRecord(side->join, side->stream)) != cudaSuccess)
      return cuda_failed(static_cast<int>(e));
    err = rpa::launch_decode(p, a, stream);
    // Join even when the decode launch failed, so that a capture in progress
    // is left with every forked stream joined.
    e = cudaStreamWaitEvent(s, side->join, 0);
    if (err) return cuda_failed(err);
    if (e != cudaSuccess) return cuda_failed(static_cast<int>(e));
  } else {
    if (decode) {
      err = rpa::launch_decode(p, a, stream);
      if (err) return cuda_failed(err);
    }
    if (prefill) {
      err = p.prefill_pairs ? rpa::launch_prefill_pair(p, a, stream)
                            : rpa::launch_prefill_tc(p, a, stream);
      if (err) return cuda_failed(err);
    }
  }
  if (p.simt_decode || p.simt_prefill) {
    err = rpa::launch_simt(p, a, stream);
    if (err) return cuda_failed(err);
  }
  return RPA_OK;
}

}  // namespace

rpa_status_t rpa_forward(const void* q, const void* k_pages, const void* v_pages,
                         const int32_t* page_table, const int32_t* cu_q_lens,
                         const int32_t* kv_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                         const int32_t* window, float sm_scale, void* out,
                         rpa_stream_t stream, const rpa_plan_t* plan, void* workspace,
                         size_t workspace_bytes) {
  if (plan == nullptr) return RPA_ERR_INVALID_ARG;
  const rpa::Plan& p = plan->p;
  if (num_seqs != p.num_seqs || num_q_heads != p.hq || num_kv_heads != p.hkv ||
      head_dim != p.d || page_size != p.p || (window != nullptr) != p.has_window || p.kv_fp8)
    return RPA_ERR_PLAN_MISMATCH;
  if (workspace == nullptr || !aligned(workspace, 256)) return RPA_ERR_INVALID_ARG;
  if (workspace_bytes < p.ws_bytes) return RPA_ERR_WORKSPACE_TOO_SMALL;
  if (p.total_q == 0) return RPA_OK;  // nothing to compute
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || page_table == nullptr ||
      cu_q_lens == nullptr || kv_lens == nullptr || out == nullptr)
    return RPA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pages, 128) ||
      !aligned(v_pages, 128) || !aligned(page_table, 4) || !aligned(cu_q_lens, 4) ||
      !aligned(kv_lens, 4) || !aligned(window, 4))
    return RPA_ERR_INVALID_ARG;

  rpa::Args a{q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window, sm_scale,
              out, static_cast<unsigned char*>(workspace)};
  return forward_launch(p, a, nullptr, stream);
}

rpa_status_t rpa_forward_fp8kv(const void* q, const void* k_pages, const void* v_pages,
                               const float* k_scale, const float* v_scale,
                               const int32_t* page_table, const int32_t* cu_q_lens,
                               const int32_t* kv_lens, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                               const int32_t* window, float sm_scale, void* out,
                               rpa_stream_t stream, const rpa_plan_t* plan, void* workspace,
                               size_t workspace_bytes) {
  if (plan == nullptr) return RPA_ERR_INVALID_ARG;
  const rpa::Plan& p = plan->p;
  if (num_seqs != p.num_seqs || num_q_heads != p.hq || num_kv_heads != p.hkv ||
      head_dim != p.d || page_size != p.p || (window != nullptr) != p.has_window || !p.kv_fp8)
    return RPA_ERR_PLAN_MISMATCH;
  if (workspace == nullptr || !aligned(workspace, 256)) return RPA_ERR_INVALID_ARG;
  if (workspace_bytes < p.ws_bytes) return RPA_ERR_WORKSPACE_TOO_SMALL;
  if (p.total_q == 0) return RPA_OK;
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || k_scale == nullptr ||
      v_scale == nullptr || page_table == nullptr || cu_q_lens == nullptr ||
      kv_lens == nullptr || out == nullptr)
    return RPA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pages, 128) ||
      !aligned(v_pages, 128) || !aligned(k_scale, 4) || !aligned(v_scale, 4) ||
      !aligned(page_table, 4) || !aligned(cu_q_lens, 4) || !aligned(kv_lens, 4) ||
      !aligned(window, 4))
    return RPA_ERR_INVALID_ARG;
  rpa::Args a{q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window, sm_scale,
              out, static_cast<unsigned char*>(workspace), k_scale, v_scale};
  return forward_launch(p, a, nullptr, stream);
}

rpa_status_t rpa_forward_kv(const void* q, const void* k_new, const void* v_new, void* k_pages,
                            void* v_pages, const int32_t* page_table, const int32_t* cu_q_lens,
                            const int32_t* kv_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                            const int32_t* window, float sm_scale, void* out,
                            rpa_stream_t stream, const rpa_plan_t* plan, void* workspace,
                            size_t workspace_bytes) {
  if (plan == nullptr) return RPA_ERR_INVALID_ARG;
  const rpa::Plan& p = plan->p;
  if (num_seqs != p.num_seqs || num_q_heads != p.hq || num_kv_heads != p.hkv ||
      head_dim != p.d || page_size != p.p || (window != nullptr) != p.has_window)
    return RPA_ERR_PLAN_MISMATCH;
  if (workspace == nullptr || !aligned(workspace, 256)) return RPA_ERR_INVALID_ARG;
  if (workspace_bytes < p.ws_bytes) return RPA_ERR_WORKSPACE_TOO_SMALL;
  if (p.total_q == 0) return RPA_OK;
  if (q == nullptr || k_new == nullptr || v_new == nullptr || k_pages == nullptr ||
      v_pages == nullptr || page_table == nullptr || cu_q_lens == nullptr ||
      kv_lens == nullptr || out == nullptr)
    return RPA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
      !aligned(k_pages, 128) || !aligned(v_pages, 128) || !aligned(page_table, 4) ||
      !aligned(cu_q_lens, 4) || !aligned(kv_lens, 4) || !aligned(window, 4))
    return RPA_ERR_INVALID_ARG;
  const int32_t esz = p.dtype == RPA_DTYPE_F32 ? 4 : 2;
  rpa::KvWriteArgs kw{k_new, v_new, k_pages, v_pages, page_table, cu_q_lens, kv_lens,
                      static_cast<unsigned char*>(workspace), p.num_seqs,
                      static_cast<int32_t>(p.total_q), p.hkv, p.d, esz, p.p, p.mpps,
                      p.num_pages};
  rpa::Args a{q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window, sm_scale,
              out, static_cast<unsigned char*>(workspace)};
  return forward_launch(p, a, &kw, stream);
}

rpa_status_t rpa_write_kv(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                          const int32_t* page_table, const int32_t* cu_q_lens,
                          const int32_t* kv_lens, int32_t num_seqs, int32_t total_q,
                          int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                          int32_t max_pages_per_seq, int32_t num_pages, int32_t dtype,
                          void* workspace, rpa_stream_t stream) {
  if (num_seqs < 1 || total_q < 0 || num_kv_heads < 1 || head_dim < 1 || page_size < 1 ||
      (page_size & (page_size - 1)) != 0 || max_pages_per_seq < 1 || num_pages < 1)
    return RPA_ERR_INVALID_ARG;
  if (dtype != RPA_DTYPE_BF16 && dtype != RPA_DTYPE_F32) return RPA_ERR_INVALID_ARG;
  const int32_t esz = dtype == RPA_DTYPE_F32 ? 4 : 2;
  if ((static_cast<int64_t>(head_dim) * esz) % 16 != 0) return RPA_ERR_UNSUPPORTED;
  if (total_q == 0) return RPA_OK;
  if (k_new == nullptr || v_new == nullptr || k_pages == nullptr || v_pages == nullptr ||
      page_table == nullptr || cu_q_lens == nullptr || kv_lens == nullptr)
    return RPA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pages, 16) ||
      !aligned(v_pages, 16) || !aligned(page_table, 4) || !aligned(cu_q_lens, 4) ||
      !aligned(kv_lens, 4) || (workspace != nullptr && !aligned(workspace, 256)))
    return RPA_ERR_INVALID_ARG;
  rpa::KvWriteArgs kw{k_new, v_new, k_pages, v_pages, page_table, cu_q_lens, kv_lens,
                      static_cast<unsigned char*>(workspace), num_seqs, total_q, num_kv_heads,
                      head_dim, esz, page_size, max_pages_per_seq, num_pages};
  rpa::trace_start(stream);
  if (int err = rpa::launch_kv_write(kw, stream)) return cuda_failed(err);
  return RPA_OK;
}

rpa_status_t rpa_qkv_prologue(const void* q, const void* k, const void* v,
                              const rpa_qkv_norm* norm, void* q_out, void* k_pages,
                              void* v_pages, const int32_t* page_table,
                              const int32_t* cu_q_lens, const int32_t* kv_lens,
                              int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                              int32_t max_pages_per_seq, int32_t num_pages, int32_t dtype,
                              void* workspace, rpa_stream_t stream) {
  if (norm == nullptr || num_seqs < 1 || total_q < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
      head_dim < 1 || page_size < 1 || (page_size & (page_size - 1)) != 0 ||
      max_pages_per_seq < 1 || num_pages < 1 || !(norm->eps >= 0.f))
    return RPA_ERR_INVALID_ARG;
  if (dtype != RPA_DTYPE_BF16 && dtype != RPA_DTYPE_F32) return RPA_ERR_INVALID_ARG;
  if (!rpa::prologue_supported(head_dim)) return RPA_ERR_UNSUPPORTED;
  if (total_q == 0) return RPA_OK;
  if (q == nullptr || k == nullptr || v == nullptr || q_out == nullptr || k_pages == nullptr ||
      v_pages == nullptr || page_table == nullptr || cu_q_lens == nullptr || kv_lens == nullptr)
    return RPA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_out, 16) ||
      !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(page_table, 4) ||
      !aligned(cu_q_lens, 4) || !aligned(kv_lens, 4) || !aligned(norm->q_weight, 4) ||
      !aligned(norm->k_weight, 4) || !aligned(norm->v_weight, 4) ||
      (workspace != nullptr && !aligned(workspace, 256)))
    return RPA_ERR_INVALID_ARG;
  rpa::PrologueArgs pa{q, k, v, norm->q_weight, norm->k_weight, norm->v_weight, norm->eps,
                       norm->rope_theta, q_out, k_pages, v_pages, page_table, cu_q_lens,
                       kv_lens, static_cast<unsigned char*>(workspace), num_seqs, total_q,
                       num_q_heads, num_kv_heads, head_dim,
                       dtype == RPA_DTYPE_F32 ? 4 : 2, page_size, max_pages_per_seq,
                       num_pages};
  rpa::trace_start(stream);
  if (int err = rpa::launch_prologue(pa, stream)) return cuda_failed(err);
  return RPA_OK;
}

rpa_status_t rpa_forward_qkv(const void* q, const void* k, const void* v,
                             const rpa_qkv_norm* norm, void* q_buf, void* k_pages,
                             void* v_pages, const int32_t* page_table,
                             const int32_t* cu_q_lens, const int32_t* kv_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t page_size, const int32_t* window,
                             float sm_scale, void* out, rpa_stream_t stream,
                             const rpa_plan_t* plan, void* workspace, size_t workspace_bytes) {
  if (plan == nullptr || norm == nullptr || !(norm->eps >= 0.f)) return RPA_ERR_INVALID_ARG;
  const rpa::Plan& p = plan->p;
  if (num_seqs != p.num_seqs || num_q_heads != p.hq || num_kv_heads != p.hkv ||
      head_dim != p.d || page_size != p.p || (window != nullptr) != p.has_window || p.kv_fp8)
    return RPA_ERR_PLAN_MISMATCH;
  if (!rpa::prologue_supported(head_dim)) return RPA_ERR_UNSUPPORTED;
  if (workspace == nullptr || !aligned(workspace, 256)) return RPA_ERR_INVALID_ARG;
  if (workspace_bytes < p.ws_bytes) return RPA_ERR_WORKSPACE_TOO_SMALL;
  if (p.total_q == 0) return RPA_OK;
  if (q == nullptr || k == nullptr || v == nullptr || q_buf == nullptr || k_pages == nullptr ||
      v_pages == nullptr || page_table == nullptr || cu_q_lens == nullptr ||
      kv_lens == nullptr || out == nullptr)
    return RPA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_buf, 16) ||
      !aligned(out, 16) || !aligned(k_pages, 128) || !aligned(v_pages, 128) ||
      !aligned(page_table, 4) || !aligned(cu_q_lens, 4) || !aligned(kv_lens, 4) ||
      !aligned(window, 4) || !aligned(norm->q_weight, 4) || !aligned(norm->k_weight, 4) ||
      !aligned(norm->v_weight, 4))
    return RPA_ERR_INVALID_ARG;
  rpa::PrologueArgs pa{q, k, v, norm->q_weight, norm->k_weight, norm->v_weight, norm->eps,
                       norm->rope_theta, q_buf, k_pages, v_pages, page_table, cu_q_lens,
                       kv_lens, static_cast<unsigned char*>(workspace), p.num_seqs,
                       static_cast<int32_t>(p.total_q), p.hq, p.hkv, p.d,
                       p.dtype == RPA_DTYPE_F32 ? 4 : 2, p.p, p.mpps, p.num_pages};
  rpa::Args a{q_buf, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window, sm_scale,
              out, static_cast<unsigned char*>(workspace)};
  return forward_launch(p, a, nullptr, stream, &pa);
}

rpa_status_t rpa_forward_decode_noalloc(const void* q, const void* k_pages,
                                        const void* v_pages, const int32_t* page_table,
                                        const int32_t* cu_q_lens, const int32_t* kv_lens,
                                        int32_t num_seqs, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t page_size, const int32_t* window,
                                        float sm_scale, void* out, rpa_stream_t stream,
                                        const rpa_plan_t* plan) {
  if (plan == nullptr) return RPA_ERR_INVALID_ARG;
  const rpa::Plan& p = plan->p;
  if (num_seqs != p.num_seqs || num_q_heads != p.hq || num_kv_heads != p.hkv ||
      head_dim != p.d || page_size != p.p || (window != nullptr) != p.has_window || p.kv_fp8)
    return RPA_ERR_PLAN_MISMATCH;
  if (p.num_prefill > 0 || p.simt_decode || p.dtype != RPA_DTYPE_BF16)
    return RPA_ERR_UNSUPPORTED;
  if (p.ws_bytes > RPA_NOALLOC_SCRATCH_BYTES) return RPA_ERR_WORKSPACE_TOO_SMALL;
  if (p.total_q == 0) return RPA_OK;
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || page_table == nullptr ||
      cu_q_lens == nullptr || kv_lens == nullptr || out == nullptr)
    return RPA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pages, 128) ||
      !aligned(v_pages, 128) || !aligned(page_table, 4) || !aligned(cu_q_lens, 4) ||
      !aligned(kv_lens, 4) || !aligned(window, 4))
    return RPA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (int err = rpa::noalloc_scratch(&scratch)) return cuda_failed(err);
  // The scratch's error word started at zero and stays sticky until
  // rpa_get_device_error(NULL, ...) reads and clears it; nothing else in the
  // scratch has to start at zero.
  rpa::Args a{q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window, sm_scale,
              out, static_cast<unsigned char*>(scratch)};
  rpa::trace_start(stream);
  if (int err = rpa::launch_decode(p, a, stream)) return cuda_failed(err);
  return RPA_OK;
}

int32_t rpa_last_cuda_error(void) { return g_last_cuda_error; }

rpa_status_t rpa_get_device_error(void* workspace, rpa_stream_t stream, int32_t* err) {
  if (err == nullptr) return RPA_ERR_INVALID_ARG;
  if (workspace == nullptr) {
    // The fixed scratch of rpa_forward_decode_noalloc on the current device.
    if (int e = rpa::noalloc_scratch(&workspace)) return cuda_failed(e);
  }
  int32_t v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, 2 * sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_failed(static_cast<int>(e));
  *err = v;
  return v == RPA_DEVERR_NONE ? RPA_OK : RPA_ERR_DEVICE;
}

rpa_status_t rpa_clear_device_error(void* workspace, rpa_stream_t stream) {
  if (workspace == nullptr) {
    if (int e = rpa::noalloc_scratch(&workspace)) return cuda_failed(e);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaError_t e = cudaMemsetAsync(workspace, 0, 2 * sizeof(int32_t), s))
    return cuda_failed(static_cast<int>(e));
  return RPA_OK;
}

const char* rpa_status_string(rpa_status_t status) {
  switch (status) {
    case RPA_OK: return "RPA_OK";
    case RPA_ERR_INVALID_ARG: return "RPA_ERR_INVALID_ARG: bad pointer, shape or metadata";
    case RPA_ERR_UNSUPPORTED: return "RPA_ERR_UNSUPPORTED: shape or dtype not supported";
    case RPA_ERR_WORKSPACE_TOO_SMALL: return "RPA_ERR_WORKSPACE_TOO_SMALL";
    case RPA_ERR_CUDA: return "RPA_ERR_CUDA: a CUDA runtime call failed";
    case RPA_ERR_DEVICE: return "RPA_ERR_DEVICE: a kernel reported an error";
    case RPA_ERR_PLAN_MISMATCH: return "RPA_ERR_PLAN_MISMATCH: arguments differ from the plan";
    default: return "unknown rpa status";
  }
}

}  // extern "C"

namespace rpa {

int ensure_dynamic_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return 0;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return static_cast<int>(e);
  done.insert({kernel, dev});
  return 0;
}

}  // namespace rpa
