/*
 * librpa: ragged paged attention on one NVIDIA GB300 (sm_103a).
 *
 * What the library computes (sources named by page title and section):
 *
 *  - "TPU Deep Dive" slides, chapter 8, "Continuous batching with static
 *    shapes": a serving step flattens every query token of every sequence into
 *    one array, and per-sequence metadata carries the ragged structure.  Here
 *    that is q[total_q, Hq, D] with cu_q_lens[num_seqs + 1] (prefix sums of the
 *    per-sequence query counts) and kv_lens[num_seqs].
 *  - Same deck, chapter 8, "KV cache layout", and "Pallas kernel / vLLM on TPU
 *    ... 19,511 tokens per second", section "Strategy 3": the KV cache is
 *    paged in fixed-size blocks (128 tokens there); each sequence reaches its
 *    blocks through a page table.  Here k_pages / v_pages are
 *    [num_pages, page_size, Hkv, D] and page_table is
 *    [num_seqs, max_pages_per_seq] int32 holding physical page ids.
 *  - "Chasing speed of light on TPU v6e", section "Attention" and footnote 5:
 *    the result is exact softmax attention over every key a query may see;
 *    sliding-window layers let a key be seen by the W queries that follow it
 *    (itself included).  Footnote 6: softmax accumulators are fp32.
 *  - "Pallas kernel / vLLM on TPU ...", section "Strategy 3": several query
 *    heads share one KV head (GQA/MQA); query head h reads KV head
 *    h / (Hq / Hkv).
 *
 * For sequence s with q_len = cu_q_lens[s+1] - cu_q_lens[s] and L = kv_lens[s],
 * query i (token t = cu_q_lens[s] + i) sits at position pos = L - q_len + i: the
 * new tokens are the last q_len entries of the cache, already written there
 * (by the caller, or first by rpa_forward_kv / rpa_forward_qkv, the fused KV
 * write of "TPU Deep Dive" chapter 8).  Key j is visible iff j <= pos and,
 * when window[s] > 0,
 * pos - j < window[s].  For every query head h:
 *     out[t][h] = sum_j softmax_j(sm_scale * q[t][h] . k_j) v_j
 * accumulated in fp32 and stored in the output dtype (bf16: round to nearest
 * even).
 *
 * Ownership and threading.  The caller owns every device buffer (q, pages,
 * metadata, out, workspace) and the CUDA stream.  rpa_forward allocates no
 * device memory, never synchronises, and enqueues its work on `stream` only.
 * A plan is a host object owned by the library between rpa_plan and
 * rpa_plan_destroy; it is read-only after creation, so one plan may serve many
 * rpa_forward calls (for instance every layer of a model step).  Two calls
 * that share a workspace must not overlap on the GPU.  Several host threads
 * may call at once, each with the stream's device current (see rpa_forward).
 * The calls enqueue kernels only, so they can be captured into CUDA graphs.
 *
 * Errors.  Every entry point returns an rpa_status_t.  Shapes, dtypes,
 * pointer alignment and the plan/argument match are checked on the host before
 * anything is enqueued; a failed check enqueues nothing.  Problems only the GPU
 * can see (a page id outside [0, num_pages), lengths that disagree with the
 * plan) are never trapped: the kernel skips the bad access, writes a code into
 * the workspace error word and carries on; rpa_get_device_error reads it.
 */
#ifndef RPA_H_
#define RPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA
 * header.  NULL means the legacy default stream. */
typedef struct CUstream_st* rpa_stream_t;

typedef int32_t rpa_status_t;
enum {
  RPA_OK = 0,
  RPA_ERR_INVALID_ARG = -1,          /* null pointer, bad shape or metadata   */
  RPA_ERR_UNSUPPORTED = -2,          /* head_dim / page_size / dtype / ratio  */
  RPA_ERR_WORKSPACE_TOO_SMALL = -3,  /* workspace_bytes below the plan's need */
  RPA_ERR_CUDA = -4,                 /* a CUDA runtime call failed            */
  RPA_ERR_DEVICE = -5,               /* the device error word is set          */
  RPA_ERR_PLAN_MISMATCH = -6         /* forward arguments differ from plan's  */
};

/* Element types of q, k_pages, v_pages and out (all four share one). */
enum { RPA_DTYPE_BF16 = 0, RPA_DTYPE_F32 = 1,
       RPA_DTYPE_FP8_E4M3 = 2 /* K/V pages only: OCP e4m3 bytes (bias 7, 3-bit
                                 mantissa, max 448), a float scale per KV head */ };

/* Codes written into the workspace error word by the kernels. */
enum {
  RPA_DEVERR_NONE = 0,
  RPA_DEVERR_PAGE_ID = 1,    /* a page-table entry outside [0, num_pages)       */
  RPA_DEVERR_LENGTHS = 2,    /* device lengths disagree with the plan's copies  */
  RPA_DEVERR_PLAN = 3,       /* the work list in the workspace is not this plan */
  RPA_DEVERR_TIMEOUT = 4,    /* a bounded wait inside a kernel gave up          */
  RPA_DEVERR_LAUNCH = 5      /* a kernel found its launch unusable (shared
                                memory base not 1024-byte aligned) and did
                                nothing                                        */
};

/* Kernel paths a plan may use. */
enum {
  RPA_PATH_AUTO = 0,   /* tensor-core prefill + split-KV decode where supported */
  RPA_PATH_SIMT = 1,   /* plain fp32 CUDA-core kernel for every sequence        */
  RPA_PATH_TC = 2      /* tensor-core paths; RPA_ERR_UNSUPPORTED if impossible  */
};

/* Split-KV decode kernels (rpa_plan_options.decode_kernel). */
enum {
  RPA_DECODE_KERNEL_AUTO = 0, /* the planner's choice                            */
  RPA_DECODE_KERNEL_MMA = 1,  /* CUDA-core warp MMAs (mma.sync): every decode
                                 shape of the tensor-core path, fp8 pages too   */
  RPA_DECODE_KERNEL_TC = 2    /* tensor cores (tcgen05.mma, accumulators in
                                 tensor memory): bf16 pages, head_dim 128 or
                                 256, G <= 8, page_size >= 16; else
                                 RPA_ERR_UNSUPPORTED                            */
};

/* Optional knobs for rpa_plan.  Zero-initialise and set struct_size. */
typedef struct rpa_plan_options {
  int32_t struct_size;      /* sizeof(rpa_plan_options)                         */
  int32_t path;             /* RPA_PATH_*                                       */
  int32_t q_block;          /* prefill query block, tokens (0: choose).  At most
                               one 128-row tile per CTA: 128 / G tokens (G =
                               num_q_heads / num_kv_heads); twice that runs on
                               SM pairs (as prefill_pairs = 2, half the block
                               per SM, head_dim 128 or 256); larger blocks are
                               refused with RPA_ERR_UNSUPPORTED             */
  int32_t kv_split;         /* decode split length, tokens (0: choose)          */
  int32_t num_sms;          /* SMs to plan for (0: ask the current device, else 152) */
  int32_t prefill_pairs;    /* tensor-core prefill on SM pairs (one M = 256 MMA
                               over two adjacent query blocks): 0 or 1 not
                               used (single-SM kernel), 2 required (else
                               RPA_ERR_UNSUPPORTED; head_dim 128 or 256)        */
  int32_t kv_dtype;         /* dtype of the K/V pages: 0 or `dtype` (the same),
                               or RPA_DTYPE_FP8_E4M3 with dtype BF16: decode
                               batches only (every q_len <= 1), head_dim 128 or
                               256, run through rpa_forward_fp8kv               */
  int32_t prefill_split;    /* 0 or -1: whole prefill work items; n > 0: lay
                               the items' key tiles (128 keys each) end to end
                               and cut them into ranges of n tiles, one per
                               CTA; items crossing a range boundary run as
                               parts whose fp32 partials a combine kernel
                               merges                                           */
  int32_t decode_sms;       /* batches with both decode and tensor-core prefill
                               work: 0 let the planner split the SMs between
                               the two persistent grids (HBM-bound decode,
                               tensor-bound prefill) and run them side by side,
                               or not when its cost model says one after the
                               other is faster; n > 0: decode on n SMs,
                               prefill on the rest; -1: one after the other,
                               each on every SM                                 */
  int32_t decode_kernel;    /* RPA_DECODE_KERNEL_* for the split-KV decode      */
  int32_t prefill_dynamic;  /* tensor-core prefill (single-SM kernel, whole
                               items): 0 items taken longest first by whichever
                               CTA gets free (a work counter in the workspace
                               header), -1 each CTA runs the list the planner
                               gave it (longest processing time first)         */
  int32_t prefill_grouping; /* dynamic prefill list: 0 group the (sequence, KV
                               head) pairs so that items sharing keys run
                               together when every prefill sequence sees its
                               whole prefix and their K and V outgrow L2
                               (DRAM reads near the algorithmic bytes, ~1%
                               longer on the causal 8k prefill), -1 longest
                               first over the whole batch                      */
} rpa_plan_options;

/* What a plan chose; filled by rpa_plan_get_info. */
typedef struct rpa_plan_info {
  int32_t path;             /* RPA_PATH_SIMT or RPA_PATH_TC                     */
  int32_t num_decode_seqs;  /* sequences with q_len == 1                        */
  int32_t num_prefill_seqs; /* sequences with q_len > 1                         */
  int32_t q_block;          /* prefill query block in tokens (query tokens of
                               one work item; on SM pairs, of both CTAs)     */
  int32_t kv_split;         /* decode split length in tokens                    */
  int32_t max_splits;       /* largest split count of any decode sequence       */
  int32_t num_prefill_items;/* (sequence, query block, kv head) work items      */
  int32_t prefill_ctas;     /* persistent prefill CTAs launched                 */
  int64_t workspace_bytes;  /* bytes rpa_forward needs                          */
  int32_t prefill_pairs;    /* 1: prefill runs on SM pairs, items are pairs of
                               query blocks                                     */
  int32_t kv_dtype;         /* dtype of the K/V pages (RPA_DTYPE_*)              */
  int32_t prefill_split_items; /* prefill items split across CTAs              */
  int32_t prefill_split_parts; /* parts those items became                     */
  int32_t prefill_max_tiles;   /* key tiles of the busiest prefill CTA        */
  int32_t decode_sms;          /* mixed batch run side by side: SMs of the
                                  decode grid (0: not side by side)          */
  int32_t prefill_sms;         /* ... and of the prefill grid                 */
  int32_t decode_kernel;       /* RPA_DECODE_KERNEL_MMA or _TC for the
                                  split-KV decode (0: no such decode)         */
  int32_t prefill_dynamic;     /* 1: prefill CTAs take items as they get free */
  int32_t prefill_groups;      /* dynamic prefill list: groups of (sequence,
                                  KV head) pairs run one after the other so
                                  that items sharing keys find them in L2
                                  (1: one group, longest first throughout)    */
} rpa_plan_info;

typedef struct rpa_plan rpa_plan_t;

/*
 * Build a plan from HOST copies of the ragged metadata (the scheduler).
 *
 * It classifies each sequence as decode (q_len == 1) or prefill (q_len > 1;
 * q_len == 0 contributes nothing), picks the decode split length and the
 * prefill query block, orders the prefill work items longest first over a
 * persistent grid, and sizes the workspace.  Host only: it launches nothing
 * and touches no device memory.
 *
 *   cu_q_lens_host [num_seqs+1], kv_lens_host [num_seqs]: host int32 arrays
 *       (cu_q_lens_host[0] == 0, non-decreasing; q_len <= kv_len).
 *   window_host: host int32 [num_seqs] (<= 0: full causal), or NULL (all
 *       full causal).  It must match what is later passed to rpa_forward.
 *   num_q_heads % num_kv_heads == 0.  head_dim in {64, 128, 256}; page_size
 *       a power of two in [1, 256] (the tensor-core prefill needs >= 16);
 *       dtype RPA_DTYPE_BF16 or RPA_DTYPE_F32 (F32 always takes the SIMT path,
 *       the fp32 debug build).
 *   max_pages_per_seq: row length of the page table; every sequence needs
 *       ceil(kv_len / page_size) <= max_pages_per_seq.
 *   num_pages: pages in the pool (page ids must lie in [0, num_pages)).
 *   opts: NULL for defaults.
 *   *plan receives a new plan (free with rpa_plan_destroy); *workspace_bytes
 *       (may be NULL) the device workspace rpa_forward needs.
 * Returns RPA_OK, RPA_ERR_INVALID_ARG or RPA_ERR_UNSUPPORTED; on error *plan
 * is set to NULL.
 * RPA_LOG=1 in the environment makes every rpa_plan print one line about
 * the plan it built (paths, CTAs, ranges, items, workspace) to stderr.
 */
rpa_status_t rpa_plan(rpa_plan_t** plan, const int32_t* cu_q_lens_host,
                      const int32_t* kv_lens_host, const int32_t* window_host,
                      int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t page_size, int32_t max_pages_per_seq,
                      int32_t num_pages, int32_t dtype, const rpa_plan_options* opts,
                      size_t* workspace_bytes);

/* Free a plan (NULL is a no-op).  Must not race with rpa_forward on it. */
rpa_status_t rpa_plan_destroy(rpa_plan_t* plan);

/* Copy out what the plan chose. */
rpa_status_t rpa_plan_get_info(const rpa_plan_t* plan, rpa_plan_info* info);

/*
 * Ragged paged attention for the batch the plan was built for.
 *
 * Device pointers (all on the current device, contiguous, row-major):
 *   q        [total_q, num_q_heads, head_dim]            dtype, 16-B aligned
 *   k_pages, v_pages [num_pages, page_size, num_kv_heads, head_dim]
 *                                                       dtype, 128-B aligned
 *   page_table [num_seqs, max_pages_per_seq] int32; entries past a sequence's
 *            last page are never read
 *   cu_q_lens [num_seqs+1] int32, kv_lens [num_seqs] int32: the same values
 *            the plan was built from
 *   window   [num_seqs] int32 (<= 0: full causal) or NULL (all full causal);
 *            NULL-ness and values must match the plan's window_host
 *   out      [total_q, num_q_heads, head_dim]            dtype, 16-B aligned
 *   workspace: at least the plan's workspace_bytes, 256-B aligned, and
 *            zero-filled before its first use (its error word must start at
 *            zero; the rest is scratch the call overwrites).
 *            Scratch owned by the call while it runs; the error word lives at
 *            its start and is sticky until rpa_get_device_error clears it.
 *   Pages: only the slots of keys some query of the batch sees are used;
 *            every other slot (the free slots of a sequence's last page past
 *            its kv_len, keys before every query's window, pages no sequence
 *            owns) may hold anything, NaN and infinities included.  The
 *            kernels load some of them along with the visible keys (whole
 *            boxes of a page) but zero them before any product uses them.
 * The scalar arguments must equal the plan's, else RPA_ERR_PLAN_MISMATCH.
 * sm_scale multiplies q.k before the softmax (1/sqrt(head_dim) is usual).
 * Enqueues on `stream` the split-KV decode kernel and, where a sequence is
 * cut across its CTAs, the log-sum-exp combine kernel (a programmatic
 * dependent launch), then the tensor-core prefill and the CUDA-core path, as
 * the batch needs, and returns without waiting for them.
 * Threads: calls from several host threads may run at once (launch
 * parameters are staged per thread); each calling thread must have the
 * stream's device current (cudaSetDevice, torch.cuda.set_device), else the
 * call fails with RPA_ERR_CUDA (rpa_last_cuda_error gives the cudaError_t),
 * and calls that share a workspace must be ordered on the GPU.
 * CUDA graphs: the call only enqueues kernel launches (no allocation, copy
 * or synchronisation), so it may be captured into a CUDA graph on `stream`;
 * every replay reruns the attention on the same buffers with the schedule
 * the plan held at capture (kernel parameters are baked into the graph), so
 * a new plan needs a new capture.
 */
rpa_status_t rpa_forward(const void* q, const void* k_pages, const void* v_pages,
                         const int32_t* page_table, const int32_t* cu_q_lens,
                         const int32_t* kv_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                         const int32_t* window, float sm_scale, void* out,
                         rpa_stream_t stream, const rpa_plan_t* plan, void* workspace,
                         size_t workspace_bytes);

/*
 * KV-cache write of a step's new tokens ("TPU Deep Dive" slides, chapter 8,
 * "Continuous batching with static shapes": ragged paged attention writes
 * the KV cache of the step's tokens itself).
 *
 * For every sequence s and each of its q_len = cu_q_lens[s+1] - cu_q_lens[s]
 * new tokens t = cu_q_lens[s] + i, at position pos = kv_lens[s] - q_len + i
 * (the query positions rpa_forward attends from), and every KV head g:
 *   k_pages[page_table[s][pos / page_size]][pos % page_size][g][:] = k_new[t][g][:]
 * and V alike.  Nothing else in the pool changes.
 *
 * Device pointers: k_new, v_new [total_q, num_kv_heads, head_dim] of `dtype`,
 * 16-B aligned; k_pages, v_pages, page_table, cu_q_lens, kv_lens as for
 * rpa_forward (kv_lens include the new tokens).  head_dim * element size must
 * be a multiple of 16 bytes; page_size a power of two.  `workspace` may be
 * NULL; otherwise its error word records a page id outside [0, num_pages)
 * or a position outside the page table (that row is skipped, never trapped).
 * Enqueues one kernel on `stream`; does not synchronise.
 */
rpa_status_t rpa_write_kv(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                          const int32_t* page_table, const int32_t* cu_q_lens,
                          const int32_t* kv_lens, int32_t num_seqs, int32_t total_q,
                          int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                          int32_t max_pages_per_seq, int32_t num_pages, int32_t dtype,
                          void* workspace, rpa_stream_t stream);

/*
 * q/k/v prologue: the step right before attention ("Chasing speed of light on
 * TPU v6e", section "The Long Tail": the q/k/v RMS norms and the rotary
 * embedding run in the kernel before attention, which takes q, k and v as
 * three arrays), fused with the KV-cache write.
 *
 * For every new token t = cu_q_lens[s] + i of sequence s, at position
 * pos = kv_lens[s] - q_len_s + i, and page = page_table[s][pos / page_size]:
 *   q_out[t][h][:]                        = rope(norm(q[t][h][:], q_weight), pos)
 *   k_pages[page][pos % page_size][g][:]  = rope(norm(k[t][g][:], k_weight), pos)
 *   v_pages[page][pos % page_size][g][:]  = norm(v[t][g][:], v_weight)
 * norm(x, w)_d = x_d / sqrt(mean_d(x_d^2) + eps) * w_d, or x itself when w is
 * NULL (a model whose norm scales by 1 + w passes 1 + w).
 * rope (halves convention): for i < D/2, with a = pos * rope_theta^(-2i/D),
 *   out_i = y_i cos a - y_{i+D/2} sin a,  out_{i+D/2} = y_{i+D/2} cos a + y_i sin a;
 * rope_theta <= 0: no rotation.  fp32 arithmetic; the angle is reduced
 * modulo 2 pi in extended precision (accurate for pos * frequency < 2^21).
 *
 * Device pointers: q, q_out [total_q, num_q_heads, head_dim]; k, v
 * [total_q, num_kv_heads, head_dim]; all of `dtype` (BF16 or F32), 16-B
 * aligned; q_out may equal q.  Weights: [head_dim] float32.  Pages, page
 * table and lengths as for rpa_write_kv (kv_lens include the new tokens).
 * head_dim in {64, 128, 256} (else RPA_ERR_UNSUPPORTED); page_size a power
 * of two.  `workspace` may be NULL; otherwise its error word records a page
 * id or position outside the table (that row is skipped, never trapped).
 * Enqueues one kernel on `stream`; does not synchronise.
 */
typedef struct rpa_qkv_norm {
  const float* q_weight; /* [head_dim] or NULL: q not normalised */
  const float* k_weight; /* [head_dim] or NULL: k not normalised */
  const float* v_weight; /* [head_dim] or NULL: v stored as given */
  float eps;             /* added to the mean square */
  float rope_theta;      /* rotary base (> 0), or <= 0 for none */
} rpa_qkv_norm;

rpa_status_t rpa_qkv_prologue(const void* q, const void* k, const void* v,
                              const rpa_qkv_norm* norm, void* q_out, void* k_pages,
                              void* v_pages, const int32_t* page_table,
                              const int32_t* cu_q_lens, const int32_t* kv_lens,
                              int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                              int32_t max_pages_per_seq, int32_t num_pages, int32_t dtype,
                              void* workspace, rpa_stream_t stream);

/*
 * The prologue, then the attention on its output, on one stream: the step
 * from the projection's q, k, v to the attention output.  q_buf receives
 * the normalised, rotated q (rpa_qkv_prologue's q_out) and is the attention's
 * query; the other arguments as rpa_qkv_prologue and rpa_forward (pool size
 * and page-table width are the plan's).
 */
rpa_status_t rpa_forward_qkv(const void* q, const void* k, const void* v,
                             const rpa_qkv_norm* norm, void* q_buf, void* k_pages,
                             void* v_pages, const int32_t* page_table,
                             const int32_t* cu_q_lens, const int32_t* kv_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t page_size, const int32_t* window,
                             float sm_scale, void* out, rpa_stream_t stream,
                             const rpa_plan_t* plan, void* workspace, size_t workspace_bytes);

/*
 * Decode over fp8 (e4m3) K/V pages with a float scale per KV head
 * ("TPU Deep Dive" slides, chapter 8, "KV cache layout": 8-bit KV packs four
 * per 32-bit word; halving the KV bytes halves decode's dominant traffic).
 * The stored keys and values are k_pages[...][g][:] * k_scale[g] and
 * v_pages[...][g][:] * v_scale[g]; otherwise exactly rpa_forward.  The plan
 * must have kv_dtype RPA_DTYPE_FP8_E4M3 (decode batch, bf16 q and out).
 * k_pages, v_pages: [num_pages, page_size, num_kv_heads, head_dim] bytes,
 * 128-B aligned; k_scale, v_scale: [num_kv_heads] float32 on the device.
 * The products run as f16 (e4m3 is exact in f16; q is converted bf16 -> f16
 * once per sequence), accumulation and softmax in fp32.
 */
rpa_status_t rpa_forward_fp8kv(const void* q, const void* k_pages, const void* v_pages,
                               const float* k_scale, const float* v_scale,
                               const int32_t* page_table, const int32_t* cu_q_lens,
                               const int32_t* kv_lens, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                               const int32_t* window, float sm_scale, void* out,
                               rpa_stream_t stream, const rpa_plan_t* plan, void* workspace,
                               size_t workspace_bytes);

/*
 * rpa_write_kv of k_new / v_new, then rpa_forward over the updated cache, in
 * order on `stream`: the step's cache update and its attention in one call.
 * Arguments as rpa_forward plus k_new, v_new (as rpa_write_kv); the pool
 * size and page-table width are the plan's.
 */
rpa_status_t rpa_forward_kv(const void* q, const void* k_new, const void* v_new, void* k_pages,
                            void* v_pages, const int32_t* page_table, const int32_t* cu_q_lens,
                            const int32_t* kv_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                            const int32_t* window, float sm_scale, void* out,
                            rpa_stream_t stream, const rpa_plan_t* plan, void* workspace,
                            size_t workspace_bytes);

/*
 * Read the device error word at the start of `workspace` after everything
 * enqueued on `stream` so far (this call synchronises `stream`), store it in
 * *err (an RPA_DEVERR_* code) and reset it to RPA_DEVERR_NONE.
 * workspace == NULL selects the fixed scratch of rpa_forward_decode_noalloc on
 * the current device (its error word, sticky in the same way).
 */
rpa_status_t rpa_get_device_error(void* workspace, rpa_stream_t stream, int32_t* err);

/* Zero the workspace error word (enqueued on `stream`, no synchronisation);
 * workspace == NULL: that of rpa_forward_decode_noalloc's fixed scratch. */
rpa_status_t rpa_clear_device_error(void* workspace, rpa_stream_t stream);

/*
 * Decode without a caller-supplied workspace: rpa_forward_decode_noalloc.
 *
 * For callers that cannot allocate device memory when they run attention:
 * code that executes inside a framework whose device memory is entirely owned
 * by another allocator, embedded or real-time serving loops that must not
 * call cudaMalloc (it can synchronise the device), and plug-ins that receive
 * only the tensors they work on.  The paper has no counterpart; this is a
 * deployment convenience.
 *
 * Same arguments as rpa_forward without the workspace.  The plan must hold
 * decode sequences only (q_len <= 1) on the split-KV decode kernel, else
 * RPA_ERR_UNSUPPORTED; a plan whose workspace_bytes exceeds
 * RPA_NOALLOC_SCRATCH_BYTES is rejected with RPA_ERR_WORKSPACE_TOO_SMALL.
 * The scratch is one fixed array inside the library (every GPU that loads the
 * library holds it until the process exits), shared by every call and keeping
 * the last call's contents; calls that overlap on the GPU (for example on two
 * streams) race on it.  Only its error word must start at zero: it does (the
 * array is zero when the library loads) and, like a workspace's, it is sticky:
 * a kernel that meets a bad page id or a length that disagrees with the plan
 * sets it and skips the access, and rpa_get_device_error(NULL, stream, &err)
 * reads and clears it.  The split partials are written before they are read
 * within a call.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, once per device, thread-safe) with that
 * device current; make that first call before any stream capture.  No device
 * memory is allocated or freed.  The call returns RPA_OK once its work is
 * enqueued (RPA_ERR_CUDA with rpa_last_cuda_error set if a CUDA call fails).
 */
#define RPA_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */

rpa_status_t rpa_forward_decode_noalloc(const void* q, const void* k_pages,
                                        const void* v_pages, const int32_t* page_table,
                                        const int32_t* cu_q_lens, const int32_t* kv_lens,
                                        int32_t num_seqs, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t page_size, const int32_t* window,
                                        float sm_scale, void* out, rpa_stream_t stream,
                                        const rpa_plan_t* plan);

/*
 * Kernel tracing (off by default).  Between rpa_trace_begin and rpa_trace_end,
 * every rpa_forward call records a CUDA event on its stream before its first
 * kernel and after each kernel it launches, so that the device time of each
 * launch can be read back.  Tracing state is process-wide and not thread-safe;
 * tracing adds one event record per launch to the stream.  A call captured
 * into a CUDA graph while tracing records its marks as event-record nodes of
 * the graph; rpa_trace_end then reads the times of the last replay.
 *
 * rpa_trace_begin: start recording up to `capacity` launches (1..65536).
 * rpa_trace_end: synchronise on the recorded events, write up to *count
 *     records (kernel id, device milliseconds) to `records`, set *count to the
 *     number written, and stop tracing.  Launches beyond `capacity` are not
 *     recorded.
 */
enum {
  RPA_KERNEL_DECODE_SPLIT = 0,   /* split-KV decode                    */
  RPA_KERNEL_DECODE_COMBINE = 1, /* log-sum-exp combine of cut sequences */
  RPA_KERNEL_PREFILL_TC = 2,     /* tensor-core prefill               */
  RPA_KERNEL_SIMT = 3,           /* CUDA-core (fp32) path             */
  RPA_KERNEL_KV_WRITE = 4,       /* KV-cache write of new tokens      */
  RPA_KERNEL_PROLOGUE = 5,       /* q/k/v norm + rotary + KV write    */
  RPA_KERNEL_PREFILL_COMBINE = 6 /* combine of split prefill items    */
};
typedef struct rpa_trace_record {
  int32_t kernel; /* RPA_KERNEL_* */
  float ms;       /* device time from the previous mark of the same call */
} rpa_trace_record;

rpa_status_t rpa_trace_begin(int32_t capacity);
rpa_status_t rpa_trace_end(rpa_trace_record* records, int32_t* count);

/* A static, human-readable name for a status code. */
const char* rpa_status_string(rpa_status_t status);

/* The cudaError_t behind the calling thread's last RPA_ERR_CUDA returned by
 * any entry point (0 if none): for diagnostics. */
int32_t rpa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RPA_H_ */
