/*
 * hdpattn.h -- C ABI of libhdpattn.so: document-masked causal attention over
 * a packed, mixed-length micro-batch, with the sequences cut into chunks of at
 * most C tokens, the causal (query chunk, key chunk) blocks computed as partial
 * (O, LSE) results, and the partials merged exactly by log-sum-exp.  One GPU
 * (sm_103a); everything runs in this library's CUDA kernels.
 *
 * Source of the method: "ByteScale: Communication-Efficient Scaling of LLM
 * Training with a 2048K Context Length on 16384 GPUs" (AI training network
 * primer research digest):
 *   section 1      capacity C: each rank holds at most C tokens;
 *   section 2      attention work grows as the square of each sequence length,
 *                  so equal-token micro-batches carry unequal FLOPs;
 *   section 3.1    a sequence longer than C spans ceil(s/C) ranks, shorter ones
 *                  are packed onto one rank by best fit (Figure 2);
 *   section 3.2    a query attends only to its own sequence; each ring step
 *                  computes one C x C block whose partial results are combined.
 *
 * Conventions for every call:
 *   - Pointers named d_* and every tensor argument are DEVICE pointers on the
 *     current CUDA device; other pointers are host pointers.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All work is enqueued asynchronously on it; the only call that blocks the
 *     host is hdp_plan_create (one small device-to-host read of totals) and
 *     hdp_device_status (which synchronizes the stream by design).
 *   - The caller owns every buffer it passes and must keep it alive until the
 *     stream has finished the work.  A plan owns its tables.
 *   - Errors are reported only through the return code; nothing aborts and no
 *     exception crosses the ABI.  hdp_last_error_message() gives a thread-local
 *     human-readable reason for the last failing call on this thread.
 *   - Layouts: Q and O are [T][hq][d] bf16, K and V are [T][hkv][d] bf16, all
 *     row-major and contiguous; LSE is [hq][T] fp32 in natural log.  Query head
 *     h reads key/value head h / (hq / hkv).  T = total tokens, at most 2^31-1.
 */
#ifndef HDPATTN_H_
#define HDPATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HDP_OK = 0,
  HDP_ERR_INVALID_ARGUMENT = 1, /* a documented precondition does not hold   */
  HDP_ERR_UNSUPPORTED = 2,      /* valid, but outside what the kernels cover  */
  HDP_ERR_OUT_OF_MEMORY = 3,    /* a device allocation failed                 */
  HDP_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed          */
  HDP_ERR_DEVICE_TIMEOUT = 5    /* a kernel's bounded wait expired (see hdp_device_status) */
} hdp_status_t;

/* Attention modes. */
#define HDP_MODE_FUSED 0 /* every query tile runs over all its causal-prior key
                            tiles; the chunk partials are merged in registers
                            by the online softmax (exactly the LSE merge) */
#define HDP_MODE_SPLIT 1 /* each causal block (qc, kc) is written as a partial
                            (O, LSE) to the workspace, then hdp_lse_merge runs */

/* Plan creation flags. */
#define HDP_PLAN_DEFAULT 0u
#define HDP_PLAN_NO_SHARDS 1u /* skip best-fit shard packing (num_shards = 0,
                                 shard_of_chunk = NULL); for callers that only
                                 need the attention tables */
#define HDP_PLAN_NO_SPLIT 2u  /* skip the SPLIT work list (num_tiles_split = 0,
                                 tiles_split = NULL), a table for callers that
                                 schedule blocks themselves; this library's
                                 FUSED and SPLIT attention both walk the fused
                                 list and run on such a plan unchanged */

typedef struct hdp_plan_s* hdp_plan_t;

/* Read-only view of a plan.  All table pointers are device pointers owned by
 * the plan; they stay valid until hdp_plan_destroy. */
typedef struct {
  int32_t num_docs;      /* n                                                  */
  int32_t capacity;      /* C                                                  */
  int32_t num_chunks;    /* N_c = sum_i ceil(s_i / C)                          */
  int32_t num_shards;    /* shards after packing (0 with HDP_PLAN_NO_SHARDS)   */
  int64_t num_blocks;    /* N_b = sum_i n_i (n_i + 1) / 2 causal (qc, kc) blocks */
  int64_t total_tokens;  /* T                                                  */
  int32_t max_doc_len;   /* longest document                                   */
  int32_t tile;          /* query/key tile rows used by the work lists (128)   */
  const int32_t* cu_seqlens;     /* [n+1] exclusive prefix sum of lengths       */
  const int32_t* chunk_offsets;  /* [n+1] first global chunk of each document   */
  const int64_t* block_offsets;  /* [n+1] first block of each document          */
  const int32_t* chunk_table;    /* [N_c][4] {doc, index in doc, first token, length} */
  const int32_t* block_table;    /* [N_b][2] {q chunk, kv chunk}, ordered by doc,
                                    then q chunk, then kv chunk ascending      */
  const int64_t* chunk_pairs;    /* [N_c] causal (query, key) pairs per chunk  */
  const int32_t* shard_of_chunk; /* [N_c] shard of each chunk (NULL if skipped) */
  /* Query-tile work lists, heaviest first (weight descending, then
   * enumeration order).  Rows of 8 int32: {q_row0, q_rows, kv_row0, kv_len,
   * block (-1 in the fused list), row offset of the tile inside its query
   * chunk (inside its document in the fused list), weight = key tiles,
   * document length (fused list; 0 in the split list)}.  Fully masked
   * (cross-document or future) tiles never appear.  In the fused list the
   * rows of query tile j of a document also describe its key tile j (same
   * rows), which the backward pass walks.  Both attention modes walk the
   * fused list; the split list is a table for callers that schedule one
   * causal block at a time. */
  const int32_t* tiles_fused;    /* [num_tiles_fused][8] one per document query tile */
  int64_t num_tiles_fused;
  const int32_t* tiles_split;    /* [num_tiles_split][8] one per block query tile
                                    (NULL unless C is a multiple of `tile`)   */
  int64_t num_tiles_split;
} hdp_plan_view_t;

/*
 * Sharding plan (section 3.1, Figure 2): chunk every document into
 * ceil(s/C) chunks of at most C tokens, enumerate the causal blocks
 * (qc, kc), kc <= qc, of each document, count the causal pairs of each chunk,
 * pack the chunks into shards (every full C-token chunk gets its own shard in
 * chunk order; shorter pieces -- short documents and tails -- are packed by
 * best-fit decreasing: length descending, document ascending, each into the
 * open piece shard with the least remaining capacity that fits, lowest id on
 * ties, else a new shard), and build the query-tile work lists.
 *   d_lengths  [num_docs] int32 device array, every entry >= 1.
 *   num_docs   >= 1.      capacity >= 1.
 *   flags      HDP_PLAN_DEFAULT, or HDP_PLAN_NO_SHARDS and / or
 *              HDP_PLAN_NO_SPLIT OR-ed together.
 *   out        receives the plan (NULL on failure).
 * Blocks the host once, to read the totals and the shard count back (best fit
 * runs on the device before that read-back).  Fails with INVALID_ARGUMENT for a
 * length < 1 or T >= 2^31, UNSUPPORTED when more than 65,536 sub-capacity
 * pieces need best-fit packing (use HDP_PLAN_NO_SHARDS), OUT_OF_MEMORY if the
 * tables cannot be allocated.  Tables are allocated stream-ordered on
 * `stream`.
 */
hdp_status_t hdp_plan_create(const int32_t* d_lengths, int32_t num_docs, int32_t capacity, void* stream,
                             hdp_plan_t* out);
hdp_status_t hdp_plan_create_ex(const int32_t* d_lengths, int32_t num_docs, int32_t capacity, uint32_t flags,
                                void* stream, hdp_plan_t* out);
hdp_status_t hdp_plan_view(hdp_plan_t plan, hdp_plan_view_t* view);
/* Frees the plan's tables, stream-ordered on the stream the plan was created
 * on; work on other streams that uses the plan must be ordered before it. */
hdp_status_t hdp_plan_destroy(hdp_plan_t plan);

/*
 * Workspace bytes hdp_attention_fwd needs for (plan, hq, d, mode).  FUSED needs
 * none (0).  SPLIT needs the partials: N_b * C * hq * (d + 1) * 4 bytes, laid
 * out as o_part [N_b][C][hq][d] fp32 followed by lse_part [N_b][hq][C] fp32
 * (256-byte aligned), the format hdp_lse_merge reads.
 */
hdp_status_t hdp_attention_workspace_bytes(hdp_plan_t plan, int32_t hq, int32_t d, int32_t mode, size_t* bytes);

/*
 * Document-masked causal attention forward (section 3.2): for every document,
 * query head h and doc-local query p,
 *   S_j = scale * q_p . k_j for doc-local keys j <= p,
 *   lse = ln sum_j exp(S_j),  o = sum_j exp(S_j - lse) v_j,
 * with query tiles scheduled heaviest first and fully masked tiles skipped.
 *   q [T][hq][d], k/v [T][hkv][d] bf16; o [T][hq][d] bf16 (round to nearest
 *   even); lse [hq][T] fp32 (natural log).
 *   hq % hkv == 0; d == 64 or 128 (else UNSUPPORTED); scale > 0.
 *   FUSED: o and lse are final.  SPLIT: needs capacity % 128 == 0 and a
 *   workspace of hdp_attention_workspace_bytes; writes the partials there,
 *   then merges them into o and lse with hdp_lse_merge on the same stream.
 *   Each partial covers exactly its block's C keys: the kernel walks the
 *   fused list and writes a partial at every chunk end of a query tile's
 *   key range.
 *   When one kv head's K and V rows of the longest document exceed the
 *   device's L2, the CTAs of a launch pace each other along the key range so
 *   that they share K/V tiles in L2.  Their positions go through one static
 *   device table (its address cached per device, like the scratch of
 *   hdp_attention_fwd_split_noalloc); concurrent launches share it, which can
 *   only weaken the pacing (every hold is bounded) and never changes the
 *   results.
 *   q, k, v, o must be 16-byte aligned.
 * Device-side wait timeouts are reported by hdp_device_status.
 */
hdp_status_t hdp_attention_fwd(hdp_plan_t plan, const void* q, const void* k, const void* v, int32_t hq,
                               int32_t hkv, int32_t d, float scale, int32_t mode, void* workspace,
                               size_t workspace_bytes, void* o, float* lse, void* stream);

/*
 * SPLIT-mode attention that allocates nothing.  The paper has no counterpart;
 * this entry exists for callers that cannot allocate device memory at the time
 * they run attention: serving processes that reserve all device memory at
 * start-up and forbid allocation on the request path, host programs whose own
 * allocator owns the device memory, and callers that must avoid the
 * device-wide synchronisation cudaMalloc/cudaFree can imply.
 * Same arguments and results as hdp_attention_fwd with mode HDP_MODE_SPLIT,
 * but the partials live in a fixed 64 MiB scratch array inside the library
 * (every GPU that loads the library holds it until the process exits).
 *   - Plans whose SPLIT workspace (hdp_attention_workspace_bytes) exceeds
 *     64 MiB are rejected with HDP_ERR_INVALID_ARGUMENT and a message.
 *   - No cudaMalloc, cudaFree or other allocating call is made.  The first
 *     call on a device resolves the scratch array's device address (once per
 *     device, with that device current) and caches it.  A cudaDeviceReset,
 *     or anything else that destroys the device's primary context,
 *     invalidates the cached address (and those of the device error word and
 *     the attention pacing table): do not call the library on that device
 *     after such a reset in the same process.
 *   - Every call shares the one scratch array, which keeps the last call's
 *     contents; every partial a call reads is written by that call first, so
 *     nothing needs to start at zero.  Calls that overlap on the GPU (other
 *     streams, other threads) race on the array and must be serialised by the
 *     caller.
 */
hdp_status_t hdp_attention_fwd_split_noalloc(hdp_plan_t plan, const void* q, const void* k, const void* v,
                                             int32_t hq, int32_t hkv, int32_t d, float scale, void* o, float* lse,
                                             void* stream);

/*
 * Backward pass of the same attention (the training step of section 5 times
 * forward and backward together; each document's gradient is independent,
 * section 3.2).  With P = exp(scale Q K^T - lse) over the causal keys of each
 * query's own document and D = rowsum(dout * o):
 *   dv = P^T dout,  dS = P * (dout V^T - D),  dk = scale dS^T Q,  dq = scale dS K
 * summed over the query heads of each GQA group for dk and dv.
 *   q, o, dout, dq: [T][hq][d] bf16;  k, v, dk, dv: [T][hkv][d] bf16;
 *   lse: [hq][T] fp32, natural log, as written by hdp_attention_fwd for this
 *   plan (FUSED or SPLIT) and `o` its output.
 * workspace: device, 256-byte aligned, at least
 * hdp_attention_bwd_workspace_bytes (D in fp32).  Deterministic: no atomics;
 * dq, dk and dv each accumulate in one CTA in a fixed order.
 * d == 64 or 128 (UNSUPPORTED otherwise); tensor pointers 16-byte aligned.
 * Every output row is written.
 */
hdp_status_t hdp_attention_bwd_workspace_bytes(hdp_plan_t plan, int32_t hq, int32_t d, size_t* bytes);
hdp_status_t hdp_attention_bwd(hdp_plan_t plan, const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, int32_t hq, int32_t hkv, int32_t d, float scale,
                               void* workspace, size_t workspace_bytes, void* dq, void* dk, void* dv, void* stream);

/*
 * Exact log-sum-exp merge of the causal blocks of every query chunk
 * (section 3.2: the partial results of the ring steps are combined):
 *   M = max_k lse_k, lse = M + ln sum_k exp(lse_k - M), o = sum_k exp(lse_k - lse) o_k
 * over the blocks (qc, kc), kc = 0..qc, of the chunk.
 *   o_part [N_b][C][hq][d] fp32, lse_part [N_b][hq][C] fp32 (the SPLIT
 *   workspace layout); o [T][hq][d] bf16, lse [hq][T] fp32.  d == 64 or 128.
 *   The plan's capacity must be a multiple of 128 (as for SPLIT attention):
 *   INVALID_ARGUMENT otherwise.
 */
hdp_status_t hdp_lse_merge(hdp_plan_t plan, const float* o_part, const float* lse_part, int32_t hq, int32_t d,
                           void* o, float* lse, void* stream);

/*
 * The same merge on plain arrays: m partials of `rows` rows of d values.
 *   o_parts [m][rows][d] fp32, lse_parts [m][rows] fp32 -> o [rows][d] bf16,
 *   lse [rows] fp32.  A partial with lse = -inf contributes nothing; a row whose
 *   partials are all -inf gets lse = -inf and o = 0.  m >= 1, d % 4 == 0,
 *   d <= 256.
 */
hdp_status_t hdp_lse_merge_rows(int32_t m, int64_t rows, int32_t d, const float* o_parts, const float* lse_parts,
                                void* o, float* lse, void* stream);

/*
 * Useful causal-attention FLOPs per shard (section 2: micro-batches of equal
 * tokens differ in FLOPs): d_out[s] = sum over the shard's chunks of
 * 4 * d * hq * chunk_pairs, exact in int64.  d_out [num_shards] int64 device.
 * INVALID_ARGUMENT if the plan was created with HDP_PLAN_NO_SHARDS.
 */
hdp_status_t hdp_flops_per_shard(hdp_plan_t plan, int32_t d, int32_t hq, int64_t* d_out, void* stream);

/*
 * Synchronizes `stream` and reports (then clears) a device-side failure
 * recorded by an earlier kernel of this library on the current device:
 * HDP_ERR_DEVICE_TIMEOUT when a bounded wait expired, HDP_ERR_CUDA when the
 * stream reports a CUDA error, else HDP_OK.
 */
hdp_status_t hdp_device_status(void* stream);

const char* hdp_status_string(hdp_status_t status);
const char* hdp_last_error_message(void);

/* Number of CUDA kernels this library has enqueued in this process (all
 * devices, all threads).  Diagnostic counter; never reset. */
uint64_t hdp_kernel_launch_count(void);

/* Number of times this library has blocked the host on a stream in this
 * process: hdp_plan_create's one read-back and hdp_device_status.  Diagnostic
 * counter; never reset. */
uint64_t hdp_host_sync_count(void);

/*
 * Budget of the bounded waits of the attention forward and backward kernels,
 * in SM clocks, for the launches this process makes after the call (all
 * devices, all threads).
 * clocks <= 0 restores the default of 2e9 clocks (about one second at
 * 2 GHz); no legitimate wait lasts more than a few microseconds.  A budget of
 * a few clocks makes the first wait that is not already satisfied expire: the
 * kernel then records the expiry, stops every role, waits (on its own,
 * unchanged budget) for the copies and tensor-core work it has in flight,
 * frees its tensor memory and returns, and hdp_device_status reports
 * HDP_ERR_DEVICE_TIMEOUT.  This is how the timeout path is tested without a
 * fault; production code leaves the default.  Always returns HDP_OK.
 */
hdp_status_t hdp_set_wait_budget(int64_t clocks);

/* ====================================================================== */
/* Cost models (host arithmetic only: no device, no stream, no allocation).
 * "ByteScale: ..." research digest, section 3.2 (ring timing model and its
 * table of worked cases) and section 3.3 (cost models T(s), Act(s) and
 * Eq. 3).  Times and bandwidths are in any consistent units. */

/*
 * Per-step compute of a ring of N ranks holding C tokens each (section 3.2):
 *   t_c = t_blk * sum_i (s_i / (N C))^2
 * where every sequence of the pack is cut into N slices and a query attends
 * only to its own sequence; t_blk is the time of one full C x C block.
 * lengths: host int32[n], n >= 1, every s_i >= 1, sum s_i <= N * C.
 * INVALID_ARGUMENT otherwise (or t_blk < 0, or a null pointer).
 */
hdp_status_t hdp_ring_step_compute(const int32_t* lengths, int32_t n, int32_t num_ranks, int32_t capacity,
                                   double t_blk, double* t_c);

/*
 * Attention time of that ring (section 3.2): each step overlaps the transfer
 * of the next K/V slice (t_x) with the compute on the current one (t_c):
 *   T_attn = (N - 1) * max(t_c, t_x) + t_c.
 * num_ranks >= 1, t_c >= 0, t_x >= 0.
 */
hdp_status_t hdp_ring_attention_time(int32_t num_ranks, double t_c, double t_x, double* t_attn);

/* Profiled cost models of section 3.3, T(s) = alpha1 s^2 + beta1 s + gamma
 * (time of one layer on a sequence of s tokens) and
 * Act(s) = alpha2 s + beta2 (activation bytes of one layer), with the
 * device-to-host and host-to-device copy bandwidths (bytes per time unit)
 * and l layers per rank. */
typedef struct {
  double alpha1, beta1, gamma;
  double alpha2, beta2;
  double bw_d2h, bw_h2d;
  int32_t layers; /* l >= 3 */
} hdp_offload_model_t;

/*
 * Selective offloading, Eq. 3 (section 3.3): the rank count of a sequence of
 * s tokens when a fraction r of the activations of l - 2 of its l layers is
 * kept in host memory,
 *   D(s) = ceil((2 Act(s) + (1 - r)(l - 2) Act(s)) / (l Act(C))),
 * subject to the copy hiding behind compute, T(s) >= r Act(s) / min(B_d2h, B_h2d),
 * and to 1 >= r >= min(1, l Act(C) / ((l - 2) Act(s))).  D does not grow with r,
 * so the rank count is smallest at the largest admissible ratio:
 *   r = min(1, T(s) min(B_d2h, B_h2d) / Act(s)) when that is at least the lower
 *   bound, else r = 0 (no offloading, D = ceil(Act(s) / Act(C))).
 * Requires s >= 1, capacity >= 1, layers >= 3, Act(C) > 0, Act(s) > 0,
 * bandwidths >= 0.  Outputs the chosen ratio and rank count.
 */
hdp_status_t hdp_offload_ranks(const hdp_offload_model_t* model, int64_t s, int64_t capacity, double* r,
                               int64_t* ranks);

/*
 * Least-squares fit of a profiled cost model (section 3.3): the polynomial of
 * the given degree (1: Act(s) = c1 s + c0; 2: T(s) = c2 s^2 + c1 s + c0)
 * minimising sum_i w_i (y_i - p(x_i))^2 over n points; coef[k] is the
 * coefficient of x^k.  w: host double[n] of weights >= 0, or NULL for all
 * ones (w_i = 1 / y_i^2 fits relative errors, for times spanning several
 * orders of magnitude).  n > degree and at least degree + 1 distinct x values
 * with positive weight; coef has degree + 1 entries.
 */
hdp_status_t hdp_fit_cost_model(const double* x, const double* y, const double* w, int32_t n, int32_t degree,
                                double* coef);

/* ====================================================================== */
/* Balance scheduler (host arithmetic only).  Research digest, section 3.4 and
 * Figure 4: micro-batches hold equal tokens but unequal attention FLOPs, so
 * workers run different numbers of them.  The section states the steps but
 * not Algorithm 2's text; the reading implemented here:
 *   1. order the micro-batches by cost, heaviest first (ties: lower index);
 *   2. cut that order into `buckets` consecutive buckets of about equal cost:
 *      the item at sorted position p goes to bucket
 *      min(B - 1, floor(B * P_p / total)), P_p the cost before it;
 *   3. HDP_BALANCE_DP: workers draw from the front of the order (the first
 *      non-empty bucket).  Each pass, every worker whose load trails the
 *      slowest worker's by more than `delta` (load + delta < max load) takes
 *      the next micro-batch, in worker order; when none trails, every worker
 *      takes one.
 *      HDP_BALANCE_PP: one bucket per pipeline (`buckets` is ignored and
 *      taken as `workers`); pipeline p runs bucket p.
 * costs: host int64[m] >= 0 (e.g. hdp_flops_per_shard copied to the host);
 * worker_of_item: host int32[m] out; worker_load: host int64[workers] out;
 * bucket_of_item: host int32[m] out, or NULL.  m >= 0, workers >= 1,
 * buckets >= 1, delta >= 0.  Time O(m log m + passes * workers); uses a
 * scratch array of m int32 allocated and freed inside the call
 * (HDP_ERR_OUT_OF_MEMORY if that fails).  The sum of the costs must fit in
 * int64. */
#define HDP_BALANCE_DP 0
#define HDP_BALANCE_PP 1
hdp_status_t hdp_balance_schedule(const int64_t* costs, int32_t m, int32_t workers, int32_t buckets, int64_t delta,
                                  int32_t mode, int32_t* worker_of_item, int64_t* worker_load,
                                  int32_t* bucket_of_item);

#ifdef __cplusplus
}
#endif

#endif /* HDPATTN_H_ */
