/*
 * unified_attention.h -- C ABI of the GB300 (sm_103a) unified paged varlen
 * attention library (libua_gb300.so).
 *
 * The operation.  One call computes attention for a flattened batch that
 * mixes prefill, chunked-prefill and decode sequences.  As the unified
 * kernel states the problem, the call has the semantics of FlashAttention's
 * varlen function for any number of new query tokens per sequence; it packs
 * the query heads that share a KV head along the query dimension and reads
 * the key cache in the FlashAttention layout ("[Kernel] Unified Triton kernel
 * that doesn't distinguish between prefill + decode", vLLM PR #16828, PR
 * description, first and third bullets).  The batch is described by the
 * usual varlen metadata (cu_seqlens_q, seqused_k, block_table), unchanged
 * from what the serving engine already keeps ("[Kernel] [V1] Improved
 * performance for V1 Triton (ROCm) backend", vLLM PR #14152, section "How is
 * this performance improvement achieved?").
 *
 * For sequence s with Lq = cu_seqlens_q[s+1] - cu_seqlens_q[s] new tokens
 * and Lk = seqused_k[s] context tokens (the new ones included, their K/V
 * already written to the cache), query head h of new token i (i < Lq, flat
 * row t = cu_seqlens_q[s] + i) attends to keys j < limit, where
 *     limit = causal ? Lk - Lq + i + 1 : Lk
 * (bottom-right alignment: the new tokens are the last Lq of the context),
 * using KV head h / (Hq / Hkv).  Key j lives in physical page
 * block_table[s][j / block_size], slot j % block_size:
 *     out[t][h] = softmax_j(scale * <q[t][h], k_j>) . v_j
 *
 * Layouts (all row-major, contiguous, bf16 = IEEE bfloat16):
 *   q        bf16  [total_q, num_q_heads, head_size]            device
 *   k_cache  bf16  [num_blocks, block_size, num_kv_heads, head_size]  device
 *   v_cache  bf16  same as k_cache                               device
 *   out      bf16  [total_q, num_q_heads, head_size]             device
 *   cu_seqlens_q int32 [num_seqs + 1], cu[0] = 0, non-decreasing  device
 *   seqused_k    int32 [num_seqs]                                 device
 *   block_table  int32 [num_seqs, block_table_stride]             device
 *   *_host       host copies of cu_seqlens_q / seqused_k, used to plan the
 *                launch without a device-to-host read; they must hold the
 *                same values as the device arrays.
 *
 * Supported set: head_size 64, 80, 96, 112, 128 or 256, block_size a
 * multiple of 16 up to 256, num_q_heads a multiple of num_kv_heads.  Anything
 * else returns UA_ERR_UNSUPPORTED before any launch.  With head_size 80, 96
 * or 112 every row, prefill rows included, runs in the decode / split-KV
 * kernel (its 128-wide instance, the columns past head_size read as zeros and
 * never written; units of two adjacent kv heads when num_kv_heads is even);
 * the tensor-core prefill kernels take head sizes 64 and 128 (one SM per
 * work item, or SM pairs for long items) and 256 (SM pairs).
 *
 * Pages of block_size = 16 r tokens (r > 1): the same memory is a cache of
 * num_blocks * r pages of 16 tokens (slot j of page b is slot j % 16 of
 * 16-token page b r + j / 16), which is what the kernels read.  Every call on
 * such a cache first expands the block table on the device (entry p becomes
 * p r .. p r + r - 1; an entry outside [0, num_blocks) becomes one the
 * kernels skip and report).  The expanded table lives in the workspace:
 * num_seqs x block_table_stride x r int32, rounded up to 256 bytes, counted
 * by every ua_workspace_size* function.  block_table_stride x r must stay
 * below 2^29.  The result is the same, bit for bit, as the call on the
 * 16-token view with the expanded table.
 *
 * Ownership: the caller owns every buffer it passes.  Split-KV partials live
 * in the caller's workspace (size from ua_workspace_size), which only the
 * call's own kernels touch, in the order of the given stream.  The launch
 * plan of a host-planned call goes to the GPU through the library's own
 * memory: per device, a ring of 8 page-locked host buffers and 8 device
 * buffers, each grown on demand (an allocation only when a plan is larger
 * than any that buffer held before; none once the sizes have settled).  The
 * plan copy runs on a library stream and is ordered only after the kernels
 * of the earlier call that used the same ring buffer, so it overlaps what
 * the caller's stream runs before the call; the caller's stream waits for it
 * before the call's kernels.  Calls are asynchronous on the given stream.
 * Two calls that share a workspace must be ordered (same stream, or
 * synchronised by the caller).
 *
 * CUDA graphs: a host-planned call (unified_attention, _lse, _append, _fp8kv)
 * fixes its plan, its grid sizes and its plan copy from this batch's host
 * lengths, so a captured replay would run them against whatever batch the
 * buffers hold by then.  Such a call made on a stream that is being captured
 * returns UA_ERR_UNSUPPORTED and enqueues nothing.  Graph users call
 * unified_attention_device_plan, which plans on the device.
 *
 * Errors are returned, never aborted on.  Invalid metadata is rejected on
 * the host before any launch.  Device-side problems (a block id outside
 * [0, num_blocks), a pipeline wait that ran out of time) never fault: the
 * kernels skip the bad access, record a code in a device status word, and
 * finish; ua_device_status() reads and clears it.
 */
#ifndef UNIFIED_ATTENTION_H
#define UNIFIED_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ua_status {
    UA_OK = 0,
    UA_ERR_INVALID_ARG = 1,   /* null pointer, bad metadata, misaligned buffer */
    UA_ERR_UNSUPPORTED = 2,   /* head_size / block_size / head ratio outside the supported set */
    UA_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small */
    UA_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, copy, device query) */
    UA_ERR_DEVICE_CHECK = 5   /* ua_device_status found a code recorded by a kernel */
} ua_status;

/* Device status word bits (ua_device_status). */
#define UA_DEVICE_BAD_BLOCK_ID 0x1   /* a block_table entry outside [0, num_blocks) was skipped */
#define UA_DEVICE_WAIT_TIMEOUT 0x2   /* a pipeline wait gave up; the output is incomplete */
#define UA_DEVICE_BAD_METADATA 0x4   /* the device planner rejected cu_seqlens_q / seqused_k
                                        (or a capacity): nothing was computed */

/*
 * unified_attention -- attention over a paged varlen batch (definition above,
 * from the unified kernel's PR description).
 *
 *   softmax_scale  multiplies every score; finite.
 *   causal         non-zero: bottom-right causal mask; zero: every one of the
 *                  Lk keys is visible (the non-causal mode requested in the
 *                  review thread of the same page, for cascade attention).
 *   num_blocks     pages in k_cache / v_cache; num_blocks * block_size < 2^31.
 *   workspace      device scratch of at least ua_workspace_size() bytes,
 *                  256-byte aligned; may be NULL only when that size is 0.
 *   stream         a cudaStream_t (NULL = legacy default stream).  All work is
 *                  ordered on it: a batch of decode rows and long prefill
 *                  items may run its decode kernel on a second stream of the
 *                  library at the same time as its prefill kernel (on other
 *                  SMs), forked from `stream` after the plan upload and
 *                  joined back into it before the call returns (see
 *                  ua_plan_inspect).
 *
 * Host-side checks (UA_ERR_INVALID_ARG): cu_seqlens_q_host[0] == 0 and
 * non-decreasing; seqused_k_host[s] >= 0; Lk > 0 whenever Lq > 0; Lk >= Lq
 * when causal; ceil(Lk / block_size) <= block_table_stride; q, k_cache,
 * v_cache, out 16-byte aligned.  Sequences with Lq = 0 are allowed and write
 * nothing.  Block-table entries at or beyond ceil(Lk / block_size) are never
 * read; entries may alias (one physical page in several sequences).
 * Every out row of every sequence is fully overwritten.
 */
ua_status unified_attention(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                            const int32_t *block_table, float softmax_scale, int32_t causal,
                            void *out, const int32_t *cu_seqlens_q_host,
                            const int32_t *seqused_k_host, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                            int32_t block_size, int32_t num_blocks, int32_t block_table_stride,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * ua_workspace_size -- bytes of device workspace unified_attention needs for
 * this batch on the current CUDA device: the launch plan (per-(sequence,
 * kv-head, query-tile) work items and their page ranges) plus the split-KV
 * partial outputs.  Host-only apart from a cached device-property query.
 * Same metadata checks as unified_attention; *bytes is written on UA_OK.
 */
ua_status ua_workspace_size(const int32_t *cu_seqlens_q_host, const int32_t *seqused_k_host,
                            int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_size, int32_t block_size, int32_t block_table_stride,
                            int32_t causal, size_t *bytes);

/* ua_status_string -- static, human-readable name of a status code. */
const char *ua_status_string(ua_status status);

/*
 * ua_device_status -- synchronises the current device, then reads and clears
 * the device status word the kernels write (UA_DEVICE_* bits).  *code gets
 * the bits; returns UA_ERR_DEVICE_CHECK if any bit was set, UA_OK if none.
 */
ua_status ua_device_status(int32_t *code);

/*
 * ua_plan_inspect -- host-only view of the work partition unified_attention
 * would launch for this batch on a GPU with num_sms multiprocessors (no CUDA
 * call is made).  This is the partition pass of the hot path: the pages
 * motivate one plan per batch because a single fixed grid fits prefill and
 * decode badly (vLLM PR #14152, section "How is this performance improvement
 * achieved?").
 *
 * counts[0..8] receives: decode CTAs, decode pieces, split units (combined),
 * partial slots, prefill tiles, prefill CTAs, decode pages in total, the
 * bytes of the plan and partials (saturated to INT32_MAX; ua_workspace_size
 * adds the expanded block table to these for pages of more than 16 tokens),
 * and the SMs the prefill kernel gets when the call runs its two kernels side
 * by side (0: one after the other, each on every SM).  A batch of decode rows
 * and long prefill items (head size 128, bf16 cache) runs them side by side
 * when that is estimated to save time: the prefill kernel on that many SMs,
 * launched first, and the decode kernel on the rest, on a second stream of
 * the library's forked from and joined back to the caller's.
 * The partition is the 16-token view's for any supported block_size.
 * If items != NULL, up to items_cap rows of 8 int32 are written:
 *   decode pieces   {0, cta, seq, kv_head, row0, nrows, page_begin, page_end}
 *                   followed by one row {1, slot or -1, unit, 0, 0, 0, 0, 0}
 *   prefill tiles   {2, cta, seq, kv_head, row0, nrows, kv_tiles, order}
 *                   (cta -1: long items, claimed by the CTAs in order as they
 *                   go; a call with head_size 128 and a positive scale)
 *   split units     {3, seq, kv_head, row0, nrows, slot_begin, nslots, 0}
 * Rows are packed (token, head-in-group) pairs: row r is token r / G, query
 * head kv_head * G + r % G, with G = num_q_heads / num_kv_heads.
 * *n_items gets the number of rows the full listing needs.
 */
ua_status ua_plan_inspect(const int32_t *cu_seqlens_q_host, const int32_t *seqused_k_host,
                          int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_size, int32_t block_size, int32_t block_table_stride,
                          int32_t causal, int32_t num_sms, int32_t *counts, int32_t *items,
                          int64_t items_cap, int64_t *n_items);

/*
 * Per-kernel timing, for roofline figures.  When enabled, unified_attention
 * records CUDA events around each kernel it launches on the caller's stream,
 * into a ring of UA_PROFILE_RING call slots per device (events are created
 * once and reused), so a caller can time many calls without synchronising
 * between them and read them afterwards.
 * ua_profile_read(calls_back, ...) synchronises on that call's last event and
 * fills, for the call calls_back calls before the latest (0 = latest):
 *   ms[0..3]       decode, prefill, combine kernel time and the plan copy
 *                  (-1 when that step did not run; the combine is always -1
 *                  now: split units are merged inside the decode kernel by
 *                  the CTA that writes a unit's last partial); for
 *                  unified_attention_device_plan, ms[3] is the planner kernel;
 *   launches[0..3] kernel launches of each kind (the copy counts as 0, the
 *                  planner kernel as 1).
 * calls_back must be below min(profiled calls, UA_PROFILE_RING).
 */
#define UA_PROFILE_RING 64
ua_status ua_profile_enable(int32_t enable);
ua_status ua_profile_read(int32_t calls_back, float *ms, int32_t *launches);

/*
 * ua_test_set_wait_limit -- test hook for the failure path of the device
 * waits: the decode / split-KV kernel of the calls made after it (any
 * thread) gives each wait of its main loop at most limit_ns nanoseconds
 * instead of the library's 4 s (0 restores that).  A wait that runs out sets
 * UA_DEVICE_WAIT_TIMEOUT in the device status word and the kernel winds
 * down: the warps that share barriers stop together, the loads it has issued
 * are waited for (with the 4 s limit) and it returns, leaving its output
 * incomplete.  Nothing else faults or stops; the next call with the normal
 * limit is correct.  Not for production use.
 */
ua_status ua_test_set_wait_limit(uint64_t limit_ns);

/*
 * unified_attention_lse -- unified_attention that also writes, for every
 * query row, the natural-log normaliser of its softmax,
 *     lse[t][h] = ln( sum over visible keys j of e^(softmax_scale * <q_t,h, k_j>) ),
 * into lse (device, fp32 [total_q, Hq], row-major, caller-owned; must not be
 * NULL, 4-byte aligned).  Rows of sequences with Lq = 0 are not written.  The
 * other arguments, the output and the errors are those of unified_attention.
 * Together with ua_merge_attn_states it gives cascade (shared-prefix)
 * attention: one call over the shared prefix with causal = 0 (every new token
 * sees the whole prefix), one over each sequence's own keys with causal = 1,
 * then the merge.  Non-causal attention for cascade attention is the review
 * request on "[Kernel] Unified Triton kernel that doesn't distinguish between
 * prefill + decode" (vLLM PR #16828, review thread).
 */
ua_status unified_attention_lse(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                                const int32_t *block_table, float softmax_scale, int32_t causal,
                                void *out, float *lse, const int32_t *cu_seqlens_q_host,
                                const int32_t *seqused_k_host, int32_t num_seqs,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                int32_t block_size, int32_t num_blocks,
                                int32_t block_table_stride, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * ua_merge_attn_states -- combine two attention results of the same query
 * rows over disjoint key sets, A and B, by their normalisers:
 *     m = max(lse_a, lse_b),  w_x = e^(lse_x - m),
 *     out = (w_a out_a + w_b out_b) / (w_a + w_b),  lse_out = m + ln(w_a + w_b).
 * A side with lse = -inf (no key) gets weight 0; both -inf gives out = 0 and
 * lse_out = -inf.  out_a, out_b, out: device bf16 [rows][head_size], 16-byte
 * aligned; lse_a, lse_b: device fp32 [rows]; lse_out: device fp32 [rows] or
 * NULL.  In-place merges are allowed: out may be out_a or out_b, and lse_out
 * may be lse_a or lse_b (the same pointer; a partial overlap is not
 * supported).  rows = total_q * Hq for the outputs of two
 * unified_attention_lse calls.  head_size: a multiple of 8, at most 2048
 * (else UA_ERR_UNSUPPORTED).  Async on stream; returns UA_ERR_INVALID_ARG for
 * bad arguments (nothing launched), UA_ERR_CUDA if the launch fails.
 */
ua_status ua_merge_attn_states(const void *out_a, const float *lse_a, const void *out_b,
                               const float *lse_b, void *out, float *lse_out, int64_t rows,
                               int32_t head_size, void *stream);

/*
 * ua_kv_append -- the step just before attention: write the new tokens' K
 * and V rows into their pages.  Token i of sequence s (0 <= i < Lq) goes to
 * context position p = seqused_k[s] - Lq + i (the new tokens are the last Lq
 * positions of the context that seqused_k counts, as in the bottom-right
 * causal mask), i.e. k_cache[block_table[s][p / block_size]][p % block_size]
 * [:][:] = k_new[t]
 * with t = cu_seqlens_q[s] + i, and the same for V.  Nothing else in the
 * caches is written.  The metadata and cache arguments are those of
 * unified_attention; k_new, v_new: device bf16 [total_q, Hkv, D], 16-byte
 * aligned.  Every sequence needs Lq <= Lk; Hkv * D up to 2048 (else
 * UA_ERR_UNSUPPORTED).  Host checks as for
 * unified_attention (nothing launched on failure); a block id outside
 * [0, num_blocks) is skipped and reported through ua_device_status.  Async on
 * stream.  The pages describe the cache layout and that seqused_k counts the
 * whole context; the append itself is the step the attention call assumes
 * has happened.
 */
ua_status ua_kv_append(const void *k_new, const void *v_new, const int32_t *cu_seqlens_q,
                       const int32_t *seqused_k, const int32_t *block_table, void *k_cache,
                       void *v_cache, const int32_t *cu_seqlens_q_host,
                       const int32_t *seqused_k_host, int32_t num_seqs, int32_t num_kv_heads,
                       int32_t head_size, int32_t block_size, int32_t num_blocks,
                       int32_t block_table_stride, void *stream);

/*
 * unified_attention_append -- ua_kv_append of k_new / v_new, then
 * unified_attention over the updated caches, in one call on one stream (the
 * new tokens' keys are in the cache before any attention kernel reads it).
 * Arguments as for the two calls; every check of both runs before anything is
 * launched.
 */
ua_status unified_attention_append(const void *q, const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *cu_seqlens_q,
                                   const int32_t *seqused_k, const int32_t *block_table,
                                   float softmax_scale, int32_t causal, void *out,
                                   const int32_t *cu_seqlens_q_host,
                                   const int32_t *seqused_k_host, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                   int32_t block_size, int32_t num_blocks,
                                   int32_t block_table_stride, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * unified_attention_fp8kv -- unified_attention over a KV cache stored as
 * FP8 e4m3 bytes with one scale per tensor: the keys are k_scale * e4m3(byte)
 * and the values v_scale * e4m3(byte) (the OCP "E4M3" format: 1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits; no infinities; 0x7f / 0xff are
 * NaN).  k_cache, v_cache: device uint8 [num_blocks, block_size, Hkv, D], 16-
 * byte aligned; q and out bf16 as for unified_attention; lse: optional fp32
 * [total_q, Hq] (as unified_attention_lse) or NULL.  Every row runs in the
 * decode kernel, whose threads widen the cache bytes to f16 in registers
 * (exact: e4m3 values are f16 values) and multiply with f16 Q (q is rounded
 * to f16, so |q| must stay below 65504) and f16 P; k_scale is folded into the
 * softmax scale and v_scale into the output.  With num_kv_heads even, each
 * work unit covers two adjacent kv heads (one 256-byte run of a page slot per
 * load).  head_size 128 only (else UA_ERR_UNSUPPORTED).
 * Workspace size from ua_workspace_size_fp8kv.  The FP8 cache is the "KV cache
 * compression" discussed on "[Kernel] [V1] Improved performance for V1 Triton
 * (ROCm) backend" (vLLM PR #14152, review thread); the pages fix neither the
 * format nor the scaling, and this reading takes e4m3 with per-tensor scales.
 */
ua_status unified_attention_fp8kv(const void *q, const void *k_cache, const void *v_cache,
                                  float k_scale, float v_scale, const int32_t *cu_seqlens_q,
                                  const int32_t *seqused_k, const int32_t *block_table,
                                  float softmax_scale, int32_t causal, void *out, float *lse,
                                  const int32_t *cu_seqlens_q_host,
                                  const int32_t *seqused_k_host, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                  int32_t block_size, int32_t num_blocks,
                                  int32_t block_table_stride, void *workspace,
                                  size_t workspace_bytes, void *stream);
ua_status ua_workspace_size_fp8kv(const int32_t *cu_seqlens_q_host,
                                  const int32_t *seqused_k_host, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                  int32_t block_size, int32_t block_table_stride, int32_t causal,
                                  size_t *bytes);

/*
 * unified_attention_no_alloc -- the same operation and arguments as
 * unified_attention, minus the workspace: the launch plan and the split-KV
 * partials go into a device array the library owns, so the caller never
 * allocates device memory.  The pages have no counterpart to this entry
 * point; it exists for callers that cannot call cudaMalloc or any other
 * device allocator -- e.g. a plugin running inside a framework whose caching
 * allocator owns all device memory and offers the plugin no way to borrow
 * it, or a latency-critical path where an allocation could synchronise the
 * device.  The caller still owns q, the caches, the metadata and out.
 *
 *   - The array holds UA_STATIC_WORKSPACE_BYTES (16 MiB).  Every GPU that
 *     loads the library's module keeps that memory until the process exits.
 *   - A batch whose workspace (as ua_workspace_size reports it) is larger
 *     returns UA_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  Nothing in it needs to start at zero: each call writes the
 *     plan and every partial before reading them.  Calls that overlap on the
 *     GPU (different streams, not ordered by the caller) race on the array.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define UA_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)

ua_status unified_attention_no_alloc(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                                     const int32_t *block_table, float softmax_scale,
                                     int32_t causal, void *out,
                                     const int32_t *cu_seqlens_q_host,
                                     const int32_t *seqused_k_host, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_size, int32_t block_size, int32_t num_blocks,
                                     int32_t block_table_stride, void *stream);

/*
 * unified_attention_device_plan -- unified_attention planned on the GPU: no
 * host copies of cu_seqlens_q / seqused_k, no host-side work that depends on
 * them, fixed launch shapes.  So one call can be captured in a CUDA graph and
 * the graph replayed after the device metadata (cu_seqlens_q, seqused_k,
 * block_table) and q have been rewritten for a new batch of the same
 * num_seqs.  The pages' unified kernel consumes the engine's existing varlen
 * metadata with no extra host step ("[Kernel] [V1] Improved performance for
 * V1 Triton (ROCm) backend", vLLM PR #14152, section "How is this performance
 * improvement achieved?").
 *
 * A planner kernel (one CTA) reads the device arrays and writes into the
 * workspace the same plan the host planner makes for that batch: the same
 * routing of rows to the decode and prefill kernels, decode page ranges, split
 * pieces and prefill item order.  Then the decode kernel (kDecCtasPerSm x SMs
 * CTAs) and, when the prefill kernel can take this head grouping and cache
 * type, the prefill kernel (SMs CTAs) run; CTAs beyond the plan's count exit.
 *
 *   q, out       bf16 [max_total_q, Hq, D]: buffers sized for max_total_q
 *                tokens; rows past cu_seqlens_q[num_seqs] are not written.
 *   lse          optional fp32 [max_total_q, Hq] or NULL.
 *   num_seqs     sequences in the batch (cu_seqlens_q has num_seqs + 1
 *                entries); sequences with no query tokens are allowed.
 *   max_total_q  the token capacity; the planner rejects a batch with
 *                cu_seqlens_q[num_seqs] > max_total_q.
 *   max_seq_q    the most query tokens one sequence may have (0: max_total_q);
 *                the planner rejects a longer sequence.  When max_seq_q x
 *                (Hq / Hkv) <= 16 no row can need the prefill kernel and it
 *                is not launched (a decode-only graph).
 *   kv_fp8       0: bf16 caches; 1: e4m3 caches with k_scale / v_scale as
 *                for unified_attention_fp8kv (head_size 128 only).
 *   workspace    ua_workspace_size_device_plan bytes, 256-byte aligned; laid
 *                out for (num_seqs, max_total_q, heads, head size,
 *                block_table_stride, kv_fp8) and the device's SM count.  With
 *                pages of more than 16 tokens the expanded block table follows
 *                the plan (it is rebuilt on every call, planned or not).
 * Other arguments as for unified_attention.  The host checks shapes,
 * pointers and the workspace; the metadata itself is checked on the device
 * (the same rules as unified_attention): a bad batch leaves an empty plan (no
 * output written) and sets UA_DEVICE_BAD_METADATA for ua_device_status.
 * Asynchronous on `stream`; no allocation, no synchronisation.
 */
ua_status unified_attention_device_plan(const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                                        const int32_t *block_table, float softmax_scale,
                                        int32_t causal, void *out, float *lse, int32_t num_seqs,
                                        int32_t max_total_q, int32_t max_seq_q, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_size,
                                        int32_t block_size, int32_t num_blocks,
                                        int32_t block_table_stride, int32_t kv_fp8,
                                        float k_scale, float v_scale, void *workspace,
                                        size_t workspace_bytes, void *stream);
/*
 * unified_attention_device_planned -- unified_attention_device_plan without the
 * planner: the decode and prefill kernels read the plan that an earlier
 * unified_attention_device_plan or ua_device_plan_build call left in the same
 * workspace for the same cu_seqlens_q / seqused_k (and the same capacities).
 * The layers of one model step share their lengths, so one plan per step
 * serves every layer's attention.  Same arguments; the metadata must be
 * unchanged since the plan was built (nothing checks that).
 */
ua_status unified_attention_device_planned(const void *q, const void *k_cache,
                                           const void *v_cache, const int32_t *cu_seqlens_q,
                                           const int32_t *seqused_k, const int32_t *block_table,
                                           float softmax_scale, int32_t causal, void *out,
                                           float *lse, int32_t num_seqs, int32_t max_total_q,
                                           int32_t max_seq_q, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_size,
                                           int32_t block_size, int32_t num_blocks,
                                           int32_t block_table_stride, int32_t kv_fp8,
                                           float k_scale, float v_scale, void *workspace,
                                           size_t workspace_bytes, void *stream);
ua_status ua_workspace_size_device_plan(int32_t num_seqs, int32_t max_total_q,
                                        int32_t max_seq_q, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_size, int32_t block_size,
                                        int32_t block_table_stride, int32_t kv_fp8,
                                        size_t *bytes);

/*
 * ua_device_plan_build -- only the planner kernel of
 * unified_attention_device_plan (same arguments), for inspecting the plan.
 * ua_device_plan_layout -- host-only: where that plan lies in the workspace
 * for a GPU with num_sms SMs.  offsets[8]: byte offsets of the header (int64
 * {dec_ctas, n_pieces, n_comb, n_slots, pre_ctas, n_tiles, dec_pages,
 * error}), cta_begin (int32), the decode pieces (8 x int32 each: seq, kvh,
 * row0, nrows, page_begin, page_end, slot, unit), the split units (8 x
 * int32), their arrival counters, the prefill items (8 x int32: seq, kvh,
 * row0, nrows, kv_tiles, q0, lq, lk), pre_begin (int32), and the workspace
 * size.  caps[8]: decode grid, unit, item, piece, split-unit and partial-slot
 * capacities, histogram buckets, num_sms.
 */
ua_status ua_device_plan_build(const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                               int32_t causal, int32_t num_seqs, int32_t max_total_q,
                               int32_t max_seq_q, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                               int32_t block_size, int32_t block_table_stride, int32_t kv_fp8,
                               void *workspace, size_t workspace_bytes, void *stream);
ua_status ua_device_plan_layout(int32_t num_seqs, int32_t max_total_q, int32_t max_seq_q,
                                int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                int32_t block_table_stride, int32_t kv_fp8, int32_t num_sms,
                                int64_t *offsets, int32_t *caps);

#ifdef __cplusplus
}
#endif

#endif /* UNIFIED_ATTENTION_H */
