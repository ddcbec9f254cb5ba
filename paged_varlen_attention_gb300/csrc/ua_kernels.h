// ua_kernels.h -- launch interface between the C ABI (ua_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ua_plan.h"
#include "unified_attention.h"

namespace ua {

struct DecodeParams {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    const int32_t *cu;           // device cu_seqlens_q
    const int32_t *seqused_k;    // device seqused_k
    const int32_t *block_table;
    int32_t bt_stride;
    int32_t num_blocks;
    int32_t hq;
    int32_t hkv;
    int32_t g;                   // hq / hkv
    int32_t causal;
    float scale_log2;            // softmax_scale * log2(e)
    const int32_t *cta_begin;    // plan: [ctas + 1]
    const DecPiece *pieces;      // plan
    float *part_o;               // [slots][kDecRows][d]
    float *part_ml;              // [slots][kDecRows][2]: running max (log2 domain), sum
    const CombUnit *comb;        // plan: split units
    int32_t *comb_count;         // plan: partials written per split unit (zero at launch; the
                                 // merging CTA zeroes it again, so a reused plan stays valid)
    float *lse;                  // optional [total_q, Hq]: natural-log normaliser per row
    float v_scale;               // scale of the V values (fp8 cache; 1 otherwise)
    int32_t heads_per_unit;      // e4m3 pages: kv heads per unit (tile rows 8j.. are head kvh + j)
    int *status;                 // device status word
    unsigned long long wait_ns;  // limit of the main loop's waits (the drains keep kWaitLimitNs)
    int32_t dq;                  // head size of q, out and the cache rows: the kernel's D, or
                                 // 80 / 96 / 112 in the D = 128 kernel (rows zero-padded)
};

struct PrefillParams {
    const __nv_bfloat16 *k_cache;
    __nv_bfloat16 *out;
    float *lse;                  // optional [total_q, Hq]: natural-log normaliser per row
    const int32_t *cu;
    const int32_t *seqused_k;
    const int32_t *block_table;
    int32_t bt_stride;
    int32_t num_blocks;
    int32_t hq;
    int32_t hkv;
    int32_t g;
    int32_t causal;
    float scale_log2;
    const PreTile *tiles;        // grouped by CTA (dealt), or longest first (claimed)
    const int32_t *tile_begin;   // dealt: [ctas + 1], CTA c runs tiles [tile_begin[c], tile_begin[c+1])
    int32_t *sched;              // claimed: [kSchedInts] next unclaimed item, CTAs done, item count
    int32_t n_tiles;
    float v_scale;               // output scale (an e4m3 cache's V scale; 1 for bf16)
    int *status;
};

// Each returns the launch error (cudaSuccess when the launch was queued).
// launch_decode: d is the head size (p.dq); for 80, 96 and 112 the D = 128
// kernel runs with tm_k / tm_v mapping the cache as (d, 16 slots, Hkv,
// blocks), two 64-column boxes per page, the second zero-filled past d.
cudaError_t launch_decode(int d, bool kv8, const DecodeParams &p, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, int ctas, cudaStream_t stream);
// claimed: the CTAs claim items from p.sched (D = 128 with a positive scale
// only); otherwise each runs its range of p.tile_begin.
cudaError_t launch_prefill(int d, bool claimed, const PrefillParams &p, const CUtensorMap &tm_q,
                           const CUtensorMap &tm_o, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           int ctas, cudaStream_t stream);
// The two-SM prefill kernel (ua_prefill_pair.cu), head size d = 128 or 256:
// `pairs` clusters of two CTAs, pair c running tiles [tile_begin[c],
// tile_begin[c+1]).  tm_vh: the page view of the V cache with d / 128
// 64-column chunks per box (the half of a page's columns one SM holds).
cudaError_t launch_prefill_pair(int d, const PrefillParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_o,
                                const CUtensorMap &tm_k, const CUtensorMap &tm_vh, int pairs,
                                cudaStream_t stream);

// The whole call behind unified_attention (arguments as declared in
// unified_attention.h).  pinned_plan: stage the plan through the library's
// page-locked ring (allocated on first use) rather than copy it from pageable
// memory; the entry point that must allocate nothing passes false.  lse:
// optional fp32 [total_q, Hq] output of the natural-log normaliser per row.
// kv_fp8: the caches hold e4m3 bytes, k = k_scale * code and v = v_scale *
// code (every row then runs in the decode kernel; D = 128 only).
ua_status run_attention(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                        const int32_t *block_table, float softmax_scale, int32_t causal, void *out,
                        const int32_t *cu_seqlens_q_host, const int32_t *seqused_k_host,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_size, int32_t block_size, int32_t num_blocks,
                        int32_t block_table_stride, void *workspace, size_t workspace_bytes,
                        void *stream, bool pinned_plan, float *lse, int kv_fp8 = 0,
                        float k_scale = 1.f, float v_scale = 1.f);

// ---- plan built on the device (ua_device_plan.cu)
// What a device-plan workspace is laid out for: the batch's sequence count,
// the query-token capacity of q / out, the longest query of one sequence, the
// heads, head size, block-table width, kv heads per decode unit, whether the
// prefill kernel may take rows, and the SM count (decode grid
// kDecCtasPerSm * num_sms, prefill grid num_sms).
struct DevPlanShape {
    int32_t page_ratio;    // caller's page size / 16 (bt_stride below counts 16-token pages)
    int32_t num_seqs;
    int32_t max_total_q;
    int32_t max_seq_q;     // query tokens of one sequence at most
    int32_t hq;
    int32_t hkv;
    int32_t d;
    int32_t bt_stride;
    int32_t hpu;
    int32_t prefill_ok;
    int32_t num_sms;
    int32_t pre_workers;   // prefill items are dealt to this many workers (<= num_sms)
    int32_t pre_pair;      // the workers are CTA pairs of the two-SM prefill kernel
};

// Workspace sections (byte offsets) and capacities for one DevPlanShape.
// The header holds int64 {dec_ctas, n_pieces, n_comb, n_slots, pre_ctas,
// n_tiles, dec_pages, error} of the last plan built.
struct DevPlanLayout {
    size_t off_header, off_cta, off_pieces, off_comb, off_comb_count, off_tiles, off_pre_begin;
    size_t off_part_o, off_part_ml, off_scratch, total_bytes;
    int32_t dec_grid, cap_units, cap_items, cap_pieces, cap_comb, cap_slots, n_buckets;
    bool valid;   // false: the capacities do not fit the planner's 32-bit counts
};

DevPlanLayout device_plan_layout(const DevPlanShape &s);

// Builds the plan of (cu, seqused_k) into the workspace (one CTA).  Bad
// metadata or an exceeded capacity leaves an empty plan and sets
// UA_DEVICE_BAD_METADATA_BIT in *status.
cudaError_t launch_device_plan(const DevPlanShape &s, const DevPlanLayout &L, const int32_t *cu,
                               const int32_t *seqused_k, int32_t causal, void *workspace,
                               int *status, cudaStream_t stream);

// Writes the new tokens' K / V rows ([total_q, Hkv, D] bf16) into their
// pages of block_size tokens: token i of sequence s to position
// seqused_k[s] - Lq + i.
cudaError_t launch_kv_append(const void *k_new, const void *v_new, const int32_t *cu,
                             const int32_t *seqused_k, const int32_t *block_table, void *k_cache,
                             void *v_cache, int32_t num_seqs, int32_t total_q, int32_t num_kv_heads,
                             int32_t head_size, int32_t block_size, int32_t num_blocks,
                             int32_t bt_stride, int *status, cudaStream_t stream);

// Pages of block_size = 16 r tokens as runs of r 16-token pages: entry j of
// each block-table row (num_seqs * stride entries), page b, becomes entries
// j r .. j r + r - 1 = b r .. b r + r - 1 of `out` (-1 for an entry outside
// [0, num_blocks)).  ua_pages.cu.
cudaError_t launch_expand_block_table(const int32_t *block_table, int32_t *out, int64_t entries,
                                      int32_t r, int32_t num_blocks, cudaStream_t stream);

// An e4m3 cache's pages for the prefill kernels: decoded page t belongs to
// sequence dq[n_dq + 1 + j] for the last j with dq[j] <= t (page t - dq[j] of
// it); its K and V (16 slots x Hkv x d e4m3 bytes each) are written as bf16
// into k16 / v16 at page t, and dq_bt[seq][page] = t.  ua_pages.cu.
cudaError_t launch_dequant_pages(const void *k8, const void *v8, const int32_t *block_table,
                                 int32_t bt_stride, int32_t num_blocks, const int32_t *dq, int32_t n_dq,
                                 int64_t dq_pages, int32_t *dq_bt, void *k16, void *v16, int32_t num_kv_heads,
                                 int32_t head_size, int *status, cudaStream_t stream);

}  // namespace ua
