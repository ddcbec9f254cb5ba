// ua_plan.h -- the work partition of unified paged varlen attention.
//
// The pages behind this library explain why one call needs a per-batch plan:
// a single fixed grid fits prefill, chunked prefill and decode badly, and
// tile sizes good for one are poor for the other ("[Kernel] [V1] Improved
// performance for V1 Triton (ROCm) backend", vLLM PR #14152, section "How is
// this performance improvement achieved?").  The unified kernel instead packs
// the query heads of one KV head along the query dimension ("[Kernel] Unified
// Triton kernel that doesn't distinguish between prefill + decode", vLLM PR
// #16828, PR description).  This plan keeps the single call and the GQA
// packing, and splits the batch into:
//
//   * decode units -- (sequence, kv head, 16-row tile) for sequences whose
//     packed rows (Lq * G) fit one 16-row warp-MMA tile.  Their KV pages are
//     concatenated and cut into equal page ranges, one per persistent CTA, so
//     every SM streams the same number of pages (split-KV).  A unit cut into
//     several pieces writes fp32 partials; the CTA that writes a unit's last
//     partial merges them with a log-sum-exp rule.  With two kv heads per
//     unit (the e4m3 cache, and heads narrower than 128 columns; Hkv even),
//     a unit is (sequence, kv heads h and h + 1, 8-row tile): tile rows 0-7
//     belong to head h, rows 8-15 to head h + 1.
//   * prefill tiles -- (sequence, kv head, 256-row tile) for the rest: two
//     128-row tensor-core tiles that share every K/V tile they load, longest
//     first.  Short items are dealt to the CTAs in advance (rounds of
//     alternating direction); long ones (2048 visible keys or more on
//     average) are claimed by the CTAs one at a time from the longest-first
//     list (an atomic counter), so that CTAs that run faster take more.
//
// Rows are packed (token, head-in-group) pairs: packed row r of a (sequence,
// kv head) is token r / G and query head kv_head * G + r % G.
//
// This header is shared by host and device code; it holds plain structs only.
#pragma once

#include <stddef.h>
#include <stdint.h>

#define UA_DEVICE_BAD_BLOCK_ID_BIT 0x1
#define UA_DEVICE_WAIT_TIMEOUT_BIT 0x2
#define UA_DEVICE_BAD_METADATA_BIT 0x4

namespace ua {

// Every wait of the kernels gives up after this long (real waits are
// microseconds), records UA_DEVICE_WAIT_TIMEOUT and winds the kernel down.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;   // 4 s

constexpr int kBlockSize = 16;      // tokens per KV page as the kernels see it
constexpr int kMaxBlockSize = 256;  // caller pages: multiples of kBlockSize up to this (viewed as
                                    // runs of 16-token pages)
constexpr int kDecRows = 16;        // packed rows per decode tile (warp MMA M)
constexpr int kPreRows = 128;       // packed rows per tcgen05 tile (MMA M)
constexpr int kPreTileRows = 256;   // packed rows per prefill work item (two MMA tiles)
constexpr int kKvTile = 128;        // keys per prefill KV tile (8 pages)
constexpr int kDecCtasPerSm = 2;    // resident decode CTAs per SM
// A decode unit's fixed cost in pages of one kv head (its Q tile and
// descriptor, the merge of the four consumer warps' partial results, the
// output): the decode CTAs get equal shares of pages + kDecUnitCost per unit,
// not of pages alone.  Measured on 256 sequences of ~40 pages: a CTA spends
// ~2 us per unit outside its pages (~5-7 pages' time), and with equal pages
// the CTAs that drew many short units ended 33 us after the median.
constexpr int64_t kDecUnitCost = 6;
constexpr size_t kAlign = 256;
// The scheduling block of claimed prefill items: the index of the next
// unclaimed item, the prefill CTAs that have finished (the last one zeroes
// both again, so a plan can be reused), the number of items.
enum : int { kSchedNext = 0, kSchedDone = 1, kSchedItems = 2, kSchedInts = 4 };
// Long prefill items: this many 128-key tiles on average (2048 keys) or more.
// They run on SM pairs when the two-SM kernel may take them (measured on the
// 2048-token chunks over 4096-token contexts: 486-497 us against 521 us for
// one SM per item, claimed), otherwise they are claimed by the one-SM CTAs
// as they go (-14% against dealing them).  Shorter items are dealt to one SM
// each: on 1000-token prompts the one-SM kernel takes 151 us against 177-183
// us on pairs (a pair spends an item's fixed costs on 128 rows per SM, one
// SM on 256), and claiming them gained nothing.
constexpr int kClaimMinMeanKvTiles = 16;

// Head sizes: 64, 128 and 256 run in kernels of their own size; 80, 96 and
// 112 run in the head-size-128 decode kernel, their rows zero-padded to 128
// columns in shared memory (the padding is never read from memory).
inline bool head_size_supported(int d) {
    return d == 64 || d == 80 || d == 96 || d == 112 || d == 128 || d == 256;
}
// The head size of the kernel that runs head size d (its partials' row length).
inline int kernel_head_size(int d) { return (d > 64 && d < 128) ? 128 : d; }

struct alignas(16) DecPiece {   // one contiguous page range of one decode unit
    int32_t seq;
    int32_t kvh;         // (first) kv head of the unit
    int32_t row0;        // first packed row of the unit
    int32_t nrows;       // packed rows in the unit, per kv head (<= kDecRows / heads per unit)
    int32_t page_begin;  // first logical page of the range
    int32_t page_end;    // one past the last logical page
    int32_t slot;        // -1: the piece is the whole unit, write bf16 output; else partial slot
    int32_t unit;        // split piece: index of its unit in the combine list; else -1
};

struct alignas(16) CombUnit {   // a decode unit split over several pieces
    int32_t seq;
    int32_t kvh;
    int32_t row0;
    int32_t nrows;
    int32_t slot_begin;
    int32_t nslots;
    int32_t pad0;
    int32_t pad1;
};

struct alignas(16) PreTile {    // one prefill work item: up to two 128-row MMA tiles
    int32_t seq;
    int32_t kvh;
    int32_t row0;
    int32_t nrows;
    int32_t kv_tiles;    // 128-key tiles its last row visits (the ordering key)
    int32_t q0;          // cu_seqlens_q[seq]: first token of the sequence
    int32_t lq;          // query tokens of the sequence
    int32_t lk;          // seqused_k[seq]
};

// Problem description as seen by the planner (host metadata).
struct Problem {
    const int32_t *cu;     // [num_seqs + 1]
    const int32_t *lk;     // [num_seqs]
    int32_t num_seqs;
    int32_t hq;
    int32_t hkv;
    int32_t d;
    int32_t bs;
    int32_t bt_stride;
    bool causal;
    int32_t kv_heads_per_unit = 1;   // decode units: 1, or 2 (adjacent heads, <= 8 rows each)
    bool prefill_claim = false;      // long prefill items may be claimed as the CTAs go
    bool prefill_pair = false;       // long prefill items may run on SM pairs (two-SM kernel)
    bool dequant_prefill = false;    // e4m3 cache: the prefill rows' pages are decoded to bf16
                                     // in the workspace first (the plan lays that region out)
    bool split_sms = false;          // a batch with both kinds of work may run its two kernels
                                     // side by side on disjoint sets of SMs
};

// Side by side.  A batch of decode rows and prefill items (head size 128,
// bf16 cache) can run its decode kernel (HBM-bound) and its prefill kernel
// (tensor-bound) at the same time on disjoint SMs: the prefill kernel is
// launched first and its CTAs (or CTA pairs) take n SMs, the decode kernel's
// 2 (N - n) CTAs take the rest.  n balances the two estimated times, each
// kernel on its own SMs: the decode kernel moves up to kSplitDecodeGBsPerSm
// GB/s per SM (~33 GB/s for each of its two CTAs, what their producer warps
// issue; at most kSplitHbmGBs in all), a unit costing kSplitUnitPages pages
// more; the two-SM prefill kernel
// runs kSplitPairGflopsPerSm GFLOP/s per SM (the pair with the most long
// items ends last), the one-SM kernel
// kSplitOneGflopsPerSm (all measured on a GB300: the Llama-3-70B long mixed
// step and the Llama-3.1-8B step of 256 decode rows beside four 512-token
// chunks).  The split is taken when it is estimated to save kSplitMinGainPct
// percent or more of the two kernels' time one after the other.
constexpr double kSplitDecodeGBsPerSm = 68.0;
constexpr double kSplitHbmGBs = 6200.0;
constexpr double kSplitUnitPages = 18.0;
constexpr double kSplitPairGflopsPerSm = 9800.0;
constexpr double kSplitOneGflopsPerSm = 5700.0;
constexpr int kSplitMinGainPct = 8;
constexpr int kSplitMinDecodeSms = 8;

// Offsets of the plan sections inside the device workspace.
struct Layout {
    size_t off_cta;        // int32 [dec_ctas + 1]
    size_t off_pieces;     // DecPiece [n_pieces]
    size_t off_comb;       // CombUnit [n_comb]
    size_t off_comb_count; // int32 [n_comb]: partials written so far (zero in the blob)
    size_t off_tiles;      // PreTile [n_tiles]
    size_t off_pre_begin;  // int32 [pre_ctas + 1] (items dealt in advance)
    size_t off_sched;      // int32 [kSchedInts] (items claimed as the CTAs go)
    size_t off_dq;         // int32 [n_dq + 1] first decoded page of each prefill sequence,
                           // then int32 [n_dq] the sequences (e4m3 cache only)
    size_t blob_bytes;     // bytes copied host -> device per call (offsets above are
                           // from the start of the workspace)
    size_t off_part_o;     // float [n_slots][kDecRows][d]
    size_t off_part_ml;    // float [n_slots][kDecRows][2]
    size_t off_dq_bt;      // int32 [num_seqs][bt_stride]: block table of the decoded pages
    size_t off_dq_k;       // bf16 [dq_pages][16][Hkv][d]: the prefill sequences' K pages
    size_t off_dq_v;       // bf16 [dq_pages][16][Hkv][d]: and V pages
    size_t total_bytes;    // workspace bytes
};

}  // namespace ua
