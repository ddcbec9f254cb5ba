// ua_planner.h -- host-side validation and work partition (no CUDA calls).
#pragma once

#include <vector>

#include "ua_plan.h"

namespace ua {

struct Plan {
    int32_t dec_ctas = 0;
    int32_t split_pre_sms = 0;          // > 0: the prefill kernel runs on this many SMs and the decode
                                        // kernel on the rest, at the same time
    int32_t dec_heads_per_unit = 1;     // kv heads per decode unit (1 or 2)
    int64_t dec_pages = 0;
    std::vector<int32_t> cta_begin;     // dec_ctas + 1
    std::vector<DecPiece> pieces;
    std::vector<CombUnit> comb;
    int32_t n_slots = 0;
    std::vector<PreTile> tiles;         // grouped by prefill CTA (dealt), or longest first (claimed)
    std::vector<int32_t> pre_begin;     // dealt: pre_ctas + 1, worker c runs tiles [pre_begin[c], pre_begin[c+1])
    int32_t pre_ctas = 0;               // prefill workers: CTAs, or CTA pairs (pre_pair)
    bool pre_claimed = false;           // the prefill CTAs claim items from the list as they go
    bool pre_pair = false;              // the items are dealt to SM pairs (two-SM kernel)
    // e4m3 cache (Problem::dequant_prefill): the sequences with prefill items, in
    // order, and the first of their pages in the decoded bf16 copy (n_dq + 1
    // entries); each sequence's whole context is decoded
    std::vector<int32_t> dq_seq;
    std::vector<int32_t> dq_base;
    int64_t dq_pages = 0;
    Layout layout{};
};

// Status codes follow ua_status (0 ok, 1 invalid arg, 2 unsupported).
int validate_problem(const Problem &p);

// Builds the partition for a GPU with num_sms multiprocessors.
// prefill_enabled = false routes every row tile to the decode kernel.
void build_plan(const Problem &p, int num_sms, bool prefill_enabled, Plan &plan);

// Packs the plan sections into one host blob laid out as plan.layout says.
void serialize_plan(const Plan &plan, std::vector<uint8_t> &blob);
// The same into dst, which holds at least plan.layout.blob_bytes bytes.
void serialize_plan_to(const Plan &plan, uint8_t *dst);

// True when the prefill (tcgen05) kernel can take this head grouping.
bool prefill_supports(const Problem &p);

}  // namespace ua
