// ua_planner.cpp -- validation and the work-partition pass (host C++).
//
// The partition follows the reasoning of "[Kernel] [V1] Improved performance
// for V1 Triton (ROCm) backend" (vLLM PR #14152, section "How is this
// performance improvement achieved?"): decode rows and prefill rows want
// different grids, so each call plans its own.  Decode units are balanced by
// pages across persistent CTAs; prefill work items go to CTAs longest first,
// dealt in rounds of alternating direction, so that the persistent CTAs
// finish together.
#include "ua_planner.h"

#include <algorithm>
#include <cmath>
#include <cstring>

namespace ua {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool prefill_supports(const Problem &p) {
    const int g = p.hq / p.hkv;
    // the one-SM tensor-core kernel is built for head sizes 64 and 128, the
    // two-SM kernel for 128 and 256
    return (p.d == 64 || p.d == 128 || (p.d == 256 && p.prefill_pair)) && g >= 1 && g <= kPreRows &&
           (kPreRows % g) == 0;
}

int validate_problem(const Problem &p) {
    if (p.num_seqs < 0 || p.hq <= 0 || p.hkv <= 0 || p.bt_stride < 0) return 1;
    if (p.num_seqs > 0 && (p.cu == nullptr || p.lk == nullptr)) return 1;
    if (p.hq % p.hkv != 0) return 2;
    if (!head_size_supported(p.d)) return 2;
    if (p.bs <= 0 || p.bs % kBlockSize != 0 || p.bs > kMaxBlockSize) return 2;
    // the block table seen in 16-token pages stays indexable in int32
    if ((int64_t)p.bt_stride * (p.bs / kBlockSize) > INT32_MAX / 4) return 1;
    if (p.num_seqs == 0) return 0;
    if (p.cu[0] != 0) return 1;
    for (int s = 0; s < p.num_seqs; ++s) {
        const int64_t lq = (int64_t)p.cu[s + 1] - p.cu[s];
        const int64_t lk = p.lk[s];
        if (lq < 0 || lk < 0) return 1;
        if (lq > 0 && lk == 0) return 1;
        if (p.causal && lk < lq) return 1;
        if ((lk + p.bs - 1) / p.bs > p.bt_stride) return 1;
    }
    // packed rows of one sequence and kv head must fit int32
    for (int s = 0; s < p.num_seqs; ++s) {
        const int64_t lq = (int64_t)p.cu[s + 1] - p.cu[s];
        if (lq * (p.hq / p.hkv) > INT32_MAX / 2) return 2;
    }
    return 0;
}

void build_plan(const Problem &p, int num_sms, bool prefill_enabled, Plan &plan) {
    // reuse the vectors' capacity across calls (the plan is thread-local in the API)
    plan.dec_ctas = 0;
    plan.split_pre_sms = 0;
    plan.dec_pages = 0;
    plan.cta_begin.clear();
    plan.pieces.clear();
    plan.comb.clear();
    plan.n_slots = 0;
    plan.tiles.clear();
    plan.pre_begin.clear();
    plan.pre_ctas = 0;
    plan.pre_claimed = false;
    plan.pre_pair = false;
    plan.layout = Layout{};
    const int g = p.hq / p.hkv;
    const bool pre_ok = prefill_enabled && prefill_supports(p);
    // decode units cover 1 kv head, or 2 adjacent heads (p.hkv even) with at
    // most kDecRows / 2 rows each
    const int hpu = (p.kv_heads_per_unit == 2 && p.hkv % 2 == 0) ? 2 : 1;
    plan.dec_heads_per_unit = hpu;

    struct Unit {
        int32_t seq, kvh, row0, nrows, pages;
    };
    // scratch kept per thread; bound to plain references once (each access to a
    // thread_local object with a constructor goes through an init check)
    thread_local std::vector<Unit> tl_units;
    thread_local std::vector<PreTile> tl_unsorted;
    thread_local std::vector<int32_t> tl_counts;
    std::vector<Unit> &units = tl_units;
    std::vector<PreTile> &unsorted = tl_unsorted;
    std::vector<int32_t> &counts = tl_counts;
    units.clear();
    unsorted.clear();
    int32_t max_kv = 0;
    // Prefill rows that would make only a few long work items (say a group's
    // new tokens against a long shared prefix) leave most SMs idle in the
    // prefill kernel, one CTA per item; they go to the decode kernel instead,
    // whose split-KV spreads the same keys over every CTA.
    bool prefill_rows_to_decode = false;
    if (pre_ok) {
        int64_t items = 0;
        int64_t max_steps = 0;
        for (int s = 0; s < p.num_seqs; ++s) {
            const int64_t lq = (int64_t)p.cu[s + 1] - p.cu[s];
            if (lq * g <= kDecRows) continue;
            items += (lq * g + kPreTileRows - 1) / kPreTileRows * p.hkv;
            max_steps = std::max<int64_t>(max_steps, ((int64_t)p.lk[s] + 63) / 64);
        }
        prefill_rows_to_decode = items > 0 && items * 4 < std::max(num_sms, 1) && max_steps >= 32;
    }
    // 32-bit arithmetic below: validate_problem bounds Lq * G and Lk well inside int32
    for (int s = 0; s < p.num_seqs; ++s) {
        const int32_t lq = p.cu[s + 1] - p.cu[s];
        const int32_t lk = p.lk[s];
        if (lq == 0) continue;
        const int32_t rows = lq * g;
        const bool decode = rows <= kDecRows || !pre_ok || prefill_rows_to_decode;
        const int32_t step = decode ? kDecRows / hpu : kPreTileRows;
        // visible keys of the last row of each row tile; the same for every kv head
        for (int32_t r0 = 0; r0 < rows; r0 += step) {
            const int32_t nr = std::min<int32_t>(step, rows - r0);
            const int32_t kend = p.causal ? std::min<int32_t>(lk, lk - lq + (r0 + nr - 1) / g + 1) : lk;
            if (decode) {
                const int32_t pages = (kend + kBlockSize - 1) / kBlockSize;
                for (int h = 0; h < p.hkv; h += hpu) units.push_back({s, h, r0, nr, pages});
            } else {
                PreTile t{};
                t.seq = s;
                t.q0 = p.cu[s];
                t.lq = lq;
                t.lk = lk;
                t.row0 = r0;
                t.nrows = nr;
                t.kv_tiles = (kend + kKvTile - 1) / kKvTile;
                max_kv = std::max(max_kv, t.kv_tiles);
                for (int h = 0; h < p.hkv; ++h) {
                    t.kvh = h;
                    unsorted.push_back(t);
                }
            }
        }
    }
    // ---- prefill: longest first (counting sort, equal lengths keep batch order).
    // Long items on average (kClaimMinMeanKvTiles) go to SM pairs when the
    // caller allows it, or else are claimed by the CTAs from this list as they
    // go.  Otherwise (and on pairs) they are dealt to the workers in rounds
    // whose direction alternates (0..n-1, then n-1..0, ...): the worker that
    // got the longest item of a round gets the shortest of the next, which
    // keeps the workers' totals within about one item of each other.
    // O(items) host cost.
    // ---- both kinds of work: the two kernels side by side on disjoint SMs
    // (head size 128, bf16 cache; see kSplitDecodeGBsPerSm)
    int32_t pre_sms = num_sms, dec_sms = num_sms;
    if (p.split_sms && !p.dequant_prefill && p.d == 128 && !units.empty() && !unsorted.empty() &&
        num_sms >= 2 * kSplitMinDecodeSms) {
        const double page_bytes = 2.0 * kBlockSize * p.d * 2 * hpu;
        double bytes = 0.0, flops = 0.0, kv_sum = 0.0;
        for (const Unit &u : units) bytes += ((double)u.pages + kSplitUnitPages) * page_bytes;
        for (const PreTile &t : unsorted) {
            flops += 4.0 * t.nrows * (double)t.kv_tiles * kKvTile * p.d;
            kv_sum += t.kv_tiles;
        }
        // long items run on SM pairs (as the deal below decides), short ones on one SM each
        const bool pairs = p.prefill_pair && kv_sum >= (double)kClaimMinMeanKvTiles * (double)unsorted.size();
        const double N = num_sms, r = kSplitDecodeGBsPerSm * 1e9, bw = kSplitHbmGBs * 1e9;
        const double f = (pairs ? kSplitPairGflopsPerSm : kSplitOneGflopsPerSm) * 1e9;
        auto t_dec = [&](double n) { return std::max(bytes / bw, bytes / (n * r)); };
        // long items on pairs: the pair with the most items (the deal gives each
        // ceil(items / pairs) or one fewer, of about equal length) ends last
        const double n_items = (double)unsorted.size();
        auto t_pre = [&](double n) {
            if (!pairs) return flops / (n * f);
            const double per = std::ceil(n_items / std::max(1.0, std::floor(n / 2)));
            return flops / n_items * per / (2.0 * f);
        };
        // F / (n f) = B / ((N - n) r)
        const double n_bal = flops * r * N / (flops * r + bytes * f);
        const int32_t step = pairs ? 2 : 1;
        int32_t best = 0;
        double best_t = t_dec(N) + t_pre(N);
        for (int32_t n = std::max<int32_t>(step, ((int32_t)n_bal - 4) / step * step);
             n <= std::min<int32_t>(num_sms - kSplitMinDecodeSms, (int32_t)n_bal + 4); n += step) {
            const double t = std::max(t_pre(n), t_dec(N - n));
            if (t < best_t) {
                best_t = t;
                best = n;
            }
        }
        if (best > 0 && best_t * 100.0 <= (t_dec(N) + t_pre(N)) * (100 - kSplitMinGainPct)) {
            pre_sms = best;
            dec_sms = num_sms - best;
            plan.split_pre_sms = best;
        }
    }
    if (!unsorted.empty()) {
        thread_local std::vector<PreTile> tl_sorted;
        thread_local std::vector<int32_t> tl_owner;
        std::vector<PreTile> &sorted = tl_sorted;
        std::vector<int32_t> &owner = tl_owner;
        counts.assign((size_t)max_kv + 2, 0);
        int64_t kv_sum = 0;
        for (const PreTile &t : unsorted) {
            ++counts[(size_t)(max_kv - t.kv_tiles) + 1];
            kv_sum += t.kv_tiles;
        }
        for (size_t b = 1; b < counts.size(); ++b) counts[b] += counts[b - 1];
        sorted.resize(unsorted.size());
        for (const PreTile &t : unsorted) sorted[(size_t)counts[(size_t)(max_kv - t.kv_tiles)]++] = t;

        const bool long_items = kv_sum >= (int64_t)kClaimMinMeanKvTiles * (int64_t)sorted.size();
        // head size 256 has only the two-SM kernel: every item goes to SM pairs
        plan.pre_pair = p.prefill_pair && (long_items || p.d == 256);
        const int32_t workers = plan.pre_pair ? std::max(pre_sms / 2, 1) : std::max(pre_sms, 1);
        const int32_t ctas = (int32_t)std::min<size_t>(sorted.size(), (size_t)workers);
        plan.pre_ctas = ctas;
        plan.pre_claimed = !plan.pre_pair && p.prefill_claim && long_items;
        if (plan.pre_claimed) {
            plan.tiles = sorted;
        } else {
            owner.resize(sorted.size());
            plan.pre_begin.assign((size_t)ctas + 1, 0);
            for (size_t i = 0; i < sorted.size(); ++i) {
                const size_t round = i / (size_t)ctas, k = i % (size_t)ctas;
                owner[i] = (int32_t)((round & 1) ? (size_t)ctas - 1 - k : k);
                ++plan.pre_begin[(size_t)owner[i] + 1];
            }
            for (int32_t c = 0; c < ctas; ++c) plan.pre_begin[(size_t)c + 1] += plan.pre_begin[(size_t)c];
            // group by CTA, keeping each CTA's items in assignment (longest-first) order
            counts.assign((size_t)ctas, 0);
            for (int32_t c = 0; c < ctas; ++c) counts[(size_t)c] = plan.pre_begin[(size_t)c];
            plan.tiles.resize(sorted.size());
            for (size_t i = 0; i < sorted.size(); ++i) plan.tiles[(size_t)counts[(size_t)owner[i]]++] = sorted[i];
        }
    }

    // ---- decode: equal shares of cost over the concatenated units, a unit
    // costing kDecUnitCost + its pages.  CTA c takes cost [T c / C, T (c+1) / C);
    // a cost position inside unit u's fixed part maps to u's first page, one in
    // its pages to that page, so the CTAs' page ranges tile the pages in order
    // (a range may be empty, always at a unit boundary).
    int64_t total = 0;
    for (const Unit &u : units) total += u.pages;
    plan.dec_pages = total;
    if (total > 0) {
        const int64_t want = (int64_t)kDecCtasPerSm * std::max(dec_sms, 1);
        const int64_t ctas = std::min<int64_t>(want, total);
        plan.dec_ctas = (int32_t)ctas;
        plan.cta_begin.assign(ctas + 1, 0);
        const int64_t cost = total + kDecUnitCost * (int64_t)units.size();
        thread_local std::vector<int64_t> tl_bound;
        std::vector<int64_t> &bound = tl_bound;      // CTA c's pages: [bound[c], bound[c + 1])
        bound.assign((size_t)ctas + 1, total);
        {
            size_t u = 0;
            int64_t ustart = 0;                      // first page of unit u
            for (int64_t c = 0; c < ctas; ++c) {
                const int64_t x = cost * c / ctas;
                // the last unit whose cost starts at or before x
                while (u + 1 < units.size() &&
                       ustart + units[u].pages + kDecUnitCost * (int64_t)(u + 1) <= x) {
                    ustart += units[u].pages;
                    ++u;
                }
                const int64_t off = x - ustart - kDecUnitCost * (int64_t)u - kDecUnitCost;
                bound[(size_t)c] = ustart + std::min<int64_t>(std::max<int64_t>(off, 0), units[u].pages);
            }
        }
        counts.assign(units.size(), 0);              // pieces per unit
        size_t ui = 0;
        int64_t unit_start = 0;                      // global page index of units[ui]'s first page
        for (int64_t c = 0; c < ctas; ++c) {
            plan.cta_begin[c] = (int32_t)plan.pieces.size();
            const int64_t lo = bound[(size_t)c];
            const int64_t hi = bound[(size_t)c + 1];
            int64_t pos = lo;
            while (pos < hi) {
                while (unit_start + units[ui].pages <= pos) {
                    unit_start += units[ui].pages;
                    ++ui;
                }
                const Unit &u = units[ui];
                const int64_t e = std::min<int64_t>(u.pages, hi - unit_start);
                DecPiece pc{};
                pc.seq = u.seq;
                pc.kvh = u.kvh;
                pc.row0 = u.row0;
                pc.nrows = u.nrows;
                pc.page_begin = (int32_t)(pos - unit_start);
                pc.page_end = (int32_t)e;
                pc.slot = counts[ui]++;              // index among the unit's pieces for now
                pc.unit = (int32_t)ui;
                plan.pieces.push_back(pc);
                pos = unit_start + e;
            }
        }
        plan.cta_begin[ctas] = (int32_t)plan.pieces.size();
        // split units get consecutive partial slots, in unit order; comb_of: a
        // unit's index in the combine list
        thread_local std::vector<int32_t> tl_comb_of;
        std::vector<int32_t> &comb_of = tl_comb_of;
        comb_of.assign(units.size(), -1);
        int32_t slot = 0;
        for (size_t u = 0; u < units.size(); ++u) {
            if (counts[u] > 1) {
                comb_of[u] = (int32_t)plan.comb.size();
                CombUnit cu{};
                cu.seq = units[u].seq;
                cu.kvh = units[u].kvh;
                cu.row0 = units[u].row0;
                cu.nrows = units[u].nrows;
                cu.slot_begin = slot;
                cu.nslots = counts[u];
                plan.comb.push_back(cu);
                counts[u] = slot;                    // now: first slot of the unit
                slot += cu.nslots;
            } else {
                counts[u] = -1;                      // whole unit in one piece
            }
        }
        plan.n_slots = slot;
        // split pieces get their partial slot and the index of their combine entry
        for (DecPiece &pc : plan.pieces) {
            const int32_t first = counts[pc.unit];
            pc.slot = first < 0 ? -1 : first + pc.slot;
            pc.unit = comb_of[pc.unit];
        }
        // A CTA's last piece is the head of a unit that the next CTA finishes
        // first thing; run it first, so that both halves of the unit are done
        // early and its merge (by whichever CTA completes it) overlaps the rest
        // of the work instead of landing at the end of the kernel.
        for (int64_t c = 0; c < ctas; ++c) {
            const int32_t b0 = plan.cta_begin[c], b1 = plan.cta_begin[c + 1];
            if (b1 - b0 > 1 && plan.pieces[b1 - 1].slot >= 0)
                std::rotate(plan.pieces.begin() + b0, plan.pieces.begin() + (b1 - 1), plan.pieces.begin() + b1);
        }
    }

    // ---- e4m3 cache: the pages the prefill items read, decoded to bf16 in the
    // workspace (a sequence's items all see its context up to the end of it,
    // so its whole context is decoded, once)
    plan.dq_seq.clear();
    plan.dq_base.clear();
    plan.dq_pages = 0;
    if (p.dequant_prefill && !plan.tiles.empty()) {
        thread_local std::vector<uint8_t> tl_has;
        std::vector<uint8_t> &has = tl_has;
        has.assign((size_t)p.num_seqs, 0);
        for (const PreTile &t : plan.tiles) has[(size_t)t.seq] = 1;
        for (int32_t s = 0; s < p.num_seqs; ++s) {
            if (!has[(size_t)s]) continue;
            plan.dq_seq.push_back(s);
            plan.dq_base.push_back((int32_t)plan.dq_pages);
            plan.dq_pages += (p.lk[s] + kBlockSize - 1) / kBlockSize;
        }
        plan.dq_base.push_back((int32_t)plan.dq_pages);
    }

    // ---- workspace layout
    Layout &L = plan.layout;
    size_t off = 0;
    L.off_cta = off;
    off = align_up(off + sizeof(int32_t) * (plan.cta_begin.size() + 1), kAlign);
    L.off_pieces = off;
    off = align_up(off + sizeof(DecPiece) * plan.pieces.size(), kAlign);
    L.off_comb = off;
    off = align_up(off + sizeof(CombUnit) * plan.comb.size(), kAlign);
    L.off_comb_count = off;
    off = align_up(off + sizeof(int32_t) * plan.comb.size(), kAlign);
    L.off_tiles = off;
    off = align_up(off + sizeof(PreTile) * plan.tiles.size(), kAlign);
    L.off_pre_begin = off;
    off = align_up(off + sizeof(int32_t) * plan.pre_begin.size(), kAlign);
    L.off_sched = off;
    off = align_up(off + sizeof(int32_t) * kSchedInts, kAlign);
    L.off_dq = off;
    off = align_up(off + sizeof(int32_t) * (plan.dq_base.size() + plan.dq_seq.size()), kAlign);
    L.blob_bytes = off;
    L.off_part_o = off;
    off = align_up(off + sizeof(float) * (size_t)plan.n_slots * kDecRows * kernel_head_size(p.d), kAlign);
    L.off_part_ml = off;
    off = align_up(off + 2 * sizeof(float) * (size_t)plan.n_slots * kDecRows, kAlign);
    const bool dq = plan.dq_pages > 0;
    const size_t dq_page_bytes = (size_t)kBlockSize * (size_t)p.hkv * (size_t)p.d * 2;
    L.off_dq_bt = off;
    off = align_up(off + (dq ? sizeof(int32_t) * (size_t)p.num_seqs * (size_t)p.bt_stride : 0), kAlign);
    L.off_dq_k = off;
    off = align_up(off + (size_t)plan.dq_pages * dq_page_bytes, kAlign);
    L.off_dq_v = off;
    off = align_up(off + (size_t)plan.dq_pages * dq_page_bytes, kAlign);
    L.total_bytes = (plan.pieces.empty() && plan.tiles.empty()) ? 0 : off;
}

void serialize_plan_to(const Plan &plan, uint8_t *dst) {
    const Layout &L = plan.layout;
    std::memset(dst, 0, L.blob_bytes);
    if (!plan.cta_begin.empty())
        std::memcpy(dst + L.off_cta, plan.cta_begin.data(), sizeof(int32_t) * plan.cta_begin.size());
    if (!plan.pieces.empty())
        std::memcpy(dst + L.off_pieces, plan.pieces.data(), sizeof(DecPiece) * plan.pieces.size());
    if (!plan.comb.empty())
        std::memcpy(dst + L.off_comb, plan.comb.data(), sizeof(CombUnit) * plan.comb.size());
    if (!plan.tiles.empty())
        std::memcpy(dst + L.off_tiles, plan.tiles.data(), sizeof(PreTile) * plan.tiles.size());
    if (!plan.pre_begin.empty())
        std::memcpy(dst + L.off_pre_begin, plan.pre_begin.data(), sizeof(int32_t) * plan.pre_begin.size());
    const int32_t sched[kSchedInts] = {0, 0, (int32_t)plan.tiles.size(), 0};
    std::memcpy(dst + L.off_sched, sched, sizeof(sched));
    if (!plan.dq_base.empty()) {
        std::memcpy(dst + L.off_dq, plan.dq_base.data(), sizeof(int32_t) * plan.dq_base.size());
        std::memcpy(dst + L.off_dq + sizeof(int32_t) * plan.dq_base.size(), plan.dq_seq.data(),
                    sizeof(int32_t) * plan.dq_seq.size());
    }
}

void serialize_plan(const Plan &plan, std::vector<uint8_t> &blob) {
    blob.resize(plan.layout.blob_bytes);
    if (!blob.empty()) serialize_plan_to(plan, blob.data());
}

}  // namespace ua
