// ua_planner.cpp -- validation and the work-partition pass (host C++).
//
// The partition follows the reasoning of "[Kernel] [V1] Improved performance
// for V1 Triton (ROCm) backend" (vLLM PR #14152, section "How is this
// performance improvement achieved?"): decode rows and prefill rows want
// different grids, so each call plans its own.  Decode units are balanced by
// pages across persistent CTAs; prefill tiles are ordered longest first.
#include "ua_planner.h"

#include <algorithm>
#include <cstring>

namespace ua {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool prefill_supports(const Problem &p) {
    const int g = p.hq / p.hkv;
    return g >= 1 && g <= kPreRows && (kPreRows % g) == 0;
}

int validate_problem(const Problem &p) {
    if (p.num_seqs < 0 || p.hq <= 0 || p.hkv <= 0 || p.bt_stride < 0) return 1;
    if (p.num_seqs > 0 && (p.cu == nullptr || p.lk == nullptr)) return 1;
    if (p.hq % p.hkv != 0) return 2;
    if (p.d != 64 && p.d != 128) return 2;
    if (p.bs != kBlockSize) return 2;
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

// Visible keys of the last packed row of a tile (all rows of the tile see a
// prefix of the context; the last row sees the longest one).
static int64_t tile_key_end(const Problem &p, int64_t lq, int64_t lk, int64_t last_row, int g) {
    if (!p.causal) return lk;
    const int64_t i_last = last_row / g;
    return std::min<int64_t>(lk, lk - lq + i_last + 1);
}

void build_plan(const Problem &p, int num_sms, bool prefill_enabled, Plan &plan) {
    // reuse the vectors' capacity across calls (the plan is thread-local in the API)
    plan.dec_ctas = 0;
    plan.dec_pages = 0;
    plan.cta_begin.clear();
    plan.pieces.clear();
    plan.comb.clear();
    plan.n_slots = 0;
    plan.tiles.clear();
    plan.pre_ctas = 0;
    plan.layout = Layout{};
    const int g = p.hq / p.hkv;
    const bool pre_ok = prefill_enabled && prefill_supports(p);

    struct Unit {
        int32_t seq, kvh, row0, nrows, pages;
    };
    std::vector<Unit> units;
    for (int s = 0; s < p.num_seqs; ++s) {
        const int64_t lq = (int64_t)p.cu[s + 1] - p.cu[s];
        const int64_t lk = p.lk[s];
        if (lq == 0) continue;
        const int64_t rows = lq * g;
        const bool decode = rows <= kDecRows || !pre_ok;
        if (decode) {
            for (int h = 0; h < p.hkv; ++h)
                for (int64_t r0 = 0; r0 < rows; r0 += kDecRows) {
                    const int64_t nr = std::min<int64_t>(kDecRows, rows - r0);
                    const int64_t kend = tile_key_end(p, lq, lk, r0 + nr - 1, g);
                    units.push_back({s, h, (int32_t)r0, (int32_t)nr,
                                     (int32_t)((kend + p.bs - 1) / p.bs)});
                }
        } else {
            for (int h = 0; h < p.hkv; ++h)
                for (int64_t r0 = 0; r0 < rows; r0 += kPreRows) {
                    const int64_t nr = std::min<int64_t>(kPreRows, rows - r0);
                    const int64_t kend = tile_key_end(p, lq, lk, r0 + nr - 1, g);
                    PreTile t{};
                    t.seq = s;
                    t.kvh = h;
                    t.row0 = (int32_t)r0;
                    t.nrows = (int32_t)nr;
                    t.kv_tiles = (int32_t)((kend + kKvTile - 1) / kKvTile);
                    plan.tiles.push_back(t);
                }
        }
    }

    // ---- prefill: longest first (stable, so equal lengths keep batch order)
    std::stable_sort(plan.tiles.begin(), plan.tiles.end(),
                     [](const PreTile &a, const PreTile &b) { return a.kv_tiles > b.kv_tiles; });
    plan.pre_ctas = (int32_t)std::min<size_t>(plan.tiles.size(), (size_t)std::max(num_sms, 1));

    // ---- decode: equal page ranges over the concatenated units
    int64_t total = 0;
    for (const Unit &u : units) total += u.pages;
    plan.dec_pages = total;
    if (total > 0) {
        const int64_t want = (int64_t)kDecCtasPerSm * std::max(num_sms, 1);
        const int64_t ctas = std::min<int64_t>(want, total);
        plan.dec_ctas = (int32_t)ctas;
        plan.cta_begin.assign(ctas + 1, 0);
        // pieces per unit, gathered first so slots can be assigned per unit
        std::vector<std::vector<DecPiece>> per_unit(units.size());
        size_t ui = 0;
        int64_t unit_start = 0;   // global page index of units[ui]'s first page
        for (int64_t c = 0; c < ctas; ++c) {
            const int64_t lo = total * c / ctas;
            const int64_t hi = total * (c + 1) / ctas;
            int64_t pos = lo;
            while (pos < hi) {
                while (unit_start + units[ui].pages <= pos) {
                    unit_start += units[ui].pages;
                    ++ui;
                }
                const Unit &u = units[ui];
                const int64_t b = pos - unit_start;
                const int64_t e = std::min<int64_t>(u.pages, hi - unit_start);
                DecPiece pc{};
                pc.seq = u.seq;
                pc.kvh = u.kvh;
                pc.row0 = u.row0;
                pc.nrows = u.nrows;
                pc.page_begin = (int32_t)b;
                pc.page_end = (int32_t)e;
                pc.slot = -1;
                pc.unit = (int32_t)ui;
                // remember which CTA owns it through the order of emission
                per_unit[ui].push_back(pc);
                pos = unit_start + e;
            }
        }
        // slots for split units
        int32_t slot = 0;
        for (size_t u = 0; u < units.size(); ++u) {
            if (per_unit[u].size() > 1) {
                CombUnit cu{};
                cu.seq = units[u].seq;
                cu.kvh = units[u].kvh;
                cu.row0 = units[u].row0;
                cu.nrows = units[u].nrows;
                cu.slot_begin = slot;
                cu.nslots = (int32_t)per_unit[u].size();
                plan.comb.push_back(cu);
                for (DecPiece &pc : per_unit[u]) pc.slot = slot++;
            }
        }
        plan.n_slots = slot;
        // emit pieces in CTA order (re-walk the same partition)
        std::vector<size_t> next(units.size(), 0);
        ui = 0;
        unit_start = 0;
        for (int64_t c = 0; c < ctas; ++c) {
            plan.cta_begin[c] = (int32_t)plan.pieces.size();
            const int64_t lo = total * c / ctas;
            const int64_t hi = total * (c + 1) / ctas;
            int64_t pos = lo;
            while (pos < hi) {
                while (unit_start + units[ui].pages <= pos) {
                    unit_start += units[ui].pages;
                    ++ui;
                }
                const int64_t e = std::min<int64_t>(units[ui].pages, hi - unit_start);
                plan.pieces.push_back(per_unit[ui][next[ui]++]);
                pos = unit_start + e;
            }
        }
        plan.cta_begin[ctas] = (int32_t)plan.pieces.size();
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
    L.off_tiles = off;
    off = align_up(off + sizeof(PreTile) * plan.tiles.size(), kAlign);
    L.blob_bytes = off;
    L.off_part_o = off;
    off = align_up(off + sizeof(float) * (size_t)plan.n_slots * kDecRows * p.d, kAlign);
    L.off_part_ml = off;
    off = align_up(off + 2 * sizeof(float) * (size_t)plan.n_slots * kDecRows, kAlign);
    L.total_bytes = (plan.pieces.empty() && plan.tiles.empty()) ? 0 : off;
}

void serialize_plan(const Plan &plan, std::vector<uint8_t> &blob) {
    const Layout &L = plan.layout;
    blob.assign(L.blob_bytes, 0);
    if (!plan.cta_begin.empty())
        std::memcpy(blob.data() + L.off_cta, plan.cta_begin.data(),
                    sizeof(int32_t) * plan.cta_begin.size());
    if (!plan.pieces.empty())
        std::memcpy(blob.data() + L.off_pieces, plan.pieces.data(),
                    sizeof(DecPiece) * plan.pieces.size());
    if (!plan.comb.empty())
        std::memcpy(blob.data() + L.off_comb, plan.comb.data(), sizeof(CombUnit) * plan.comb.size());
    if (!plan.tiles.empty())
        std::memcpy(blob.data() + L.off_tiles, plan.tiles.data(),
                    sizeof(PreTile) * plan.tiles.size());
}

}  // namespace ua
