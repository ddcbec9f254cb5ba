// ua_device_plan.cu -- the work partition of unified attention, built on the GPU.
//
// The pages' unified kernel takes the engine's varlen metadata as it is, with
// no extra host-side step ("[Kernel] [V1] Improved performance for V1 Triton
// (ROCm) backend", vLLM PR #14152, section "How is this performance
// improvement achieved?").  The library's default call plans on the host from
// host copies of cu_seqlens_q and seqused_k; this file makes the same plan
// from the device arrays, so that a call needs no host copies and can be
// captured once in a CUDA graph and replayed with new lengths.
//
// ua_plan_kernel (one CTA of 1024 threads) produces exactly what build_plan
// in ua_planner.cpp produces -- the same routing of rows to the two kernels,
// the same equal page ranges of the decode units and split pieces (a CTA's
// last split piece moved to the front), the same longest-first prefill items
// dealt in rounds of alternating direction -- into a workspace laid out for
// capacities (sequences, query tokens, block-table width) instead of for one
// batch.  The grids are fixed (kDecCtasPerSm * SMs decode CTAs, SMs prefill
// CTAs); CTAs past the plan's count get empty ranges.
//
// Everything is scans, binary searches and one stable counting sort; the
// plan is a deterministic function of the metadata (no atomics decide an
// order).
#include <algorithm>
#include <climits>

#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {

namespace {

constexpr int kPlanThreads = 1024;
// The scratch arrays move into shared memory when they fit (most batches):
// the planner is a chain of dependent lookups, which then cost shared-memory
// rather than L2 latency.
constexpr size_t kPlanSmemMax = 192 * 1024;
constexpr int kPlanMaxGrid = 1024;    // decode CTAs the planner can partition over

struct UnitRec {          // one decode unit (a run of one or two kv heads' pages)
    int32_t seq, kvh, row0, nrows, pages, npieces, comb, slot0;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Exclusive prefix sum of v[0, n) in place by the whole block; returns the
// total.  Thread t takes a contiguous run of ceil(n / blockDim) entries.
template <typename T>
__device__ T block_scan(T *v, int n, T *s_part) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int b = min(n, tid * per), e = min(n, b + per);
    T sum = 0;
    for (int i = b; i < e; ++i) sum += v[i];
    T x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_part[w] = x;
    __syncthreads();
    if (w == 0) {
        T t = lane < nw ? s_part[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const T y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        s_part[lane] = t;
    }
    __syncthreads();
    const T total = s_part[nw - 1];
    T base = (w > 0 ? s_part[w - 1] : T(0)) + x - sum;
    for (int i = b; i < e; ++i) {
        const T t = v[i];
        v[i] = base;
        base += t;
    }
    __syncthreads();   // v complete and s_part free for the next scan
    return total;
}

// Two exclusive prefix sums (int32) in one pass; returns both totals.
__device__ int2 block_scan2(int32_t *v, int32_t *w2, int n, int32_t *s_part /* [64] */) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int b = min(n, tid * per), e = min(n, b + per);
    int s1 = 0, s2 = 0;
    for (int i = b; i < e; ++i) {
        s1 += v[i];
        s2 += w2[i];
    }
    int x1 = s1, x2 = s2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y1 = __shfl_up_sync(0xffffffffu, x1, o), y2 = __shfl_up_sync(0xffffffffu, x2, o);
        if (lane >= o) {
            x1 += y1;
            x2 += y2;
        }
    }
    if (lane == 31) {
        s_part[w] = x1;
        s_part[32 + w] = x2;
    }
    __syncthreads();
    if (w == 0) {
        int t1 = lane < nw ? s_part[lane] : 0, t2 = lane < nw ? s_part[32 + lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y1 = __shfl_up_sync(0xffffffffu, t1, o), y2 = __shfl_up_sync(0xffffffffu, t2, o);
            if (lane >= o) {
                t1 += y1;
                t2 += y2;
            }
        }
        s_part[lane] = t1;
        s_part[32 + lane] = t2;
    }
    __syncthreads();
    const int2 total = make_int2(s_part[nw - 1], s_part[32 + nw - 1]);
    int b1 = (w > 0 ? s_part[w - 1] : 0) + x1 - s1, b2 = (w > 0 ? s_part[32 + w - 1] : 0) + x2 - s2;
    for (int i = b; i < e; ++i) {
        const int t1 = v[i], t2 = w2[i];
        v[i] = b1;
        w2[i] = b2;
        b1 += t1;
        b2 += t2;
    }
    __syncthreads();
    return total;
}

// Block-wide reductions (every thread gets the result): warps reduce with
// shuffles, warp 0 reduces the warps' values, one shared slot broadcasts.
// block_sum_max2 returns (sum of a, max of b, max of c) in one pass.
__device__ void block_sum_max2(long long &a, long long &b, long long &c, long long *s_red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b = max(b, (long long)__shfl_xor_sync(0xffffffffu, b, o));
        c = max(c, (long long)__shfl_xor_sync(0xffffffffu, c, o));
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) {
        s_red[w] = a;
        s_red[32 + w] = b;
        s_red[64 + w] = c;
    }
    __syncthreads();
    if (w == 0) {
        long long x = lane < nw ? s_red[lane] : 0, y = lane < nw ? s_red[32 + lane] : LLONG_MIN,
                  z = lane < nw ? s_red[64 + lane] : LLONG_MIN;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            x += __shfl_xor_sync(0xffffffffu, x, o);
            y = max(y, (long long)__shfl_xor_sync(0xffffffffu, y, o));
            z = max(z, (long long)__shfl_xor_sync(0xffffffffu, z, o));
        }
        if (lane == 0) {
            s_red[96] = x;
            s_red[97] = y;
            s_red[98] = z;
        }
    }
    __syncthreads();
    a = s_red[96];
    b = s_red[97];
    c = s_red[98];
    __syncthreads();   // s_red free for the next reduction
}

__device__ long long block_max(long long v, long long *s_red) {
    long long zero = 0, dummy = LLONG_MIN;
    block_sum_max2(zero, v, dummy, s_red);
    return v;
}

// Last index i in [0, n) with a[i] <= x (a non-decreasing, a[0] <= x).
template <typename T>
__device__ int last_le(const T *a, int n, T x) {
    int lo = 0, hi = n;   // answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

struct PlanArgs {
    const int32_t *cu;
    const int32_t *lk;
    int32_t num_seqs, max_total_q, max_seq_q, hq, hkv, g, bt_stride, hpu, prefill_ok, num_sms, causal;
    int32_t pre_workers;      // prefill items are dealt to this many workers
    int32_t dec_grid, cap_units, cap_items, cap_pieces, cap_comb, cap_slots, n_buckets;
    long long *header;
    int32_t *cta_begin;       // [dec_grid + 1]
    DecPiece *pieces;         // [cap_pieces]
    CombUnit *comb;           // [cap_comb]
    int32_t *comb_count;      // [cap_comb]
    PreTile *tiles;           // [cap_items]
    int32_t *pre_begin;       // [num_sms + 1]
    // scratch
    int32_t *seq_u;           // [num_seqs + 1]
    int32_t *seq_i;           // [num_seqs + 1]
    UnitRec *urec;            // [cap_units]
    long long *ustart;        // [cap_units + 1]
    PreTile *irec;            // [cap_items] (batch order)
    int32_t *ikey;            // [cap_items]
    int32_t *hist;            // [n_buckets]
    int32_t *tmp;             // [max(cap_units, dec_grid) + 1]
    int32_t *tmp2;            // [max(cap_units, dec_grid) + 1]
    uint32_t smem_bytes;      // dynamic shared memory for scratch arrays that fit
    int *status;
};

__device__ void empty_plan(const PlanArgs &a, long long err) {
    for (int c = threadIdx.x; c <= a.dec_grid; c += blockDim.x) a.cta_begin[c] = 0;
    for (int c = threadIdx.x; c <= a.num_sms; c += blockDim.x) a.pre_begin[c] = 0;
    if (threadIdx.x < 8) a.header[threadIdx.x] = threadIdx.x == 7 ? err : 0;
    if (threadIdx.x == 0 && err) record_status(a.status, UA_DEVICE_BAD_METADATA_BIT);
}

__global__ void __launch_bounds__(kPlanThreads, 1) ua_plan_kernel(const PlanArgs args) {
    extern __shared__ __align__(16) uint8_t plan_smem[];
    // Scratch arrays that fit go to shared memory (generic pointers reach both;
    // the decisions depend only on counts every thread knows).
    PlanArgs a = args;
    size_t sm_used = 0;
    auto carve = [&](size_t bytes) -> uint8_t * {
        uint8_t *p = plan_smem + sm_used;
        sm_used = (sm_used + bytes + 15) & ~size_t(15);
        return p;
    };
    if (8 * ((size_t)a.num_seqs + 1) <= a.smem_bytes) {
        a.seq_u = reinterpret_cast<int32_t *>(carve(4 * ((size_t)a.num_seqs + 1)));
        a.seq_i = reinterpret_cast<int32_t *>(carve(4 * ((size_t)a.num_seqs + 1)));
    }
    __shared__ long long s_red[100];
    __shared__ int32_t s_part32[64];
    __shared__ long long s_part64[32];
    // decode CTA c: pages [s_clo[c], s_clo[c + 1]), units s_uf[c] .. s_ul[c],
    // pieces from s_cb[c]
    __shared__ long long s_clo[kPlanMaxGrid + 1];
    __shared__ int32_t s_uf[kPlanMaxGrid];
    __shared__ int32_t s_ul[kPlanMaxGrid];
    __shared__ int32_t s_cb[kPlanMaxGrid + 1];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int ns = a.num_seqs;

    // ---- validation (as validate_problem) and the few-long-prefill-items rule
    long long err = 0, items = 0, max_steps = 0;
    if (tid == 0 && ns > 0 && (a.cu[0] != 0 || a.cu[ns] > a.max_total_q)) err = 1;
    for (int s = tid; s < ns; s += nt) {
        const long long lq = (long long)a.cu[s + 1] - a.cu[s];
        const long long lk = a.lk[s];
        if (lq < 0 || lq > a.max_seq_q || lk < 0 || (lq > 0 && lk == 0) || (a.causal && lk < lq) ||
            (lk + kBlockSize - 1) / kBlockSize > a.bt_stride || lq * a.g > INT32_MAX / 2) {
            err = 1;
            continue;
        }
        const long long rows = lq * a.g;
        if (a.prefill_ok && rows > kDecRows) {
            items += (rows + kPreTileRows - 1) / kPreTileRows * a.hkv;
            max_steps = max(max_steps, (lk + 63) / 64);
        }
    }
    block_sum_max2(items, err, max_steps, s_red);
    if (err) {
        empty_plan(a, 1);
        return;
    }
    const bool pre_on =
        a.prefill_ok && !(items > 0 && items * 4 < max(a.num_sms, 1) && max_steps >= 32);
    const int step = kDecRows / a.hpu;        // rows per decode unit and kv head
    const int upt = a.hkv / a.hpu;            // decode units per row tile

    // ---- per sequence: decode units and prefill items (exclusive scans)
    for (int s = tid; s < ns; s += nt) {
        const int lq = a.cu[s + 1] - a.cu[s];
        const int rows = lq * a.g;
        const bool dec = rows <= kDecRows || !pre_on;
        a.seq_u[s] = (lq > 0 && dec) ? (rows + step - 1) / step * upt : 0;
        a.seq_i[s] = (lq > 0 && !dec) ? (rows + kPreTileRows - 1) / kPreTileRows * a.hkv : 0;
    }
    if (tid == 0) {
        a.seq_u[ns] = 0;
        a.seq_i[ns] = 0;
    }
    __syncthreads();
    const int2 tot = block_scan2(a.seq_u, a.seq_i, ns + 1, s_part32);
    const int n_units = tot.x, n_items = tot.y;
    if (n_units > a.cap_units || n_items > a.cap_items) {
        empty_plan(a, 2);
        return;
    }
    {
        const size_t nb = (size_t)a.n_buckets, nu = (size_t)n_units, ni = (size_t)n_items;
        const size_t need = 16 * 8 + sizeof(UnitRec) * nu + 8 * (nu + 1) + sizeof(PreTile) * ni + 4 * ni +
                            4 * nb + 8 * (max(nu, (size_t)a.dec_grid) + 1);
        if (sm_used + need <= a.smem_bytes) {
            a.urec = reinterpret_cast<UnitRec *>(carve(sizeof(UnitRec) * nu));
            sm_used = (sm_used + 7) & ~size_t(7);
            a.ustart = reinterpret_cast<long long *>(carve(8 * (nu + 1)));
            a.irec = reinterpret_cast<PreTile *>(carve(sizeof(PreTile) * ni));
            a.ikey = reinterpret_cast<int32_t *>(carve(4 * ni));
            a.hist = reinterpret_cast<int32_t *>(carve(4 * nb));
            a.tmp = reinterpret_cast<int32_t *>(carve(4 * (max(nu, (size_t)a.dec_grid) + 1)));
            a.tmp2 = reinterpret_cast<int32_t *>(carve(4 * (max(nu, (size_t)a.dec_grid) + 1)));
        }
    }

    // ---- units (order: sequence, row tile, kv head) and their page counts
    for (int u = tid; u < n_units; u += nt) {
        const int s = last_le(a.seq_u, ns + 1, u);
        const int local = u - a.seq_u[s];
        const int lq = a.cu[s + 1] - a.cu[s], lk = a.lk[s];
        const int rows = lq * a.g;
        const int r0 = (local / upt) * step;
        const int nr = min(step, rows - r0);
        const int kend = a.causal ? min(lk, lk - lq + (r0 + nr - 1) / a.g + 1) : lk;
        UnitRec r;
        r.seq = s;
        r.kvh = (local % upt) * a.hpu;
        r.row0 = r0;
        r.nrows = nr;
        r.pages = (kend + kBlockSize - 1) / kBlockSize;
        r.npieces = 0;
        r.comb = -1;
        r.slot0 = -1;
        a.urec[u] = r;
        a.ustart[u] = r.pages;
    }
    // ---- prefill items (order: sequence, row tile, kv head) and their sort keys
    for (int i = tid; i < n_items; i += nt) {
        const int s = last_le(a.seq_i, ns + 1, i);
        const int local = i - a.seq_i[s];
        const int lq = a.cu[s + 1] - a.cu[s], lk = a.lk[s];
        const int rows = lq * a.g;
        PreTile t;
        t.seq = s;
        t.kvh = local % a.hkv;
        t.row0 = (local / a.hkv) * kPreTileRows;
        t.nrows = min(kPreTileRows, rows - t.row0);
        const int kend = a.causal ? min(lk, lk - lq + (t.row0 + t.nrows - 1) / a.g + 1) : lk;
        t.kv_tiles = (kend + kKvTile - 1) / kKvTile;
        t.q0 = a.cu[s];
        t.lq = lq;
        t.lk = lk;
        a.irec[i] = t;
        a.ikey[i] = t.kv_tiles;
    }
    if (tid == 0) a.ustart[n_units] = 0;
    __syncthreads();
    const long long total_pages = block_scan(a.ustart, n_units + 1, s_part64);

    // ---- decode: equal shares of cost (kDecUnitCost + pages per unit), one per CTA
    int dec_ctas = 0, n_pieces = 0, n_comb = 0, n_slots = 0;
    if (total_pages > 0) {
        const long long P = total_pages;
        dec_ctas = (int)min((long long)a.dec_grid, P);
        const int C = dec_ctas;
        const long long T = P + kDecUnitCost * (long long)n_units;
        // the CTAs' page ranges (the only 64-bit divisions): cost T c / C mapped to
        // a page (the first page of the unit whose fixed part holds it, or the page
        // it falls on), then first and last units and pieces per CTA
        for (int c = tid; c <= C; c += nt) {
            if (c == C) {
                s_clo[c] = P;
                continue;
            }
            const long long x = T * c / C;
            int lo = 0, hi = n_units;    // the last unit u with ustart[u] + K u <= x
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (a.ustart[mid] + kDecUnitCost * (long long)mid <= x) lo = mid;
                else hi = mid;
            }
            const long long off = x - a.ustart[lo] - kDecUnitCost * (long long)lo - kDecUnitCost;
            const long long pages = a.ustart[lo + 1] - a.ustart[lo];
            s_clo[c] = a.ustart[lo] + min(max(off, 0LL), pages);
        }
        __syncthreads();
        for (int c = tid; c < C; c += nt) {
            if (s_clo[c + 1] == s_clo[c]) {      // an empty share (at a unit boundary)
                s_uf[c] = 0;
                s_ul[c] = -1;
                s_cb[c] = 0;
                continue;
            }
            const int uf = last_le(a.ustart, n_units, s_clo[c]);
            const int ul = last_le(a.ustart, n_units, s_clo[c + 1] - 1);
            s_uf[c] = uf;
            s_ul[c] = ul;
            s_cb[c] = ul - uf + 1;
        }
        if (tid == 0) s_cb[C] = 0;
        __syncthreads();
        n_pieces = block_scan(s_cb, C + 1, s_part32);
        for (int c = tid; c <= a.dec_grid; c += nt) a.cta_begin[c] = c <= C ? s_cb[c] : n_pieces;
        if (n_pieces > a.cap_pieces) {
            empty_plan(a, 2);
            return;
        }
        // pieces per unit: the CTAs its pages fall in; split units get a combine
        // entry and consecutive partial slots, in unit order
        for (int u = tid; u < n_units; u += nt) {
            const int cf = last_le(s_clo, C, a.ustart[u]);            // CTA holding its first page
            const int cl = last_le(s_clo, C, a.ustart[u + 1] - 1);    // and its last
            const int np = cl - cf + 1;
            a.urec[u].npieces = np;
            a.urec[u].comb = np > 1 ? 1 : 0;
            a.urec[u].slot0 = np > 1 ? np : 0;
        }
        __syncthreads();
        // one pass of scans over the split flags and the split units' piece
        // counts (urec's fields are strided: copy them to two arrays)
        for (int u = tid; u < n_units; u += nt) {
            a.tmp[u] = a.urec[u].comb;
            a.tmp2[u] = a.urec[u].slot0;
        }
        if (tid == 0) {
            a.tmp[n_units] = 0;
            a.tmp2[n_units] = 0;
        }
        __syncthreads();
        const int2 cs = block_scan2(a.tmp, a.tmp2, n_units + 1, s_part32);
        n_comb = cs.x;
        n_slots = cs.y;
        for (int u = tid; u < n_units; u += nt) {
            const bool split = a.urec[u].npieces > 1;
            a.urec[u].comb = split ? a.tmp[u] : -1;
            a.urec[u].slot0 = split ? a.tmp2[u] : -1;
        }
        __syncthreads();
        if (n_comb > a.cap_comb || n_slots > a.cap_slots) {
            empty_plan(a, 2);
            return;
        }
        // the pieces, at their place in their CTA's list (a CTA whose last piece
        // belongs to a split unit runs that piece first)
        for (int u = tid; u < n_units; u += nt) {
            const UnitRec r = a.urec[u];
            const long long st = a.ustart[u], en = a.ustart[u + 1];
            const int cf = last_le(s_clo, C, st);
            for (int k = 0; k < r.npieces; ++k) {
                const int c = cf + k;
                const long long lo = s_clo[c], hi = s_clo[c + 1];
                const int n = s_cb[c + 1] - s_cb[c];
                int pos = u - s_uf[c];
                if (n > 1 && a.urec[s_ul[c]].npieces > 1) pos = pos + 1 == n ? 0 : pos + 1;
                DecPiece pc;
                pc.seq = r.seq;
                pc.kvh = r.kvh;
                pc.row0 = r.row0;
                pc.nrows = r.nrows;
                pc.page_begin = (int32_t)(max(lo, st) - st);
                pc.page_end = (int32_t)(min(hi, en) - st);
                pc.slot = r.npieces > 1 ? r.slot0 + k : -1;
                pc.unit = r.comb;
                a.pieces[s_cb[c] + pos] = pc;
            }
            if (r.npieces > 1) {
                CombUnit cu;
                cu.seq = r.seq;
                cu.kvh = r.kvh;
                cu.row0 = r.row0;
                cu.nrows = r.nrows;
                cu.slot_begin = r.slot0;
                cu.nslots = r.npieces;
                cu.pad0 = 0;
                cu.pad1 = 0;
                a.comb[r.comb] = cu;
                a.comb_count[r.comb] = 0;
            }
        }
    } else {
        for (int c = tid; c <= a.dec_grid; c += nt) a.cta_begin[c] = 0;
    }

    // ---- prefill: longest first (stable), dealt in rounds of alternating direction
    int pre_ctas = 0;
    if (n_items > 0) {
        long long mk = 0;
        for (int i = tid; i < n_items; i += nt) mk = max(mk, (long long)a.ikey[i]);
        const int max_kv = (int)block_max(mk, s_red);
        if (max_kv + 2 > a.n_buckets) {
            empty_plan(a, 2);
            return;
        }
        // bucket b = max_kv - key (longest first); cursor = items in earlier buckets
        for (int b = tid; b <= max_kv + 1; b += nt) a.hist[b] = 0;
        __syncthreads();
        for (int i = tid; i < n_items; i += nt) atomicAdd(a.hist + (max_kv - a.ikey[i]), 1);
        __syncthreads();
        block_scan(a.hist, max_kv + 2, s_part32);
        // ranks, in batch order within a bucket: chunks of nt items; in a chunk,
        // the warps take their turn, each group of equal keys in a warp reading
        // and advancing its bucket's cursor once
        const int C = min(n_items, a.pre_workers);
        pre_ctas = C;
        const int R = n_items / C, rem = n_items % C;
        for (int c = tid; c <= a.num_sms; c += nt) {
            const int cc = min(c, C);
            const int extra = (R & 1) ? max(0, cc - (C - rem)) : min(cc, rem);
            a.pre_begin[c] = R * cc + extra;
        }
        for (int base = 0; base < n_items; base += nt) {
            const int i = base + tid;
            const bool valid = i < n_items;
            const int key = valid ? a.ikey[i] : -1;
            const unsigned same = __match_any_sync(0xffffffffu, key);
            const int leader = __ffs(same) - 1;
            const int before = __popc(same & ((1u << lane) - 1u));
            int rank = 0;
            for (int w = 0; w < (nt >> 5); ++w) {
                if (warp == w) {
                    int b0 = 0;
                    if (valid && lane == leader) {
                        int *cur = a.hist + (max_kv - key);
                        b0 = *cur;
                        *cur = b0 + __popc(same);
                    }
                    rank = __shfl_sync(0xffffffffu, b0, leader) + before;
                }
                __syncthreads();
            }
            if (valid) {
                const int round = rank / C, k = rank % C;
                const int owner = (round & 1) ? C - 1 - k : k;
                a.tiles[a.pre_begin[owner] + round] = a.irec[i];
            }
        }
    } else {
        for (int c = tid; c <= a.num_sms; c += nt) a.pre_begin[c] = 0;
    }

    if (tid == 0) {
        a.header[0] = dec_ctas;
        a.header[1] = n_pieces;
        a.header[2] = n_comb;
        a.header[3] = n_slots;
        a.header[4] = pre_ctas;
        a.header[5] = n_items;
        a.header[6] = total_pages;
        a.header[7] = 0;
    }
}

}  // namespace

DevPlanLayout device_plan_layout(const DevPlanShape &s) {
    DevPlanLayout L{};
    const int g = s.hq / s.hkv;
    const int hpu = s.hpu;
    const int64_t rows = (int64_t)s.max_total_q * g;
    const int64_t step = kDecRows / hpu;
    // units of a sequence: ceil(rows_s / step) row tiles, so at most
    // rows_s / step + 1 of them; the sum over sequences is bounded by the totals
    L.dec_grid = kDecCtasPerSm * std::max(s.num_sms, 1);
    const int64_t units = (int64_t)(s.hkv / hpu) * ((int64_t)s.num_seqs + (rows + step - 1) / step);
    const int64_t items =
        s.prefill_ok ? (int64_t)s.hkv * ((int64_t)s.num_seqs + (rows + kPreTileRows - 1) / kPreTileRows) : 0;
    // keys of a sequence <= bt_stride * kBlockSize, so kv_tiles <= that / kKvTile rounded up
    const int64_t buckets = ((int64_t)s.bt_stride * kBlockSize + kKvTile - 1) / kKvTile + 2;
    // the planner counts in 32-bit integers
    L.valid = units + L.dec_grid < INT32_MAX / 4 && items < INT32_MAX / 4 &&
              buckets < INT32_MAX / 4 && L.dec_grid <= kPlanMaxGrid;
    if (!L.valid) return L;
    L.cap_units = (int32_t)units;
    L.cap_items = (int32_t)items;
    // every CTA boundary cuts at most one unit: at most dec_grid - 1 extra pieces,
    // dec_grid - 1 split units and 2 (dec_grid - 1) pieces of split units
    L.cap_pieces = L.cap_units + L.dec_grid;
    L.cap_comb = std::min(L.cap_units, L.dec_grid);
    L.cap_slots = 2 * L.dec_grid;
    L.n_buckets = (int32_t)buckets;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, kAlign);
        return at;
    };
    L.off_header = take(8 * sizeof(long long));
    L.off_cta = take(sizeof(int32_t) * ((size_t)L.dec_grid + 1));
    L.off_pieces = take(sizeof(DecPiece) * (size_t)L.cap_pieces);
    L.off_comb = take(sizeof(CombUnit) * (size_t)L.cap_comb);
    L.off_comb_count = take(sizeof(int32_t) * (size_t)L.cap_comb);
    L.off_tiles = take(sizeof(PreTile) * (size_t)L.cap_items);
    L.off_pre_begin = take(sizeof(int32_t) * ((size_t)s.num_sms + 1));
    L.off_part_o = take(sizeof(float) * (size_t)L.cap_slots * kDecRows * kernel_head_size(s.d));
    L.off_part_ml = take(2 * sizeof(float) * (size_t)L.cap_slots * kDecRows);
    L.off_scratch = off;
    take(sizeof(int32_t) * ((size_t)s.num_seqs + 1));                  // seq_u
    take(sizeof(int32_t) * ((size_t)s.num_seqs + 1));                  // seq_i
    take(sizeof(UnitRec) * (size_t)L.cap_units);                        // urec
    take(sizeof(long long) * ((size_t)L.cap_units + 1));               // ustart
    take(sizeof(PreTile) * (size_t)L.cap_items);                        // irec
    take(sizeof(int32_t) * (size_t)L.cap_items);                        // ikey
    take(sizeof(int32_t) * (size_t)L.n_buckets);                        // hist
    take(sizeof(int32_t) * ((size_t)std::max(L.cap_units, L.dec_grid) + 1));   // tmp
    take(sizeof(int32_t) * ((size_t)std::max(L.cap_units, L.dec_grid) + 1));   // tmp2
    L.total_bytes = off;
    return L;
}

cudaError_t launch_device_plan(const DevPlanShape &s, const DevPlanLayout &L, const int32_t *cu,
                               const int32_t *seqused_k, int32_t causal, void *workspace,
                               int *status, cudaStream_t stream) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    PlanArgs a{};
    a.cu = cu;
    a.lk = seqused_k;
    a.num_seqs = s.num_seqs;
    a.max_total_q = s.max_total_q;
    a.max_seq_q = s.max_seq_q;
    a.hq = s.hq;
    a.hkv = s.hkv;
    a.g = s.hq / s.hkv;
    a.bt_stride = s.bt_stride;
    a.hpu = s.hpu;
    a.prefill_ok = s.prefill_ok;
    a.num_sms = s.num_sms;
    a.pre_workers = s.pre_workers;
    a.causal = causal != 0;
    a.dec_grid = L.dec_grid;
    a.cap_units = L.cap_units;
    a.cap_items = L.cap_items;
    a.cap_pieces = L.cap_pieces;
    a.cap_comb = L.cap_comb;
    a.cap_slots = L.cap_slots;
    a.n_buckets = L.n_buckets;
    a.header = reinterpret_cast<long long *>(ws + L.off_header);
    a.cta_begin = reinterpret_cast<int32_t *>(ws + L.off_cta);
    a.pieces = reinterpret_cast<DecPiece *>(ws + L.off_pieces);
    a.comb = reinterpret_cast<CombUnit *>(ws + L.off_comb);
    a.comb_count = reinterpret_cast<int32_t *>(ws + L.off_comb_count);
    a.tiles = reinterpret_cast<PreTile *>(ws + L.off_tiles);
    a.pre_begin = reinterpret_cast<int32_t *>(ws + L.off_pre_begin);
    size_t off = L.off_scratch;
    auto take = [&](size_t bytes) {
        uint8_t *p = ws + off;
        off = align_up(off + bytes, kAlign);
        return p;
    };
    a.seq_u = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * ((size_t)s.num_seqs + 1)));
    a.seq_i = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * ((size_t)s.num_seqs + 1)));
    a.urec = reinterpret_cast<UnitRec *>(take(sizeof(UnitRec) * (size_t)L.cap_units));
    a.ustart = reinterpret_cast<long long *>(take(sizeof(long long) * ((size_t)L.cap_units + 1)));
    a.irec = reinterpret_cast<PreTile *>(take(sizeof(PreTile) * (size_t)L.cap_items));
    a.ikey = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * (size_t)L.cap_items));
    a.hist = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * (size_t)L.n_buckets));
    a.tmp = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * ((size_t)std::max(L.cap_units, L.dec_grid) + 1)));
    a.tmp2 = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * ((size_t)std::max(L.cap_units, L.dec_grid) + 1)));
    a.status = status;
    a.smem_bytes = (uint32_t)kPlanSmemMax;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        const cudaError_t e = cudaFuncSetAttribute(ua_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)kPlanSmemMax);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    ua_plan_kernel<<<1, kPlanThreads, kPlanSmemMax, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ua
