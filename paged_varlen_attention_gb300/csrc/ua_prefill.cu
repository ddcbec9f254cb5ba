// ua_prefill.cu -- tensor-core prefill / chunked-prefill kernel (tcgen05 + TMEM + TMA).
//
// Query runs longer than one 16-row tile go here.  The query heads that share
// a KV head are stacked along M, so one 128-row MMA tile holds 128/G tokens x
// G heads and every K/V tile loaded from the paged cache feeds all of them
// (the GQA packing of "[Kernel] Unified Triton kernel that doesn't
// distinguish between prefill + decode", vLLM PR #16828, PR description,
// where it serves to keep the tensor cores busy).
//
// One persistent CTA per SM walks its work items, longest first: the items
// dealt to it in advance, or (kClaimed: long items) items it claims from the
// plan's longest-first list one at a time (an atomic counter), so that an SM
// that runs faster takes more of them.  A work item is a pair of 128-row MMA
// tiles, A and B, of the same (sequence, KV head); both use every K/V step
// the CTA loads.  A step is 64 keys (4 pages).
//
// TMEM (512 columns) holds, per tile X: two S buffers of 64 fp32 columns
// (steps alternate between them; P is written as bf16 pairs over the first 32
// columns of its S) and O (D fp32 columns).  With two S buffers the scores of
// step j+1 are computed while the softmax of step j runs and while P V of
// step j-1 is still reading its P, so each tile keeps up to three MMA groups
// (S, S, P V) in flight and the tensor core overlaps them across A and B: a
// chain of MMAs into one accumulator is latency-bound, independent chains are
// not.
//
// Roles (12 warps):
//   warps 0-3   softmax of tile A, one thread per row (TMEM lane): scale into
//               the log2 domain, bottom-right causal mask, row max, exp2, row
//               sum, P as bf16 into TMEM.  O is rescaled only when a row max
//               grows by more than 2^8 (the stale max cancels in O / l).  The
//               epilogue divides by l and writes bf16 rows of out.
//   warps 4-7   the same for tile B
//   warp 8      allocates TMEM; issues tile A's MMAs (whole warp, one elected
//               lane):  S_A = Q_A K_j^T  (M 128, N 64, K D; K-major operands)
//                       O_A += P_A V_j   (A = P in TMEM, B = V MN-major)
//               in the order S(0), S(1), then P V(j) and S(j+2) as each buffer
//               frees up.
//   warp 11     the same for tile B
//   warp 9      (kClaimed) claims the CTA's items: lane 0 takes the next
//               index with an atomic add and puts the item's record into a
//               4-slot ring in shared memory that every role reads in order;
//               and TMA producer of the Q tiles (box {64, G, 128/G} of [T, Hq, D])
//               and of V (one box per 16-token page: a 5-D view of the cache,
//               so one box holds all D columns of the page).  The step that
//               holds a sequence's last, partial page lands on a barrier of its
//               own: this warp zeroes the rows past the context (they may hold
//               anything, NaN included, and 0 x NaN is NaN in P V) before it
//               releases the step.
//   warp 10     TMA producer of K: per page one {64, 1, 16} box per 64 columns
//               of [pages*16, Hkv, D], into [chunk][key][64] so that each
//               64-wide column chunk of the step is one K-major operand.
// Pages past a step's last visible key are read out of bounds (zero fill)
// instead of from the block table.  Every wait is bounded (see
// ua_device.cuh); TMEM is always freed.
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {

constexpr int kStep = 64;                            // keys per KV step
constexpr int kStepPages = kStep / kBlockSize;       // 4 pages

template <int D>
struct PreCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kQBytes = kPreRows * D * 2;          // one 128-row Q tile
    static constexpr int kKvBytes = kStep * D * 2;            // one step of K (or V)
    static constexpr int kKChunkBytes = kStep * 128;          // K: 64 keys x 64 columns
    static constexpr int kPageBytes = kBlockSize * D * 2;     // V: one 16-token page
    static constexpr int kThreads = 384;                      // 12 warps: 3 per SMSP, 168 regs
    static constexpr int kKStages = 3;
    static constexpr int kVStages = 3;
    static constexpr int kTmemCols = 512;
    static constexpr uint32_t kColO = 128;                    // + 256 * tile; S buffers at 0, 64
    // output staging per tile: D/64 buffers of 128 rows x 64 columns of bf16
    // (one TMA store box each), so the passes of an epilogue never wait for
    // each other's stores
    static constexpr int kStageBytes = kPreRows * 128 * kChunks;
    // Q x2 (A, B), K x4, V x4, staging x2, barriers; one CTA owns the SM (and its TMEM)
    static constexpr size_t kUsed = 1024 + 2 * (size_t)kQBytes +
                                    (size_t)(kKStages + kVStages) * kKvBytes + 2 * kStageBytes + 512;
    static constexpr size_t kSmemBytes = kUsed < 120 * 1024 ? 120 * 1024 : kUsed;
    static constexpr float kRescaleThreshold = 8.0f;          // log2 units
};

// mbarrier slots.  [2]: one per tile X; [4] of S / P / P V: index 2 * X + b,
// b the S buffer.
enum : int {
    kBarQFull = 0,      // [2]
    kBarQEmpty = 2,     // [2]
    kBarKFull = 4,      // [4] K stages
    kBarKEmpty = 8,     // [4] 2 arrivals: both MMA warps
    kBarVFull = 12,     // [4] V stages
    kBarVEmpty = 16,    // [4] 2 arrivals: both MMA warps
    kBarVTail = 20,     // TMA of a step that holds a sequence's partial last page
    kBarSFull = 21,     // [4]
    kBarPFull = 25,     // [4] 128 arrivals
    kBarPvDone = 29,    // [4]
    kBarDrain = 33,     // [2]
    kBarItemFull = 35,  // [kItemRing] (kClaimed) an item record is in the ring slot
    kBarItemEmpty = 39, // [kItemRing] (kClaimed) kItemReaders arrivals: every reader has taken it
    kNumBars = 43
};

struct SubInfo {
    int row0, nrows, n;      // packed rows of this 128-row tile; its KV steps
    int kend_max, kend_lo;   // keys visible to its last / first row
};

struct PairInfo {
    int seq, q0, lq, lk, kvh, n;   // n: KV steps of the pair (= max over tiles)
    SubInfo sub[2];
};

__device__ __forceinline__ int visible_keys(const PrefillParams &p, int lq, int lk, int row) {
    if (!p.causal) return lk;
    return min(lk, lk - lq + row / p.g + 1);
}

// The work item's geometry from its plan record (sequence offsets and lengths
// are in the record, so no dependent loads of the metadata arrays).
__device__ __forceinline__ PairInfo make_pair(const PrefillParams &p, const PreTile &pt) {
    PairInfo pi;
    pi.seq = pt.seq;
    pi.q0 = pt.q0;
    pi.lq = pt.lq;
    pi.lk = pt.lk;
    pi.kvh = pt.kvh;
    pi.n = 0;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        SubInfo &s = pi.sub[x];
        s.row0 = pt.row0 + x * kPreRows;
        s.nrows = max(0, min(kPreRows, pt.nrows - x * kPreRows));
        if (s.nrows > 0) {
            s.kend_max = visible_keys(p, pi.lq, pi.lk, s.row0 + s.nrows - 1);
            s.kend_lo = visible_keys(p, pi.lq, pi.lk, s.row0);
            s.n = (s.kend_max + kStep - 1) / kStep;
        } else {
            s.kend_max = s.kend_lo = 0;
            s.n = 0;
        }
        pi.n = max(pi.n, s.n);
    }
    return pi;
}

// Walks this CTA's work items (its range of the plan).  Records are loaded two
// items ahead: take() hands out the record loaded one item earlier and starts
// the load of the one after next, so no role waits on a record's load at an
// item boundary (only the first two loads are waited for).
struct ItemCursor {
    int t, end;
    PreTile cur, nxt;
    __device__ __forceinline__ ItemCursor(const PrefillParams &p)
        : t(p.tile_begin[blockIdx.x]), end(p.tile_begin[blockIdx.x + 1]) {
        if (t < end) cur = p.tiles[t];
        if (t + 1 < end) nxt = p.tiles[t + 1];
    }
    __device__ __forceinline__ bool valid(const PrefillParams &) const { return t < end; }
    __device__ __forceinline__ PreTile take(const PrefillParams &p) {
        const PreTile out = cur;
        cur = nxt;
        if (t + 2 < end) nxt = p.tiles[t + 2];
        ++t;
        return out;
    }
};

// Claimed items pass through a ring of kItemRing records in shared memory:
// slot k % kItemRing holds the CTA's k-th item (or an end marker, seq = -1)
// once ItemFull completes its phase k / kItemRing; the kItemReaders reader
// warps (10; 8 and 11; 0-7) arrive on ItemEmpty after reading it, which lets
// warp 9 refill the slot.
constexpr int kItemRing = 4;
constexpr int kItemReaders = 11;

// A role's walk over this CTA's items: dealt ones through ItemCursor, claimed
// ones from the ring (reader warps release each slot).  take() returns 1 with
// an item, 0 at the end, -1 when a wait gave up.
template <bool kClaimed>
struct ItemIter;

// A record made warp-uniform: every field from lane 0 (the compiler then sees
// values derived from it, such as MMA operands and loop bounds, as uniform).
__device__ __forceinline__ PreTile uniform_tile(const PreTile &t) {
    PreTile u;
    u.seq = __shfl_sync(0xffffffffu, t.seq, 0);
    u.kvh = __shfl_sync(0xffffffffu, t.kvh, 0);
    u.row0 = __shfl_sync(0xffffffffu, t.row0, 0);
    u.nrows = __shfl_sync(0xffffffffu, t.nrows, 0);
    u.kv_tiles = __shfl_sync(0xffffffffu, t.kv_tiles, 0);
    u.q0 = __shfl_sync(0xffffffffu, t.q0, 0);
    u.lq = __shfl_sync(0xffffffffu, t.lq, 0);
    u.lk = __shfl_sync(0xffffffffu, t.lk, 0);
    return u;
}

template <>
struct ItemIter<false> {
    ItemCursor it;
    __device__ __forceinline__ ItemIter(const PrefillParams &p, const PreTile *, uint32_t, uint32_t)
        : it(p) {}
    __device__ __forceinline__ int take(const PrefillParams &p, uint32_t, bool, int, PreTile &out) {
        if (!it.valid(p)) return 0;
        out = uniform_tile(it.take(p));
        return 1;
    }
};

template <>
struct ItemIter<true> {
    const PreTile *ring;
    uint32_t full0, empty0;
    __device__ __forceinline__ ItemIter(const PrefillParams &, const PreTile *r, uint32_t f, uint32_t e)
        : ring(r), full0(f), empty0(e) {}
    __device__ __forceinline__ int take(const PrefillParams &p, uint32_t k, bool release, int lane,
                                        PreTile &out) {
        const uint32_t slot = k % kItemRing;
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * slot, (k / kItemRing) & 1, p.status))) return -1;
        out = uniform_tile(ring[slot]);
        __syncwarp();
        if (release && lane == 0) mbar_arrive(empty0 + 8 * slot);
        return out.seq < 0 ? 0 : 1;
    }
};

// Block ids of the 4 pages of KV step j (lanes 0-3 load; out-of-range or
// not-needed pages give num_blocks, which TMA reads as zeros).
__device__ __forceinline__ int step_block_id(const PrefillParams &p, const int32_t *bt_row, int j,
                                             int kend, int lane) {
    int bid = p.num_blocks;
    const int page = j * kStepPages + lane;
    if (lane < kStepPages && page * kBlockSize < kend) {
        bid = __ldg(bt_row + page);
        if (bid < 0 || bid >= p.num_blocks) {
            record_status(p.status, UA_DEVICE_BAD_BLOCK_ID_BIT);
            bid = p.num_blocks;
        }
    }
    return bid;
}

// tcgen05.mma / commit issued by one elected lane of a converged warp.
__device__ __forceinline__ void umma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// Rows [0, nrows) of a staged 64-column slice of O (layout of a Q tile: row r
// at r * 128 bytes, 16-byte pieces XOR-ed with r % 8) to out, by the tile's
// 128 threads.  Used for a tile that ends before 128 rows; kept out of line.
template <int D>
__device__ __noinline__ void copy_partial_rows(__nv_bfloat16 *out, const uint8_t *stg, int tid, int nrows,
                                               int row0, int q0, int kvh, int g, int hq, int col0) {
    for (int u = tid; u < nrows * 8; u += 128) {
        const int row = u >> 3, piece = u & 7;
        const uint4 val = *reinterpret_cast<const uint4 *>(stg + row * 128 + ((piece ^ (row & 7)) << 4));
        const int prr = row0 + row;
        *reinterpret_cast<uint4 *>(out + ((int64_t)(q0 + prr / g) * hq + kvh * g + prr % g) * D + col0 + 8 * piece) =
            val;
    }
}

template <int D, bool kPos, bool kClaimed>
__global__ void __launch_bounds__(PreCfg<D>::kThreads, 1)
    ua_prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_vp) {
    using C = PreCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sq = smem_u32(smem);                         // Q[2]: A, B
    const uint32_t sk = sq + 2 * C::kQBytes;                    // K[4]: [chunk][64 keys][64]
    const uint32_t sv = sk + C::kKStages * C::kKvBytes;         // V[4]: [page][chunk][16][64]
    uint8_t *sv_ptr = smem + 2 * C::kQBytes + C::kKStages * C::kKvBytes;
    uint8_t *stage_ptr = sv_ptr + C::kVStages * C::kKvBytes;     // [tile][128 rows][64] bf16, 128B swizzle
    const uint32_t sstage = smem_u32(stage_ptr);
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage_ptr + 2 * C::kStageBytes);
    PreTile *ring = reinterpret_cast<PreTile *>(bars + ((kNumBars + 1) & ~1));   // 16-byte aligned
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ring + kItemRing);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

    // the warp index and TMEM base broadcast from lane 0, so that the compiler
    // sees them as warp-uniform (MMA operands built from them need no per-lane loop)
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    // a CTA with no item (a fixed grid whose plan, built on the device, has
    // fewer items than CTAs) leaves before touching barriers or TMEM (the same
    // answer for every thread)
    int n_items = 0;
    if constexpr (kClaimed) {
        n_items = p.sched[kSchedItems];
        if (n_items == 0) return;
    } else {
        if (p.tile_begin[blockIdx.x] == p.tile_begin[blockIdx.x + 1]) return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarQFull + i), 1);
            mbar_init(bar(kBarQEmpty + i), 1);
            mbar_init(bar(kBarDrain + i), 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(kBarKFull + i), 1);
            mbar_init(bar(kBarKEmpty + i), 2);
            mbar_init(bar(kBarVFull + i), 1);
            mbar_init(bar(kBarVEmpty + i), 2);
            mbar_init(bar(kBarSFull + i), 1);
            mbar_init(bar(kBarPFull + i), 128);
            mbar_init(bar(kBarPvDone + i), 1);
        }
        mbar_init(bar(kBarVTail), 1);
        if constexpr (kClaimed)
            for (int i = 0; i < kItemRing; ++i) {
                mbar_init(bar(kBarItemFull + i), 1);
                mbar_init(bar(kBarItemEmpty + i), kItemReaders);
            }
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
    if (warp == 9) {
        // ================================================================ Q + V producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_vp);
        }
        const uint64_t pol_kv = l2_policy_evict_last();   // K/V steps are re-read by sibling items
        bool ok = true;
        uint32_t e = 0, v_issued = 0, tails = 0;
        uint32_t q_issued[2] = {0, 0};
        // (kClaimed) lane 0 claims items and publishes them in the ring.
        // claim: the next index of the longest-first list (atomic add) and a
        // load of its record, not waited for here; publish: once every reader
        // has taken the slot's previous item, the record (or the end marker)
        // goes into slot f % kItemRing; it returns 1 for an item, 0 for the end
        // marker, -1 when the wait gave up.  Item k + 1 is claimed when item k
        // starts and published once item k's loads are all issued (the claim's
        // latency hides behind item k, and a CTA holds at most one unstarted
        // item); with at most two items per CTA it is claimed only then, as
        // claiming ahead would let the CTAs that start first take the items of
        // those that start later.
        uint32_t fetched = 0;
        int more = 1;
        int next_idx = 0;
        PreTile next_rec{};
        auto claim = [&]() {
            next_idx = atomicAdd(p.sched + kSchedNext, 1);
            next_rec = p.tiles[min(next_idx, n_items - 1)];
        };
        auto publish = [&]() -> int {
            const uint32_t f = fetched, slot = f % kItemRing;
            if (f >= (uint32_t)kItemRing &&
                !mbar_wait(bar(kBarItemEmpty + slot), ((f / kItemRing) - 1) & 1, p.status))
                return -1;
            PreTile t = next_rec;
            if (next_idx >= n_items) t.seq = -1;
            ring[slot] = t;
            mbar_arrive(bar(kBarItemFull + slot));   // release: the record is visible
            ++fetched;
            return next_idx < n_items ? 1 : 0;
        };
        const bool ahead = n_items > 2 * (int)gridDim.x;
        if constexpr (kClaimed) {
            if (lane == 0) {
                claim();
                more = publish();
            }
        }
        ItemIter<kClaimed> items(p, ring, bar(kBarItemFull), bar(kBarItemEmpty));
        for (uint32_t k = 0; ok; ++k) {
            if constexpr (kClaimed) {
                if (lane == 0 && more == 1 && ahead) claim();
                if (__shfl_sync(0xffffffffu, more, 0) < 0) {
                    ok = false;
                    break;
                }
            }
            PreTile cur;
            const int got = items.take(p, k, false, lane, cur);
            if (got < 0) ok = false;
            if (got <= 0) break;
            const PairInfo pi = make_pair(p, cur);
            int good = 1;
            if (lane == 0) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    if (!good || pi.sub[x].nrows == 0) continue;
                    // Q buffer x is free once the last S of its previous tile is done
                    if (q_issued[x] > 0 &&
                        !mbar_wait(bar(kBarQEmpty + x), (q_issued[x] - 1) & 1, p.status)) {
                        good = 0;
                        continue;
                    }
                    mbar_arrive_expect_tx(bar(kBarQFull + x), C::kQBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sq + x * C::kQBytes + c * (kPreRows * 128), &tm_q, c * 64,
                                    pi.kvh * p.g, pi.q0 + pi.sub[x].row0 / p.g, bar(kBarQFull + x));
                    ++q_issued[x];
                }
            }
            ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            const int kend = max(pi.sub[0].kend_max, pi.sub[1].kend_max);
            const int32_t *bt_row = p.block_table + (int64_t)pi.seq * p.bt_stride;
            // the step holding the sequence's partial last page, if a row sees it
            const int last_page_start = (pi.lk - 1) & ~(kBlockSize - 1);
            const int tail_step = ((pi.lk & (kBlockSize - 1)) != 0 && last_page_start < kend)
                                      ? last_page_start / kStep : -1;
            for (int j = 0; j < pi.n && ok; ++j, ++e) {
                const int bid = step_block_id(p, bt_row, j, kend, lane);
                int b[kStepPages];
#pragma unroll
                for (int i = 0; i < kStepPages; ++i) b[i] = __shfl_sync(0xffffffffu, bid, i);
                const uint32_t vs = e % C::kVStages, vph = (e / C::kVStages) & 1;
                const bool tail = (j == tail_step);
                const uint32_t land = tail ? bar(kBarVTail) : bar(kBarVFull + vs);
                good = 1;
                if (lane == 0) {
                    if (!mbar_wait(bar(kBarVEmpty + vs), vph ^ 1, p.status)) {
                        good = 0;
                    } else {
                        mbar_arrive_expect_tx(land, C::kKvBytes);
#pragma unroll
                        for (int i = 0; i < kStepPages; ++i)
                            tma_load_5d_hint(sv + vs * C::kKvBytes + i * C::kPageBytes, &tm_vp, 0, 0, 0,
                                             pi.kvh, b[i], land, pol_kv);
                        ++v_issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                if (ok && tail) {
                    // wait for this step's data, zero the key rows past the context in the
                    // last page, then release the step to the MMA warps
                    const bool landed = mbar_wait(bar(kBarVTail), tails & 1, p.status);
                    ++tails;
                    if (!__all_sync(0xffffffffu, landed)) {
                        ok = false;
                    } else {
                        const int k0 = pi.lk - j * kStep;                       // first row to clear
                        const int k1 = last_page_start + kBlockSize - j * kStep;  // end of the page
                        constexpr int per_row = C::kChunks * 8;                 // 16-byte pieces per key row
                        for (int u = lane; u < (k1 - k0) * per_row; u += 32) {
                            const int key = k0 + u / per_row;
                            const int c = (u % per_row) / 8;
                            const int piece = u % 8;
                            *reinterpret_cast<uint4 *>(sv_ptr + vs * C::kKvBytes +
                                                       (key / kBlockSize) * C::kPageBytes + c * 2048 +
                                                       (key % kBlockSize) * 128 + piece * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(kBarVFull + vs));
                    }
                }
            }
            if constexpr (kClaimed) {
                // this item's loads are all issued: publish the next item
                if (lane == 0 && more == 1) {
                    if (!ahead) claim();
                    more = publish();
                }
            }
        }
        // drain: the last loads issued must land before the CTA can exit
        if (lane == 0) {
            for (uint32_t x = (v_issued > (uint32_t)C::kVStages ? v_issued - C::kVStages : 0); x < v_issued; ++x)
                mbar_wait(bar(kBarVFull + x % C::kVStages), (x / C::kVStages) & 1, p.status);
            for (int x = 0; x < 2; ++x)
                if (q_issued[x] > 0) mbar_wait(bar(kBarQFull + x), (q_issued[x] - 1) & 1, p.status);
            if constexpr (kClaimed) {
                // this CTA claims no more; the last CTA to get here zeroes the
                // counters for the next launch that reuses the plan
                __threadfence();
                if (atomicAdd(p.sched + kSchedDone, 1) == (int)gridDim.x - 1) {
                    atomicExch(p.sched + kSchedNext, 0);
                    atomicExch(p.sched + kSchedDone, 0);
                }
            }
        }
    } else if (warp == 10) {
        // ================================================================ K producer
        if (lane == 0) prefetch_tensormap(&tm_k);
        const uint64_t pol_kv = l2_policy_evict_last();
        bool ok = true;
        uint32_t e = 0, k_issued = 0;
        ItemIter<kClaimed> items(p, ring, bar(kBarItemFull), bar(kBarItemEmpty));
        for (uint32_t k = 0; ok; ++k) {
            PreTile cur;
            const int got = items.take(p, k, true, lane, cur);
            if (got < 0) ok = false;
            if (got <= 0) break;
            const PairInfo pi = make_pair(p, cur);
            const int kend = max(pi.sub[0].kend_max, pi.sub[1].kend_max);
            const int32_t *bt_row = p.block_table + (int64_t)pi.seq * p.bt_stride;
            for (int j = 0; j < pi.n && ok; ++j, ++e) {
                const int bid = step_block_id(p, bt_row, j, kend, lane);
                int b[kStepPages];
#pragma unroll
                for (int i = 0; i < kStepPages; ++i) b[i] = __shfl_sync(0xffffffffu, bid, i);
                const uint32_t ks = e % C::kKStages, kph = (e / C::kKStages) & 1;
                int good = 1;
                if (lane == 0) {
                    if (!mbar_wait(bar(kBarKEmpty + ks), kph ^ 1, p.status)) {
                        good = 0;
                    } else {
                        mbar_arrive_expect_tx(bar(kBarKFull + ks), C::kKvBytes);
#pragma unroll
                        for (int i = 0; i < kStepPages; ++i)
#pragma unroll
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d_hint(sk + ks * C::kKvBytes + c * C::kKChunkBytes + i * 2048,
                                                 &tm_k, c * 64, pi.kvh, b[i] * kBlockSize,
                                                 bar(kBarKFull + ks), pol_kv);
                        ++k_issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            }
        }
        if (lane == 0) {
            for (uint32_t x = (k_issued > (uint32_t)C::kKStages ? k_issued - C::kKStages : 0); x < k_issued; ++x)
                mbar_wait(bar(kBarKFull + x % C::kKStages), (x / C::kKStages) & 1, p.status);
        }
    } else if (warp == 8 || warp == 11) {
        // ================================================================ MMA issuers (A: warp 8, B: warp 11)
        const int x = warp == 8 ? 0 : 1;
        constexpr uint32_t idesc_s = umma_idesc_bf16(kPreRows, kStep, 0, 0);
        constexpr uint32_t idesc_pv = umma_idesc_bf16(kPreRows, D, 0, 1);
        const uint32_t tbase = tmem + (uint32_t)x * 256;
        const uint32_t qbase = sq + (uint32_t)x * C::kQBytes;
        bool ok = true;
        bool issued_any = false;
        uint32_t e = 0, qcnt = 0;
        uint32_t scnt = 0, pcnt = 0;   // S and P V issued by this warp over all items; P V k reads S k
        // S of KV event ev into buffer scnt % 2, which is free once P V scnt-2 has read its P
        auto issue_s = [&](uint32_t ev) -> bool {
            const uint32_t b = scnt & 1;
            if (scnt >= 2 &&
                !mbar_wait(bar(kBarPvDone + 2 * x + b), ((scnt - 2) >> 1) & 1, p.status))
                return false;
            const uint32_t ks = ev % C::kKStages, kph = (ev / C::kKStages) & 1;
            if (!mbar_wait(bar(kBarKFull + ks), kph, p.status)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t qoff = (kk >> 2) * (kPreRows * 128) + (kk & 3) * 32;
                const uint32_t koff = (kk >> 2) * C::kKChunkBytes + (kk & 3) * 32;
                umma_ss_warp(tbase + b * kStep, umma_desc_sw128(qbase + qoff, 16, 1024),
                             umma_desc_sw128(sk + ks * C::kKvBytes + koff, 16, 1024), idesc_s,
                             kk > 0 ? 1u : 0u);
            }
            umma_commit_warp(bar(kBarSFull + 2 * x + b));
            umma_commit_warp(bar(kBarKEmpty + ks));
            ++scnt;
            issued_any = true;
            return true;
        };
        // O += P V for S pcnt, V of KV event ev; first: O starts from zero
        auto issue_pv = [&](uint32_t ev, bool first) -> bool {
            const uint32_t b = pcnt & 1;
            if (!mbar_wait(bar(kBarPFull + 2 * x + b), (pcnt >> 1) & 1, p.status)) return false;
            const uint32_t vs = ev % C::kVStages, vph = (ev / C::kVStages) & 1;
            if (!mbar_wait(bar(kBarVFull + vs), vph, p.status)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kStepPages; ++kk) {
                // 16 keys per MMA = one page of V: P columns b*64 + kk*8 .. +8 (bf16
                // pairs); V page kk is [chunk][16 keys][64], MN-major: 64-wide d
                // chunks 2 KB apart (LBO), 8-key groups 1 KB apart (SBO)
                const uint64_t bdesc =
                    umma_desc_sw128(sv + vs * C::kKvBytes + kk * C::kPageBytes, kBlockSize * 128, 1024);
                umma_ts_warp(tbase + C::kColO, tbase + b * kStep + kk * 8, bdesc, idesc_pv,
                             (first && kk == 0) ? 0u : 1u);
            }
            umma_commit_warp(bar(kBarPvDone + 2 * x + b));
            umma_commit_warp(bar(kBarVEmpty + vs));
            ++pcnt;
            return true;
        };
        ItemIter<kClaimed> items(p, ring, bar(kBarItemFull), bar(kBarItemEmpty));
        for (uint32_t k = 0; ok; ++k) {
            PreTile cur;
            const int got = items.take(p, k, true, lane, cur);
            if (got < 0) ok = false;
            if (got <= 0) break;
            const PairInfo pi = make_pair(p, cur);
            const int nx = x ? pi.sub[1].n : pi.sub[0].n;
            if (nx > 0) {
                if (!mbar_wait(bar(kBarQFull + x), qcnt & 1, p.status)) {
                    ok = false;
                    break;
                }
                ++qcnt;
                // S(0), S(1), then P V(t-2) and S(t) as each S buffer frees up; Q is
                // released after the last S.  (One loop, so that each issue sequence
                // exists once in the code: the kernel's speed depends on its size.)
                for (int t = 0; t < nx + 2 && ok; ++t) {
                    if (t >= 2) ok = issue_pv(e + t - 2, t == 2);
                    if (ok && t < nx) {
                        ok = issue_s(e + t);
                        if (ok && t == nx - 1) umma_commit_warp(bar(kBarQEmpty + x));
                    }
                }
            }
            // KV steps of the pair this tile does not see: release them, in order
            for (int j = nx; j < pi.n && ok; ++j) {
                const uint32_t ev = e + j;
                if (!mbar_wait(bar(kBarKFull + ev % C::kKStages), (ev / C::kKStages) & 1, p.status) ||
                    !mbar_wait(bar(kBarVFull + ev % C::kVStages), (ev / C::kVStages) & 1, p.status)) {
                    ok = false;
                    break;
                }
                mbar_arrive_warp(bar(kBarKEmpty + ev % C::kKStages));
                mbar_arrive_warp(bar(kBarVEmpty + ev % C::kVStages));
            }
            e += pi.n;
        }
        // every MMA issued has completed before TMEM is released
        if (issued_any) {
            umma_commit_warp(bar(kBarDrain + x));
            mbar_wait(bar(kBarDrain + x), 0, p.status);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ================================================================ softmax + epilogue
        const int x = warp >> 2;                        // tile A (0) or B (1)
        const int quarter = warp & 3;                   // TMEM lanes this warp may touch
        const int r = quarter * 32 + lane;              // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + (uint32_t)x * 256;
        const uint32_t o_addr = s_addr + C::kColO;
        bool ok = true;
        uint32_t ex = 0;    // steps of this tile slot over all items (S k lives in buffer k % 2)
        ItemIter<kClaimed> items(p, ring, bar(kBarItemFull), bar(kBarItemEmpty));
        for (uint32_t k = 0; ok; ++k) {
            PreTile cur;
            const int got = items.take(p, k, true, lane, cur);
            if constexpr (kClaimed) {
                // the tile's four warps wait for the item each; they give up together
                if (!named_barrier_and(1 + x, 128, got >= 0)) {
                    ok = false;
                    break;
                }
            }
            if (got <= 0) break;
            const PairInfo pi = make_pair(p, cur);
            const SubInfo si = x ? pi.sub[1] : pi.sub[0];
            if (si.nrows == 0) continue;
            const int pr = si.row0 + r;
            const bool valid = r < si.nrows;
            const int i = pr / p.g;
            const int kend = (p.causal && valid) ? min(pi.lk, pi.lk - pi.lq + i + 1) : pi.lk;
            float m_run = -INFINITY;
            float l = 0.f;
            for (int j = 0; j < si.n; ++j, ++ex) {
                const uint32_t b = ex & 1;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(bar(kBarSFull + 2 * x + b), (ex >> 1) & 1, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // The 64 scores of this row.  With a positive scale (kPos, the usual case)
                // the max is taken on the raw scores and the scale is folded into the
                // exponent's FMA; otherwise the scores are scaled first.  Keys at or
                // past the row's limit (diagonal and tail steps only) become -inf.
                uint32_t xs[kStep];
                tmem_ld64(s_addr + b * kStep, xs);
                if (!kPos) {
#pragma unroll
                    for (int k = 0; k < kStep; ++k)
                        xs[k] = __float_as_uint(__uint_as_float(xs[k]) * p.scale_log2);
                }
                constexpr uint32_t kNegInf = 0xff800000u;
                if ((j + 1) * kStep > si.kend_lo) {
                    const int lim = kend - j * kStep;               // visible keys of this step
#pragma unroll
                    for (int k = 0; k < kStep; ++k) xs[k] = k < lim ? xs[k] : kNegInf;
                }
                float m8[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) m8[a] = __uint_as_float(xs[a]);
#pragma unroll
                for (int k = 8; k < kStep; k += 2)
                    m8[(k >> 1) & 7] = fmax3(m8[(k >> 1) & 7], __uint_as_float(xs[k]),
                                             __uint_as_float(xs[k + 1]));
                float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                                 fmaxf(m8[6], m8[7]));
                if (kPos) mx *= p.scale_log2;
                if (j == 0) {
                    m_run = mx;
                } else if (__any_sync(0xffffffffu, mx > m_run + C::kRescaleThreshold)) {
                    // a row max of this warp grew a lot: move the warp's rows to their
                    // new max and rescale O (after the P V of the previous step) and l.
                    // TMEM loads / stores are warp-wide, so the whole warp takes this path.
                    const float m_new = fmaxf(m_run, mx);
                    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
                    const uint32_t pb = (ex - 1) & 1;
                    const bool waited =
                        mbar_wait(bar(kBarPvDone + 2 * x + pb), ((ex - 1) >> 1) & 1, p.status);
                    if (!__all_sync(0xffffffffu, waited)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // a rare path: kept rolled, out of the instruction cache's way
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(o_addr + 32 * c, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                        tmem_st32(o_addr + 32 * c, v);
                    }
                    l *= alpha;
                    m_run = m_new;
                }
                const float mu = (m_run == -INFINITY) ? 0.f : m_run;
                // p = 2^(s * c - mu), two lanes of work per FMA, summed in 4 chains,
                // packed to bf16 pairs over the first 32 columns of this S buffer
                const float2 c2 = kPos ? make_float2(p.scale_log2, p.scale_log2) : make_float2(1.f, 1.f);
                const float2 nmu2 = make_float2(-mu, -mu);
                float2 l4[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) l4[a] = make_float2(0.f, 0.f);
                uint32_t pk[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float2 y = ffma2(make_float2(__uint_as_float(xs[2 * k]), __uint_as_float(xs[2 * k + 1])),
                                           c2, nmu2);
                    const float2 pv = make_float2(fast_exp2(y.x), fast_exp2(y.y));
                    l4[k & 3] = fadd2(l4[k & 3], pv);
                    pk[k] = pack_bf16x2(pv.x, pv.y);
                }
                tmem_st32(s_addr + b * kStep, pk);
                l += ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + 2 * x + b));
            }
            // ---- epilogue: O / l -> bf16 rows of out (after the last P V of this tile).
            // The tile's four warps decide together whether they go on: a warp
            // whose wait ran out must not leave the others at the barriers below.
            bool eok = ok;
            if (eok) {
                const uint32_t lb = (ex - 1) & 1;
                eok = __all_sync(0xffffffffu,
                                 mbar_wait(bar(kBarPvDone + 2 * x + lb), ((ex - 1) >> 1) & 1, p.status));
            }
            ok = named_barrier_and(1 + x, 128, eok);
            if (!ok) break;
            tc_fence_after();
            // O / l as bf16, 64 columns per pass, into the tile's staging buffer in
            // the layout of a Q tile (row r at r * 128 bytes, 16-byte pieces XOR-ed
            // with r % 8); then one TMA store per pass writes the 128 rows into
            // out.  A tile that ends before 128 rows (the last of its sequence)
            // copies its rows out by hand instead, as the box would run into the
            // next sequence's rows.
            const float inv = l > 0.f ? p.v_scale / l : 0.f;
            if (p.lse != nullptr && valid)
                p.lse[(int64_t)(pi.q0 + i) * p.hq + pi.kvh * p.g + pr % p.g] = row_lse(m_run, l);
            const bool leader = quarter == 0 && lane == 0;
            const int tid = quarter * 32 + lane;        // thread of the tile = row r
            // the previous item's stores have read the staging buffers
            if (leader) bulk_wait_read_all();
            named_barrier_sync(1 + x, 128);
#pragma unroll 1
            for (int h = 0; h < D / 64; ++h) {
                uint8_t *stg = stage_ptr + x * C::kStageBytes + h * (kPreRows * 128);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + 64 * h + 32 * c, v);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4 *>(stg + r * 128 + (((4 * c + k) ^ (r & 7)) << 4)) = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * k]) * inv, __uint_as_float(v[8 * k + 1]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv));
                }
                fence_proxy_async_smem();
                named_barrier_sync(1 + x, 128);
                if (si.nrows == kPreRows) {
                    if (leader) {
                        tma_store_3d(&tm_o, sstage + x * C::kStageBytes + h * (kPreRows * 128), 64 * h,
                                     pi.kvh * p.g, pi.q0 + si.row0 / p.g);
                        bulk_commit_group();
                    }
                } else {
                    copy_partial_rows<D>(p.out, stg, tid, si.nrows, si.row0, pi.q0, pi.kvh, p.g, p.hq, 64 * h);
                    named_barrier_sync(1 + x, 128);     // the buffer is free for the next pass
                }
            }
            // O is read: the next item's first P V (which overwrites O) waits for this
            // warpgroup's P of that item, which comes after these loads
        }
    }

    // the output stores have completed before the CTA's shared memory goes away
    if (warp < 8 && (warp & 3) == 0 && lane == 0) bulk_wait_all();
    // ---- teardown: every role is done with TMEM before it is freed
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool kPos, bool kClaimed>
static cudaError_t launch_prefill_t(const PrefillParams &p, const CUtensorMap &tm_q,
                                    const CUtensorMap &tm_o, const CUtensorMap &tm_k, const CUtensorMap &tm_vp, int ctas,
                                    cudaStream_t stream) {
    using C = PreCfg<D>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(ua_prefill_kernel<D, kPos, kClaimed>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    ua_prefill_kernel<D, kPos, kClaimed><<<ctas, C::kThreads, C::kSmemBytes, stream>>>(p, tm_q, tm_o, tm_k, tm_vp);
    return cudaGetLastError();
}

cudaError_t launch_prefill(int d, bool claimed, const PrefillParams &p, const CUtensorMap &tm_q,
                           const CUtensorMap &tm_o, const CUtensorMap &tm_k, const CUtensorMap &tm_vp,
                           int ctas, cudaStream_t stream) {
    const bool pos = p.scale_log2 > 0.f;
    if (claimed) {
        // the claiming kernel exists for D = 128 with a positive scale (the
        // planner claims only then)
        if (d != 128 || !pos) return cudaErrorInvalidValue;
        return launch_prefill_t<128, true, true>(p, tm_q, tm_o, tm_k, tm_vp, ctas, stream);
    }
    if (d == 64)
        return pos ? launch_prefill_t<64, true, false>(p, tm_q, tm_o, tm_k, tm_vp, ctas, stream)
                   : launch_prefill_t<64, false, false>(p, tm_q, tm_o, tm_k, tm_vp, ctas, stream);
    return pos ? launch_prefill_t<128, true, false>(p, tm_q, tm_o, tm_k, tm_vp, ctas, stream)
               : launch_prefill_t<128, false, false>(p, tm_q, tm_o, tm_k, tm_vp, ctas, stream);
}

}  // namespace ua
