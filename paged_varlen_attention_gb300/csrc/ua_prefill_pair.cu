// ua_prefill_pair.cu -- tensor-core prefill on pairs of SMs (tcgen05 cta_group::2),
// head size 128.
//
// The same operation as the one-SM prefill kernel (ua_prefill.cu): query runs
// longer than one 16-row decode tile, the query heads of one KV head stacked
// along M so that every K/V tile feeds all of them (the GQA packing of
// "[Kernel] Unified Triton kernel that doesn't distinguish between prefill +
// decode", vLLM PR #16828, PR description, where it keeps the tensor cores
// busy).  Here a work item -- 256 packed rows of one (sequence, KV head) --
// runs on a cluster of two CTAs on two SMs: CTA r holds rows 128 r .. 128 r +
// 127 of the item, and one MMA instruction computes all 256 rows (M = 256).
// What the pair buys:
//   * 128-key score tiles (N = 128).  Each SM reads its own 128 Q rows and
//     half of the K tile per instruction from shared memory (96 bytes per
//     cycle at full rate, against 128 available); with one SM per 128-row
//     tile and N = 64 (the one-SM kernel) it reads 192, so score MMAs ran
//     at about two thirds of the rate.
//   * K and V are loaded once per pair: CTA r loads keys 64 r .. 64 r + 63 of
//     each 128-key step (the B operand of S = Q K^T is split by N) and the
//     columns 64 r .. 64 r + 63 of V for all 128 keys (the B operand of
//     O += P V is split by N = D).
//   * TMEM per SM: three 128-column score buffers and O (128 columns), so
//     the scores of step j + 1 and j + 2 can be computed while the softmax of
//     step j runs, and S(j + 2) reuses the buffer of P V(j - 1), which had a
//     whole step to complete.
//
// Roles (12 warps per CTA):
//   warps 0-7  softmax of the CTA's 128 rows: warp w takes the rows of TMEM lane
//              quarter w % 4 (one row per thread) and half w / 4 of each step's
//              keys (each reads the other half's scores too, for the row max).  Scale into the log2 domain, bottom-right causal
//              mask, row max, exp2, row sum, P as bf16 over the first 64
//              columns of the step's score buffer; every warp then arrives on
//              the leader's P barrier (the peer's warps remotely).  O is
//              rescaled only when a row max grows by more than 2^8.  After an
//              item's last P V: O / l as bf16 rows of out (each warp its half
//              of the columns; TMA store of the 128-row tile, or by hand for a
//              tile that ends early).
//   warp 8     allocates TMEM (warp 8 of both CTAs, collectively).  Leader
//              CTA: one lane issues the pair's score MMAs S(x) = Q K^T over the
//              KV steps of the pair's items in order, each once its buffer's
//              previous P has been read (P V(x - 3) done).  Peer CTA: one lane
//              relays "this CTA's Q tile / K half has landed" to the leader's
//              barriers (the leader's MMAs read both halves).
//   warp 11    leader CTA: one lane issues O += P(y) V(y) once the pair's P(y)
//              and both V halves are there.  Peer CTA: relays its V halves.
//              Two issuing lanes, because one lane that waits for its barriers
//              and issues 16 MMAs and their commits per step was measured to
//              take longer than the tensor core needs for them.
//              Commits arrive on the barrier at the same offset in both CTAs.
//   warp 9     TMA producer of the CTA's Q tiles (double-buffered, so the next
//              item's scores can start before this item ends) and K halves
//              (four {64, 1, 16} boxes per 64 columns of [pages*16, Hkv, D]).
//   warp 10    TMA producer of the CTA's V halves (one {64, 16, 1, 1, 1} box
//              per page: its 64 columns of the page); zeroes the rows past
//              the context of a sequence's last, partial page (they may hold
//              anything, NaN included, and 0 x NaN is NaN) before it releases
//              that step.
// Pages past a step's last visible key are read out of bounds (zero fill).
// Every wait is bounded (see ua_device.cuh); TMEM is always freed.
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {
namespace {

constexpr int kPStep = 128;                      // keys per KV step
constexpr int kPStepPages = kPStep / kBlockSize; // 8
constexpr int kPHalfPages = kPStepPages / 2;     // K pages per CTA per step
constexpr int kPThreads = 384;                   // 12 warps
constexpr int kPStgBytes = kPreRows * 128 * 2;   // epilogue staging: a 64-column slice per half
constexpr int kPTmemCols = 512;
constexpr float kPRescaleThreshold = 8.0f;       // log2 units
constexpr int kPRedBytes = 2 * kPreRows * 4;      // row sums of the two halves at an item's end

// Sizes by head size.  Per SM: Q is this CTA's 128 rows x D, a K stage its 64
// of the step's 128 keys x D, a V stage all 128 keys x its D / 2 columns (the
// B operand of P V is split by N = D), and TMEM holds the score buffers (128
// columns each) and O (D columns).  D = 256 fits 512 TMEM columns and 227 KB
// of shared memory with two stages and one Q tile.
template <int D>
struct PairCfg {
    static_assert(D == 128 || D == 256, "head sizes 128 and 256");
    static constexpr int kChunks = D / 64;                   // 64-column chunks of a Q / K row
    static constexpr int kHalfChunks = D / 128;              // of the D / 2 columns of V and O a half holds
    static constexpr int kStages = D == 128 ? 3 : 2;         // K / V stages = score buffers
    static constexpr int kQBufs = D == 128 ? 2 : 1;          // Q tiles (two: the next item's S starts early)
    static constexpr int kQBytes = kPreRows * D * 2;
    static constexpr int kKBytes = (kPStep / 2) * D * 2;
    static constexpr int kVPage = kBlockSize * (D / 2) * 2;  // one page of this SM's V columns
    static constexpr int kVBytes = kPStepPages * kVPage;
    static constexpr uint32_t kColO = kStages * kPStep;      // O after the score buffers
    static_assert(kColO + D <= (uint32_t)kPTmemCols, "TMEM: score buffers + O");
    static constexpr size_t kSmemUsed = 1024 + kQBufs * (size_t)kQBytes +
                                        kStages * (size_t)(kKBytes + kVBytes) + kPStgBytes + 512 + kPRedBytes;
    static_assert(kSmemUsed <= 232448, "dynamic shared memory above 227 KB");
};

enum : int {
    bQFull = 0,     // [2] this CTA's Q tile landed (TMA tx)
    bQEmpty = 2,    // [2] the item's last S is done (commit, both CTAs)
    bQPeer = 4,     // [2] leader: the peer's Q tile landed (relayed)
    bKFull = 6,     // [3]
    bKEmpty = 9,    // [3]
    bKPeer = 12,    // [3] leader
    bVFull = 15,    // [3]
    bVEmpty = 18,   // [3]
    bVPeer = 21,    // [3] leader
    bVTail = 24,    // a step that holds a sequence's partial last page lands here first
    bSFull = 25,    // [3] scores of the step are in the buffer (commit, both CTAs)
    bPFull = 28,    // [3] leader: P of the step written by the 16 softmax warps of the pair
    bPvDone = 31,   // [3] P V of the step completed (commit, both CTAs)
    bDrain = 34,    // the S issuer's MMAs have completed
    bDrain2 = 35,   // the P V issuer's MMAs have completed
    kPNumBars = 36
};

// A work item as one CTA of the pair sees it.
struct PairItem {
    int seq, q0, lq, lk, kvh;
    int n;                 // 128-key steps of the pair (its last valid row's keys)
    int kend;              // keys visible to the pair's last valid row
    int my_row0;           // first packed row of this CTA's tile
    int my_nrows;          // valid rows of this CTA's tile (0 .. 128)
    int my_kend_lo;        // keys visible to this tile's first row
};

__device__ __forceinline__ int pair_visible(const PrefillParams &p, int lq, int lk, int row) {
    if (!p.causal) return lk;
    return min(lk, lk - lq + row / p.g + 1);
}

__device__ __forceinline__ PairItem make_item(const PrefillParams &p, const PreTile &t, uint32_t rank) {
    PairItem it;
    it.seq = t.seq;
    it.q0 = t.q0;
    it.lq = t.lq;
    it.lk = t.lk;
    it.kvh = t.kvh;
    it.kend = pair_visible(p, t.lq, t.lk, t.row0 + t.nrows - 1);
    it.n = (it.kend + kPStep - 1) / kPStep;
    it.my_row0 = t.row0 + (int)rank * kPreRows;
    it.my_nrows = max(0, min(kPreRows, t.nrows - (int)rank * kPreRows));
    it.my_kend_lo = it.my_nrows > 0 ? pair_visible(p, t.lq, t.lk, it.my_row0) : it.kend;
    return it;
}

// The pair's items: its range of the plan's list (dealt in advance).  Records
// are loaded two items ahead: next() hands out the one loaded an item earlier.
struct PairCursor {
    int t, end;
    PreTile cur, nxt;
    __device__ __forceinline__ PairCursor(const PrefillParams &p, int pair)
        : t(p.tile_begin[pair]), end(p.tile_begin[pair + 1]) {
        if (t < end) cur = p.tiles[t];
        if (t + 1 < end) nxt = p.tiles[t + 1];
    }
    __device__ __forceinline__ bool next(const PrefillParams &p, PreTile &out) {
        if (t >= end) return false;
        out = cur;
        cur = nxt;
        if (t + 2 < end) nxt = p.tiles[t + 2];
        ++t;
        return true;
    }
};

// Block id of page `page` of the sequence for a step whose pair sees `kend`
// keys (out-of-range or not-needed pages give num_blocks: TMA reads zeros).
__device__ __forceinline__ int page_block_id(const PrefillParams &p, const int32_t *bt_row, int page,
                                             int kend) {
    int bid = p.num_blocks;
    if (page * kBlockSize < kend) {
        bid = __ldg(bt_row + page);
        if (bid < 0 || bid >= p.num_blocks) {
            record_status(p.status, UA_DEVICE_BAD_BLOCK_ID_BIT);
            bid = p.num_blocks;
        }
    }
    return bid;
}

// tcgen05 issue by one thread (the issuing warps run their loops on lane 0).
__device__ __forceinline__ void umma_pair_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at offset `bar` in both CTAs once this thread's MMAs so far have completed.
__device__ __forceinline__ void umma_pair_commit(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .b16 m;\n\t"
        "mov.b16 m, 3;\n\t"
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], m;\n\t}" ::"r"(bar)
        : "memory");
}

// The same on this CTA's barrier only.
__device__ __forceinline__ void umma_local_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Rows [r_lo, r_hi) of a staged 64-column slice of O (row r at r * 128 bytes,
// 16-byte pieces XOR-ed with r % 8) to out, by the tile's 128 threads.
template <int D>
__device__ __noinline__ void pair_copy_rows(__nv_bfloat16 *out, const uint8_t *stg, int tid, int nrows,
                                            int row0, int q0, int kvh, int g, int hq, int col0) {
    for (int u = tid; u < nrows * 8; u += 128) {
        const int row = u >> 3, piece = u & 7;
        const uint4 val = *reinterpret_cast<const uint4 *>(stg + row * 128 + ((piece ^ (row & 7)) << 4));
        const int prr = row0 + row;
        *reinterpret_cast<uint4 *>(out + ((int64_t)(q0 + prr / g) * hq + kvh * g + prr % g) * D + col0 +
                                   8 * piece) = val;
    }
}

}  // namespace

template <bool kPos, int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    ua_prefill_pair_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_vh) {
    using C = PairCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sq = smem_u32(smem);                              // Q[kQBufs]: [chunk][128 rows][64]
    const uint32_t sk = sq + C::kQBufs * C::kQBytes;                 // K[kStages]: [chunk][64 keys][64]
    const uint32_t sv = sk + C::kStages * C::kKBytes;                // V[kStages]: [page][chunk][16 keys][64]
    uint8_t *sv_ptr = smem + C::kQBufs * C::kQBytes + C::kStages * C::kKBytes;
    uint8_t *stage_ptr = sv_ptr + C::kStages * C::kVBytes;           // [half][128 rows][64] bf16
    const uint32_t sstage = smem_u32(stage_ptr);
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage_ptr + kPStgBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kPNumBars + 1);
    float *red = reinterpret_cast<float *>(stage_ptr + kPStgBytes + 512);   // [2][128]
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

    // the warp index and TMEM base broadcast from lane 0, so that the compiler
    // sees them as warp-uniform
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = (int)(blockIdx.x >> 1);
    // a pair with no item leaves before touching barriers or TMEM (both CTAs
    // of the pair read the same range)
    if (p.tile_begin[pair] == p.tile_begin[pair + 1]) return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(bQFull + i), 1);
            mbar_init(bar(bQEmpty + i), 1);
            mbar_init(bar(bQPeer + i), 1);
        }
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(bar(bKFull + i), 1);
            mbar_init(bar(bKEmpty + i), 1);
            mbar_init(bar(bKPeer + i), 1);
            mbar_init(bar(bVFull + i), 1);
            mbar_init(bar(bVEmpty + i), 1);
            mbar_init(bar(bVPeer + i), 1);
            mbar_init(bar(bSFull + i), 1);
            mbar_init(bar(bPFull + i), 16);
            mbar_init(bar(bPvDone + i), 1);
        }
        mbar_init(bar(bVTail), 1);
        mbar_init(bar(bDrain), 1);
        mbar_init(bar(bDrain2), 1);
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc_pair(smem_u32(tmem_slot), kPTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();       // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
    const uint64_t pol_kv = l2_policy_evict_last();   // K/V steps are re-read by sibling items

    if (warp == 9) {
        // ================================================================ Q + K producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
        }
        bool ok = true;
        uint32_t e = 0, k_issued = 0, q_issued = 0;
        PairCursor cur(p, pair);
        PreTile t;
        for (uint32_t k = 0; ok && cur.next(p, t); ++k) {
            const PairItem it = make_item(p, t, rank);
            int good = 1;
            if (lane == 0) {
                const uint32_t qb = k % C::kQBufs;
                // buffer qb is free once the last S of item k - kQBufs is done
                if (k >= (uint32_t)C::kQBufs &&
                    !mbar_wait(bar(bQEmpty + qb), ((k / C::kQBufs) - 1) & 1, p.status)) {
                    good = 0;
                } else {
                    mbar_arrive_expect_tx(bar(bQFull + qb), C::kQBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sq + qb * C::kQBytes + c * (kPreRows * 128), &tm_q, c * 64, it.kvh * p.g,
                                    it.q0 + it.my_row0 / p.g, bar(bQFull + qb));
                    ++q_issued;
                }
            }
            ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            const int32_t *bt_row = p.block_table + (int64_t)it.seq * p.bt_stride;
            for (int j = 0; j < it.n && ok; ++j, ++e) {
                // lanes 0-3: this CTA's four pages of the step
                int bid = p.num_blocks;
                if (lane < kPHalfPages)
                    bid = page_block_id(p, bt_row, j * kPStepPages + (int)rank * kPHalfPages + lane, it.kend);
                int b[kPHalfPages];
#pragma unroll
                for (int i = 0; i < kPHalfPages; ++i) b[i] = __shfl_sync(0xffffffffu, bid, i);
                const uint32_t s = e % C::kStages, ph = (e / C::kStages) & 1;
                good = 1;
                if (lane == 0) {
                    if (!mbar_wait(bar(bKEmpty + s), ph ^ 1, p.status)) {
                        good = 0;
                    } else {
                        mbar_arrive_expect_tx(bar(bKFull + s), C::kKBytes);
#pragma unroll
                        for (int i = 0; i < kPHalfPages; ++i)
#pragma unroll
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d_hint(sk + s * C::kKBytes + c * 8192 + i * 2048, &tm_k, c * 64,
                                                 it.kvh, b[i] * kBlockSize, bar(bKFull + s), pol_kv);
                        ++k_issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            }
        }
        // drain: the last loads issued land before the CTA can exit
        if (lane == 0) {
            for (uint32_t x = (k_issued > (uint32_t)C::kStages ? k_issued - C::kStages : 0); x < k_issued; ++x)
                mbar_wait(bar(bKFull + x % C::kStages), (x / C::kStages) & 1, p.status);
            for (uint32_t x = (q_issued > (uint32_t)C::kQBufs ? q_issued - C::kQBufs : 0); x < q_issued; ++x)
                mbar_wait(bar(bQFull + x % C::kQBufs), (x / C::kQBufs) & 1, p.status);
        }
    } else if (warp == 10) {
        // ================================================================ V producer
        if (lane == 0) prefetch_tensormap(&tm_vh);
        bool ok = true;
        uint32_t e = 0, v_issued = 0, tails = 0;
        PairCursor cur(p, pair);
        PreTile t;
        while (ok && cur.next(p, t)) {
            const PairItem it = make_item(p, t, rank);
            const int32_t *bt_row = p.block_table + (int64_t)it.seq * p.bt_stride;
            // the step holding the sequence's partial last page, if a row of the pair sees it
            const int last_page_start = (it.lk - 1) & ~(kBlockSize - 1);
            const int tail_step = ((it.lk & (kBlockSize - 1)) != 0 && last_page_start < it.kend)
                                      ? last_page_start / kPStep : -1;
            for (int j = 0; j < it.n && ok; ++j, ++e) {
                int bid = p.num_blocks;
                if (lane < kPStepPages) bid = page_block_id(p, bt_row, j * kPStepPages + lane, it.kend);
                int b[kPStepPages];
#pragma unroll
                for (int i = 0; i < kPStepPages; ++i) b[i] = __shfl_sync(0xffffffffu, bid, i);
                const uint32_t s = e % C::kStages, ph = (e / C::kStages) & 1;
                const bool tail = (j == tail_step);
                const uint32_t land = tail ? bar(bVTail) : bar(bVFull + s);
                int good = 1;
                if (lane == 0) {
                    if (!mbar_wait(bar(bVEmpty + s), ph ^ 1, p.status)) {
                        good = 0;
                    } else {
                        mbar_arrive_expect_tx(land, C::kVBytes);
#pragma unroll
                        for (int i = 0; i < kPStepPages; ++i)
                            tma_load_5d_hint(sv + s * C::kVBytes + i * C::kVPage, &tm_vh, 0, 0,
                                             (int)rank * C::kHalfChunks, it.kvh, b[i], land, pol_kv);
                        ++v_issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                if (ok && tail) {
                    // wait for the step, zero the key rows past the context in the last
                    // page (this CTA's 64 columns), then release the step to the MMAs
                    const bool landed = mbar_wait(bar(bVTail), tails & 1, p.status);
                    ++tails;
                    if (!__all_sync(0xffffffffu, landed)) {
                        ok = false;
                    } else {
                        const int k0 = it.lk - j * kPStep;                       // first key to clear
                        const int k1 = last_page_start + kBlockSize - j * kPStep;  // end of the page
                        for (int u = lane; u < (k1 - k0) * 8 * C::kHalfChunks; u += 32) {
                            const int piece = u & 7;
                            const int cc = (u >> 3) % C::kHalfChunks;            // this SM's 64-column chunk
                            const int key = k0 + (u >> 3) / C::kHalfChunks;
                            *reinterpret_cast<uint4 *>(sv_ptr + s * C::kVBytes + (key / kBlockSize) * C::kVPage +
                                                       cc * 2048 + (key % kBlockSize) * 128 + piece * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(bVFull + s));
                    }
                }
            }
        }
        if (lane == 0) {
            for (uint32_t x = (v_issued > (uint32_t)C::kStages ? v_issued - C::kStages : 0); x < v_issued; ++x)
                mbar_wait(bar(bVFull + x % C::kStages), (x / C::kStages) & 1, p.status);
        }
    } else if ((warp == 8 || warp == 11) && rank == 1) {
        // ================================================================ relays (peer CTA)
        // The leader's MMAs read this CTA's halves of Q, K (warp 8) and V (warp 11);
        // tell it when each has landed, in the order the leader consumes them.
        // The loads are complete once this lane has seen their barrier, so the
        // arrivals need no ordering of their own (relaxed: a release at cluster
        // scope cost 500-1,400 ns per arrival here).
        if (lane == 0) {
            const bool qk = warp == 8;
            const uint32_t lead_q = mapa_shared(bar(bQPeer), 0);
            const uint32_t lead_kv = mapa_shared(bar(qk ? bKPeer : bVPeer), 0);
            const int full = qk ? bKFull : bVFull;
            bool ok = true;
            uint32_t e = 0;
            PairCursor cur(p, pair);
            PreTile t;
            for (uint32_t k = 0; ok && cur.next(p, t); ++k) {
                const PairItem it = make_item(p, t, rank);
                const uint32_t qb = k % C::kQBufs;
                if (qk) {
                    if (!mbar_wait(bar(bQFull + qb), (k / C::kQBufs) & 1, p.status)) break;
                    mbar_arrive_cluster_relaxed(lead_q + 8 * qb);
                }
                for (int j = 0; j < it.n; ++j, ++e) {
                    const uint32_t s = e % C::kStages, ph = (e / C::kStages) & 1;
                    if (!mbar_wait(bar(full + s), ph, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster_relaxed(lead_kv + 8 * s);
                }
            }
        }
        __syncwarp();
    } else if (warp == 8) {
        // ================================================================ S issuer (leader CTA)
        // One lane issues S(x) = Q K^T into score buffer x % 3 for the pair's
        // KV steps in order, as soon as that buffer's previous P has been read
        // (P V(x - 3) done) and both CTAs' K halves of the step have landed.
        if (lane == 0) {
            constexpr uint32_t idesc_s = umma_idesc_bf16(2 * kPreRows, kPStep, 0, 0);
            bool ok = true, issued_any = false;
            uint32_t x = 0;
            PairCursor cur(p, pair);
            PreTile t;
            for (uint32_t k = 0; ok && cur.next(p, t); ++k) {
                const PairItem it = make_item(p, t, rank);
                const uint32_t qb = k % C::kQBufs, qph = (k / C::kQBufs) & 1;
                if (!mbar_wait(bar(bQFull + qb), qph, p.status) ||
                    !mbar_wait_cluster(bar(bQPeer + qb), qph, p.status))
                    break;
                const uint64_t qd = umma_desc_sw128(sq + qb * C::kQBytes, 16, 1024);
                for (int j = 0; j < it.n; ++j, ++x) {
                    const uint32_t b = x % C::kStages, ph = (x / C::kStages) & 1;
                    if ((x >= (uint32_t)C::kStages &&
                         !mbar_wait(bar(bPvDone + b), ((x - C::kStages) / C::kStages) & 1, p.status)) ||
                        !mbar_wait(bar(bKFull + b), ph, p.status) ||
                        !mbar_wait_cluster(bar(bKPeer + b), ph, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t kd = umma_desc_sw128(sk + b * C::kKBytes, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_pair_ss(tmem + b * kPStep, qd + (uint64_t)(((kk >> 2) * (kPreRows * 128) + (kk & 3) * 32) >> 4),
                                     kd + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), idesc_s,
                                     kk > 0 ? 1u : 0u);
                    umma_pair_commit(bar(bSFull + b));
                    umma_pair_commit(bar(bKEmpty + b));
                    issued_any = true;
                }
                if (ok) umma_pair_commit(bar(bQEmpty + qb));   // the item's last S: its Q buffer is free
            }
            // every MMA issued has completed before TMEM is released
            if (issued_any) {
                umma_local_commit(bar(bDrain));
                mbar_wait(bar(bDrain), 0, p.status);
            }
        }
        __syncwarp();
    } else if (warp == 11) {
        // ================================================================ P V issuer (leader CTA)
        // One lane issues O += P(y) V(y) once the pair's 8 softmax warps have
        // written P(y) and both CTAs' V halves of the step have landed; an
        // item's first step starts O from zero.
        if (lane == 0) {
            constexpr uint32_t idesc_pv = umma_idesc_bf16(2 * kPreRows, D, 0, 1);
            bool ok = true, issued_any = false;
            uint32_t y = 0;
            PairCursor cur(p, pair);
            PreTile t;
            while (ok && cur.next(p, t)) {
                const PairItem it = make_item(p, t, rank);
                for (int j = 0; j < it.n; ++j, ++y) {
                    const uint32_t b = y % C::kStages, ph = (y / C::kStages) & 1;
                    if (!mbar_wait_cluster(bar(bPFull + b), ph, p.status) ||
                        !mbar_wait(bar(bVFull + b), ph, p.status) ||
                        !mbar_wait_cluster(bar(bVPeer + b), ph, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // 16 keys per MMA = one page of V: P columns b*128 + kk*8 .. +8 (bf16
                    // pairs); V page kk is [chunk][16 keys][64 columns], MN-major: this SM's
                    // 64-column chunks 2 KB apart, 8-key groups 1 KB apart
                    const uint64_t vd = umma_desc_sw128(sv + b * C::kVBytes, 2048, 1024);
#pragma unroll
                    for (int kk = 0; kk < kPStepPages; ++kk)
                        umma_pair_ts(tmem + C::kColO, tmem + b * kPStep + kk * 8,
                                     vd + (uint64_t)((kk * C::kVPage) >> 4), idesc_pv,
                                     (j == 0 && kk == 0) ? 0u : 1u);
                    umma_pair_commit(bar(bPvDone + b));
                    umma_pair_commit(bar(bVEmpty + b));
                    issued_any = true;
                }
            }
            if (issued_any) {
                umma_local_commit(bar(bDrain2));
                mbar_wait(bar(bDrain2), 0, p.status);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ================================================================ softmax + epilogue
        // Warp w takes the rows of TMEM lane quarter q = w % 4 (one row per
        // thread) and half h = w / 4 of each step's 128 keys and of O's 128
        // columns; each warp reads the other half's scores too, for the row max,
        // and the two warps of a quarter (one SMSP) combine each row's sum at
        // the item's end through shared memory.
        const int q = warp & 3, h = warp >> 2;
        const int r = q * 32 + lane;                    // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t s_base = tmem + lane_off;
        const uint32_t o_addr = s_base + C::kColO + (D / 2) * h;   // this half's O columns
        const uint32_t lead_p = mapa_shared(bar(bPFull), 0);
        const int qbar = 2 + q;                         // named barrier of the quarter's two warps
        bool ok = true;
        uint32_t y = 0;     // KV steps over all items (step y lives in buffer y % 3)
        PairCursor cur(p, pair);
        PreTile t;
        while (ok && cur.next(p, t)) {
            const PairItem it = make_item(p, t, rank);
            const int pr = it.my_row0 + r;
            const bool valid = r < it.my_nrows;
            const int i = pr / p.g;
            const int kend = (p.causal && valid) ? min(it.lk, it.lk - it.lq + i + 1) : it.lk;
            float m_run = -INFINITY;
            float l = 0.f;          // this half's share of the row sum
            for (int j = 0; j < it.n; ++j, ++y) {
                const uint32_t b = y % C::kStages, ph = (y / C::kStages) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(bar(bSFull + b), ph, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t xs[64];
                tmem_ld64(s_base + b * kPStep + 64 * h, xs);
                if (!kPos) {
#pragma unroll
                    for (int k = 0; k < 64; ++k) xs[k] = __float_as_uint(__uint_as_float(xs[k]) * p.scale_log2);
                }
                constexpr uint32_t kNegInf = 0xff800000u;
                const bool masked = (j + 1) * kPStep > it.my_kend_lo;
                const int lim = kend - j * kPStep;              // visible keys of this step
                if (masked) {
#pragma unroll
                    for (int k = 0; k < 64; ++k) xs[k] = (64 * h + k) < lim ? xs[k] : kNegInf;
                }
                float m8[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) m8[a] = __uint_as_float(xs[a]);
#pragma unroll
                for (int k = 8; k < 64; k += 2)
                    m8[(k >> 1) & 7] = fmax3(m8[(k >> 1) & 7], __uint_as_float(xs[k]), __uint_as_float(xs[k + 1]));
                // the other half's scores, for the row max only (each warp computes the
                // full max itself: no exchange with its partner, which would hold the
                // two warps of an SMSP in step)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t ys[32];
                    tmem_ld32(s_base + b * kPStep + 64 * (1 - h) + 32 * c, ys);
                    if (!kPos) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) ys[k] = __float_as_uint(__uint_as_float(ys[k]) * p.scale_log2);
                    }
                    if (masked) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) ys[k] = (64 * (1 - h) + 32 * c + k) < lim ? ys[k] : kNegInf;
                    }
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        m8[(k >> 2) & 7] = fmax3(m8[(k >> 2) & 7], fmax3(__uint_as_float(ys[k]), __uint_as_float(ys[k + 1]),
                                                                         __uint_as_float(ys[k + 2])),
                                                 __uint_as_float(ys[k + 3]));
                }
                float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                if (kPos) mx *= p.scale_log2;
                if (j == 0) {
                    m_run = mx;
                } else if (__any_sync(0xffffffffu, mx > m_run + kPRescaleThreshold)) {
                    // a row max of this quarter grew a lot (both warps of the quarter see
                    // the same maxes, so both take this path): move the rows to their new
                    // max and rescale this half of O (after the P V of the previous step) and l
                    const float m_new = fmaxf(m_run, mx);
                    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
                    const uint32_t pb = (y - 1) % C::kStages, pph = ((y - 1) / C::kStages) & 1;
                    if (!__all_sync(0xffffffffu, mbar_wait(bar(bPvDone + pb), pph, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
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
                // packed to bf16 pairs: keys 64 h .. 64 h + 63 go over columns 32 h ..
                // 32 h + 31 of this score buffer
                const float2 c2 = kPos ? make_float2(p.scale_log2, p.scale_log2) : make_float2(1.f, 1.f);
                const float2 nmu2 = make_float2(-mu, -mu);
                float2 l4[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) l4[a] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int e2 = 32 * c + 2 * k;
                        const float2 yv = ffma2(make_float2(__uint_as_float(xs[e2]), __uint_as_float(xs[e2 + 1])), c2, nmu2);
                        const float2 pv = make_float2(fast_exp2(yv.x), fast_exp2(yv.y));
                        l4[k & 3] = fadd2(l4[k & 3], pv);
                        pk[k] = pack_bf16x2(pv.x, pv.y);
                    }
                    tmem_st16(s_base + b * kPStep + 32 * h + 16 * c, pk);
                }
                l += ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
                // P is in TMEM once tcgen05.wait::st returns; the leader's MMA reads it
                // after seeing this arrival.  The leader's own warps arrive locally; the
                // peer's with relaxed ordering (a release at cluster scope would wait
                // for the SM's tensor work in flight: 1,000-2,700 cycles a step)
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0)
                        mbar_arrive(bar(bPFull + b));
                    else
                        mbar_arrive_cluster_relaxed(lead_p + 8 * b);
                }
            }
            // ---- epilogue: O / l -> bf16 rows of out (after the item's last P V).
            // The eight softmax warps decide together whether they go on: a warp
            // whose wait ran out must not leave the others at the barriers below.
            bool eok = ok;
            if (eok) {
                const uint32_t lb = (y - 1) % C::kStages, lph = ((y - 1) / C::kStages) & 1;
                eok = __all_sync(0xffffffffu, mbar_wait(bar(bPvDone + lb), lph, p.status));
            }
            ok = named_barrier_and(1, 256, eok);
            if (!ok) break;
            tc_fence_after();
            // the row sum over both halves (the barrier before the next item's write to
            // these slots is the epilogue's first 256-thread barrier, which the partner
            // reaches only after this read)
            float *xl = red;
            xl[h * kPreRows + r] = l;
            named_barrier_sync(qbar, 64);
            const float lt = l + xl[(1 - h) * kPreRows + r];
            const float inv = lt > 0.f ? p.v_scale / lt : 0.f;
            if (p.lse != nullptr && valid && h == 0)
                p.lse[(int64_t)(it.q0 + i) * p.hq + it.kvh * p.g + pr % p.g] = row_lse(m_run, lt);
            const bool leader = warp == 0 && lane == 0;
            // O / l in passes of one 64-column chunk per half: each warp writes its
            // rows of the chunk into its half of the staging buffer, then the
            // leader stores both chunks (TMA), or each half copies its rows by hand
            // for a tile that ends before 128 rows (a box would run into the next
            // sequence's rows)
#pragma unroll 1
            for (int pass = 0; pass < C::kHalfChunks; ++pass) {
                // the previous pass's (or item's) stores have read the staging buffer
                if (leader) bulk_wait_read_all();
                named_barrier_sync(1, 256);
                uint8_t *stg = stage_ptr + h * (kPreRows * 128);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + 64 * pass + 32 * c, v);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4 *>(stg + r * 128 + (((4 * c + k) ^ (r & 7)) << 4)) = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * k]) * inv, __uint_as_float(v[8 * k + 1]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv));
                }
                fence_proxy_async_smem();
                named_barrier_sync(1, 256);
                if (it.my_nrows == kPreRows) {
                    if (leader) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            tma_store_3d(&tm_o, sstage + hh * (kPreRows * 128), 64 * (hh * C::kHalfChunks + pass),
                                         it.kvh * p.g, it.q0 + it.my_row0 / p.g);
                        bulk_commit_group();
                    }
                } else if (it.my_nrows > 0) {
                    pair_copy_rows<D>(p.out, stg, r, it.my_nrows, it.my_row0, it.q0, it.kvh, p.g, p.hq,
                                      64 * (h * C::kHalfChunks + pass));
                    named_barrier_sync(1, 256);     // the buffer is free for the next pass
                }
            }
            // O is read: the next item's first P V (which overwrites O) waits for this
            // CTA's P of that item, which comes after these loads
        }
        // the output stores have completed before the CTA's shared memory goes away
        if (warp == 0 && lane == 0) bulk_wait_all();
    }

    // ---- teardown: both CTAs are done with TMEM and with each other's barriers
    tc_fence_before();
    cluster_sync_all();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kPTmemCols);
    }
    cluster_sync_all();
}

template <bool kPos, int D>
static cudaError_t launch_pair_t(const PrefillParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_o,
                                 const CUtensorMap &tm_k, const CUtensorMap &tm_vh, int pairs,
                                 cudaStream_t stream) {
    using C = PairCfg<D>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(ua_prefill_pair_kernel<kPos, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemUsed);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    ua_prefill_pair_kernel<kPos, D><<<2 * pairs, kPThreads, C::kSmemUsed, stream>>>(p, tm_q, tm_o, tm_k, tm_vh);
    return cudaGetLastError();
}

cudaError_t launch_prefill_pair(int d, const PrefillParams &p, const CUtensorMap &tm_q, const CUtensorMap &tm_o,
                                const CUtensorMap &tm_k, const CUtensorMap &tm_vh, int pairs,
                                cudaStream_t stream) {
    const bool pos = p.scale_log2 > 0.f;
    switch (d) {
        case 128:
            return pos ? launch_pair_t<true, 128>(p, tm_q, tm_o, tm_k, tm_vh, pairs, stream)
                       : launch_pair_t<false, 128>(p, tm_q, tm_o, tm_k, tm_vh, pairs, stream);
        case 256:
            return pos ? launch_pair_t<true, 256>(p, tm_q, tm_o, tm_k, tm_vh, pairs, stream)
                       : launch_pair_t<false, 256>(p, tm_q, tm_o, tm_k, tm_vh, pairs, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace ua
