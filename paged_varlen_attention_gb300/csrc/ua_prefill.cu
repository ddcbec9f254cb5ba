// ua_prefill.cu -- tensor-core prefill / chunked-prefill kernel (tcgen05 + TMEM + TMA).
//
// Query runs longer than one 16-row tile go here.  The query heads that share
// a KV head are stacked along M, so one 128-row tile holds 128/G tokens x G
// heads and every K/V tile loaded from the paged cache feeds all of them
// (the GQA packing of "[Kernel] Unified Triton kernel that doesn't
// distinguish between prefill + decode", vLLM PR #16828, PR description,
// there done "to ensure the Tensor cores are well used").
//
// One persistent CTA per SM walks its 128-row tiles (longest first).  Roles:
//   warp 0    TMA producer: the Q tile (box {64, G, 128/G} of [T, Hq, D]) and,
//             per 128-key tile, eight 16-token pages of K and of V
//             (box {64, 1, 16} of [pages*16, Hkv, D]), 128-byte swizzled;
//             pages past the tile's last visible key are read out of bounds,
//             which fills zeros.
//   warp 1    allocates TMEM and issues the MMAs from one thread:
//               S[e%2] = Q K_e^T      (M 128, N 128, K D; both operands K-major)
//               O     += P_e V_e      (A = P in TMEM as bf16, B = V MN-major)
//             in the order S0, S1, PV0, S2, PV1, ... so that the scores of
//             tile e+1 are computed while the softmax of tile e runs.
//   warps 2-5 softmax, one thread per row (TMEM lane): scale into the log2
//             domain, bottom-right causal mask, row max, exp2, row sum, P as
//             bf16 written over S in TMEM.  O is rescaled only when a row max
//             grows by more than 2^8 (the stale max cancels in O / l); the
//             epilogue divides by l and writes bf16 rows.
// Every wait is bounded (see ua_device.cuh); TMEM is always freed.
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {

template <int D>
struct PreCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kQBytes = kPreRows * D * 2;          // one 128-row Q tile
    static constexpr int kKvBytes = kKvTile * D * 2;          // one 128-key K (or V) tile
    static constexpr int kChunkBytes = kKvTile * 128;         // 128 rows x 64 columns
    static constexpr int kThreads = 192;
    static constexpr int kTmemCols = 512;
    static constexpr uint32_t kColS0 = 0;
    static constexpr uint32_t kColS1 = 128;
    static constexpr uint32_t kColO = 256;
    // Q x2, K x2, V x2, barriers; padded so one CTA owns the SM (and its TMEM)
    static constexpr size_t kUsed = 1024 + 2 * (size_t)kQBytes + 4 * (size_t)kKvBytes + 256;
    static constexpr size_t kSmemBytes = kUsed < 120 * 1024 ? 120 * 1024 : kUsed;
    static constexpr float kRescaleThreshold = 8.0f;          // log2 units
};

// mbarrier slots
enum : int {
    kBarQFull = 0,      // [2]
    kBarQEmpty = 2,     // [2]
    kBarKFull = 4,      // [2]
    kBarKEmpty = 6,     // [2]
    kBarVFull = 8,      // [2]
    kBarVEmpty = 10,    // [2]
    kBarSFull = 12,     // [2]
    kBarPFull = 14,     // [2]
    kBarSFree = 16,     // [2]
    kBarPvDone = 18,
    kBarOFull = 19,
    kBarDrain = 20,
    kNumBars = 21
};

struct TileInfo {
    int q0, lq, lk, kvh, row0, nrows, n;
    int kend_max;   // keys visible to the last row of the tile
    int kend_lo;    // keys visible to the first row of the tile
};

__device__ __forceinline__ TileInfo load_tile(const PrefillParams &p, int t) {
    const PreTile pt = p.tiles[t];
    TileInfo ti;
    ti.q0 = p.cu[pt.seq];
    ti.lq = p.cu[pt.seq + 1] - ti.q0;
    ti.lk = p.seqused_k[pt.seq];
    ti.kvh = pt.kvh;
    ti.row0 = pt.row0;
    ti.nrows = pt.nrows;
    ti.n = pt.kv_tiles;
    if (p.causal) {
        const int i_last = (pt.row0 + pt.nrows - 1) / p.g;
        const int i_first = pt.row0 / p.g;
        ti.kend_max = min(ti.lk, ti.lk - ti.lq + i_last + 1);
        ti.kend_lo = min(ti.lk, ti.lk - ti.lq + i_first + 1);
    } else {
        ti.kend_max = ti.lk;
        ti.kend_lo = ti.lk;
    }
    return ti;
}

template <int D>
__global__ void __launch_bounds__(PreCfg<D>::kThreads, 1)
    ua_prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
    using C = PreCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sq = smem_u32(smem);                         // Q[2]
    const uint32_t sk = sq + 2 * C::kQBytes;                    // K[2]
    const uint32_t sv = sk + 2 * C::kKvBytes;                   // V[2]
    uint8_t *sv_ptr = smem + 2 * C::kQBytes + 2 * C::kKvBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * C::kQBytes + 4 * C::kKvBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarQFull + i), 1);
            mbar_init(bar(kBarQEmpty + i), 1);
            mbar_init(bar(kBarKFull + i), 1);
            mbar_init(bar(kBarKEmpty + i), 1);
            mbar_init(bar(kBarVFull + i), 1);
            mbar_init(bar(kBarVEmpty + i), 1);
            mbar_init(bar(kBarSFull + i), 1);
            mbar_init(bar(kBarPFull + i), 128);
            mbar_init(bar(kBarSFree + i), 1);
        }
        mbar_init(bar(kBarPvDone), 1);
        mbar_init(bar(kBarOFull), 1);
        mbar_init(bar(kBarDrain), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================================ producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const uint64_t pol_kv = l2_policy_evict_last();   // K/V tiles are re-read by sibling tiles
        bool ok = true;
        uint32_t e = 0, tc = 0;
        for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tc) {
            const TileInfo ti = load_tile(p, t);
            const uint32_t qb = tc & 1;
            int good = 1;
            if (lane == 0) {
                if (!mbar_wait(bar(kBarQEmpty + qb), ((tc >> 1) & 1) ^ 1, p.status)) {
                    good = 0;
                } else {
                    mbar_arrive_expect_tx(bar(kBarQFull + qb), C::kQBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sq + qb * C::kQBytes + c * (kPreRows * 128), &tm_q, c * 64,
                                    ti.kvh * p.g, ti.q0 + ti.row0 / p.g, bar(kBarQFull + qb));
                }
            }
            ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            const int32_t *bt_row = p.block_table + (int64_t)(p.tiles[t].seq) * p.bt_stride;
            for (int j = 0; j < ti.n && ok; ++j, ++e) {
                // block ids of the tile's 8 pages; pages past the last visible key
                // are never read from the table and load as zeros
                int bid = p.num_blocks;
                const int page = j * (kKvTile / kBlockSize) + lane;
                if (lane < kKvTile / kBlockSize && page * kBlockSize < ti.kend_max) {
                    bid = __ldg(bt_row + page);
                    if (bid < 0 || bid >= p.num_blocks) {
                        record_status(p.status, UA_DEVICE_BAD_BLOCK_ID_BIT);
                        bid = p.num_blocks;
                    }
                }
                int b[kKvTile / kBlockSize];
#pragma unroll
                for (int i = 0; i < kKvTile / kBlockSize; ++i) b[i] = __shfl_sync(0xffffffffu, bid, i);
                const uint32_t st = e & 1, ph = (e >> 1) & 1;
                good = 1;
                if (lane == 0) {
                    if (!mbar_wait(bar(kBarKEmpty + st), ph ^ 1, p.status)) {
                        good = 0;
                    } else {
                        mbar_arrive_expect_tx(bar(kBarKFull + st), C::kKvBytes);
#pragma unroll
                        for (int i = 0; i < kKvTile / kBlockSize; ++i)
#pragma unroll
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d_hint(sk + st * C::kKvBytes + c * C::kChunkBytes + i * 2048,
                                                 &tm_k, c * 64, ti.kvh, b[i] * kBlockSize,
                                                 bar(kBarKFull + st), pol_kv);
                    }
                    if (good && !mbar_wait(bar(kBarVEmpty + st), ph ^ 1, p.status)) {
                        good = 0;
                    } else if (good) {
                        mbar_arrive_expect_tx(bar(kBarVFull + st), C::kKvBytes);
#pragma unroll
                        for (int i = 0; i < kKvTile / kBlockSize; ++i)
#pragma unroll
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d_hint(sv + st * C::kKvBytes + c * C::kChunkBytes + i * 2048,
                                                 &tm_v, c * 64, ti.kvh, b[i] * kBlockSize,
                                                 bar(kBarVFull + st), pol_kv);
                    }
                }
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            }
        }
        // drain: the last loads issued must land before the CTA can exit
        if (lane == 0) {
            for (uint32_t x = (e > 2 ? e - 2 : 0); x < e; ++x) {
                mbar_wait(bar(kBarKFull + (x & 1)), (x >> 1) & 1, p.status);
                mbar_wait(bar(kBarVFull + (x & 1)), (x >> 1) & 1, p.status);
            }
            for (uint32_t x = (tc > 2 ? tc - 2 : 0); x < tc; ++x)
                mbar_wait(bar(kBarQFull + (x & 1)), (x >> 1) & 1, p.status);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        constexpr uint32_t idesc_s = umma_idesc_bf16(kPreRows, kKvTile, 0, 0);
        constexpr uint32_t idesc_pv = umma_idesc_bf16(kPreRows, D, 0, 1);
        bool ok = true;
        uint32_t e = 0, tc = 0, issued_any = 0;
        // O += P_e V_e for KV tile event ev; `first` starts a fresh accumulator.
        auto issue_pv = [&](uint32_t ev, bool first) -> bool {
            const uint32_t sb = ev & 1, ph = (ev >> 1) & 1;
            if (!mbar_wait(bar(kBarPFull + sb), ph, p.status)) return false;
            if (!mbar_wait(bar(kBarVFull + sb), ph, p.status)) return false;
            tc_fence_after();
            const uint32_t p_col = tmem + (sb ? C::kColS1 : C::kColS0);
#pragma unroll
            for (int kk = 0; kk < kKvTile / 16; ++kk) {
                // 16 keys per step: P columns kk*8 .. +8 (bf16 pairs), V rows kk*16 .. +16
                const uint64_t bdesc = umma_desc_sw128(sv + sb * C::kKvBytes + kk * 2048,
                                                       C::kChunkBytes, 1024);
                umma_ts(tmem + C::kColO, p_col + kk * 8, bdesc, idesc_pv, (first && kk == 0) ? 0u : 1u);
            }
            umma_commit(bar(kBarVEmpty + sb));
            umma_commit(bar(kBarSFree + sb));
            umma_commit(bar(kBarPvDone));
            return true;
        };
        if (lane == 0) {
            for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tc) {
                const int n = p.tiles[t].kv_tiles;
                const uint32_t qb = tc & 1;
                if (!mbar_wait(bar(kBarQFull + qb), (tc >> 1) & 1, p.status)) {
                    ok = false;
                    break;
                }
                for (int j = 0; j < n && ok; ++j, ++e) {
                    const uint32_t sb = e & 1, ph = (e >> 1) & 1;
                    if (!mbar_wait(bar(kBarKFull + sb), ph, p.status) ||
                        (e >= 2 && !mbar_wait(bar(kBarSFree + sb), ph ^ 1, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t s_col = tmem + (sb ? C::kColS1 : C::kColS0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                        const uint64_t adesc = umma_desc_sw128(sq + qb * C::kQBytes + off, 16, 1024);
                        const uint64_t bdesc = umma_desc_sw128(sk + sb * C::kKvBytes + off, 16, 1024);
                        umma_ss(s_col, adesc, bdesc, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    issued_any = 1;
                    umma_commit(bar(kBarSFull + sb));
                    umma_commit(bar(kBarKEmpty + sb));
                    if (j == n - 1) umma_commit(bar(kBarQEmpty + qb));
                    if (j >= 1 && !issue_pv(e - 1, j == 1)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                if (!issue_pv(e - 1, n == 1)) {
                    ok = false;
                    break;
                }
                umma_commit(bar(kBarOFull));
            }
            // every MMA issued has completed before TMEM is released
            if (issued_any) {
                umma_commit(bar(kBarDrain));
                mbar_wait(bar(kBarDrain), 0, p.status);
            }
        }
        __syncwarp();
    } else {
        // ================================================================ softmax + epilogue
        const int quarter = warp & 3;                   // TMEM lanes this warp may touch
        const int r = quarter * 32 + lane;              // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        bool ok = true;
        uint32_t e = 0, tc = 0;
        for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tc) {
            const TileInfo ti = load_tile(p, t);
            const int pr = ti.row0 + r;
            const bool valid = r < ti.nrows;
            const int i = pr / p.g;
            const int kend = (p.causal && valid) ? min(ti.lk, ti.lk - ti.lq + i + 1) : ti.lk;
            float m_run = -INFINITY;
            float l = 0.f;
            for (int j = 0; j < ti.n; ++j, ++e) {
                const uint32_t sb = e & 1, ph = (e >> 1) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + sb), ph, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_off + (sb ? C::kColS1 : C::kColS0);
                float x[kKvTile];
#pragma unroll
                for (int c = 0; c < kKvTile / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(s_addr + 32 * c, v);
#pragma unroll
                    for (int k = 0; k < 32; ++k) x[32 * c + k] = __uint_as_float(v[k]) * p.scale_log2;
                }
                if ((j + 1) * kKvTile > ti.kend_lo) {       // diagonal / tail tile: mask
                    const int lim = kend - j * kKvTile;
#pragma unroll
                    for (int k = 0; k < kKvTile; ++k)
                        if (k >= lim) x[k] = -INFINITY;
                }
                float mx = x[0];
#pragma unroll
                for (int k = 1; k < kKvTile; ++k) mx = fmaxf(mx, x[k]);
                if (j == 0) {
                    m_run = mx;
                } else if (__any_sync(0xffffffffu, mx > m_run + C::kRescaleThreshold)) {
                    // a row max of this warp grew a lot: move the warp's rows to their
                    // new max and rescale O (after P V of the previous tile) and l.
                    // TMEM loads / stores are warp-wide, so the whole warp takes this path.
                    const float m_new = fmaxf(m_run, mx);
                    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
                    const bool waited = mbar_wait(bar(kBarPvDone), (e - 1) & 1, p.status);
                    if (!__all_sync(0xffffffffu, waited)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_off + C::kColO + 32 * c, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                        tmem_st32(tmem + lane_off + C::kColO + 32 * c, v);
                    }
                    l *= alpha;
                    m_run = m_new;
                }
                const float mu = (m_run == -INFINITY) ? 0.f : m_run;
                float lsum = 0.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float p0 = fast_exp2(x[64 * c + 2 * k] - mu);
                        const float p1 = fast_exp2(x[64 * c + 2 * k + 1] - mu);
                        lsum += p0 + p1;
                        pk[k] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(s_addr + 32 * c, pk);      // P (bf16 pairs) over the first 64 columns of S
                }
                l += lsum;
                // V rows past the context in the sequence's last page may hold
                // anything (NaN included): zero them before P V reads them.
                const int last_page_start = (ti.lk - 1) & ~(kBlockSize - 1);
                if (warp == 2 && (ti.lk & (kBlockSize - 1)) != 0 && ((ti.lk - 1) / kKvTile) == j &&
                    last_page_start < ti.kend_max) {
                    if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarVFull + sb), ph, p.status))) {
                        ok = false;
                    } else {
                        const int k0 = ti.lk - j * kKvTile;
                        const int k1 = last_page_start + kBlockSize - j * kKvTile;
                        const int per_row = C::kChunks * 8;     // 16-byte pieces per key row
                        for (int u = lane; u < (k1 - k0) * per_row; u += 32) {
                            const int key = k0 + u / per_row;
                            const int c = (u % per_row) / 8;
                            const int piece = u % 8;
                            *reinterpret_cast<uint4 *>(sv_ptr + sb * C::kKvBytes + c * C::kChunkBytes +
                                                       key * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + sb));
                if (!ok) break;
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16 rows of out
            if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarOFull), tc & 1, p.status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = p.out + ((int64_t)(ti.q0 + i) * p.hq + ti.kvh * p.g + pr % p.g) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + C::kColO + 32 * c, v);
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    pk[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * inv, __uint_as_float(v[2 * k + 1]) * inv);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
        }
    }

    // ---- teardown: every role is done with TMEM before it is freed
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D>
static cudaError_t launch_prefill_t(const PrefillParams &p, const CUtensorMap &tm_q,
                                    const CUtensorMap &tm_k, const CUtensorMap &tm_v, int ctas,
                                    cudaStream_t stream) {
    using C = PreCfg<D>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(ua_prefill_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    ua_prefill_kernel<D><<<ctas, C::kThreads, C::kSmemBytes, stream>>>(p, tm_q, tm_k, tm_v);
    return cudaGetLastError();
}

cudaError_t launch_prefill(int d, const PrefillParams &p, const CUtensorMap &tm_q,
                           const CUtensorMap &tm_k, const CUtensorMap &tm_v, int ctas,
                           cudaStream_t stream) {
    return d == 64 ? launch_prefill_t<64>(p, tm_q, tm_k, tm_v, ctas, stream)
                   : launch_prefill_t<128>(p, tm_q, tm_k, tm_v, ctas, stream);
}

}  // namespace ua
