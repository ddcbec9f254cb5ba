// ua_decode.cu -- memory-bound decode / split-KV kernel with the LSE merge of
// split units done by the CTA that finishes a unit's last partial.
//
// The decode rows of a unified batch (a handful of new tokens per sequence)
// are HBM-bound: every KV page of every sequence is read once per KV head and
// used by the G query heads that share it.  Packing those G heads (times the
// few new tokens) into the M dimension of one 16-row warp MMA tile is the GQA
// packing of the unified kernel ("[Kernel] Unified Triton kernel that doesn't
// distinguish between prefill + decode", vLLM PR #16828, PR description):
// each page is fetched once and feeds all heads of its group.
//
// Structure (one persistent CTA = 4 consumer warps + 2 producer warps):
//   * the K producer walks the CTA's pieces (contiguous page ranges of
//     (sequence, kv head, row tile) units), reads 32 block-table entries at a
//     time, and issues one TMA box per K page (a 5-D view of the cache, so
//     one box holds all D columns of the page's 16 tokens) into a ring of
//     shared-memory stages (128-byte swizzle); the V producer walks the same
//     pages and issues their V boxes into the same stages;
//   * consumer warp w takes pages w, w+4, ... of each piece: S = Q K^T with
//     mma.sync m16n8k16 (bf16 in, fp32 accumulate), bottom-right causal mask,
//     online softmax in the exp2 domain (O and l rescaled only when a row
//     max grows by more than 2^8), O += P V;
//   * at the end of each piece the four warps merge their (m, l, O) through
//     shared memory and write the bf16 output, or an fp32 partial plus its
//     running (max, sum) when the unit was split across CTAs (split-KV);
//   * a split unit is merged by the CTA whose partial completes it: each CTA
//     counts its partial in (device-scope fence, then an atomic add on the
//     unit's counter, zeroed by the plan copy of every call), and the one that
//     brings the count to the unit's number of pieces reads all partials back
//     from L2 and writes the bf16 output, in slot order (so the result does
//     not depend on which CTA finished last).
// Offsets into the cache are 64-bit; TMA coordinates stay 32-bit
// (num_blocks * block_size < 2^31 is checked on the host).
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {

// KV8: the cache holds e4m3 bytes (per-tensor scales).  Each consumer
// thread reads its MMA fragments' bytes straight from the stage (16-byte
// loads) and widens them to f16 in registers; the MMAs run on f16 operands
// (Q converted once per piece, in shared memory).  A unit may hold two
// adjacent kv heads (heads_per_unit = 2): one TMA box then brings both
// heads' 128-byte rows of a slot, a 256-byte run of the cache, and the
// 16-row tile holds head kvh in rows 0-7 and head kvh + 1 in rows 8-15.  Each
// head's 8 rows run as the N side of transposed MMAs (S^T = K Q^T, then
// O^T += V^T P^T, see kv8_page), so no MMA carries the other head's rows;
// the contraction index d of K Q^T and the d rows of O^T are permuted so
// that a thread's K and V bytes are contiguous.  D = 128 only.
//
// D = 256: a thread holds 64 registers of Q fragments and 128 of the O
// accumulator, so the kernel runs one CTA per SM (up to 255 registers a
// thread) with a deeper ring of 16 KB stages; every row of such a batch
// comes here (the tensor-core prefill kernels are built for D 64 and 128).
//
// Head sizes 80, 96 and 112 run in the D = 128 kernel (p.dq < D): the K / V
// pages arrive through a 4-D view of the cache whose rows end at dq, two
// 64-column boxes per page, and TMA fills the columns past dq with zeros
// (they are not read from memory); Q's tile rows are zero past dq; the output
// keeps the first dq columns.  Every row of such a batch comes here too; the
// k-steps of Q K^T past dq and the n-tiles of P V past dq (all zeros) are
// skipped.  A unit takes two adjacent kv heads when Hkv is even (rows 0-7
// head kvh, rows 8-15 head kvh + 1, as for e4m3 pages): their rows of a slot
// are one run of 2 dq elements in the cache, which for dq = 96 is three whole
// 128-byte lines, where one head's 192 bytes share a line with a neighbour
// head's row (a head fetched alone read 4/3 of its bytes from memory).  The
// MMAs then run once per head over the 16-row tile, each head keeping its
// own rows.
template <int D, bool KV8, bool kNarrow = false>
struct DecCfg {
    static_assert(!KV8 || D == 128, "the e4m3 path is laid out for D = 128");
    static_assert(D == 64 || D == 128 || D == 256, "head sizes 64, 128 and 256");
    static_assert(!kNarrow || (D == 128 && !KV8), "narrower heads run in the bf16 D = 128 kernel");
    static constexpr int kChunks = D / 64;                        // 64-column TMA boxes per row
    static constexpr int kHeadPageBytes = kBlockSize * D * (KV8 ? 1 : 2);   // one page of one kv head
    // K (or V) part of a stage: room for two kv heads' pages (e4m3, narrower heads)
    static constexpr int kPageBytes = (KV8 || kNarrow ? 2 : 1) * kHeadPageBytes;
    static constexpr int kStageBytes = 2 * kPageBytes;           // K + V
    // 64 KB of stages at two CTAs per SM; 128 KB at one (D = 256)
    static constexpr int kStages = (D == 64) ? 16 : kNarrow ? 4 : 8;
    static constexpr int kMinCtasPerSm = (D == 256) ? 1 : 2;
    static constexpr int kConsumerWarps = 4;
    // consumer warps, then the K producer (descriptors, Q rows, K boxes), then
    // the V producer (V boxes): one warp issuing both boxes of every page
    // held a CTA to ~30 GB/s (a copy of the kernel without its page compute
    // moved no more, nor with 16 stages instead of 8).  A narrower head's
    // kernel keeps one producer warp for both (measured faster there: the
    // Phi-3-mini-shaped decode 405 us against 420 with two, 424 with an idle
    // sixth warp)
    static constexpr int kProducerWarps = kNarrow ? 1 : 2;
    static constexpr int kThreads = (kConsumerWarps + kProducerWarps) * 32;
    static constexpr int kMergeFloats = kDecRows * D + 2 * kDecRows;   // per warp
    // ring of piece descriptors + Q tiles, filled by the producer ahead of use
    static constexpr int kRing = 3;
    static constexpr int kQTileBytes = kDecRows * D * 2;
    static constexpr int kDescInts = 16;
    static constexpr size_t kMergeBytes = (size_t)kConsumerWarps * kMergeFloats * 4;
    static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes +
                                         kMergeBytes + (size_t)kRing * (kQTileBytes + kDescInts * 4) +
                                         (2 * kStages + 2 * kRing) * 8;
    static_assert(kSmemBytes + 64 <= 232448, "dynamic shared memory above 227 KB");
};

constexpr float kDecRescale = 8.0f;   // log2 units

// Fields of a piece descriptor in the shared-memory ring.
enum : int {
    kDq0 = 0, kDlq, kDlk, kDkvh, kDrow0, kDnrows, kDpb, kDpe, kDslot, kDcomb, kDslot0, kDnslots
};

// e4m3 pages (D = 128).  The tile's 16 rows are two groups of 8: group j
// holds head kvh + j's rows (two heads per unit) or rows 8j .. 8j + 7 of
// head kvh (one).  Each group runs transposed, with its rows as the N = 8
// side of the m16n8k16 MMA, so no MMA carries another head's rows:
//   S^T = K Q^T  (M = 16 keys, N = 8 rows, K = d: eight k-steps),
//   O^T += V^T P^T  (M = 16 columns of d per m-tile, eight m-tiles, K = 16 keys).
// A thread (n = lane / 4, t = lane % 4) then holds S^T at keys n, n + 8 and
// rows 2t, 2t + 1, and O^T at columns 16n + i, 16n + 8 + i (m-tile i) and the
// same two rows.  P^T reaches the B-operand layout of the second MMA by an
// 8 x 8 transpose in registers (movmatrix).

// The Q tile of an e4m3 piece ([16 rows][128] at 256 bytes a row) is
// converted in place from bf16 to f16 before the pages, 16-byte chunk c of
// row r moving to chunk c ^ kv8_qswz(r, c): the reads of kv8_qk_t are then
// free of bank conflicts.  The map swaps chunks within {2q, 2q + 1} (q < 4)
// and within {8, 9, 10, 11} and {12, 13, 14, 15}.
__device__ __forceinline__ int kv8_qswz(int r, int c) { return (((c >> 3) & 1) << 1) | (r & 1); }

// S^T += K Q^T for group J: the K page at shared address kb ([slot][128 B],
// 128-byte swizzle: 16-byte chunk c of slot r sits at c ^ (r % 8)), the f16
// Q tile at qt.  Thread (n, t) reads key rows n and 8 + n, chunks 2t and
// 2t + 1; word w of chunk 2t + h holds the 4 bytes of k-step 4h + w, which
// are logical k (2t, 2t + 1 | 2t + 8, 2t + 9): d = 32t + 16(ks / 4) +
// 4(ks % 4) + (0, 1 | 2, 3).  The B operand (Q^T, row 8J + n) takes the same
// columns of Q: chunk 4t + 2h + x of the row holds k-steps 4h + 2x and
// 4h + 2x + 1.
template <int J>
__device__ __forceinline__ void kv8_qk_t(float (&s)[4], uint32_t qt, uint32_t kb, int lane) {
    const int n = lane >> 2, t = lane & 3;
    const int row = 8 * J + n;
    uint32_t kr[2][2][4];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 v = lds128(kb + (rr * 8 + n) * 128 + (((2 * t + h) ^ n) << 4));
            kr[rr][h][0] = v.x;
            kr[rr][h][1] = v.y;
            kr[rr][h][2] = v.z;
            kr[rr][h][3] = v.w;
        }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int c = 4 * t + 2 * h + x;
            const uint4 q = lds128(qt + row * 256 + ((c ^ kv8_qswz(row, c)) << 4));
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t w0 = kr[0][h][2 * x + u], w1 = kr[1][h][2 * x + u];
                const uint32_t a[4] = {e4m3x2_to_f16x2((uint16_t)(w0 & 0xffffu)),
                                       e4m3x2_to_f16x2((uint16_t)(w1 & 0xffffu)),
                                       e4m3x2_to_f16x2((uint16_t)(w0 >> 16)),
                                       e4m3x2_to_f16x2((uint16_t)(w1 >> 16))};
                mma_f16_16816(s, a, u ? q.z : q.x, u ? q.w : q.y);
            }
        }
}

// O^T += V^T P^T for one group: the V page at vb.  Thread (n, t) reads chunk
// n (d = 16n .. 16n + 15) of value rows 2t, 2t + 1, 2t + 8, 2t + 9; m-tile i
// takes bytes i and 8 + i of the chunk, the byte pairs of rows (2t, 2t + 1)
// and (2t + 8, 2t + 9) interleaved into f16 pairs.  vm0 / vm1 zero the keys
// past the context; pb: P^T in the B-operand layout; o: this group's eight
// m-tiles.
template <bool kMask>
__device__ __forceinline__ void kv8_pv_t(float (*o)[4], const uint32_t (&pb)[2], uint32_t vb, int lane,
                                         uint32_t vm0, uint32_t vm1) {
    const int n = lane >> 2;
    uint32_t vr[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 2 * (lane & 3) + (i & 1) + (i >> 1) * 8;
        const uint4 v = lds128(vb + r * 128 + ((n ^ (r & 7)) << 4));
        vr[i][0] = v.x;
        vr[i][1] = v.y;
        vr[i][2] = v.z;
        vr[i][3] = v.w;
    }
#pragma unroll
    for (int w = 0; w < 2; ++w)
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            // bytes 2hb, 2hb + 1 of word w (d = 16n + 4w + 2hb + (0, 1)) and of word
            // w + 2 (d + 8), rows (2t, 2t + 1) and (2t + 8, 2t + 9) interleaved
            const uint32_t sel = hb ? 0x7362u : 0x5140u;
            const uint32_t x0 = __byte_perm(vr[0][w], vr[1][w], sel);
            const uint32_t x1 = __byte_perm(vr[2][w], vr[3][w], sel);
            const uint32_t x0h = __byte_perm(vr[0][w + 2], vr[1][w + 2], sel);
            const uint32_t x1h = __byte_perm(vr[2][w + 2], vr[3][w + 2], sel);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int sh = 16 * b;
                uint32_t a[4] = {e4m3x2_to_f16x2((uint16_t)(x0 >> sh)), e4m3x2_to_f16x2((uint16_t)(x0h >> sh)),
                                 e4m3x2_to_f16x2((uint16_t)(x1 >> sh)), e4m3x2_to_f16x2((uint16_t)(x1h >> sh))};
                if (kMask) {
                    a[0] &= vm0;
                    a[1] &= vm0;
                    a[2] &= vm1;
                    a[3] &= vm1;
                }
                mma_f16_16816(o[4 * w + 2 * hb + b], a, pb[0], pb[1]);
            }
        }
}

// One e4m3 page for the groups j < ng: S^T, the mask, the online softmax
// (per thread: rows 2t + r of group j, m[j][r] the running max, l[j][r] this
// thread's part of the running sum, summed over the warp at the end of the
// piece) and O^T += V^T P^T.  kpage: bytes from one head's page to the
// next (two heads per unit) or 0.  kend[j][r]: visible-key limit of the row.
__device__ __forceinline__ void kv8_page(float (&o)[16][4], float (&m)[2][2], float (&l)[2][2],
                                         uint32_t qt, uint32_t kb, uint32_t vb,
                                         uint32_t kpage, int ng, int key0, const int (&kend)[2][2],
                                         int lk, float scale_log2, float rescale, int lane) {
    const int n = lane >> 2, t2 = (lane & 3) * 2;
    float s[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
    // both groups without a branch between them (a group that does not run has
    // zero Q rows and every key masked), so their MMA chains interleave
    kv8_qk_t<0>(s[0], qt, kb, lane);
    kv8_qk_t<1>(s[1], qt, kb + kpage, lane);
    // scale into the log2 domain and mask (entry e: key n + 8(e / 2), row 2t + e % 2)
    float lm[2][2];
    bool grow = false;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = key0 + n + (e >> 1) * 8;
            s[j][e] = key < kend[j][e & 1] ? s[j][e] * scale_log2 : -INFINITY;
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            lm[j][r] = fmaxf(s[j][r], s[j][r + 2]);
            grow |= lm[j][r] > m[j][r] + rescale;
        }
    }
    // The running max moves only when a row max grows by more than `rescale`
    // (log2 units); the test needs no reduction: a row's max grows that much
    // exactly when one of its eight threads sees it.
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float mx = lm[j][r];
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(m[j][r], mx);
                const float alpha = fast_exp2(m[j][r] - ((mn == -INFINITY) ? 0.f : mn));
                m[j][r] = mn;
                l[j][r] *= alpha;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[8 * j + i][r] *= alpha;
                    o[8 * j + i][r + 2] *= alpha;
                }
            }
    }
    // V rows past the context (last page) may hold anything, NaN included:
    // zero them so 0 * NaN never reaches O.
    const bool tail = key0 + kBlockSize > lk;
    const uint32_t vm0 = (key0 + t2 < lk ? 0x0000ffffu : 0u) | (key0 + t2 + 1 < lk ? 0xffff0000u : 0u);
    const uint32_t vm1 = (key0 + 8 + t2 < lk ? 0x0000ffffu : 0u) | (key0 + 9 + t2 < lk ? 0xffff0000u : 0u);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        if (j == 1 && ng < 2) break;
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float mu = m[j][e & 1] == -INFINITY ? 0.f : m[j][e & 1];
            p[e] = fast_exp2(s[j][e] - mu);
            l[j][e & 1] += p[e];
        }
        // P^T (keys n, n + 8 x rows 2t, 2t + 1) to the B layout (keys 2t, 2t + 1
        // | 2t + 8, 2t + 9 x row n)
        const uint32_t pb[2] = {movmatrix_trans(pack_f16x2(p[0], p[1])),
                                movmatrix_trans(pack_f16x2(p[2], p[3]))};
        if (tail)
            kv8_pv_t<true>(o + 8 * j, pb, vb + (j ? kpage : 0u), lane, vm0, vm1);
        else
            kv8_pv_t<false>(o + 8 * j, pb, vb + (j ? kpage : 0u), lane, vm0, vm1);
    }
}

// Tile row r of a unit with hp kv heads: its head offset and its packed row
// index within that head.
__device__ __forceinline__ int tile_row_head(int r, int hp) { return hp == 2 ? r >> 3 : 0; }
__device__ __forceinline__ int tile_row_idx(int r, int hp) { return hp == 2 ? r & 7 : r; }

// Merge of the partials of split unit u (log2 domain) by the 128 consumer
// threads of the CTA that wrote the unit's last partial.  Partial s holds
// O_s = sum_j 2^(x_j - m_s) v_j, its max m_s and l_s = sum_j 2^(x_j - m_s):
//   M = max_s m_s,  out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// The partials of other CTAs are read through L2 (ld.global.cg).
template <int D, bool kNarrow>
__device__ __forceinline__ void merge_unit(const DecodeParams &p, int q0, int kvh, int row0, int nrows,
                                           int hp, int slot0, int nslots, int tid, int nthreads) {
    const int tile_rows = hp == 2 ? kDecRows : nrows;
    for (int gi = tid; gi < tile_rows * (D / 4); gi += nthreads) {
        const int row = gi / (D / 4);
        const int col = (gi % (D / 4)) * 4;
        if (tile_row_idx(row, hp) >= nrows) continue;
        float M = -INFINITY;
        for (int s = 0; s < nslots; ++s)
            M = fmaxf(M, __ldcg(p.part_ml + 2 * ((int64_t)(slot0 + s) * kDecRows + row)));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float W = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < nslots; ++s) {
                const int64_t base = (int64_t)(slot0 + s) * kDecRows + row;
                const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + 2 * base));
                const float w = fast_exp2(ml.x - M);     // 0 for an empty partial (m = -inf)
                W += w * ml.y;
                const float4 ov = __ldcg(reinterpret_cast<const float4 *>(p.part_o + base * D + col));
                acc.x += w * ov.x;
                acc.y += w * ov.y;
                acc.z += w * ov.z;
                acc.w += w * ov.w;
            }
        }
        const float inv = W > 0.f ? p.v_scale / W : 0.f;
        const int pr = row0 + tile_row_idx(row, hp);
        const int64_t t = (int64_t)q0 + pr / p.g;
        const int h = (kvh + tile_row_head(row, hp)) * p.g + pr % p.g;
        if (p.lse != nullptr && col == 0) p.lse[t * p.hq + h] = row_lse(M, W);
        const int dq = kNarrow ? p.dq : D;
        if (kNarrow && col >= dq) continue;          // zero padding of a narrower head
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2 *>(p.out + (t * p.hq + h) * dq + col) = packed;
    }
}

// One page's box(es) of one tensor into dst, completing on bar: the 5-D view
// (all D columns of 16 slots, [chunk][slot][64], 128-byte swizzle; hp heads
// of an e4m3 page in one box), or for a narrower head one box per 64
// columns of (dq, slot, kv head, block), zeros past dq, each box the unit's
// hp heads: [chunk][head][slot][64].
template <bool kNarrow, int kChunks>
__device__ __forceinline__ void issue_page(uint32_t dst, const CUtensorMap *tm, int kvh, int b, int hp,
                                           uint32_t bar, uint64_t policy) {
    if constexpr (!kNarrow) {
        tma_load_5d_hint(dst, tm, 0, 0, 0, kvh, b, bar, policy);
    } else {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tma_load_4d_hint(dst + c * hp * 2048, tm, 64 * c, 0, kvh, b, bar, policy);
    }
}

// kNarrow: a head narrower than D (p.dq < D, see above).
template <int D, bool KV8, bool kNarrow>
__global__ void __launch_bounds__(DecCfg<D, KV8, kNarrow>::kThreads,
                                  DecCfg<D, KV8, kNarrow>::kMinCtasPerSm)
    ua_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
    using C = DecCfg<D, KV8, kNarrow>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    float *merge = reinterpret_cast<float *>(smem + (size_t)C::kStages * C::kStageBytes);
    uint8_t *qring = reinterpret_cast<uint8_t *>(merge) + C::kMergeBytes;       // [kRing][16][D] bf16
    int *dring = reinterpret_cast<int *>(qring + C::kRing * C::kQTileBytes);   // [kRing][kDescInts]
    uint64_t *bars = reinterpret_cast<uint64_t *>(dring + C::kRing * C::kDescInts);
    const uint32_t stage0 = smem_u32(stages);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + C::kStages);
    const uint32_t pfull0 = smem_u32(bars + 2 * C::kStages);
    const uint32_t pempty0 = smem_u32(bars + 2 * C::kStages + C::kRing);
    const uint32_t qring0 = smem_u32(qring);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    __shared__ int s_merge;   // this CTA completed the split unit of its current piece
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < C::kRing; ++i) {
            mbar_init(pfull0 + 8 * i, 1);
            mbar_init(pempty0 + 8 * i, 1);
        }
        fence_barrier_init();
    }
    // A head narrower than D (80, 96, 112 in the D = 128 kernel): the Q tiles'
    // columns dq .. D - 1 are zero for good (the copies below fill only the
    // first dq), and so are those of K and V (the tensor map ends at dq).
    if constexpr (kNarrow) {
        const int pad = D - p.dq;
        for (int u = threadIdx.x; u < C::kRing * kDecRows * pad; u += C::kThreads) {
            const int row = u / pad, c = p.dq + u % pad;
            reinterpret_cast<__nv_bfloat16 *>(qring)[row * D + c] = __float2bfloat16_rn(0.f);
        }
        fence_proxy_async_smem();
    }
    __syncthreads();

    const int pbeg = p.cta_begin[blockIdx.x];
    const int pend = p.cta_begin[blockIdx.x + 1];
    uint32_t issued = 0;   // producer: pages issued (kept for the final drain)

    if (warp == C::kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            if constexpr (kNarrow) prefetch_tensormap(&tm_v);
        }
        const uint64_t policy = l2_policy_evict_first();
        const int hp = KV8 || kNarrow ? p.heads_per_unit : 1;   // kv heads per unit (and per box)
        bool ok = true;
        uint32_t filled = 0;   // ring entries filled
        DecPiece nxt{};
        if (pbeg < pend) nxt = p.pieces[pbeg];
        for (int pi = pbeg; pi < pend && ok; ++pi) {
            // this piece (loaded one piece ahead) and the next one's struct
            const DecPiece pc = nxt;
            if (pi + 1 < pend) nxt = p.pieces[pi + 1];
            const int32_t *bt_row = p.block_table + (int64_t)pc.seq * p.bt_stride;
            const int q0 = p.cu[pc.seq];
            const int lq = p.cu[pc.seq + 1] - q0;
            const int lk = p.seqused_k[pc.seq];
            // ---- ring entry: descriptor + the piece's Q rows (bulk copies, one per token)
            int good = 1;
            if (lane == 0) {
                const uint32_t slot = filled % C::kRing, ph = (filled / C::kRing) & 1;
                if (!mbar_wait(pempty0 + 8 * slot, ph ^ 1, p.status, p.wait_ns)) {
                    good = 0;
                } else {
                    int *d = dring + slot * C::kDescInts;
                    d[kDq0] = q0;
                    d[kDlq] = lq;
                    d[kDlk] = lk;
                    d[kDkvh] = pc.kvh;
                    d[kDrow0] = pc.row0;
                    d[kDnrows] = pc.nrows;
                    d[kDpb] = pc.page_begin;
                    d[kDpe] = pc.page_end;
                    d[kDslot] = pc.slot;
                    if (pc.unit >= 0) {
                        const CombUnit cu = p.comb[pc.unit];
                        d[kDcomb] = pc.unit;
                        d[kDslot0] = cu.slot_begin;
                        d[kDnslots] = cu.nslots;
                    }
                    const uint32_t pb = pfull0 + 8 * slot;
                    const int dq = kNarrow ? p.dq : D;
                    mbar_arrive_expect_tx(pb, (uint32_t)(pc.nrows * hp) * dq * 2);
                    // head kvh + j's rows go to tile rows 8j + r (hp = 2) or r; a row of
                    // dq < D columns is copied alone (the tile's rows are D wide)
                    for (int j = 0; j < hp; ++j)
                        for (int r = 0; r < pc.nrows;) {
                            const int pr = pc.row0 + r;
                            const int h0 = pr % p.g;
                            const int cnt = dq == D ? min(p.g - h0, pc.nrows - r) : 1;
                            const __nv_bfloat16 *src =
                                p.q + ((int64_t)(q0 + pr / p.g) * p.hq + (pc.kvh + j) * p.g + h0) * dq;
                            bulk_load(qring0 + slot * C::kQTileBytes + (8 * j + r) * D * 2, src,
                                      (uint32_t)cnt * dq * 2, pb);
                            r += cnt;
                        }
                    ++filled;
                }
            }
            ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            if (!ok) break;
            // ---- the piece's pages, 32 block-table entries at a time
            for (int base = pc.page_begin; base < pc.page_end && ok; base += 32) {
                const int n = min(32, pc.page_end - base);
                int bid = 0;
                if (lane < n) {
                    bid = __ldg(bt_row + base + lane);
                    if (bid < 0 || bid >= p.num_blocks) {
                        record_status(p.status, UA_DEVICE_BAD_BLOCK_ID_BIT);
                        bid = p.num_blocks;   // outside the tensor map: TMA fills zeros
                    }
                }
                for (int k = 0; k < n; ++k) {
                    const int b = __shfl_sync(0xffffffffu, bid, k);
                    good = 1;
                    if (lane == 0) {
                        const uint32_t st = issued % C::kStages;
                        const uint32_t ph = (issued / C::kStages) & 1;
                        if (!mbar_wait(empty0 + 8 * st, ph ^ 1, p.status, p.wait_ns)) {
                            good = 0;
                        } else {
                            const uint32_t fb = full0 + 8 * st;
                            // the stage's K and V bytes (the V producer's boxes complete
                            // on the same barrier, before or after this)
                            mbar_arrive_expect_tx(fb, 2u * hp * C::kHeadPageBytes);
                            const uint32_t kdst = stage0 + st * C::kStageBytes;
                            if constexpr (!kNarrow) {
                                issue_page<kNarrow, C::kChunks>(kdst, &tm_k, pc.kvh, b, hp, fb, policy);
                            } else {
                                // a narrower head's kernel has no V producer warp: both
                                // tensors' boxes, one per 64 columns (see issue_page)
                                const uint32_t vdst = kdst + C::kPageBytes;
#pragma unroll
                                for (int c = 0; c < C::kChunks; ++c) {
                                    tma_load_4d_hint(kdst + c * hp * 2048, &tm_k, 64 * c, 0, pc.kvh, b, fb, policy);
                                    tma_load_4d_hint(vdst + c * hp * 2048, &tm_v, 64 * c, 0, pc.kvh, b, fb, policy);
                                }
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                    if (!ok) break;
                    ++issued;
                }
            }
        }
        // the ring's last bulk copies must land before the CTA can exit
        if (lane == 0)
            for (uint32_t x = (filled > (uint32_t)C::kRing ? filled - C::kRing : 0); x < filled; ++x)
                mbar_wait(pfull0 + 8 * (x % C::kRing), (x / C::kRing) & 1, p.status);
    } else if (warp == C::kConsumerWarps + 1) {
        // (no such warp in a narrower head's kernel: its V boxes come from the K producer)
        if constexpr (!kNarrow) {
            // ------------------------------------------------------------ V producer
            // The same pages in the same order as the K producer, into the same
            // stages: each V box once the stage is free (the K producer's
            // expect-tx covers its bytes; a box that lands first leaves the
            // barrier's transaction count below zero until then, and the phase
            // cannot complete before the K producer's arrival).
            if (lane == 0) prefetch_tensormap(&tm_v);
            const uint64_t policy = l2_policy_evict_first();
            const int hp = KV8 || kNarrow ? p.heads_per_unit : 1;
            bool ok = true;
            uint32_t vissued = 0;
            for (int pi = pbeg; pi < pend && ok; ++pi) {
                const DecPiece pc = p.pieces[pi];
                const int32_t *bt_row = p.block_table + (int64_t)pc.seq * p.bt_stride;
                for (int base = pc.page_begin; base < pc.page_end && ok; base += 32) {
                    const int n = min(32, pc.page_end - base);
                    int bid = 0;
                    if (lane < n) {
                        bid = __ldg(bt_row + base + lane);
                        if (bid < 0 || bid >= p.num_blocks) bid = p.num_blocks;   // reported by the K producer
                    }
                    for (int k = 0; k < n; ++k) {
                        const int b = __shfl_sync(0xffffffffu, bid, k);
                        int good = 1;
                        if (lane == 0) {
                            const uint32_t st = vissued % C::kStages;
                            const uint32_t ph = (vissued / C::kStages) & 1;
                            if (!mbar_wait(empty0 + 8 * st, ph ^ 1, p.status, p.wait_ns))
                                good = 0;
                            else
                                issue_page<kNarrow, C::kChunks>(stage0 + st * C::kStageBytes + C::kPageBytes, &tm_v,
                                                                pc.kvh, b, hp, full0 + 8 * st, policy);
                        }
                        ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                        if (!ok) break;
                        ++vissued;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int w = warp;
        const int qr = lane >> 2;          // fragment row (and row + 8)
        const int qc = (lane & 3) * 2;     // fragment column pair
        float *mrg_o = merge + w * C::kMergeFloats;
        float *mrg_m = mrg_o + kDecRows * D;
        float *mrg_l = mrg_m + kDecRows;
        uint32_t gbase = 0;
        bool ok = true;
        const int hp = KV8 || kNarrow ? p.heads_per_unit : 1;   // kv heads per unit
        // Every consumer warp walks every piece (the merges use a named barrier),
        // even after a failed wait: a piece it could not get counts as empty.  The
        // four warps decide together whether they have the piece (a barrier that
        // ANDs their results), so that they agree on the merge steps below.
        for (int pi = pbeg; pi < pend; ++pi) {
            // the piece's descriptor and Q rows, prepared by the producer
            const uint32_t ring = (uint32_t)(pi - pbeg);
            const uint32_t slot = ring % C::kRing;
            if (ok && !__all_sync(0xffffffffu,
                                  mbar_wait(pfull0 + 8 * slot, (ring / C::kRing) & 1, p.status, p.wait_ns)))
                ok = false;
            if constexpr (KV8) {
                // the Q tile to f16 in place (rows past the unit to zeros), swizzled for
                // kv8_qk_t: thread (r, q) moves chunks c1, c2 of row r, a pair the
                // swizzle maps onto itself
                if (ok) {
                    const int r = threadIdx.x >> 3, q = threadIdx.x & 7;
                    const int c1 = q < 4 ? 2 * q : 8 + 4 * ((q - 4) >> 1) + ((q - 4) & 1);
                    const int c2 = q < 4 ? c1 + 1 : c1 ^ kv8_qswz(r, c1);
                    const bool live = tile_row_idx(r, hp) < dring[slot * C::kDescInts + kDnrows];
                    uint8_t *rowp = qring + slot * C::kQTileBytes + r * (D * 2);
                    uint4 v1 = *reinterpret_cast<const uint4 *>(rowp + c1 * 16);
                    uint4 v2 = *reinterpret_cast<const uint4 *>(rowp + c2 * 16);
                    v1 = live ? make_uint4(bf16x2_to_f16x2(v1.x), bf16x2_to_f16x2(v1.y), bf16x2_to_f16x2(v1.z),
                                           bf16x2_to_f16x2(v1.w))
                              : make_uint4(0u, 0u, 0u, 0u);
                    v2 = live ? make_uint4(bf16x2_to_f16x2(v2.x), bf16x2_to_f16x2(v2.y), bf16x2_to_f16x2(v2.z),
                                           bf16x2_to_f16x2(v2.w))
                              : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(rowp + (c1 ^ kv8_qswz(r, c1)) * 16) = v1;
                    *reinterpret_cast<uint4 *>(rowp + (c2 ^ kv8_qswz(r, c2)) * 16) = v2;
                    // the ring slot is refilled by bulk copies (async proxy) later
                    fence_proxy_async_smem();
                }
            }
            ok = named_barrier_and(1, C::kConsumerWarps * 32, ok);
            const int *d = dring + slot * C::kDescInts;
            struct {
                int kvh, row0, nrows, page_begin, page_end, slot, comb, slot0, nslots;
            } pc;
            const int q0 = ok ? d[kDq0] : 0;
            const int lq = ok ? d[kDlq] : 0;
            const int lk = ok ? d[kDlk] : 0;
            pc.kvh = ok ? d[kDkvh] : 0;
            pc.row0 = ok ? d[kDrow0] : 0;
            pc.nrows = ok ? d[kDnrows] : 0;
            pc.page_begin = ok ? d[kDpb] : 0;
            pc.page_end = ok ? d[kDpe] : 0;
            pc.slot = ok ? d[kDslot] : -1;
            if (pc.slot >= 0) {
                pc.comb = d[kDcomb];
                pc.slot0 = d[kDslot0];
                pc.nslots = d[kDnslots];
            }
            const uint8_t *qtile = qring + slot * C::kQTileBytes;
            const int npages = pc.page_end - pc.page_begin;

            // visible-key limit of this thread's two rows (bottom-right causal)
            int kend[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = tile_row_idx(qr + 8 * rr, hp);
                const int i = (pc.row0 + r) / p.g;
                kend[rr] = (p.causal && r < pc.nrows) ? min(lk, lk - lq + i + 1) : lk;
            }
            // KV8: groups of 8 tile rows (head kvh + j, or rows 8j.. of head kvh);
            // the second one runs when it holds rows.  kend8[j][r]: row 8j + 2t + r
            // (0 for a group that does not run: every key masked)
            const int ng = (hp == 2 || pc.nrows > 8) ? 2 : 1;
            int kend8[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = tile_row_idx(8 * j + qc + rr, hp);
                    const int i = (pc.row0 + r) / p.g;
                    kend8[j][rr] = j >= ng ? 0 : (p.causal && r < pc.nrows) ? min(lk, lk - lq + i + 1) : lk;
                }
            // Q fragments (A operand), zero for rows past the unit (bf16 pages; the
            // e4m3 path reads its f16 tile from shared memory)
            uint32_t qa[KV8 ? 1 : D / 16][4];
            if constexpr (!KV8) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                    for (int ri = 0; ri < 4; ++ri) {
                        const int r = qr + (ri & 1) * 8;
                        const int col = ks * 16 + qc + (ri >> 1) * 8;
                        qa[ks][ri] = tile_row_idx(r, hp) < pc.nrows
                                         ? *reinterpret_cast<const uint32_t *>(qtile + (r * D + col) * 2)
                                         : 0u;
                    }
            }

            float o[D / 8][4];
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
            float m[2] = {-INFINITY, -INFINITY};
            float l[2] = {0.f, 0.f};
            float m8[2][2] = {{-INFINITY, -INFINITY}, {-INFINITY, -INFINITY}};
            float l8[2][2] = {{0.f, 0.f}, {0.f, 0.f}};

            for (int k = w; k < npages && ok; k += C::kConsumerWarps) {
                const uint32_t gidx = gbase + k;
                const uint32_t st = gidx % C::kStages;
                const uint32_t ph = (gidx / C::kStages) & 1;
                if (!mbar_wait(full0 + 8 * st, ph, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t kb = stage0 + st * C::kStageBytes;
                const uint32_t vb = kb + C::kPageBytes;
                const int key0 = (pc.page_begin + k) * kBlockSize;

                if constexpr (KV8) {
                    kv8_page(o, m8, l8, qring0 + slot * C::kQTileBytes, kb, vb,
                             hp == 2 ? (uint32_t)C::kHeadPageBytes : 0u, ng, key0,
                             kend8, lk, p.scale_log2, kDecRescale, lane);
                } else {
                    // S = Q K^T for 16 rows x 16 keys
                    float s[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
                    if constexpr (kNarrow) {
                        // head j's page at kb + 2048 j (chunks hp * 2048 apart); with two
                        // heads, rows 8-15 (entries 2, 3) take the second head's scores
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if (j >= hp) break;
                            float sj[2][4];
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                                for (int e = 0; e < 4; ++e) sj[nt][e] = 0.f;
#pragma unroll
                            for (int ks = 0; ks < D / 16; ++ks) {
                                if (ks * 16 >= p.dq) break;     // zero columns of both operands
                                const int c = ks >> 2;
                                const int ch = (ks & 3) * 2 + ((lane >> 3) & 1);
                                const int r = ((lane >> 4) << 3) + (lane & 7);
                                uint32_t b0, b1, b2, b3;
                                ldmatrix_x4(kb + (c * hp + j) * 2048 + r * 128 + ((ch ^ (r & 7)) << 4), b0,
                                            b1, b2, b3);
                                mma_bf16_16816(sj[0], qa[ks], b0, b1);
                                mma_bf16_16816(sj[1], qa[ks], b2, b3);
                            }
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (j == 0 || e >= 2) s[nt][e] = sj[nt][e];
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const int c = ks >> 2;
                            const int ch = (ks & 3) * 2 + ((lane >> 3) & 1);
                            const int r = ((lane >> 4) << 3) + (lane & 7);
                            uint32_t b0, b1, b2, b3;
                            ldmatrix_x4(kb + c * 2048 + r * 128 + ((ch ^ (r & 7)) << 4), b0, b1, b2, b3);
                            mma_bf16_16816(s[0], qa[ks], b0, b1);
                            mma_bf16_16816(s[1], qa[ks], b2, b3);
                        }
                    }
                    // scale into the log2 domain and mask
                    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int rr = e >> 1;
                            const int key = key0 + nt * 8 + qc + (e & 1);
                            const float x = key < kend[rr] ? s[nt][e] * p.scale_log2 : -INFINITY;
                            s[nt][e] = x;
                            mx[rr] = fmaxf(mx[rr], x);
                        }
                    // The running max moves only when a row max of this warp grows by
                    // more than kDecRescale (log2 units): until then p = 2^(s - m) <= 2^8,
                    // exact after O / l, and O and l need no rescaling (most pages).
                    float mu[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
                        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
                    }
                    if (__any_sync(0xffffffffu, mx[0] > m[0] + kDecRescale || mx[1] > m[1] + kDecRescale)) {
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const float mn = fmaxf(m[rr], mx[rr]);
                            const float alpha = fast_exp2(m[rr] - ((mn == -INFINITY) ? 0.f : mn));
                            m[rr] = mn;
                            l[rr] *= alpha;
#pragma unroll
                            for (int nt = 0; nt < D / 8; ++nt) {
                                o[nt][2 * rr] *= alpha;
                                o[nt][2 * rr + 1] *= alpha;
                            }
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) mu[rr] = (m[rr] == -INFINITY) ? 0.f : m[rr];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float pv = fast_exp2(s[nt][e] - mu[e >> 1]);
                            s[nt][e] = pv;
                            l[e >> 1] += pv;
                        }
                    uint32_t pa[4];
                    pa[0] = pack_bf16x2(s[0][0], s[0][1]);
                    pa[1] = pack_bf16x2(s[0][2], s[0][3]);
                    pa[2] = pack_bf16x2(s[1][0], s[1][1]);
                    pa[3] = pack_bf16x2(s[1][2], s[1][3]);
                    // V rows past the context (last page) may hold anything, NaN
                    // included: zero them so 0 * NaN never reaches O.
                    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
                    if (key0 + kBlockSize > lk) {
                        vm0 = (key0 + qc < lk ? 0x0000ffffu : 0u) | (key0 + qc + 1 < lk ? 0xffff0000u : 0u);
                        vm1 = (key0 + 8 + qc < lk ? 0x0000ffffu : 0u) |
                              (key0 + 9 + qc < lk ? 0xffff0000u : 0u);
                    }
                    if constexpr (kNarrow) {
                        // each head's P rows against its own V page
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if (j >= hp) break;
                            uint32_t pj[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) pj[i] = (hp == 1 || (i & 1) == j) ? pa[i] : 0u;
#pragma unroll
                            for (int np = 0; np < D / 16; ++np) {
                                if (np * 16 >= p.dq) break;     // output columns past the head
                                const int c = np >> 2;
                                const int ch = (np & 3) * 2 + (lane >> 4);
                                const int r = ((lane >> 3) & 1) * 8 + (lane & 7);
                                uint32_t v0, v1, v2, v3;
                                ldmatrix_x4_trans(vb + (c * hp + j) * 2048 + r * 128 + ((ch ^ (r & 7)) << 4), v0,
                                                  v1, v2, v3);
                                mma_bf16_16816(o[2 * np], pj, v0 & vm0, v1 & vm1);
                                mma_bf16_16816(o[2 * np + 1], pj, v2 & vm0, v3 & vm1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int np = 0; np < D / 16; ++np) {
                            const int c = np >> 2;
                            const int ch = (np & 3) * 2 + (lane >> 4);
                            const int r = ((lane >> 3) & 1) * 8 + (lane & 7);
                            uint32_t v0, v1, v2, v3;
                            ldmatrix_x4_trans(vb + c * 2048 + r * 128 + ((ch ^ (r & 7)) << 4), v0, v1, v2, v3);
                            mma_bf16_16816(o[2 * np], pa, v0 & vm0, v1 & vm1);
                            mma_bf16_16816(o[2 * np + 1], pa, v2 & vm0, v3 & vm1);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * st);
            }
            gbase += npages;

            // ---- merge the four warps' states and write the result
            if constexpr (KV8) {
                // row 8j + 2t + r: l8 summed over the row's eight threads; o[8j + i][r + 2h]
                // is column 16n + 8h + i, so a thread holds 16 consecutive columns of
                // each of its rows: four float4 stores at column d ^ 4 ((row / 2) % 8)
                // (conflict-free; groups of 4 columns stay together for the readers)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        float lt = l8[j][rr];
                        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
                        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
                        const int row = 8 * j + qc + rr;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int i0 = 8 * j + 4 * (q4 & 1), e = rr + 2 * (q4 >> 1);
                            const int d = 16 * qr + 4 * q4;
                            *reinterpret_cast<float4 *>(mrg_o + row * D + (d ^ (((row >> 1) & 7) << 2))) =
                                make_float4(o[i0][e], o[i0 + 1][e], o[i0 + 2][e], o[i0 + 3][e]);
                        }
                        if (qr == 0) {
                            mrg_m[row] = m8[j][rr];
                            mrg_l[row] = lt;
                        }
                    }
            } else {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
                    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
                }
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    const int col = nt * 8 + qc;
                    *reinterpret_cast<float2 *>(mrg_o + qr * D + col) = make_float2(o[nt][0], o[nt][1]);
                    *reinterpret_cast<float2 *>(mrg_o + (qr + 8) * D + col) = make_float2(o[nt][2], o[nt][3]);
                }
                if ((lane & 3) == 0) {
                    mrg_m[qr] = m[0];
                    mrg_m[qr + 8] = m[1];
                    mrg_l[qr] = l[0];
                    mrg_l[qr + 8] = l[1];
                }
            }
            named_barrier_sync(1, C::kConsumerWarps * 32);
            // every consumer has its copy of the descriptor and Q: free the ring slot
            if (threadIdx.x == 0) mbar_arrive(pempty0 + 8 * slot);
            const int tid = threadIdx.x;
            for (int gi = tid; gi < kDecRows * (D / 4); gi += C::kConsumerWarps * 32) {
                const int row = gi / (D / 4);
                const int col = (gi % (D / 4)) * 4;
                if (tile_row_idx(row, hp) >= pc.nrows) continue;
                float mw[C::kConsumerWarps];
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < C::kConsumerWarps; ++ww) {
                    mw[ww] = merge[ww * C::kMergeFloats + kDecRows * D + row];
                    M = fmaxf(M, mw[ww]);
                }
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float L = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int ww = 0; ww < C::kConsumerWarps; ++ww) {
                        const float f = fast_exp2(mw[ww] - M);
                        L += f * merge[ww * C::kMergeFloats + kDecRows * D + kDecRows + row];
                        const int scol = KV8 ? col ^ (((row >> 1) & 7) << 2) : col;
                        const float4 ov =
                            *reinterpret_cast<const float4 *>(merge + ww * C::kMergeFloats + row * D + scol);
                        acc.x += f * ov.x;
                        acc.y += f * ov.y;
                        acc.z += f * ov.z;
                        acc.w += f * ov.w;
                    }
                }
                if (pc.slot < 0) {
                    const float inv = L > 0.f ? p.v_scale / L : 0.f;
                    const int pr = pc.row0 + tile_row_idx(row, hp);
                    const int64_t t = (int64_t)q0 + pr / p.g;
                    const int h = (pc.kvh + tile_row_head(row, hp)) * p.g + pr % p.g;
                    if (p.lse != nullptr && col == 0) p.lse[t * p.hq + h] = row_lse(M, L);
                    const int dq = kNarrow ? p.dq : D;
                    if (!kNarrow || col < dq) {       // not the zero padding of a narrower head
                        uint2 packed;
                        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                        *reinterpret_cast<uint2 *>(p.out + (t * p.hq + h) * dq + col) = packed;
                    }
                } else {
                    // partial: unnormalised sum relative to M, plus (M, L)
                    const int64_t base = ((int64_t)pc.slot * kDecRows + row);
                    *reinterpret_cast<float4 *>(p.part_o + base * D + col) = acc;
                    if (col == 0) *reinterpret_cast<float2 *>(p.part_ml + 2 * base) = make_float2(M, L);
                }
            }
            if (pc.slot >= 0) {
                // count this partial in; the CTA that completes the unit merges it
                __threadfence();
                named_barrier_sync(1, C::kConsumerWarps * 32);
                if (tid == 0) s_merge = atomicAdd(p.comb_count + pc.comb, 1) == pc.nslots - 1;
                named_barrier_sync(1, C::kConsumerWarps * 32);
                if (s_merge) {
                    __threadfence();
                    merge_unit<D, kNarrow>(p, q0, pc.kvh, pc.row0, pc.nrows, hp, pc.slot0, pc.nslots, tid,
                                           C::kConsumerWarps * 32);
                    // every piece has arrived: nothing else touches the counter in this
                    // launch; zero it for the next launch that reuses the plan
                    if (tid == 0) p.comb_count[pc.comb] = 0;
                }
            }
            named_barrier_sync(1, C::kConsumerWarps * 32);
        }
    }

    // Drain: every TMA load this CTA issued must have landed before the CTA
    // exits (on the normal path they all have; this matters after a timeout).
    __syncthreads();
    if (warp == C::kConsumerWarps && lane == 0) {
        const uint32_t first = issued > (uint32_t)C::kStages ? issued - C::kStages : 0;
        for (uint32_t gidx = first; gidx < issued; ++gidx)
            mbar_wait(full0 + 8 * (gidx % C::kStages), (gidx / C::kStages) & 1, p.status);
    }
}

template <int D, bool KV8, bool kNarrow = false>
static cudaError_t launch_decode_t(const DecodeParams &p, const CUtensorMap &tm_k,
                                   const CUtensorMap &tm_v, int ctas, cudaStream_t stream) {
    using C = DecCfg<D, KV8, kNarrow>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(ua_decode_kernel<D, KV8, kNarrow>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    ua_decode_kernel<D, KV8, kNarrow><<<ctas, C::kThreads, C::kSmemBytes, stream>>>(p, tm_k, tm_v);
    return cudaGetLastError();
}

cudaError_t launch_decode(int d, bool kv8, const DecodeParams &p, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, int ctas, cudaStream_t stream) {
    if (kv8) {
        if (d != 128) return cudaErrorInvalidValue;
        return launch_decode_t<128, true>(p, tm_k, tm_v, ctas, stream);
    }
    if (p.dq != d) return cudaErrorInvalidValue;
    switch (d) {
        case 64: return launch_decode_t<64, false>(p, tm_k, tm_v, ctas, stream);
        case 80:
        case 96:
        case 112: return launch_decode_t<128, false, true>(p, tm_k, tm_v, ctas, stream);
        case 128: return launch_decode_t<128, false>(p, tm_k, tm_v, ctas, stream);
        case 256: return launch_decode_t<256, false>(p, tm_k, tm_v, ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ua
