// ua_kv_append.cu -- the step just before attention: write the new tokens'
// K and V rows into their pages of the paged cache.
//
// The unified call reads the context of sequence s from the cache up to
// seqused_k[s], which counts the new tokens too ("[Kernel] Unified Triton
// kernel that doesn't distinguish between prefill + decode", vLLM PR #16828,
// PR description: the FlashAttention-layout cache and the engine's varlen
// metadata); the new tokens are the last Lq positions of that context
// (bottom-right, as in the causal mask), so token i of sequence s goes to
// position p = Lk - Lq + i: page block_table[s][p / block_size], slot
// p % block_size.
//
// A CTA per run of consecutive tokens: its threads copy the run's K and V
// rows as a flat array of 16-byte pieces (Hkv * D * 2 / 16 per row, Hkv * D
// <= 2048; larger heads are refused on the host).  Each token's slot is found
// first, before any row moves, so the lookup's dependent loads meet an idle
// memory system: the CTA stages cu_seqlens_q and seqused_k in shared memory
// (one round trip, all threads), one lane per token finds its sequence by
// binary search there and reads its page from the block table (a second
// round trip); then the rows stream, a few 16-byte pieces of K and of V in
// flight per thread.  A block id outside [0, num_blocks) is skipped and
// reported in the device status word, like in the attention kernels.
// HBM-bound: per token 2 * Hkv * D * 2 bytes read and the same written; the
// grid is sized so every CTA is resident at once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "unified_attention.h"
#include "ua_kernels.h"
#include "ua_plan.h"

namespace ua {

constexpr int kAppendThreads = 256;
constexpr int kAppendMaxTokens = 64;    // tokens per CTA, at most
constexpr int kAppendBatch = 4;         // 16-byte pieces of K (and of V) a thread has in flight
constexpr int kAppendSmemSeqs = 4096;   // sequences staged in shared memory, at most

// kStaged: cu_seqlens_q and seqused_k staged in shared memory (num_seqs <=
// kAppendSmemSeqs); else the search reads them from global memory.
template <bool kStaged>
__global__ void __launch_bounds__(kAppendThreads, 4)
    ua_kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                        const int32_t *__restrict__ cu, const int32_t *__restrict__ seqused_k,
                        const int32_t *__restrict__ block_table, uint4 *__restrict__ k_cache,
                        uint4 *__restrict__ v_cache, int32_t num_seqs, int32_t total_q,
                        int32_t row_vec, int32_t tokens_per_cta, int32_t block_size,
                        int32_t num_blocks, int32_t bt_stride, int *status) {
    extern __shared__ int32_t s_seq[];                    // [num_seqs + 1] cu, [num_seqs] seqused_k
    __shared__ int64_t s_dst[kAppendMaxTokens];
    const int64_t t0 = (int64_t)blockIdx.x * tokens_per_cta;
    if (t0 >= total_q) return;
    const int32_t nt = (int32_t)((int64_t)total_q - t0 < tokens_per_cta ? (int64_t)total_q - t0
                                                                        : tokens_per_cta);
    const int32_t *c_cu = cu, *c_sk = seqused_k;
    if constexpr (kStaged) {
        for (int32_t i = (int32_t)threadIdx.x; i <= num_seqs; i += kAppendThreads) {
            s_seq[i] = __ldg(cu + i);
            if (i < num_seqs) s_seq[num_seqs + 1 + i] = __ldg(seqused_k + i);
        }
        __syncthreads();
        c_cu = s_seq;
        c_sk = s_seq + num_seqs + 1;
    }
    if (threadIdx.x < (unsigned)nt) {
        const int32_t t = (int32_t)(t0 + threadIdx.x);
        // the sequence of token t: the last s with cu[s] <= t
        int32_t lo = 0, hi = num_seqs - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (c_cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int32_t q0 = c_cu[lo], lq = c_cu[lo + 1] - q0;
        const int32_t pos = c_sk[lo] - lq + (t - q0);
        int32_t page = -1;
        if (pos >= 0 && pos / block_size < bt_stride)
            page = __ldg(block_table + (int64_t)lo * bt_stride + pos / block_size);
        int64_t dst = -1;
        if (page < 0 || page >= num_blocks)
            atomicOr(status, UA_DEVICE_BAD_BLOCK_ID_BIT);
        else
            dst = ((int64_t)page * block_size + pos % block_size) * row_vec;
        s_dst[threadIdx.x] = dst;
    }
    __syncthreads();

    const int32_t pieces = nt * row_vec;                 // per tensor
    const uint4 *ksrc = k_new + t0 * row_vec;
    const uint4 *vsrc = v_new + t0 * row_vec;
    for (int32_t base = 0; base < pieces; base += kAppendThreads * kAppendBatch) {
        uint4 kv[kAppendBatch], vv[kAppendBatch];
#pragma unroll
        for (int u = 0; u < kAppendBatch; ++u) {
            const int32_t f = base + (int32_t)threadIdx.x + kAppendThreads * u;
            if (f < pieces) {
                kv[u] = __ldg(ksrc + f);
                vv[u] = __ldg(vsrc + f);
            }
        }
#pragma unroll
        for (int u = 0; u < kAppendBatch; ++u) {
            const int32_t f = base + (int32_t)threadIdx.x + kAppendThreads * u;
            if (f < pieces) {
                const int32_t tok = f / row_vec;
                const int64_t dst = s_dst[tok];
                if (dst >= 0) {
                    const int32_t i = f - tok * row_vec;
                    k_cache[dst + i] = kv[u];
                    v_cache[dst + i] = vv[u];
                }
            }
        }
    }
}

cudaError_t launch_kv_append(const void *k_new, const void *v_new, const int32_t *cu,
                             const int32_t *seqused_k, const int32_t *block_table, void *k_cache,
                             void *v_cache, int32_t num_seqs, int32_t total_q, int32_t num_kv_heads,
                             int32_t head_size, int32_t block_size, int32_t num_blocks,
                             int32_t bt_stride, int *status, cudaStream_t stream) {
    const int32_t row_vec = num_kv_heads * head_size * 2 / 16;
    if (row_vec > 256) return cudaErrorInvalidValue;
    if (total_q <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // as many tokens per CTA as it takes for one resident wave (4 CTAs per
    // SM), at least 8 (short rows) and at most kAppendMaxTokens
    const int64_t resident = (int64_t)std::max(sms, 1) * 4;
    int32_t per = (int32_t)std::min<int64_t>(
        kAppendMaxTokens, std::max<int64_t>(8, ((int64_t)total_q + resident - 1) / resident));
    const int64_t blocks = ((int64_t)total_q + per - 1) / per;
    if (num_seqs <= kAppendSmemSeqs) {
        const size_t smem = sizeof(int32_t) * (2 * (size_t)num_seqs + 1);
        ua_kv_append_kernel<true><<<(unsigned)blocks, kAppendThreads, smem, stream>>>(
            static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu, seqused_k,
            block_table, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_seqs,
            total_q, row_vec, per, block_size, num_blocks, bt_stride, status);
    } else {
        ua_kv_append_kernel<false><<<(unsigned)blocks, kAppendThreads, 0, stream>>>(
            static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu, seqused_k,
            block_table, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_seqs,
            total_q, row_vec, per, block_size, num_blocks, bt_stride, status);
    }
    return cudaGetLastError();
}

}  // namespace ua
