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
// A warp per token (grid-stride): it finds its sequence by binary search in
// cu_seqlens_q and copies Hkv * D bf16 of K and of V with 16-byte loads and
// stores (Hkv * D <= 2048; larger heads are refused on the host).  A
// block id outside [0, num_blocks) is skipped and reported in the device
// status word, like in the attention kernels.  HBM-bound: per token
// 2 * Hkv * D * 2 bytes read and the same written.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "unified_attention.h"
#include "ua_kernels.h"
#include "ua_plan.h"

namespace ua {

// One warp per token row at a time (grid-stride over tokens): each lane
// copies row_vec / 32 sixteen-byte pieces of K and of V, all loads issued
// before the stores, so a warp keeps its whole row in flight.
constexpr int kAppendMaxVec = 8;    // Hkv * D * 2 / 16 / 32 pieces per lane, up to Hkv * D = 2048

__global__ void __launch_bounds__(256)
    ua_kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                        const int32_t *__restrict__ cu, const int32_t *__restrict__ seqused_k,
                        const int32_t *__restrict__ block_table, uint4 *__restrict__ k_cache,
                        uint4 *__restrict__ v_cache, int32_t num_seqs, int32_t total_q,
                        int32_t row_vec, int32_t block_size, int32_t num_blocks, int32_t bt_stride,
                        int *status) {
    const int lane = threadIdx.x & 31;
    const int32_t warps = (int32_t)(gridDim.x * (blockDim.x >> 5));
    for (int32_t t = (int32_t)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)); t < total_q;
         t += warps) {
        // the sequence of token t: the last s with cu[s] <= t
        int32_t lo = 0, hi = num_seqs - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
        }
        const int32_t q0 = __ldg(cu + lo), lq = __ldg(cu + lo + 1) - q0;
        const int32_t pos = __ldg(seqused_k + lo) - lq + (t - q0);
        int32_t page = -1;
        if (pos >= 0 && pos / block_size < bt_stride)
            page = __ldg(block_table + (int64_t)lo * bt_stride + pos / block_size);
        if (page < 0 || page >= num_blocks) {
            if (lane == 0) atomicOr(status, UA_DEVICE_BAD_BLOCK_ID_BIT);
            continue;
        }
        const int64_t dst = ((int64_t)page * block_size + pos % block_size) * row_vec;
        const int64_t src = (int64_t)t * row_vec;
        uint4 kv[kAppendMaxVec], vv[kAppendMaxVec];
#pragma unroll
        for (int u = 0; u < kAppendMaxVec; ++u) {
            const int32_t i = lane + 32 * u;
            if (i < row_vec) {
                kv[u] = __ldg(k_new + src + i);
                vv[u] = __ldg(v_new + src + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kAppendMaxVec; ++u) {
            const int32_t i = lane + 32 * u;
            if (i < row_vec) {
                k_cache[dst + i] = kv[u];
                v_cache[dst + i] = vv[u];
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
    if (row_vec > 32 * kAppendMaxVec) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // 8 warps per CTA, up to 8 CTAs per SM, no more warps than tokens
    const int64_t want = ((int64_t)total_q + 7) / 8;
    const int blocks = (int)std::min<int64_t>(want, (int64_t)std::max(sms, 1) * 8);
    ua_kv_append_kernel<<<blocks, 256, 0, stream>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), cu, seqused_k,
        block_table, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_seqs, total_q,
        row_vec, block_size, num_blocks, bt_stride, status);
    return cudaGetLastError();
}

}  // namespace ua
