// ua_merge.cu -- merge of two attention results over disjoint key sets by
// their log-sum-exp: the combination step of cascade (shared-prefix)
// attention, where the keys of a prefix common to many sequences are
// attended once without the causal mask and the sequences' own keys with it.
// Non-causal attention for cascade attention is the review request on "[Kernel]
// Unified Triton kernel that doesn't distinguish between prefill + decode"
// (vLLM PR #16828, review thread); the two passes combine exactly like the
// split-KV partials of one call:
//   m = max(lse_a, lse_b),  w_x = e^(lse_x - m),
//   out = (w_a out_a + w_b out_b) / (w_a + w_b),  lse = m + ln(w_a + w_b).
// HBM-bound: per row it reads two bf16 rows and two floats and writes one row
// and one float; 16-byte accesses, one thread per 8 elements of a row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "unified_attention.h"

namespace ua {

// out may alias out_a or out_b, and lse_out may alias lse_a or lse_b (the API
// allows merging in place, and chained cascade merges do), so no pointer is
// __restrict__ and every read is a plain load.  Each thread reads its 8
// elements of a row before it writes them, and no other thread touches them.
// A row's lse is read by all of the row's threads, which may span warps
// (head_size / 8 threads per row), so the block reads every lse of its chunk
// of rows before any thread writes lse_out: the chunk loop runs the same
// number of times in every thread of the block, with a barrier between the
// reads and the writes.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads)
    ua_merge_kernel(const __nv_bfloat16 *out_a, const float *lse_a, const __nv_bfloat16 *out_b,
                    const float *lse_b, __nv_bfloat16 *out, float *lse_out, int64_t rows, int d) {
    const int per_row = d / 8;
    const int rows_per_chunk = kMergeThreads / per_row;     // >= 1: d <= 8 * kMergeThreads
    const int64_t chunks = (rows + rows_per_chunk - 1) / rows_per_chunk;
    const int rr = threadIdx.x / per_row;                    // row within the chunk
    const int c = (threadIdx.x % per_row) * 8;
    for (int64_t ch = blockIdx.x; ch < chunks; ch += gridDim.x) {
        const int64_t r = ch * rows_per_chunk + rr;
        const bool active = rr < rows_per_chunk && r < rows;
        float a = -INFINITY, b = -INFINITY;
        uint4 va = make_uint4(0, 0, 0, 0), vb = va;
        if (active) {
            a = lse_a[r];
            b = lse_b[r];
            va = *reinterpret_cast<const uint4 *>(out_a + r * d + c);
            vb = *reinterpret_cast<const uint4 *>(out_b + r * d + c);
        }
        __syncthreads();      // every lse of the chunk has been read
        if (active) {
            const float m = fmaxf(a, b);
            float wa = 0.f, wb = 0.f, lse = -INFINITY;
            if (m != -INFINITY) {
                wa = expf(a - m);      // 0 when that side saw no key (lse = -inf)
                wb = expf(b - m);
                lse = m + logf(wa + wb);
            }
            const float inv = (wa + wb) > 0.f ? 1.f / (wa + wb) : 0.f;
            const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&va);
            const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&vb);
            uint4 vo;
            __nv_bfloat162 *po = reinterpret_cast<__nv_bfloat162 *>(&vo);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 fa = __bfloat1622float2(pa[k]);
                const float2 fb = __bfloat1622float2(pb[k]);
                po[k] = __floats2bfloat162_rn((wa * fa.x + wb * fb.x) * inv,
                                              (wa * fa.y + wb * fb.y) * inv);
            }
            *reinterpret_cast<uint4 *>(out + r * d + c) = vo;
            if (lse_out != nullptr && c == 0) lse_out[r] = lse;
        }
        __syncthreads();      // this chunk's writes come before the next chunk's reads
    }
}

}  // namespace ua

extern "C" ua_status ua_merge_attn_states(const void *out_a, const float *lse_a, const void *out_b,
                                         const float *lse_b, void *out, float *lse_out, int64_t rows,
                                         int32_t head_size, void *stream) {
    if (rows < 0 || head_size <= 0 || head_size % 8 != 0) return UA_ERR_INVALID_ARG;
    if (head_size > 8 * ua::kMergeThreads) return UA_ERR_UNSUPPORTED;
    if (rows == 0) return UA_OK;
    if (!out_a || !lse_a || !out_b || !lse_b || !out) return UA_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(out_a) | reinterpret_cast<uintptr_t>(out_b) |
                          reinterpret_cast<uintptr_t>(out);
    if (mis & 15) return UA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    const int64_t rows_per_chunk = ua::kMergeThreads / (head_size / 8);
    const int64_t chunks = (rows + rows_per_chunk - 1) / rows_per_chunk;
    const int64_t blocks = std::min<int64_t>(chunks, (int64_t)sms * 8);
    ua::ua_merge_kernel<<<(unsigned)blocks, ua::kMergeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(out_a), lse_a, static_cast<const __nv_bfloat16 *>(out_b), lse_b,
        static_cast<__nv_bfloat16 *>(out), lse_out, rows, head_size);
    if (cudaGetLastError() != cudaSuccess) return UA_ERR_CUDA;
    return UA_OK;
}
