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

// out may alias out_a or out_b (the API allows merging in place), so the three
// row pointers are not __restrict__ and are read with plain loads: each thread
// reads its 8 elements of a row before it writes them, and no other thread
// touches them.
__global__ void __launch_bounds__(256)
    ua_merge_kernel(const __nv_bfloat16 *out_a, const float *__restrict__ lse_a,
                    const __nv_bfloat16 *out_b, const float *__restrict__ lse_b,
                    __nv_bfloat16 *out, float *__restrict__ lse_out, int64_t rows, int d) {
    const int per_row = d / 8;
    const int64_t total = rows * per_row;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / per_row;
        const int c = (int)(idx % per_row) * 8;
        const float a = __ldg(lse_a + r), b = __ldg(lse_b + r);
        const float m = fmaxf(a, b);
        float wa = 0.f, wb = 0.f, lse = -INFINITY;
        if (m != -INFINITY) {
            wa = expf(a - m);      // 0 when that side saw no key (lse = -inf)
            wb = expf(b - m);
            lse = m + logf(wa + wb);
        }
        const float inv = (wa + wb) > 0.f ? 1.f / (wa + wb) : 0.f;
        const uint4 va = *reinterpret_cast<const uint4 *>(out_a + r * d + c);
        const uint4 vb = *reinterpret_cast<const uint4 *>(out_b + r * d + c);
        const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&va);
        const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&vb);
        uint4 vo;
        __nv_bfloat162 *po = reinterpret_cast<__nv_bfloat162 *>(&vo);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 fa = __bfloat1622float2(pa[k]);
            const float2 fb = __bfloat1622float2(pb[k]);
            po[k] = __floats2bfloat162_rn((wa * fa.x + wb * fb.x) * inv, (wa * fa.y + wb * fb.y) * inv);
        }
        *reinterpret_cast<uint4 *>(out + r * d + c) = vo;
        if (lse_out != nullptr && c == 0) lse_out[r] = lse;
    }
}

}  // namespace ua

extern "C" ua_status ua_merge_attn_states(const void *out_a, const float *lse_a, const void *out_b,
                                         const float *lse_b, void *out, float *lse_out, int64_t rows,
                                         int32_t head_size, void *stream) {
    if (rows < 0 || head_size <= 0 || head_size % 8 != 0) return UA_ERR_INVALID_ARG;
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
    const int64_t work = rows * (head_size / 8);
    const int64_t blocks = std::min<int64_t>((work + 255) / 256, (int64_t)sms * 8);
    ua::ua_merge_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(out_a), lse_a, static_cast<const __nv_bfloat16 *>(out_b), lse_b,
        static_cast<__nv_bfloat16 *>(out), lse_out, rows, head_size);
    if (cudaGetLastError() != cudaSuccess) return UA_ERR_CUDA;
    return UA_OK;
}
