// ua_pages.cu -- caches whose pages hold a multiple of 16 tokens.
//
// The pages' unified kernel reads the cache in the FlashAttention layout,
// [num_blocks, block_size, Hkv, D] ("[Kernel] Unified Triton kernel that
// doesn't distinguish between prefill + decode", vLLM PR #16828, PR
// description).  With block_size = 16 r that memory is also a
// [num_blocks * r, 16, Hkv, D] cache: slot t of page b is slot t % 16 of
// 16-token page b * r + t / 16.  The kernels work on 16-token pages, so a call
// with larger pages first expands the block table: entry j of a sequence,
// page b, becomes entries j r .. j r + r - 1 = b r .. b r + r - 1.  An entry
// outside [0, num_blocks) becomes -1, which the kernels skip and report.
//
// ua_dequant_pages_kernel -- an e4m3 cache's pages, decoded for the prefill
// kernels.  The tensor-core prefill kernels read bf16 operands; with an e4m3
// cache the call first decodes the pages its prefill sequences read (each one's
// whole context) into a bf16 copy in the workspace, contiguous per sequence,
// and writes the block table of that copy.  The values are decoded exactly
// (an e4m3 value has 4 significant bits) and left unscaled: the prefill kernels
// apply k_scale through the softmax scale and v_scale to the output.  A block
// id outside [0, num_blocks) is reported in the device status word and its
// page decoded as zeros.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "unified_attention.h"
#include "ua_kernels.h"

namespace ua {

__global__ void __launch_bounds__(256)
    ua_expand_block_table_kernel(const int32_t *__restrict__ bt, int32_t *__restrict__ out, int64_t n,
                                 int32_t r, int32_t num_blocks) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t b = bt[i];
        const bool ok = b >= 0 && b < num_blocks;
        for (int32_t k = 0; k < r; ++k) out[i * r + k] = ok ? b * r + k : -1;
    }
}

cudaError_t launch_expand_block_table(const int32_t *block_table, int32_t *out, int64_t entries,
                                      int32_t r, int32_t num_blocks, cudaStream_t stream) {
    if (entries <= 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((entries + 255) / 256, 4096);
    ua_expand_block_table_kernel<<<(unsigned)blocks, 256, 0, stream>>>(block_table, out, entries, r,
                                                                       num_blocks);
    return cudaGetLastError();
}

// Eight e4m3 values (two 32-bit words) as eight bf16 values (four words).
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint32_t lo, uint32_t hi) {
    uint32_t out[4];
    const uint32_t w[2] = {lo, hi};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint16_t pair = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        const float a = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
        const float b = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
        const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        out[k] = *reinterpret_cast<const uint32_t *>(&v);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// dq: [n_dq + 1] first decoded page of each listed sequence, then [n_dq] the
// sequences.  A CTA takes decoded page t at a time (grid-stride); its threads
// convert the page's 16-byte pieces of K and V (page_vec per tensor).
__global__ void __launch_bounds__(256)
    ua_dequant_pages_kernel(const uint4 *__restrict__ k8, const uint4 *__restrict__ v8,
                            const int32_t *__restrict__ block_table, int32_t bt_stride, int32_t num_blocks,
                            const int32_t *__restrict__ dq, int32_t n_dq, int32_t *__restrict__ dq_bt,
                            uint4 *__restrict__ k16, uint4 *__restrict__ v16, int32_t page_vec, int *status) {
    const int32_t pages = __ldg(dq + n_dq);
    for (int32_t t = blockIdx.x; t < pages; t += gridDim.x) {
        // the sequence of decoded page t: the last j with dq[j] <= t
        int32_t lo = 0, hi = n_dq - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (__ldg(dq + mid) <= t) lo = mid; else hi = mid - 1;
        }
        const int32_t s = __ldg(dq + n_dq + 1 + lo);
        const int32_t pg = t - __ldg(dq + lo);
        const int32_t b = __ldg(block_table + (int64_t)s * bt_stride + pg);
        const bool ok = b >= 0 && b < num_blocks;
        if (threadIdx.x == 0) {
            dq_bt[(int64_t)s * bt_stride + pg] = t;
            if (!ok) atomicOr(status, UA_DEVICE_BAD_BLOCK_ID_BIT);
        }
        const uint4 *ks = k8 + (int64_t)b * page_vec;
        const uint4 *vs = v8 + (int64_t)b * page_vec;
        uint4 *kd = k16 + (int64_t)t * 2 * page_vec;
        uint4 *vd = v16 + (int64_t)t * 2 * page_vec;
        for (int32_t i = threadIdx.x; i < page_vec; i += blockDim.x) {
            const uint4 kr = ok ? __ldg(ks + i) : make_uint4(0, 0, 0, 0);
            const uint4 vr = ok ? __ldg(vs + i) : make_uint4(0, 0, 0, 0);
            kd[2 * i] = e4m3x8_to_bf16x8(kr.x, kr.y);
            kd[2 * i + 1] = e4m3x8_to_bf16x8(kr.z, kr.w);
            vd[2 * i] = e4m3x8_to_bf16x8(vr.x, vr.y);
            vd[2 * i + 1] = e4m3x8_to_bf16x8(vr.z, vr.w);
        }
    }
}

cudaError_t launch_dequant_pages(const void *k8, const void *v8, const int32_t *block_table,
                                 int32_t bt_stride, int32_t num_blocks, const int32_t *dq, int32_t n_dq,
                                 int64_t dq_pages, int32_t *dq_bt, void *k16, void *v16, int32_t num_kv_heads,
                                 int32_t head_size, int *status, cudaStream_t stream) {
    if (dq_pages <= 0 || n_dq <= 0) return cudaSuccess;
    const int64_t page_bytes = (int64_t)16 * num_kv_heads * head_size;     // e4m3
    if (page_bytes % 16 != 0) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t grid = std::min<int64_t>(dq_pages, (int64_t)std::max(sms, 1) * 8);
    ua_dequant_pages_kernel<<<(unsigned)grid, 256, 0, stream>>>(
        static_cast<const uint4 *>(k8), static_cast<const uint4 *>(v8), block_table, bt_stride, num_blocks,
        dq, n_dq, dq_bt, static_cast<uint4 *>(k16), static_cast<uint4 *>(v16), (int32_t)(page_bytes / 16),
        status);
    return cudaGetLastError();
}

}  // namespace ua
