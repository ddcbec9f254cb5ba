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
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

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

}  // namespace ua
