// ua_static_ws.cu -- unified_attention_no_alloc: the same call as
// unified_attention, with its scratch memory in a fixed device array that the
// library owns, so the caller never has to allocate device memory.
//
// Who needs this: code that is not allowed to call cudaMalloc (or any other
// device allocator) -- for example a plugin inside a framework whose caching
// allocator owns all device memory and gives the plugin no handle to it, or a
// latency-critical path where an allocation could synchronise the device.
// Such callers still own q, the caches, the metadata and out; only the
// workspace (launch plan + split-KV partials) moves into this array.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library's module holds UA_STATIC_WORKSPACE_BYTES of device memory for it
// until the process exits.  In host code the symbol is only a stand-in, not a
// device address, so the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "unified_attention.h"
#include "ua_kernels.h"

namespace {

constexpr size_t kStaticBytes = UA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_ua_static_workspace[kStaticBytes];

std::mutex g_static_mutex;
void *g_static_addr[kMaxDevices] = {};

// Device address of the array on the current device (set-up on first use).
ua_status static_workspace(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ua_static_workspace) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
        g_static_addr[dev] = p;
    }
    *addr = g_static_addr[dev];
    return UA_OK;
}

}  // namespace

extern "C" ua_status unified_attention_no_alloc(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *cu_seqlens_q,
    const int32_t *seqused_k, const int32_t *block_table, float softmax_scale, int32_t causal,
    void *out, const int32_t *cu_seqlens_q_host, const int32_t *seqused_k_host, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
    int32_t num_blocks, int32_t block_table_stride, void *stream) {
    // Size check first: a batch whose plan and partials do not fit is refused
    // before anything is launched.
    size_t need = 0;
    ua_status st = ua_workspace_size(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                                     num_kv_heads, head_size, block_size, block_table_stride,
                                     causal, &need);
    if (st != UA_OK) return st;
    if (need > kStaticBytes) return UA_ERR_WORKSPACE;
    void *ws = nullptr;
    st = static_workspace(&ws);
    if (st != UA_OK) return st;
    // the plan goes up from pageable memory: no page-locked buffer is allocated
    return ua::run_attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                             softmax_scale, causal, out, cu_seqlens_q_host, seqused_k_host,
                             num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                             num_blocks, block_table_stride, ws, kStaticBytes, stream,
                             /*pinned_plan=*/false, /*lse=*/nullptr);
}
