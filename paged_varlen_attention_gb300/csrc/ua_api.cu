// ua_api.cu -- the C ABI of the library: validation, the partition pass, the
// host-to-device copy of the plan, tensor-map set-up, and the kernel launches.
//
// The operation is the unified kernel's ("[Kernel] Unified Triton kernel that
// doesn't distinguish between prefill + decode", vLLM PR #16828, PR
// description): one call for a batch that mixes prefill, chunked prefill and
// decode, over the FlashAttention-layout paged cache.  Inside the call the
// batch is split into decode units (memory-bound, split-KV, warp MMA) and
// prefill tiles (tensor-core tcgen05 tiles), as the planner decides.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "unified_attention.h"
#include "ua_kernels.h"
#include "ua_planner.h"

namespace ua {

// The device status word the kernels write (bounded waits, bad block ids).
__device__ int g_ua_device_status = 0;

// Prefill rows go to the tcgen05 kernel when this is set; otherwise every
// row tile runs in the decode kernel (correct for any shape, slower for long
// query runs).
constexpr bool kPrefillEnabled = UA_PREFILL_ENABLED;
// Head-size-128 prefill rows run on pairs of SMs (ua_prefill_pair.cu) when
// this is set; otherwise on one SM per work item (ua_prefill.cu).
constexpr bool kPairPrefill = UA_PREFILL_PAIR;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int dev = 0;
    int sms = 0;
    int *status = nullptr;             // device address of g_ua_device_status
    bool events = false;
    // profiling ring: per call, events before the plan copy, after it, after
    // decode, after prefill, after combine; what ran and how many launches
    cudaEvent_t ev[UA_PROFILE_RING][5] = {};
    bool ran[UA_PROFILE_RING][4] = {};
    bool split[UA_PROFILE_RING] = {};  // the call ran its two kernels side by side
    // a second stream for the decode kernel of a call whose two kernels run side by
    // side, and the events that fork it from the caller's stream and join it back
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex side_mutex;             // a record of fork / join and the wait on it go together
    int launches[UA_PROFILE_RING][4] = {};
    int64_t calls = 0;                 // profiled calls so far
};

static std::mutex g_mutex;
static DeviceState g_devices[kMaxDevices];
static bool g_profile = false;
// Limit of the decode kernel's main-loop waits for calls made from now on
// (ua_test_set_wait_limit; 0: the library's limit, kWaitLimitNs).
static std::atomic<unsigned long long> g_wait_limit_ns{0};

// The device's second stream and fork / join events (created on first use).
static ua_status side_stream(DeviceState *ds) {
    if (ds->side) return UA_OK;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ds->side) return UA_OK;
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ds->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ds->join, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    ds->side = s;
    return UA_OK;
}

static unsigned long long wait_limit_ns() {
    const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
    return v ? v : kWaitLimitNs;
}

// The plan of a host-planned call goes to the GPU through two rings per
// device, both owned by the library and grown on demand (an allocation only
// when a plan is larger than any that slot held before):
//   * page-locked host buffers the plan is serialised into (from page-locked
//     memory the copy is one DMA that does not hold up the host thread); a
//     buffer is rewritten only after the copy that last read it has finished;
//   * device buffers the kernels read the plan from; a buffer is overwritten
//     only after the kernels of the call that last used it have finished (an
//     event recorded on that call's stream behind its kernels).
// The copy runs on a library-owned stream and touches library memory only,
// so it needs no ordering with the caller's stream beyond that event: it
// overlaps whatever the caller's stream runs before the call (other layers'
// kernels, the previous call's own kernels), and the caller's stream waits
// for the copy before this call's kernels.  The caller's workspace holds the
// split-KV partials, which only this call's kernels touch, in stream order.
struct PlanStaging {
    static constexpr int kSlots = 8;
    uint8_t *buf[kSlots] = {};             // page-locked host
    size_t cap[kSlots] = {};
    cudaEvent_t done[kSlots] = {};         // behind the copy that read buf[i]
    bool busy[kSlots] = {};
    uint8_t *dbuf[kSlots] = {};            // device
    size_t dcap[kSlots] = {};
    cudaEvent_t used[kSlots] = {};         // behind the kernels of the call that read dbuf[i]
    bool used_pending[kSlots] = {};        // used[i] has been recorded and may not have completed
    bool held[kSlots] = {};                // a call between its copy and its kernels owns slot i
    int next = 0;
    cudaStream_t side = nullptr;           // copy stream
    cudaEvent_t copied = nullptr;          // behind the latest copy
};
static std::mutex g_stage_mutex;
static PlanStaging g_staging[kMaxDevices];

static ua_status cuda_failed() {
    cudaGetLastError();
    return UA_ERR_CUDA;
}

// Copies the plan into a device buffer of the ring (see above) and makes the
// caller's stream wait for it; *dplan is where the kernels read it, *slot the
// ring slot, which release_plan_slot must give back once the call's kernels
// are enqueued (or the call gave up).
static ua_status stage_plan(int dev, const Plan &plan, cudaStream_t stream, uint8_t **dplan,
                            int *slot) {
    const size_t bytes = plan.layout.blob_bytes;
    std::unique_lock<std::mutex> lock(g_stage_mutex);
    PlanStaging &st = g_staging[dev];
    if (!st.side) {
        cudaStream_t sd = nullptr;
        if (cudaStreamCreateWithFlags(&sd, cudaStreamNonBlocking) != cudaSuccess) return cuda_failed();
        if (cudaEventCreateWithFlags(&st.copied, cudaEventDisableTiming) != cudaSuccess) {
            cudaStreamDestroy(sd);
            return cuda_failed();
        }
        st.side = sd;
    }
    // a slot that no other call holds (more than kSlots calls between their
    // copy and their launches at once, from several host threads: wait)
    int i = -1;
    while (i < 0) {
        for (int k = 0; k < PlanStaging::kSlots && i < 0; ++k) {
            const int c = (st.next + k) % PlanStaging::kSlots;
            if (!st.held[c]) i = c;
        }
        if (i < 0) {
            lock.unlock();
            std::this_thread::yield();
            lock.lock();
        }
    }
    st.next = (i + 1) % PlanStaging::kSlots;
    if (st.busy[i]) {
        if (cudaEventSynchronize(st.done[i]) != cudaSuccess) return cuda_failed();
        st.busy[i] = false;
    }
    if (!st.done[i] && cudaEventCreateWithFlags(&st.done[i], cudaEventDisableTiming) != cudaSuccess) {
        st.done[i] = nullptr;
        return cuda_failed();
    }
    if (!st.used[i] && cudaEventCreateWithFlags(&st.used[i], cudaEventDisableTiming) != cudaSuccess) {
        st.used[i] = nullptr;
        return cuda_failed();
    }
    if (st.cap[i] < bytes) {
        if (st.buf[i]) cudaFreeHost(st.buf[i]);
        st.buf[i] = nullptr;
        st.cap[i] = 0;
        const size_t want = bytes + bytes / 2 + 4096;
        void *h = nullptr;
        if (cudaHostAlloc(&h, want, cudaHostAllocDefault) != cudaSuccess) return cuda_failed();
        st.buf[i] = static_cast<uint8_t *>(h);
        st.cap[i] = want;
    }
    if (st.dcap[i] < bytes) {
        // the kernels that last read the old buffer finish before it is freed
        if (st.used_pending[i]) {
            if (cudaEventSynchronize(st.used[i]) != cudaSuccess) return cuda_failed();
            st.used_pending[i] = false;
        }
        if (st.dbuf[i]) cudaFree(st.dbuf[i]);
        st.dbuf[i] = nullptr;
        st.dcap[i] = 0;
        const size_t want = (bytes + bytes / 2 + 4096 + kAlign - 1) / kAlign * kAlign;
        void *d = nullptr;
        if (cudaMalloc(&d, want) != cudaSuccess) return cuda_failed();
        st.dbuf[i] = static_cast<uint8_t *>(d);
        st.dcap[i] = want;
    }
    serialize_plan_to(plan, st.buf[i]);
    if ((st.used_pending[i] && cudaStreamWaitEvent(st.side, st.used[i], 0) != cudaSuccess) ||
        cudaMemcpyAsync(st.dbuf[i], st.buf[i], bytes, cudaMemcpyHostToDevice, st.side) != cudaSuccess ||
        cudaEventRecord(st.done[i], st.side) != cudaSuccess ||
        cudaEventRecord(st.copied, st.side) != cudaSuccess ||
        cudaStreamWaitEvent(stream, st.copied, 0) != cudaSuccess)
        return cuda_failed();
    st.busy[i] = true;
    st.held[i] = true;
    *dplan = st.dbuf[i];
    *slot = i;
    return UA_OK;
}

// After this call's kernels are enqueued on stream (or the call gave up after
// its copy): the slot's device buffer may be rewritten once they finish.
static ua_status release_plan_slot(int dev, int slot, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_stage_mutex);
    PlanStaging &st = g_staging[dev];
    st.held[slot] = false;
    if (cudaEventRecord(st.used[slot], stream) != cudaSuccess) {
        // nothing tells when the buffer is free again: wait for the whole device
        cudaGetLastError();
        cudaDeviceSynchronize();
        st.used_pending[slot] = false;
        return UA_ERR_CUDA;
    }
    st.used_pending[slot] = true;
    return UA_OK;
}

static ua_status device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &s = g_devices[dev];
    if (!s.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_ua_device_status) != cudaSuccess) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
        s.dev = dev;
        s.sms = sms;
        s.status = static_cast<int *>(addr);
        s.ready = true;
    }
    *out = &s;
    return UA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// L2 fill width for boxes whose rows hold `run` contiguous useful bytes: a
// 256-byte fill over a 128-byte run drags in bytes that another CTA reads much
// later (the next KV head's row), which costs DRAM bandwidth, not hits.
static CUtensorMapL2promotion l2_fill(uint64_t run) {
    return run >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
}

// 3-D bf16 map over a [outer, mid, inner] tensor with 128-byte swizzled boxes
// of {64, box_mid, box_outer} elements.  Out-of-range boxes read zeros.
static bool encode_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t mid,
                       uint64_t outer, uint32_t box_mid, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {inner, mid, outer};
    cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
    cuuint32_t box[3] = {64, box_mid, box_outer};
    cuuint32_t estr[3] = {1, 1, 1};
    // a box row's useful run: all of `inner` (the other 64-column boxes of a
    // row follow), times box_mid when that spans the whole middle extent
    const uint64_t run = inner * 2 * (box_mid == mid ? mid : box_mid);
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, l2_fill(run), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 5-D bf16 map over the paged cache [num_blocks][16][Hkv][D] viewed as
// (64 columns, 16 slots, D/64 chunks, Hkv, blocks): one box {64, 16, D/64, 1, 1}
// is one 16-token page of one KV head, laid out [chunk][slot][64] in shared
// memory with the 128-byte swizzle.  Out-of-range blocks read zeros.
// eb: bytes per element, 2 (bf16) or 1 (e4m3): a 128-byte chunk is 64 or 128
// elements, and a page row D * eb bytes.  box_heads: KV heads per box (1, or
// 2 adjacent heads laid out [head][chunk][slot][128 B]).
// box_chunks: 128-byte chunks per box (all D * eb / 128 of them, or 1: one
// 64-column slice of the page, chosen by the chunk coordinate).
static bool encode_page_map(CUtensorMap *map, const void *base, int d, int hkv,
                            uint64_t num_blocks, int eb = 2, int box_heads = 1, int box_chunks = 0) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const uint64_t row = (uint64_t)hkv * d * eb;   // bytes between slots
    const cuuint32_t inner = 128 / eb, chunks = (cuuint32_t)(d * eb / 128);
    cuuint64_t dims[5] = {inner, (cuuint64_t)kBlockSize, chunks, (cuuint64_t)hkv, num_blocks};
    cuuint64_t strides[4] = {row, 128, (cuuint64_t)d * eb, row * kBlockSize};
    const cuuint32_t bch = box_chunks > 0 ? (cuuint32_t)box_chunks : chunks;
    cuuint32_t box[5] = {inner, (cuuint32_t)kBlockSize, bch, (cuuint32_t)box_heads, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    // the box's heads of one slot are the useful run (the whole slot when
    // they are all Hkv heads); with 128-byte runs (one e4m3 head at D = 128)
    // a 256-byte fill read 1.38x the algorithmic DRAM bytes
    const CUtensorMapL2promotion promo =
        l2_fill(bch != chunks ? (uint64_t)128 * bch
                              : (hkv == box_heads ? row * kBlockSize : (uint64_t)d * eb * box_heads));
    CUresult r = enc(map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                     const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D bf16 map over the paged cache of a head narrower than 128 columns (80,
// 96, 112): (d, 16 slots, Hkv, blocks), boxes of {64, 16, box_heads, 1} with
// the 128-byte swizzle.  The box at column 64 runs past d, and TMA fills those
// columns with zeros without reading them: each head's page lands in the
// layout of a 128-column page, [chunk][head][slot][64], with zeros past d.
static bool encode_page_map_narrow(CUtensorMap *map, const void *base, int d, int hkv,
                                   uint64_t num_blocks, int box_heads) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const uint64_t row = (uint64_t)hkv * d * 2;   // bytes between slots
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)kBlockSize, (cuuint64_t)hkv, num_blocks};
    cuuint64_t strides[3] = {row, (cuuint64_t)d * 2, row * kBlockSize};
    cuuint32_t box[4] = {64, (cuuint32_t)kBlockSize, (cuuint32_t)box_heads, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     l2_fill((uint64_t)d * 2), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The decode kernel's K / V maps of a call: the 5-D page view (whole pages of
// D = 64, 128, 256 or of an e4m3 cache), or the narrow view above.
static bool encode_decode_maps(CUtensorMap *tk, CUtensorMap *tv, const void *k, const void *v, int d,
                               int hkv, uint64_t num_blocks, int eb, int box_heads) {
    if (kernel_head_size(d) != d)
        return encode_page_map_narrow(tk, k, d, hkv, num_blocks, box_heads) &&
               encode_page_map_narrow(tv, v, d, hkv, num_blocks, box_heads);
    return encode_page_map(tk, k, d, hkv, num_blocks, eb, box_heads) &&
           encode_page_map(tv, v, d, hkv, num_blocks, eb, box_heads);
}

static bool aligned(const void *p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// A host-planned call is not captured into a CUDA graph: its plan, grid
// sizes and plan copy are fixed by this batch's host lengths, and a replay
// would run them against whatever batch the buffers hold by then.  Called
// after the host-side checks and before anything is enqueued.
static ua_status refuse_capture(cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return UA_ERR_UNSUPPORTED;
    }
    return cs == cudaStreamCaptureStatusNone ? UA_OK : UA_ERR_UNSUPPORTED;
}

// Whether the prefill rows of this call may run on SM pairs: head size 128
// (long items), 256 (every item: the one-SM kernel is built for 64 and 128).
static bool use_pair_prefill(int32_t head_size) {
    return kPairPrefill && (head_size == 128 || head_size == 256);
}

// The prefill scheduling options of a call: long items on SM pairs
// (two-SM kernel, head size 128), or else claimed by the one-SM CTAs as they
// go (head size 128 with a positive scale); the planner decides per batch.
// An e4m3 cache's prefill rows read a bf16 copy of their pages that the call
// decodes first (ua_pages.cu), so they take the same kernels.
static void configure_prefill(Problem &pr, bool scale_positive, int kv_fp8) {
    pr.prefill_pair = use_pair_prefill(pr.d);
    pr.prefill_claim = !pr.prefill_pair && pr.d == 128 && scale_positive;
    pr.dequant_prefill = kv_fp8 != 0;
}

// Workspace bytes of the block table expanded to 16-token pages (pages of
// block_size = 16 r tokens); 0 for 16-token pages.
static size_t expanded_table_bytes(int32_t num_seqs, int32_t stride, int32_t block_size) {
    if (block_size == kBlockSize || num_seqs <= 0 || stride <= 0) return 0;
    const size_t n = (size_t)num_seqs * (size_t)stride * (size_t)(block_size / kBlockSize);
    return (n * sizeof(int32_t) + kAlign - 1) / kAlign * kAlign;
}

}  // namespace ua

using namespace ua;

extern "C" const char *ua_status_string(ua_status s) {
    switch (s) {
        case UA_OK: return "UA_OK";
        case UA_ERR_INVALID_ARG: return "UA_ERR_INVALID_ARG";
        case UA_ERR_UNSUPPORTED: return "UA_ERR_UNSUPPORTED";
        case UA_ERR_WORKSPACE: return "UA_ERR_WORKSPACE";
        case UA_ERR_CUDA: return "UA_ERR_CUDA";
        case UA_ERR_DEVICE_CHECK: return "UA_ERR_DEVICE_CHECK";
    }
    return "UA_ERR_UNKNOWN";
}

static Problem make_problem(const int32_t *cu, const int32_t *lk, int32_t num_seqs, int32_t hq,
                            int32_t hkv, int32_t d, int32_t bs, int32_t bt_stride,
                            int32_t causal) {
    Problem p;
    p.cu = cu;
    p.lk = lk;
    p.num_seqs = num_seqs;
    p.hq = hq;
    p.hkv = hkv;
    p.d = d;
    p.bs = bs;
    p.bt_stride = bt_stride;
    p.causal = causal != 0;
    // heads narrower than 128 columns: decode units of two adjacent kv heads,
    // whose rows of a slot are one run of the cache (see the decode kernel)
    if (kernel_head_size(d) != d) p.kv_heads_per_unit = 2;
    p.split_sms = true;
    return p;
}

// The problem as the kernels see it: 16-token pages, a block table r times as
// wide (the plan of a call with larger pages is built on that view).
static void to_16_token_pages(Problem &p) {
    if (p.bs == kBlockSize) return;
    p.bt_stride *= p.bs / kBlockSize;
    p.bs = kBlockSize;
}

extern "C" ua_status ua_workspace_size(const int32_t *cu_seqlens_q_host,
                                       const int32_t *seqused_k_host, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_size, int32_t block_size,
                                       int32_t block_table_stride, int32_t causal,
                                       size_t *bytes) {
    if (!bytes) return UA_ERR_INVALID_ARG;
    Problem pr = make_problem(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                              num_kv_heads, head_size, block_size, block_table_stride, causal);
    int v = validate_problem(pr);
    if (v) return static_cast<ua_status>(v);
    to_16_token_pages(pr);
    DeviceState *ds = nullptr;
    ua_status st = device_state(&ds);
    if (st != UA_OK) return st;
    // items dealt in advance (the plan of either sign of the scale fits in this)
    configure_prefill(pr, false, 0);
    thread_local Plan plan;
    build_plan(pr, ds->sms, kPrefillEnabled, plan);
    *bytes = plan.layout.total_bytes + expanded_table_bytes(num_seqs, block_table_stride, block_size);
    return UA_OK;
}

extern "C" ua_status ua_workspace_size_fp8kv(const int32_t *cu_seqlens_q_host,
                                             const int32_t *seqused_k_host, int32_t num_seqs,
                                             int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_size, int32_t block_size,
                                             int32_t block_table_stride, int32_t causal,
                                             size_t *bytes) {
    if (!bytes) return UA_ERR_INVALID_ARG;
    Problem pr = make_problem(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                              num_kv_heads, head_size, block_size, block_table_stride, causal);
    pr.kv_heads_per_unit = 2;
    int v = validate_problem(pr);
    if (v) return static_cast<ua_status>(v);
    if (head_size != 128) return UA_ERR_UNSUPPORTED;
    to_16_token_pages(pr);
    DeviceState *ds = nullptr;
    ua_status st = device_state(&ds);
    if (st != UA_OK) return st;
    // items dealt in advance (the plan of either sign of the scale fits in this),
    // the decoded bf16 copy of the prefill sequences' pages included
    configure_prefill(pr, false, 1);
    thread_local Plan plan;
    build_plan(pr, ds->sms, kPrefillEnabled, plan);
    *bytes = plan.layout.total_bytes + expanded_table_bytes(num_seqs, block_table_stride, block_size);
    return UA_OK;
}

extern "C" ua_status ua_plan_inspect(const int32_t *cu_seqlens_q_host,
                                     const int32_t *seqused_k_host, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int32_t block_table_stride,
                                     int32_t causal, int32_t num_sms, int32_t *counts,
                                     int32_t *items, int64_t items_cap, int64_t *n_items) {
    if (!counts || num_sms <= 0) return UA_ERR_INVALID_ARG;
    Problem pr = make_problem(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                              num_kv_heads, head_size, block_size, block_table_stride, causal);
    configure_prefill(pr, true, 0);   // as a call with a positive softmax scale
    int v = validate_problem(pr);
    if (v) return static_cast<ua_status>(v);
    thread_local Plan plan;
    build_plan(pr, num_sms, kPrefillEnabled, plan);
    counts[0] = plan.dec_ctas;
    counts[1] = (int32_t)plan.pieces.size();
    counts[2] = (int32_t)plan.comb.size();
    counts[3] = plan.n_slots;
    counts[4] = (int32_t)plan.tiles.size();
    counts[5] = plan.pre_ctas;
    counts[6] = (int32_t)std::min<int64_t>(plan.dec_pages, INT32_MAX);
    counts[7] = (int32_t)std::min<size_t>(plan.layout.total_bytes, (size_t)INT32_MAX);
    counts[8] = plan.split_pre_sms;
    const int64_t need = 2 * (int64_t)plan.pieces.size() + (int64_t)plan.tiles.size() +
                         (int64_t)plan.comb.size();
    if (n_items) *n_items = need;
    if (!items) return UA_OK;
    int64_t row = 0;
    auto put = [&](int32_t a, int32_t b, int32_t c, int32_t d, int32_t e, int32_t f, int32_t g,
                   int32_t h) {
        if (row >= items_cap) return;
        int32_t *r = items + 8 * row;
        r[0] = a; r[1] = b; r[2] = c; r[3] = d; r[4] = e; r[5] = f; r[6] = g; r[7] = h;
        ++row;
    };
    for (int c = 0; c < plan.dec_ctas; ++c)
        for (int i = plan.cta_begin[c]; i < plan.cta_begin[c + 1]; ++i) {
            const DecPiece &pc = plan.pieces[i];
            put(0, c, pc.seq, pc.kvh, pc.row0, pc.nrows, pc.page_begin, pc.page_end);
            put(1, pc.slot, pc.unit, 0, 0, 0, 0, 0);
        }
    for (size_t i = 0; i < plan.tiles.size(); ++i) {
        const PreTile &t = plan.tiles[i];
        const int32_t cta = plan.pre_claimed
                                ? -1
                                : (int32_t)(std::upper_bound(plan.pre_begin.begin(), plan.pre_begin.end(),
                                                             (int32_t)i) - plan.pre_begin.begin()) - 1;
        put(2, cta, t.seq, t.kvh, t.row0, t.nrows, t.kv_tiles, (int32_t)i);
    }
    for (const CombUnit &u : plan.comb)
        put(3, u.seq, u.kvh, u.row0, u.nrows, u.slot_begin, u.nslots, 0);
    return UA_OK;
}

extern "C" ua_status ua_device_status(int32_t *code) {
    if (!code) return UA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_ua_device_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    *code = value;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_ua_device_status, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
        return UA_ERR_DEVICE_CHECK;
    }
    return UA_OK;
}

extern "C" ua_status ua_test_set_wait_limit(uint64_t limit_ns) {
    g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
    return UA_OK;
}

extern "C" ua_status ua_profile_enable(int32_t enable) {
    std::lock_guard<std::mutex> lock(g_mutex);
    g_profile = enable != 0;
    return UA_OK;
}

extern "C" ua_status ua_profile_read(int32_t calls_back, float *ms, int32_t *launches) {
    if (!ms || !launches) return UA_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    ua_status st = device_state(&ds);
    if (st != UA_OK) return st;
    if (calls_back < 0 || calls_back >= std::min<int64_t>(ds->calls, UA_PROFILE_RING))
        return UA_ERR_INVALID_ARG;
    const int slot = (int)((ds->calls - 1 - calls_back) % UA_PROFILE_RING);
    if (cudaEventSynchronize(ds->ev[slot][4]) != cudaSuccess) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    // ev 0 before the plan copy, 1 after it, 2 after decode, 3 after prefill, 4 after combine
    // a call whose kernels ran side by side: both timed from the fork (event 1)
    const int from[4] = {1, ds->split[slot] ? 1 : 2, 3, 0};
    const int to[4] = {2, 3, 4, 1};
    for (int i = 0; i < 4; ++i) {
        ms[i] = -1.f;
        launches[i] = 0;
        if (!ds->ran[slot][i]) continue;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, ds->ev[slot][from[i]], ds->ev[slot][to[i]]) != cudaSuccess) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
        ms[i] = t;
        launches[i] = ds->launches[slot][i];
    }
    return UA_OK;
}

namespace ua {

ua_status run_attention(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                        const int32_t *block_table, float softmax_scale, int32_t causal, void *out,
                        const int32_t *cu_seqlens_q_host, const int32_t *seqused_k_host,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_size, int32_t block_size, int32_t num_blocks,
                        int32_t block_table_stride, void *workspace, size_t workspace_bytes,
                        void *stream_ptr, bool pinned_plan, float *lse, int kv_fp8, float k_scale,
                        float v_scale) {
    // Pages of block_size = 16 r tokens: the same memory is a cache of 16-token
    // pages; expand the block table into the front of the workspace and run
    // the call on that view.
    if (block_size != kBlockSize) {
        Problem chk = make_problem(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                                   num_kv_heads, head_size, block_size, block_table_stride, causal);
        const int v = validate_problem(chk);
        if (v) return static_cast<ua_status>(v);
        if (num_seqs == 0 || cu_seqlens_q_host[num_seqs] == 0) return UA_OK;
        const int32_t r = block_size / kBlockSize;
        if (!block_table || num_blocks <= 0 ||
            (int64_t)num_blocks * block_size >= ((int64_t)1 << 31))
            return UA_ERR_INVALID_ARG;
        const size_t xb = expanded_table_bytes(num_seqs, block_table_stride, block_size);
        if (!workspace || workspace_bytes < xb || !aligned(workspace, kAlign)) return UA_ERR_WORKSPACE;
        int32_t *xbt = static_cast<int32_t *>(workspace);
        const ua_status cap = refuse_capture(static_cast<cudaStream_t>(stream_ptr));
        if (cap != UA_OK) return cap;
        if (launch_expand_block_table(block_table, xbt, (int64_t)num_seqs * block_table_stride, r,
                                      num_blocks, static_cast<cudaStream_t>(stream_ptr)) != cudaSuccess) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
        return run_attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, xbt, softmax_scale, causal,
                             out, cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                             num_kv_heads, head_size, kBlockSize, num_blocks * r,
                             block_table_stride * r, static_cast<uint8_t *>(workspace) + xb,
                             workspace_bytes - xb, stream_ptr, pinned_plan, lse, kv_fp8, k_scale,
                             v_scale);
    }
    // ---- host-side checks, before any CUDA call
    Problem pr = make_problem(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                              num_kv_heads, head_size, block_size, block_table_stride, causal);
    // e4m3 pages: decode units take two adjacent kv heads (256-byte rows per slot)
    if (kv_fp8) pr.kv_heads_per_unit = 2;
    // the entry point that must allocate nothing creates no second stream either:
    // its two kernels run one after the other (its plan is sized that way)
    if (!pinned_plan) pr.split_sms = false;
    int v = validate_problem(pr);
    if (v) return static_cast<ua_status>(v);
    if (!std::isfinite(softmax_scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return UA_ERR_INVALID_ARG;
    if (kv_fp8 && head_size != 128) return UA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return UA_OK;
    const int64_t total_q = cu_seqlens_q_host[num_seqs];
    if (total_q == 0) return UA_OK;
    if (!q || !k_cache || !v_cache || !out || !cu_seqlens_q || !seqused_k || !block_table)
        return UA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(lse, 4))
        return UA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || (int64_t)num_blocks * block_size >= ((int64_t)1 << 31))
        return UA_ERR_INVALID_ARG;
    if (total_q >= ((int64_t)1 << 31)) return UA_ERR_INVALID_ARG;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    ua_status st = refuse_capture(stream);
    if (st != UA_OK) return st;
    DeviceState *ds = nullptr;
    st = device_state(&ds);
    if (st != UA_OK) return st;

    // ---- partition pass
    thread_local Plan plan;
    thread_local std::vector<uint8_t> blob;
    configure_prefill(pr, softmax_scale * k_scale > 0.f, kv_fp8);
    build_plan(pr, ds->sms, kPrefillEnabled, plan);
    const bool pair_prefill = plan.pre_pair;
    const Layout &L = plan.layout;
    if (L.total_bytes > 0) {
        if (!workspace || workspace_bytes < L.total_bytes || !aligned(workspace, kAlign))
            return UA_ERR_WORKSPACE;
    }
    if (!pinned_plan) serialize_plan(plan, blob);

    // ---- tensor maps: K/V page views (5-D), Q as [total_q, Hq, D]
    const int g = num_q_heads / num_kv_heads;
    CUtensorMap tm_kp, tm_vp, tm_q, tm_o, tm_k3, tm_vh;
    const int eb = kv_fp8 ? 1 : 2;
    const int box_heads = plan.dec_heads_per_unit;   // 2 only for e4m3 pages and narrower heads
                                                     // (no prefill tiles for either)
    if (!encode_decode_maps(&tm_kp, &tm_vp, k_cache, v_cache, head_size, num_kv_heads,
                            (uint64_t)num_blocks, eb, box_heads))
        return UA_ERR_CUDA;
    // prefill: Q tiles (loads) and out tiles (stores) as [total_q, Hq, D], and K as
    // [num_blocks * 16, Hkv, D] with one box per 64 columns.  With an e4m3 cache
    // the prefill kernels read the bf16 copy of their sequences' pages that the
    // call decodes into the workspace, through its own block table.
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const bool dq = plan.dq_pages > 0;
    const void *k_pre = dq ? static_cast<const void *>(ws + L.off_dq_k) : k_cache;
    const void *v_pre = dq ? static_cast<const void *>(ws + L.off_dq_v) : v_cache;
    const int32_t *bt_pre = dq ? reinterpret_cast<const int32_t *>(ws + L.off_dq_bt) : block_table;
    const int64_t blocks_pre = dq ? plan.dq_pages : num_blocks;
    CUtensorMap tm_vpre = tm_vp, tm_kpre_unused;
    if (!plan.tiles.empty() &&
        (!encode_map(&tm_q, q, head_size, num_q_heads, (uint64_t)total_q, g, kPreRows / g) ||
         !encode_map(&tm_o, out, head_size, num_q_heads, (uint64_t)total_q, g, kPreRows / g) ||
         !encode_map(&tm_k3, k_pre, head_size, num_kv_heads, (uint64_t)blocks_pre * block_size, 1,
                     kBlockSize)))
        return UA_ERR_CUDA;
    if (!plan.tiles.empty() && dq && !pair_prefill &&
        !encode_decode_maps(&tm_kpre_unused, &tm_vpre, k_pre, v_pre, head_size, num_kv_heads,
                            (uint64_t)blocks_pre, 2, 1))
        return UA_ERR_CUDA;
    if (!plan.tiles.empty() && pair_prefill &&
        !encode_page_map(&tm_vh, v_pre, head_size, num_kv_heads, (uint64_t)blocks_pre, 2, 1, head_size / 128))
        return UA_ERR_CUDA;

    const bool prof = g_profile;
    if (prof && !ds->events) {
        for (int c = 0; c < UA_PROFILE_RING; ++c)
            for (int i = 0; i < 5; ++i)
                if (cudaEventCreate(&ds->ev[c][i]) != cudaSuccess) {
                    cudaGetLastError();
                    return UA_ERR_CUDA;
                }
        ds->events = true;
    }
    const int pslot = (int)(ds->calls % UA_PROFILE_RING);
    auto mark = [&](int i) {
        if (prof) cudaEventRecord(ds->ev[pslot][i], stream);
    };
    const float scale_log2 = softmax_scale * k_scale * 1.4426950408889634f;

    mark(0);
    // The plan: in a device buffer of the library's ring (pinned_plan), or at
    // the start of the workspace, copied in stream order from pageable memory
    // (which allocates nothing).  Once a ring slot is taken, every way out of
    // this call gives it back behind whatever kernels the call launched.
    struct SlotGuard {
        int dev = -1, slot = -1;
        cudaStream_t stream = nullptr;
        ~SlotGuard() {
            if (slot >= 0) release_plan_slot(dev, slot, stream);
        }
    } guard;
    uint8_t *pl = ws;
    if (L.blob_bytes > 0) {
        if (pinned_plan) {
            int slot = -1;
            st = stage_plan(ds->dev, plan, stream, &pl, &slot);
            if (st != UA_OK) return st;
            guard.dev = ds->dev;
            guard.slot = slot;
            guard.stream = stream;
        } else if (cudaMemcpyAsync(ws, blob.data(), L.blob_bytes, cudaMemcpyHostToDevice,
                                   stream) != cudaSuccess) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
    }
    mark(1);
    cudaError_t e = cudaSuccess;
    auto launch_dec = [&](cudaStream_t s) -> ua_status {
        if (plan.dec_ctas > 0) {
            DecodeParams dp{};
            dp.q = static_cast<const __nv_bfloat16 *>(q);
            dp.out = static_cast<__nv_bfloat16 *>(out);
            dp.cu = cu_seqlens_q;
            dp.seqused_k = seqused_k;
            dp.block_table = block_table;
            dp.bt_stride = block_table_stride;
            dp.num_blocks = num_blocks;
            dp.hq = num_q_heads;
            dp.hkv = num_kv_heads;
            dp.g = g;
            dp.causal = causal != 0;
            dp.scale_log2 = scale_log2;
            dp.cta_begin = reinterpret_cast<const int32_t *>(pl + L.off_cta);
            dp.pieces = reinterpret_cast<const DecPiece *>(pl + L.off_pieces);
            dp.part_o = reinterpret_cast<float *>(ws + L.off_part_o);
            dp.part_ml = reinterpret_cast<float *>(ws + L.off_part_ml);
            dp.comb = reinterpret_cast<const CombUnit *>(pl + L.off_comb);
            dp.comb_count = reinterpret_cast<int32_t *>(pl + L.off_comb_count);
            dp.lse = lse;
            dp.v_scale = v_scale;
            dp.heads_per_unit = plan.dec_heads_per_unit;
            dp.status = ds->status;
            dp.wait_ns = wait_limit_ns();
            dp.dq = head_size;
            e = launch_decode(head_size, kv_fp8 != 0, dp, tm_kp, tm_vp, plan.dec_ctas, s);
            if (e != cudaSuccess) return UA_ERR_CUDA;
        }
        return UA_OK;
    };
    auto launch_pre = [&](cudaStream_t s) -> ua_status {
        if (!plan.tiles.empty()) {
            if (dq) {
                e = launch_dequant_pages(k_cache, v_cache, block_table, block_table_stride, num_blocks,
                                         reinterpret_cast<const int32_t *>(pl + L.off_dq),
                                         (int32_t)plan.dq_seq.size(), plan.dq_pages,
                                         reinterpret_cast<int32_t *>(ws + L.off_dq_bt), ws + L.off_dq_k,
                                         ws + L.off_dq_v, num_kv_heads, head_size, ds->status, s);
                if (e != cudaSuccess) return UA_ERR_CUDA;
            }
            PrefillParams pp{};
            pp.k_cache = static_cast<const __nv_bfloat16 *>(k_pre);
            pp.out = static_cast<__nv_bfloat16 *>(out);
            pp.lse = lse;
            pp.cu = cu_seqlens_q;
            pp.seqused_k = seqused_k;
            pp.block_table = bt_pre;
            pp.bt_stride = block_table_stride;
            pp.num_blocks = (int32_t)blocks_pre;
            pp.v_scale = v_scale;
            pp.hq = num_q_heads;
            pp.hkv = num_kv_heads;
            pp.g = g;
            pp.causal = causal != 0;
            pp.scale_log2 = scale_log2;
            pp.tiles = reinterpret_cast<const PreTile *>(pl + L.off_tiles);
            pp.tile_begin = reinterpret_cast<const int32_t *>(pl + L.off_pre_begin);
            pp.sched = reinterpret_cast<int32_t *>(pl + L.off_sched);
            pp.n_tiles = (int32_t)plan.tiles.size();
            pp.status = ds->status;
            e = pair_prefill ? launch_prefill_pair(head_size, pp, tm_q, tm_o, tm_k3, tm_vh, plan.pre_ctas, s)
                             : launch_prefill(head_size, plan.pre_claimed, pp, tm_q, tm_o, tm_k3, tm_vpre,
                                              plan.pre_ctas, s);
            if (e != cudaSuccess) return UA_ERR_CUDA;
        }
        return UA_OK;
    };
    const bool split = plan.split_pre_sms > 0;
    if (split) {
        // side by side: the prefill kernel first (its CTAs take their SMs), the
        // decode kernel on the library's second stream (the rest of the SMs)
        st = side_stream(ds);
        if (st != UA_OK) return st;
        {
            std::lock_guard<std::mutex> lock(ds->side_mutex);
            if (cudaEventRecord(ds->fork, stream) != cudaSuccess ||
                cudaStreamWaitEvent(ds->side, ds->fork, 0) != cudaSuccess) {
                cudaGetLastError();
                return UA_ERR_CUDA;
            }
        }
        st = launch_pre(stream);
        if (st != UA_OK) return st;
        mark(3);
        st = launch_dec(ds->side);
        if (st != UA_OK) return st;
        if (prof) cudaEventRecord(ds->ev[pslot][2], ds->side);
        std::lock_guard<std::mutex> lock(ds->side_mutex);
        if (cudaEventRecord(ds->join, ds->side) != cudaSuccess ||
            cudaStreamWaitEvent(stream, ds->join, 0) != cudaSuccess) {
            cudaGetLastError();
            return UA_ERR_CUDA;
        }
    } else {
        st = launch_dec(stream);
        if (st != UA_OK) return st;
        mark(2);
        st = launch_pre(stream);
        if (st != UA_OK) return st;
        mark(3);
    }
    // (split units are merged inside the decode kernel: no separate combine step)
    mark(4);
    if (guard.slot >= 0) {
        const int slot = guard.slot;
        guard.slot = -1;
        st = release_plan_slot(ds->dev, slot, stream);
        if (st != UA_OK) return st;
    }
    if (prof) {
        std::lock_guard<std::mutex> lock(g_mutex);
        ds->ran[pslot][0] = plan.dec_ctas > 0;
        ds->ran[pslot][1] = !plan.tiles.empty();
        ds->ran[pslot][2] = false;
        ds->ran[pslot][3] = L.blob_bytes > 0;
        ds->split[pslot] = split;
        ds->launches[pslot][0] = plan.dec_ctas > 0 ? 1 : 0;
        ds->launches[pslot][1] = plan.tiles.empty() ? 0 : (dq ? 2 : 1);   // page decode + prefill
        ds->launches[pslot][2] = 0;
        ds->launches[pslot][3] = 0;
        ++ds->calls;
    }
    return UA_OK;
}

}  // namespace ua

extern "C" ua_status unified_attention(const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                                       const int32_t *block_table, float softmax_scale,
                                       int32_t causal, void *out,
                                       const int32_t *cu_seqlens_q_host,
                                       const int32_t *seqused_k_host, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_size, int32_t block_size, int32_t num_blocks,
                                       int32_t block_table_stride, void *workspace,
                                       size_t workspace_bytes, void *stream) {
    return ua::run_attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                             softmax_scale, causal, out, cu_seqlens_q_host, seqused_k_host,
                             num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                             num_blocks, block_table_stride, workspace, workspace_bytes, stream,
                             /*pinned_plan=*/true, /*lse=*/nullptr);
}

extern "C" ua_status unified_attention_lse(const void *q, const void *k_cache, const void *v_cache,
                                           const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                                           const int32_t *block_table, float softmax_scale,
                                           int32_t causal, void *out, float *lse,
                                           const int32_t *cu_seqlens_q_host,
                                           const int32_t *seqused_k_host, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_size, int32_t block_size, int32_t num_blocks,
                                           int32_t block_table_stride, void *workspace,
                                           size_t workspace_bytes, void *stream) {
    if (lse == nullptr) return UA_ERR_INVALID_ARG;
    return ua::run_attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                             softmax_scale, causal, out, cu_seqlens_q_host, seqused_k_host,
                             num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                             num_blocks, block_table_stride, workspace, workspace_bytes, stream,
                             /*pinned_plan=*/true, lse);
}

extern "C" ua_status ua_kv_append(const void *k_new, const void *v_new, const int32_t *cu_seqlens_q,
                                  const int32_t *seqused_k, const int32_t *block_table,
                                  void *k_cache, void *v_cache, const int32_t *cu_seqlens_q_host,
                                  const int32_t *seqused_k_host, int32_t num_seqs,
                                  int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  int32_t num_blocks, int32_t block_table_stride, void *stream) {
    // the attention call's checks with causal = 1 (every sequence has Lq <= Lk:
    // its new tokens fit in its context)
    Problem pr = make_problem(cu_seqlens_q_host, seqused_k_host, num_seqs, num_kv_heads,
                              num_kv_heads, head_size, block_size, block_table_stride, 1);
    const int v = validate_problem(pr);
    if (v) return static_cast<ua_status>(v);
    if (num_seqs == 0 || cu_seqlens_q_host[num_seqs] == 0) return UA_OK;
    if (!k_new || !v_new || !cu_seqlens_q || !seqused_k || !block_table || !k_cache || !v_cache)
        return UA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return UA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || (int64_t)num_blocks * block_size >= ((int64_t)1 << 31)) return UA_ERR_INVALID_ARG;
    if ((int64_t)num_kv_heads * head_size > 2048) return UA_ERR_UNSUPPORTED;
    DeviceState *ds = nullptr;
    ua_status st = device_state(&ds);
    if (st != UA_OK) return st;
    if (launch_kv_append(k_new, v_new, cu_seqlens_q, seqused_k, block_table, k_cache, v_cache,
                         num_seqs, cu_seqlens_q_host[num_seqs], num_kv_heads, head_size, block_size,
                         num_blocks, block_table_stride, ds->status,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return UA_ERR_CUDA;
    }
    return UA_OK;
}

extern "C" ua_status unified_attention_append(
    const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
    const int32_t *cu_seqlens_q, const int32_t *seqused_k, const int32_t *block_table,
    float softmax_scale, int32_t causal, void *out, const int32_t *cu_seqlens_q_host,
    const int32_t *seqused_k_host, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_size, int32_t block_size, int32_t num_blocks, int32_t block_table_stride,
    void *workspace, size_t workspace_bytes, void *stream) {
    // everything the attention call checks, first, so that a rejected call writes nothing
    Problem pr = make_problem(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                              num_kv_heads, head_size, block_size, block_table_stride, causal);
    const int v = validate_problem(pr);
    if (v) return static_cast<ua_status>(v);
    size_t need = 0;
    ua_status st = ua_workspace_size(cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                                     num_kv_heads, head_size, block_size, block_table_stride,
                                     causal, &need);
    if (st != UA_OK) return st;
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, kAlign)))
        return UA_ERR_WORKSPACE;
    if (!std::isfinite(softmax_scale) || !q || !out || !aligned(q, 16) || !aligned(out, 16))
        return UA_ERR_INVALID_ARG;
    st = refuse_capture(static_cast<cudaStream_t>(stream));
    if (st != UA_OK) return st;
    st = ua_kv_append(k_new, v_new, cu_seqlens_q, seqused_k, block_table, k_cache, v_cache,
                      cu_seqlens_q_host, seqused_k_host, num_seqs, num_kv_heads, head_size,
                      block_size, num_blocks, block_table_stride, stream);
    if (st != UA_OK) return st;
    return unified_attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table, softmax_scale,
                             causal, out, cu_seqlens_q_host, seqused_k_host, num_seqs, num_q_heads,
                             num_kv_heads, head_size, block_size, num_blocks, block_table_stride,
                             workspace, workspace_bytes, stream);
}

extern "C" ua_status unified_attention_fp8kv(
    const void *q, const void *k_cache, const void *v_cache, float k_scale, float v_scale,
    const int32_t *cu_seqlens_q, const int32_t *seqused_k, const int32_t *block_table,
    float softmax_scale, int32_t causal, void *out, float *lse, const int32_t *cu_seqlens_q_host,
    const int32_t *seqused_k_host, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_size, int32_t block_size, int32_t num_blocks, int32_t block_table_stride,
    void *workspace, size_t workspace_bytes, void *stream) {
    return ua::run_attention(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                             softmax_scale, causal, out, cu_seqlens_q_host, seqused_k_host,
                             num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                             num_blocks, block_table_stride, workspace, workspace_bytes, stream,
                             /*pinned_plan=*/true, lse, /*kv_fp8=*/1, k_scale, v_scale);
}

// ---------------------------------------------------------------------------
// Calls planned on the device (no host copies of the lengths; graph-capturable)

namespace ua {

// Host-side checks of a device-plan call's shapes; fills the workspace shape.
static ua_status device_plan_shape(int32_t num_seqs, int32_t max_total_q, int32_t max_seq_q,
                                   int32_t hq, int32_t hkv, int32_t d, int32_t bs,
                                   int32_t bt_stride, int32_t kv_fp8, int sms, DevPlanShape *s) {
    if (num_seqs < 0 || max_total_q < 0 || max_seq_q < 0 || hq <= 0 || hkv <= 0 || bt_stride < 0)
        return UA_ERR_INVALID_ARG;
    if (hq % hkv != 0 || !head_size_supported(d)) return UA_ERR_UNSUPPORTED;
    if (bs <= 0 || bs % kBlockSize != 0 || bs > kMaxBlockSize) return UA_ERR_UNSUPPORTED;
    if (kv_fp8 && d != 128) return UA_ERR_UNSUPPORTED;
    if ((int64_t)bt_stride * (bs / kBlockSize) > INT32_MAX / 4) return UA_ERR_INVALID_ARG;
    if ((int64_t)max_total_q * (hq / hkv) > INT32_MAX / 2) return UA_ERR_INVALID_ARG;
    Problem pr = make_problem(nullptr, nullptr, 0, hq, hkv, d, kBlockSize, bt_stride, 1);
    s->page_ratio = bs / kBlockSize;
    s->num_seqs = num_seqs;
    s->max_total_q = max_total_q;
    s->max_seq_q = (max_seq_q == 0 || max_seq_q > max_total_q) ? max_total_q : max_seq_q;
    s->hq = hq;
    s->hkv = hkv;
    s->d = d;
    s->bt_stride = bt_stride * s->page_ratio;   // in 16-token pages
    s->hpu = ((kv_fp8 || kernel_head_size(d) != d) && hkv % 2 == 0) ? 2 : 1;
    // no sequence can fill more than one decode tile: the prefill kernel never has work
    const bool can_prefill = (int64_t)s->max_seq_q * (hq / hkv) > kDecRows;
    s->prefill_ok = (kPrefillEnabled && !kv_fp8 && can_prefill && prefill_supports(pr)) ? 1 : 0;
    s->num_sms = sms;
    // dealt to one SM per item: the kernel is fixed at capture, before the
    // batch (and so its item lengths) is known
    s->pre_pair = 0;
    s->pre_workers = sms;
    return UA_OK;
}

static ua_status run_attention_device_plan(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *cu_seqlens_q,
    const int32_t *seqused_k, const int32_t *block_table, float softmax_scale, int32_t causal,
    void *out, float *lse, int32_t num_seqs, int32_t max_total_q, int32_t max_seq_q,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
    int32_t num_blocks, int32_t block_table_stride, int32_t kv_fp8, float k_scale, float v_scale,
    void *workspace, size_t workspace_bytes, void *stream_ptr, int mode) {
    // mode 0: plan, then attend; 1: plan only; 2: attend with the plan already
    // in the workspace (built by an earlier call on the same metadata)
    const bool plan_only = mode == 1;
    DeviceState *ds = nullptr;
    ua_status st = device_state(&ds);
    if (st != UA_OK) return st;
    DevPlanShape shape{};
    st = device_plan_shape(num_seqs, max_total_q, max_seq_q, num_q_heads, num_kv_heads, head_size,
                           block_size, block_table_stride, kv_fp8, ds->sms, &shape);
    if (st != UA_OK) return st;
    if (!std::isfinite(softmax_scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return UA_ERR_INVALID_ARG;
    if (num_seqs == 0 || max_total_q == 0) return UA_OK;
    if (!cu_seqlens_q || !seqused_k) return UA_ERR_INVALID_ARG;
    if (!plan_only) {
        if (!q || !k_cache || !v_cache || !out || !block_table) return UA_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
            !aligned(lse, 4))
            return UA_ERR_INVALID_ARG;
        if (num_blocks <= 0 || (int64_t)num_blocks * block_size >= ((int64_t)1 << 31))
            return UA_ERR_INVALID_ARG;
    }
    const DevPlanLayout L = device_plan_layout(shape);
    if (!L.valid) return UA_ERR_UNSUPPORTED;
    // pages of 16 r tokens: the block table expanded to 16-token pages, after
    // the plan's sections
    const size_t xb = expanded_table_bytes(num_seqs, block_table_stride, block_size);
    if (!workspace || workspace_bytes < L.total_bytes + xb || !aligned(workspace, kAlign))
        return UA_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (plan_only) {
        if (launch_device_plan(shape, L, cu_seqlens_q, seqused_k, causal, ws, ds->status, stream) !=
            cudaSuccess)
            return UA_ERR_CUDA;
        return UA_OK;
    }

    if (shape.page_ratio > 1) {
        int32_t *xbt = reinterpret_cast<int32_t *>(ws + L.total_bytes);
        if (launch_expand_block_table(block_table, xbt, (int64_t)num_seqs * block_table_stride,
                                      shape.page_ratio, num_blocks, stream) != cudaSuccess)
            return UA_ERR_CUDA;
        block_table = xbt;
        num_blocks *= shape.page_ratio;
        block_table_stride = shape.bt_stride;
        block_size = kBlockSize;
    }
    // tensor maps over the caller's buffers (q / out sized for max_total_q tokens)
    const int g = num_q_heads / num_kv_heads;
    CUtensorMap tm_kp, tm_vp, tm_q, tm_o, tm_k3, tm_vh;
    const int eb = kv_fp8 ? 1 : 2;
    if (!encode_decode_maps(&tm_kp, &tm_vp, k_cache, v_cache, head_size, num_kv_heads,
                            (uint64_t)num_blocks, eb, shape.hpu))
        return UA_ERR_CUDA;
    if (shape.prefill_ok && shape.pre_pair &&
        !encode_page_map(&tm_vh, v_cache, head_size, num_kv_heads, (uint64_t)num_blocks, 2, 1,
                         std::max(head_size / 128, 1)))
        return UA_ERR_CUDA;
    if (shape.prefill_ok &&
        (!encode_map(&tm_q, q, head_size, num_q_heads, (uint64_t)max_total_q, g, kPreRows / g) ||
         !encode_map(&tm_o, out, head_size, num_q_heads, (uint64_t)max_total_q, g, kPreRows / g) ||
         !encode_map(&tm_k3, k_cache, head_size, num_kv_heads, (uint64_t)num_blocks * block_size, 1,
                     kBlockSize)))
        return UA_ERR_CUDA;

    const bool prof = g_profile;
    if (prof && !ds->events) {
        for (int c = 0; c < UA_PROFILE_RING; ++c)
            for (int i = 0; i < 5; ++i)
                if (cudaEventCreate(&ds->ev[c][i]) != cudaSuccess) {
                    cudaGetLastError();
                    return UA_ERR_CUDA;
                }
        ds->events = true;
    }
    const int pslot = (int)(ds->calls % UA_PROFILE_RING);
    auto mark = [&](int i) {
        if (prof) cudaEventRecord(ds->ev[pslot][i], stream);
    };
    const float scale_log2 = softmax_scale * k_scale * 1.4426950408889634f;

    mark(0);
    if (mode == 0 &&
        launch_device_plan(shape, L, cu_seqlens_q, seqused_k, causal, ws, ds->status, stream) !=
            cudaSuccess)
        return UA_ERR_CUDA;
    mark(1);
    DecodeParams dp{};
    dp.q = static_cast<const __nv_bfloat16 *>(q);
    dp.out = static_cast<__nv_bfloat16 *>(out);
    dp.cu = cu_seqlens_q;
    dp.seqused_k = seqused_k;
    dp.block_table = block_table;
    dp.bt_stride = block_table_stride;
    dp.num_blocks = num_blocks;
    dp.hq = num_q_heads;
    dp.hkv = num_kv_heads;
    dp.g = g;
    dp.causal = causal != 0;
    dp.scale_log2 = scale_log2;
    dp.cta_begin = reinterpret_cast<const int32_t *>(ws + L.off_cta);
    dp.pieces = reinterpret_cast<const DecPiece *>(ws + L.off_pieces);
    dp.part_o = reinterpret_cast<float *>(ws + L.off_part_o);
    dp.part_ml = reinterpret_cast<float *>(ws + L.off_part_ml);
    dp.comb = reinterpret_cast<const CombUnit *>(ws + L.off_comb);
    dp.comb_count = reinterpret_cast<int32_t *>(ws + L.off_comb_count);
    dp.lse = lse;
    dp.v_scale = v_scale;
    dp.heads_per_unit = shape.hpu;
    dp.status = ds->status;
    dp.wait_ns = wait_limit_ns();
    dp.dq = head_size;
    if (launch_decode(head_size, kv_fp8 != 0, dp, tm_kp, tm_vp, L.dec_grid, stream) != cudaSuccess)
        return UA_ERR_CUDA;
    mark(2);
    if (shape.prefill_ok) {
        PrefillParams pp{};
        pp.k_cache = static_cast<const __nv_bfloat16 *>(k_cache);
        pp.out = static_cast<__nv_bfloat16 *>(out);
        pp.lse = lse;
        pp.cu = cu_seqlens_q;
        pp.seqused_k = seqused_k;
        pp.block_table = block_table;
        pp.bt_stride = block_table_stride;
        pp.num_blocks = num_blocks;
        pp.hq = num_q_heads;
        pp.hkv = num_kv_heads;
        pp.g = g;
        pp.causal = causal != 0;
        pp.scale_log2 = scale_log2;
        pp.tiles = reinterpret_cast<const PreTile *>(ws + L.off_tiles);
        pp.tile_begin = reinterpret_cast<const int32_t *>(ws + L.off_pre_begin);
        pp.n_tiles = L.cap_items;
        pp.v_scale = v_scale;
        pp.status = ds->status;
        const cudaError_t pe =
            shape.pre_pair ? launch_prefill_pair(head_size, pp, tm_q, tm_o, tm_k3, tm_vh, shape.pre_workers, stream)
                           : launch_prefill(head_size, /*claimed=*/false, pp, tm_q, tm_o, tm_k3, tm_vp,
                                            shape.num_sms, stream);
        if (pe != cudaSuccess) return UA_ERR_CUDA;
    }
    mark(3);
    mark(4);
    if (prof) {
        std::lock_guard<std::mutex> lock(g_mutex);
        ds->ran[pslot][0] = true;
        ds->ran[pslot][1] = shape.prefill_ok != 0;
        ds->ran[pslot][2] = false;
        ds->ran[pslot][3] = mode == 0;
        ds->launches[pslot][0] = 1;
        ds->launches[pslot][1] = shape.prefill_ok ? 1 : 0;
        ds->launches[pslot][2] = 0;
        ds->launches[pslot][3] = mode == 0 ? 1 : 0;   // the planner kernel
        ++ds->calls;
    }
    return UA_OK;
}

}  // namespace ua

extern "C" ua_status ua_workspace_size_device_plan(int32_t num_seqs, int32_t max_total_q,
                                                   int32_t max_seq_q, int32_t num_q_heads,
                                                   int32_t num_kv_heads, int32_t head_size,
                                                   int32_t block_size, int32_t block_table_stride,
                                                   int32_t kv_fp8, size_t *bytes) {
    if (!bytes) return UA_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    ua_status st = device_state(&ds);
    if (st != UA_OK) return st;
    DevPlanShape shape{};
    st = device_plan_shape(num_seqs, max_total_q, max_seq_q, num_q_heads, num_kv_heads, head_size,
                           block_size, block_table_stride, kv_fp8, ds->sms, &shape);
    if (st != UA_OK) return st;
    const DevPlanLayout L = device_plan_layout(shape);
    if (!L.valid) return UA_ERR_UNSUPPORTED;
    *bytes = L.total_bytes + expanded_table_bytes(num_seqs, block_table_stride, block_size);
    return UA_OK;
}

extern "C" ua_status ua_device_plan_layout(int32_t num_seqs, int32_t max_total_q,
                                           int32_t max_seq_q, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_size,
                                           int32_t block_size, int32_t block_table_stride,
                                           int32_t kv_fp8, int32_t num_sms, int64_t *offsets,
                                           int32_t *caps) {
    if (!offsets || !caps || num_sms <= 0) return UA_ERR_INVALID_ARG;
    DevPlanShape shape{};
    ua_status st = device_plan_shape(num_seqs, max_total_q, max_seq_q, num_q_heads, num_kv_heads,
                                     head_size, block_size, block_table_stride, kv_fp8, num_sms,
                                     &shape);
    if (st != UA_OK) return st;
    const DevPlanLayout L = device_plan_layout(shape);
    if (!L.valid) return UA_ERR_UNSUPPORTED;
    const size_t total = L.total_bytes + expanded_table_bytes(num_seqs, block_table_stride, block_size);
    const size_t off[8] = {L.off_header, L.off_cta,       L.off_pieces,    L.off_comb,
                           L.off_comb_count, L.off_tiles, L.off_pre_begin, total};
    for (int i = 0; i < 8; ++i) offsets[i] = (int64_t)off[i];
    const int32_t cap[8] = {L.dec_grid, L.cap_units, L.cap_items, L.cap_pieces,
                            L.cap_comb, L.cap_slots, L.n_buckets, shape.num_sms};
    for (int i = 0; i < 8; ++i) caps[i] = cap[i];
    return UA_OK;
}

extern "C" ua_status ua_device_plan_build(const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                                          int32_t causal, int32_t num_seqs, int32_t max_total_q,
                                          int32_t max_seq_q, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_size,
                                          int32_t block_size, int32_t block_table_stride,
                                          int32_t kv_fp8, void *workspace, size_t workspace_bytes,
                                          void *stream) {
    return ua::run_attention_device_plan(nullptr, nullptr, nullptr, cu_seqlens_q, seqused_k, nullptr,
                                         1.f, causal, nullptr, nullptr, num_seqs, max_total_q,
                                         max_seq_q, num_q_heads, num_kv_heads, head_size, block_size, 0,
                                         block_table_stride, kv_fp8, 1.f, 1.f, workspace,
                                         workspace_bytes, stream, /*mode=*/1);
}

extern "C" ua_status unified_attention_device_plan(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *cu_seqlens_q,
    const int32_t *seqused_k, const int32_t *block_table, float softmax_scale, int32_t causal,
    void *out, float *lse, int32_t num_seqs, int32_t max_total_q, int32_t max_seq_q,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
    int32_t num_blocks, int32_t block_table_stride, int32_t kv_fp8, float k_scale, float v_scale,
    void *workspace, size_t workspace_bytes, void *stream) {
    return ua::run_attention_device_plan(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                                         softmax_scale, causal, out, lse, num_seqs, max_total_q,
                                         max_seq_q, num_q_heads, num_kv_heads, head_size, block_size,
                                         num_blocks, block_table_stride, kv_fp8, k_scale, v_scale,
                                         workspace, workspace_bytes, stream, /*mode=*/0);
}

extern "C" ua_status unified_attention_device_planned(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *cu_seqlens_q,
    const int32_t *seqused_k, const int32_t *block_table, float softmax_scale, int32_t causal,
    void *out, float *lse, int32_t num_seqs, int32_t max_total_q, int32_t max_seq_q,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
    int32_t num_blocks, int32_t block_table_stride, int32_t kv_fp8, float k_scale, float v_scale,
    void *workspace, size_t workspace_bytes, void *stream) {
    return ua::run_attention_device_plan(q, k_cache, v_cache, cu_seqlens_q, seqused_k, block_table,
                                         softmax_scale, causal, out, lse, num_seqs, max_total_q,
                                         max_seq_q, num_q_heads, num_kv_heads, head_size, block_size,
                                         num_blocks, block_table_stride, kv_fp8, k_scale, v_scale,
                                         workspace, workspace_bytes, stream, /*mode=*/2);
}
