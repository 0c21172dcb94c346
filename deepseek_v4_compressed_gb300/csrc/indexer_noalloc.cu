// indexer_noalloc.cu -- dsv4_indexer_topk for callers that cannot allocate
// device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// inside a host runtime whose allocator they do not control (a plugin of a
// serving engine that owns every device allocation, an embedded or
// restricted-process deployment where cudaMalloc is forbidden or pre-budgeted
// to zero), or tools that must not change the device's memory footprint
// while they run.  For them this entry point keeps the indexer's scratch (the
// per-query logits) in a file-scope device array instead of a caller-provided
// workspace.  Every GPU that loads the library holds this array until the
// process exits.
#include <mutex>

#include "dsv4_common.cuh"
#include "plan.h"

namespace {

// Scratch for the logits of one call: batch x max_slots fp32 values, i.e. up to
// 1,048,576 logits (batch 32 at context 131072, batch 4 at context 1M).
constexpr size_t kNoAllocScratchBytes = 4u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code cannot use the array's name as a device pointer).
dsv4_status scratch_for_current_device(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSV4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_dev[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return DSV4_ERR_CUDA;
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return DSV4_OK;
}

}  // namespace

extern "C" dsv4_status dsv4_indexer_topk_noalloc(const dsv4_plan* plan, const dsv4_indexer_args* args,
                                                 dsv4_stream_t stream)
{
    if (plan == nullptr || args == nullptr) return DSV4_ERR_INVALID;
    if (plan->ws_bytes > kNoAllocScratchBytes) return DSV4_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const dsv4_status s = scratch_for_current_device(&scratch);
    if (s != DSV4_OK) return s;
    // The logits region needs no clearing: every logit a call reads is written
    // by the same call first.
    return dsv4_indexer_topk(plan, args, scratch, kNoAllocScratchBytes, stream);
}
