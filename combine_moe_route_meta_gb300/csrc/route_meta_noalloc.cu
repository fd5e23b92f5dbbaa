// route_meta_noalloc.cu -- moe_route_meta for callers that cannot allocate device memory.
//
// moe_route_meta needs a caller-provided scratch buffer once the pairs span several
// thread blocks (the per-block histogram table [B][E]). Some callers
// have no way to provide one: an inference engine that has already reserved the GPU's
// memory for its own pool, a plugin interface that passes in nothing but input and
// output pointers, or a code path where a cudaMalloc (which can synchronise the device)
// is not acceptable. moe_route_meta_noalloc serves them: it routes the same computation
// through a fixed scratch array that lives in this library's own device memory.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes bytes. Every GPU
// that loads the library holds it until the process exits. Its device address is looked
// up once per device, with that device current, on the first call made on that device.
// All calls share the array, so calls whose kernels overlap on the GPU race with each
// other. Nothing in it has to start at zero: the count kernel writes every table cell the
// place kernel reads, so a call never sees what an earlier call left there. No call
// allocates or frees memory, and no call issues anything but the kernels of moe_route_meta.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "moe_dispatch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once per device).
moe_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_route_meta_noalloc(const int32_t* topk_ids, int64_t num_tokens, int topk,
                                               int num_experts, int num_partitions,
                                               int max_tokens_per_expert, int64_t* seg_indptr,
                                               int32_t* src2dst, int32_t* reorder_topk_ids,
                                               int32_t* masked_m, int32_t* partition_counts,
                                               int32_t* expected_m_host, int32_t* dev_status,
                                               moe_stream_t stream) {
    if (num_tokens < 0 || topk < 1 || num_experts < 1) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_route_meta_workspace_size(num_tokens, topk, num_experts);
    if (need > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        moe_status_t st = scratch_address(&scratch);
        if (st != MOE_OK) return st;
    }
    return moe_route_meta(topk_ids, num_tokens, topk, num_experts, num_partitions, max_tokens_per_expert,
                          seg_indptr, src2dst, reorder_topk_ids, masked_m, partition_counts, expected_m_host,
                          scratch, need > 0 ? kNoAllocScratchBytes : 0, dev_status, stream);
}
