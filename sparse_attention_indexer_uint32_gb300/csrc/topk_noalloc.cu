// topk_noalloc.cu -- topk_transform_noalloc: plan + select + transform for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs where an allocation would break an allocator's or a framework's
// accounting, or a plugin that only receives input and output pointers from
// its host.  This entry point runs the same kernels as topk_plan +
// topk_transform, but the plan's work lists live in a fixed array in device
// memory that belongs to this library.  Every GPU that loads the library
// holds that array (kNoAllocWorkspaceBytes) until the process exits.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "topk_internal.h"
#include "topkidx.h"

namespace topkidx {
namespace {

constexpr int32_t kNoAllocMaxBatch = TOPK_NOALLOC_MAX_BATCH;
constexpr size_t kNoAllocWorkspaceBytes = plan_bytes(kNoAllocMaxBatch);

// The shared scratch: one plan workspace for up to kNoAllocMaxBatch rows
// (the plan's lists, and the segment-split path's candidate buffers for its
// first kSplitMaxRows rows: about 8.6 MB).
// In host code this name is only a stand-in for the device symbol; its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_workspace_ptr[kMaxDevices] = {};

// Looks up (once per device, with that device current) the device address of
// the scratch array.
cudaError_t workspace_for_current_device(void** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_workspace_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        g_workspace_ptr[dev] = p;
    }
    *ptr = g_workspace_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace topkidx

extern "C" topk_status_t topk_transform_noalloc(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                                                int32_t batch, int32_t max_seq_len, const int32_t* page_table,
                                                int64_t page_table_stride, int32_t page_size, int32_t k,
                                                int32_t* out_indices, int32_t* out_raw_indices_or_null,
                                                topk_stream_t stream) {
    using namespace topkidx;
    if (batch > kNoAllocMaxBatch) return TOPK_ENOSPACE;
    // The transform's own checks, repeated so that a bad call enqueues nothing.
    if (!scores || !seq_lens || !page_table || !out_indices) return TOPK_EINVAL;
    if (batch < 1 || max_seq_len < 0 || k < 1 || k > kMaxK) return TOPK_EINVAL;
    if (page_size < 1 || (page_size & (page_size - 1)) != 0 || page_size > (1 << 30)) return TOPK_EINVAL;
    if (row_stride < max_seq_len || row_stride < 1) return TOPK_EINVAL;
    if (page_table_stride < (static_cast<int64_t>(max_seq_len) + page_size - 1) / page_size || page_table_stride < 1)
        return TOPK_EINVAL;
    if (reinterpret_cast<uintptr_t>(scores) % 16 != 0 || row_stride % 4 != 0) return TOPK_EALIGN;
    if (reinterpret_cast<uintptr_t>(seq_lens) % 4 || reinterpret_cast<uintptr_t>(page_table) % 4 ||
        reinterpret_cast<uintptr_t>(out_indices) % 4 || reinterpret_cast<uintptr_t>(out_raw_indices_or_null) % 4)
        return TOPK_EALIGN;
    void* ws = nullptr;
    if (workspace_for_current_device(&ws) != cudaSuccess) return TOPK_ECUDA;
    // The plan kernel rewrites every header field and list entry that the
    // select kernels read, so the previous call's contents need no clearing.
    const topk_status_t st = topk_plan(seq_lens, batch, max_seq_len, ws, kNoAllocWorkspaceBytes, stream);
    if (st != TOPK_OK) return st;
    return topk_transform(scores, row_stride, seq_lens, batch, max_seq_len, page_table, page_table_stride,
                          page_size, k, out_indices, out_raw_indices_or_null, ws, stream);
}
