// route_noalloc.cu -- gg_route_hist_offsets_noalloc: the routing-metadata
// entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: for
// example a runtime that owns all device memory through its own arena and
// gives a plugin only the input and output buffers, or a latency-critical path
// where an allocation (and the device synchronisation it can imply) is not
// acceptable.  For them the per-chunk counts of the counting sort live in a
// fixed static device array of this library instead of a caller workspace.
//
// The array holds GG_ROUTE_NOALLOC_SCRATCH_BYTES bytes; every GPU that loads
// the library keeps its own copy until the process exits.  All calls on one
// device share that device's copy: calls that overlap on the same device (on
// concurrent streams) race on it and must be serialised by the caller; calls
// on different devices do not interfere.  Devices numbered kMaxDevices (64) or
// higher are refused with GG_ERR_UNSUPPORTED.  Nothing in the array needs
// clearing between calls: the count pass writes every entry the later passes
// read.
#include <mutex>

#include "common.cuh"

namespace gg {
int route_launch(const int32_t* ids, int64_t T, int topk, int E, int pad_block, int32_t* m_sizes,
                 int32_t* offsets, int32_t* padded, int32_t* gather_idx, int32_t* row_id_map,
                 int32_t* counts, int32_t* status, cudaStream_t stream);
size_t route_workspace_bytes(int64_t T, int topk, int E);
}  // namespace gg

namespace {

constexpr size_t kScratchInts = GG_ROUTE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);

// The counts[E][chunks] table of the counting sort.  In host code this name is
// only a stand-in for the device symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_route_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on each device does this set-up).
int scratch_for_current_device(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { gg::record_cuda_error(e); return GG_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return GG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess || p == nullptr) {
            gg::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            return GG_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return GG_OK;
}

}  // namespace

extern "C" int gg_route_hist_offsets_noalloc(const int32_t* topk_ids, int64_t T, int topk, int E,
                                             int pad_block, int32_t* m_sizes, int32_t* offsets,
                                             int32_t* padded_offsets, int32_t* gather_idx,
                                             int32_t* row_id_map, int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || !m_sizes || !offsets) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31)) return GG_ERR_UNSUPPORTED;
    if (R > 0 && (!topk_ids || !gather_idx)) return GG_ERR_INVALID_ARG;
    if (pad_block > 0 && !padded_offsets) return GG_ERR_INVALID_ARG;
    // route_workspace_bytes rounds up to 256 bytes; the array is a multiple of 256.
    if (gg::route_workspace_bytes(T, topk, E) > GG_ROUTE_NOALLOC_SCRATCH_BYTES)
        return GG_ERR_WORKSPACE;
    int32_t* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != GG_OK) return rc;
    return gg::route_launch(topk_ids, T, topk, E, pad_block, m_sizes, offsets, padded_offsets,
                            gather_idx, row_id_map, scratch, status,
                            reinterpret_cast<cudaStream_t>(stream));
}
