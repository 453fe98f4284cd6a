// abi.cu -- host side of the C ABI: status strings, CUDA error capture, TMA
// tensor-map encoding, and the argument validation + launch of the routing
// and row-moving entry points.  The grouped-GEMM entry points live beside
// their kernels (gemm_ragged_m.cu, gemm_dw.cu, gemm_dual.cu).
#include <cudaTypedefs.h>

#include <cstdio>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace gg {

int route_launch(const int32_t* ids, int64_t T, int topk, int E, int pad_block, int32_t* m_sizes,
                 int32_t* offsets, int32_t* padded, int32_t* gather_idx, int32_t* row_id_map,
                 int32_t* counts, int32_t* status, cudaStream_t stream);
size_t route_workspace_bytes(int64_t T, int topk, int E);
int permute_launch(const uint16_t* X, const int32_t* row_id_map, int64_t T, int topk, int64_t K,
                   uint16_t* Xp, int32_t* status, cudaStream_t stream);
int combine_launch(const uint16_t* Y, const int32_t* row_id_map, const float* topk_w, int64_t T,
                   int topk, int64_t N, uint16_t* out, int32_t* status, cudaStream_t stream);
int swiglu_bwd_launch(const uint16_t* H, const uint16_t* dA, int64_t rows, int64_t I, uint16_t* dH,
                      cudaStream_t stream);
int combine_bwd_launch(const uint16_t* G, const uint16_t* Y, const int32_t* row_id_map,
                       const float* topk_w, int64_t T, int topk, int64_t N, uint16_t* dY, float* dw,
                       int32_t* status, cudaStream_t stream);
size_t backward_dw_workspace_bytes(int64_t T, int topk, int64_t N, int64_t K, int flags);

namespace {
thread_local char g_last_error[256] = "no error";
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

void record_cuda_error(cudaError_t e) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (cache[dev] == 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = sms > 0 ? sms : 1;
    }
    return cache[dev];
}

static bool encode(CUtensorMap* m, uint32_t rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled unavailable");
        return false;
    }
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    // The swizzle span equals the box's inner extent (rows of 64 or 128 bytes),
    // which is the layout the MMA descriptors expect for that tile.
    const CUtensorMapSwizzle sw = box[0] * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base),
                                dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
        return false;
    }
    return true;
}

// 2-D bf16 tensor [outer, inner] (inner contiguous), rows row_stride elements apart.
bool encode_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_elems * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    return encode(m, 2, base, dims, strides, box);
}

// 3-D bf16 tensor [d2, d1, d0] (d0 contiguous), box {b0, b1, 1}.
bool encode_map_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_elems, uint64_t stride2_elems, uint32_t b0, uint32_t b1) {
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_elems * 2, stride2_elems * 2};
    const cuuint32_t box[3] = {b0, b1, 1};
    return encode(m, 3, base, dims, strides, box);
}

// An MN-major operand [rows, cols] (cols contiguous, a multiple of 64) viewed
// as 3-D {64, rows, cols / 64}: the third dimension steps 128 bytes along a
// row, so one box {64, box_rows, box_chunks} brings box_chunks adjacent
// 64-column chunks of box_rows rows, chunk after chunk, in one copy.
bool encode_map_mn_chunks(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                          uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_chunks) {
    if (cols % 64) return false;
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {row_stride_elems * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, box_chunks};
    return encode(m, 3, base, dims, strides, box);
}

// The same view per plane of a 3-D tensor [planes, rows, cols] (the expert
// weights): {64, rows, cols / 64, planes}, box {64, box_rows, box_chunks, 1}.
bool encode_map_mn_chunks_planes(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                                 uint64_t planes, uint64_t row_stride_elems,
                                 uint64_t plane_stride_elems, uint32_t box_rows,
                                 uint32_t box_chunks) {
    if (cols % 64) return false;
    const cuuint64_t dims[4] = {64, rows, cols / 64, planes};
    const cuuint64_t strides[3] = {row_stride_elems * 2, 128, plane_stride_elems * 2};
    const cuuint32_t box[4] = {64, box_rows, box_chunks, 1};
    return encode(m, 4, base, dims, strides, box);
}

}  // namespace gg

namespace gg {
namespace {
// One CTA waits, through the same bounded wait every pipelined kernel uses,
// on an mbarrier phase that can never complete (nothing arrives on it).
__global__ void selftest_wait_kernel(int32_t* status, uint64_t limit_ns, int32_t* result) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = mbar_wait(&bar, 0, &abort_flag, status, 0, limit_ns);
        *result = ok ? 1 : 0;
    }
}
}  // namespace

std::atomic<int> g_gemm_schedule{GG_SCHEDULE_AUTO};
}  // namespace gg

using namespace gg;

namespace {
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
}  // namespace

extern "C" {

const char* gg_status_string(int code) {
    switch (code) {
        case GG_OK: return "ok";
        case GG_ERR_INVALID_ARG: return "invalid argument";
        case GG_ERR_UNSUPPORTED: return "unsupported shape, alignment or size";
        case GG_ERR_CUDA: return "CUDA error (see gg_last_cuda_error)";
        case GG_ERR_DEVICE_CHECK: return "a kernel found bad input data (see the device status code)";
        case GG_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case GG_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

const char* gg_device_status_string(int code) {
    switch (code) {
        case GG_DEV_OK: return "ok";
        case GG_DEV_BAD_EXPERT_ID: return "expert id outside [0, E)";
        case GG_DEV_BAD_ROW_INDEX: return "row index outside its tensor";
        case GG_DEV_SIZES_MISMATCH: return "m_sizes negative or not summing to T*topk";
        case GG_DEV_TIMEOUT: return "a bounded wait inside a kernel ran out";
        default: return "unknown device status";
    }
}

const char* gg_last_cuda_error(void) { return g_last_error; }

size_t gg_route_workspace_size(int64_t T, int topk, int E) {
    if (T < 0 || topk < 1 || E < 1) return 0;
    return route_workspace_bytes(T, topk, E);
}

size_t gg_workspace_size(int op, int64_t T, int topk, int E, int64_t N, int64_t K, int flags) {
    if (T < 0 || topk < 1 || E < 1 || N < 0 || K < 0) return 0;
    switch (op) {
        case GG_OP_ROUTE: return route_workspace_bytes(T, topk, E);
        case GG_OP_BACKWARD_DW: return backward_dw_workspace_bytes(T, topk, N, K, flags);
        case GG_OP_FORWARD_COMBINE: return static_cast<size_t>(T) * static_cast<size_t>(N) * sizeof(float);
        default: return 0;
    }
}

int gg_read_status(const int32_t* status, int32_t* code, void* stream) {
    if (!status) return GG_ERR_INVALID_ARG;
    int32_t v = 0;
    // a copy into this stack word: the runtime stages it, nothing is allocated here
    cudaError_t e = cudaMemcpyAsync(&v, status, sizeof v, cudaMemcpyDeviceToHost, as_stream(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
    if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
    if (code) *code = v;
    if (v == GG_DEV_OK) return GG_OK;
    return v == GG_DEV_TIMEOUT ? GG_ERR_TIMEOUT : GG_ERR_DEVICE_CHECK;
}

int gg_set_gemm_schedule(int mode) {
    if (mode != GG_SCHEDULE_AUTO && mode != GG_SCHEDULE_STATIC && mode != GG_SCHEDULE_DYNAMIC)
        return GG_ERR_INVALID_ARG;
    return g_gemm_schedule.exchange(mode);
}

int gg_route_hist_offsets(const int32_t* topk_ids, int64_t T, int topk, int E, int pad_block,
                          int32_t* m_sizes, int32_t* offsets, int32_t* padded_offsets,
                          int32_t* gather_idx, int32_t* row_id_map, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || !m_sizes || !offsets) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31)) return GG_ERR_UNSUPPORTED;
    if (R > 0 && (!topk_ids || !gather_idx)) return GG_ERR_INVALID_ARG;
    if (pad_block > 0 && !padded_offsets) return GG_ERR_INVALID_ARG;
    const size_t need = route_workspace_bytes(T, topk, E);
    if (R > 0 && (!workspace || workspace_bytes < need)) return GG_ERR_WORKSPACE;
    return route_launch(topk_ids, T, topk, E, pad_block, m_sizes, offsets, padded_offsets,
                        gather_idx, row_id_map, static_cast<int32_t*>(workspace), status,
                        as_stream(stream));
}

int gg_permute(const gg_bf16* X, const int32_t* row_id_map, int64_t T, int topk, int64_t K,
               gg_bf16* Xp, int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || K < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || K % 8) return GG_ERR_UNSUPPORTED;
    if (T * topk >= (int64_t(1) << 31)) return GG_ERR_UNSUPPORTED;
    if (T == 0 || K == 0) return GG_OK;
    if (!X || !row_id_map || !Xp) return GG_ERR_INVALID_ARG;
    if (!al16(X) || !al16(Xp)) return GG_ERR_UNSUPPORTED;
    return permute_launch(X, row_id_map, T, topk, K, Xp, status, as_stream(stream));
}

int gg_unpermute_combine(const gg_bf16* Y, const int32_t* row_id_map, const float* topk_w,
                         int64_t T, int topk, int64_t N, gg_bf16* out, int32_t* status,
                         void* stream) {
    if (T < 0 || topk < 1 || N < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || N % 8) return GG_ERR_UNSUPPORTED;
    if (T * topk >= (int64_t(1) << 31)) return GG_ERR_UNSUPPORTED;
    if (T == 0 || N == 0) return GG_OK;
    if (!Y || !out) return GG_ERR_INVALID_ARG;
    if (!al16(Y) || !al16(out)) return GG_ERR_UNSUPPORTED;
    return combine_launch(Y, row_id_map, topk_w, T, topk, N, out, status, as_stream(stream));
}

int gg_unpermute_combine_bwd(const gg_bf16* G, const gg_bf16* Y, const int32_t* row_id_map,
                             const float* topk_w, int64_t T, int topk, int64_t N, gg_bf16* dY,
                             float* dw, int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || N < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || N % 8) return GG_ERR_UNSUPPORTED;
    if (T * topk >= (int64_t(1) << 31)) return GG_ERR_UNSUPPORTED;
    if (T == 0) return GG_OK;
    if (dw && !Y && N > 0) return GG_ERR_INVALID_ARG;
    if (N == 0) {
        if (!dw) return GG_OK;
        const cudaError_t e = cudaMemsetAsync(dw, 0, sizeof(float) * static_cast<size_t>(T * topk),
                                              as_stream(stream));
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
        return GG_OK;
    }
    if (!G || !dY) return GG_ERR_INVALID_ARG;
    if (!al16(G) || !al16(dY) || (Y && !al16(Y))) return GG_ERR_UNSUPPORTED;
    return combine_bwd_launch(G, dw ? Y : nullptr, row_id_map, topk_w, T, topk, N, dY, dw, status,
                              as_stream(stream));
}

int gg_swiglu_bwd(const gg_bf16* H, const gg_bf16* dA, int64_t rows, int64_t I, gg_bf16* dH,
                  void* stream) {
    if (rows < 0 || I < 0) return GG_ERR_INVALID_ARG;
    if (I % 8) return GG_ERR_UNSUPPORTED;
    if (rows == 0 || I == 0) return GG_OK;
    if (!H || !dA || !dH) return GG_ERR_INVALID_ARG;
    if (!al16(H) || !al16(dA) || !al16(dH)) return GG_ERR_UNSUPPORTED;
    return swiglu_bwd_launch(H, dA, rows, I, dH, as_stream(stream));
}

int gg_selftest_bounded_wait(int32_t* status, int32_t* result, uint64_t limit_ns, void* stream) {
    if (!status || !result || limit_ns == 0 || limit_ns > kWaitLimitNs) return GG_ERR_INVALID_ARG;
    clear_pending_launch_error();
    selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(status, limit_ns, result);
    return launch_result();
}

}  // extern "C"
