// gemm_dw.cu -- backward dW: dW[e] = dY_e^T . X_e with each expert's own rows
// as the (ragged) reduction dimension (interface.py, grouped_gemm_dW;
// matmul_ogs.py, the ragged dw comment).  Both operands are MN-major tiles of
// reduction rows; dense operands come in by TMA and the rows past an expert's
// end are zeroed in shared memory before the MMA, gathered operands come in
// by cp.async with zero fill.
#include "gemm_engine.cuh"

using namespace gg;

namespace {
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}

extern "C" int gg_backward_dW(const gg_bf16* X, const gg_bf16* dY, const int32_t* m_sizes,
                              const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N,
                              int64_t K, int permute_x, int permute_y, gg_bf16* dW,
                              int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || N < 0 || K < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS || N % 8 || K % 8) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return GG_ERR_UNSUPPORTED;
    if ((permute_x || permute_y) && !gather_idx) return GG_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return GG_OK;
    if (!dW || !m_sizes) return GG_ERR_INVALID_ARG;
    if (!al16(dW)) return GG_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (R == 0) {
        const cudaError_t e = cudaMemsetAsync(dW, 0, static_cast<size_t>(E) * N * K * 2, st);
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
        return GG_OK;
    }
    if (!X || !dY) return GG_ERR_INVALID_ARG;
    if (!al16(X) || !al16(dY)) return GG_ERR_UNSUPPORTED;
    GemmParams p{};
    p.E = E;
    p.topk = topk;
    p.R = R;
    p.M = static_cast<int>(N);
    p.N = static_cast<int>(K);
    p.m_sizes = m_sizes;
    p.gather_idx = gather_idx;
    p.out = dW;
    p.ld_out = K;
    p.status = status;
    CUtensorMap mA{}, mB{};
    if (permute_y) p.ga = GatherSrc{dY, N, R, N, ROW_SLOT};
    else if (!encode_map_2d(&mA, dY, N, R, N, 64, kBK)) return GG_ERR_CUDA;
    if (permute_x) p.gb = GatherSrc{X, K, T, K, ROW_TOKEN};
    else if (!encode_map_2d(&mB, X, K, R, K, 64, kBK)) return GG_ERR_CUDA;
    const int64_t bound = static_cast<int64_t>(E) * ((N + kBM - 1) / kBM) * ((K + kBN - 1) / kBN);
    if (permute_y && permute_x)
        return launch_gemm<KIND_RAGGED_K, true, true, true, true, false>(mA, mB, mA, mB, p, bound, st);
    if (permute_y)
        return launch_gemm<KIND_RAGGED_K, true, true, true, false, false>(mA, mB, mA, mB, p, bound, st);
    if (permute_x)
        return launch_gemm<KIND_RAGGED_K, true, true, false, true, false>(mA, mB, mA, mB, p, bound, st);
    // both dense: when the widths allow, read each operand's stage as one box of
    // 64-column chunks (one TMA copy per operand and stage, not two)
    if (N % 64 == 0 && K % 64 == 0) {
        if (!encode_map_mn_chunks(&mA, dY, N, R, N, kBK, kBM / 64)) return GG_ERR_CUDA;
        if (!encode_map_mn_chunks(&mB, X, K, R, K, kBK, (kBN / 2) / 64)) return GG_ERR_CUDA;
        p.mn_chunk_view = 1;
    }
    return launch_gemm<KIND_RAGGED_K, true, true, false, false, true>(mA, mB, mA, mB, p, bound, st);
}
