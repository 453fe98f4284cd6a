// gemm_dw.cu -- backward dW: dW[e] = dY_e^T . X_e with each expert's own rows
// as the (ragged) reduction dimension (interface.py, grouped_gemm_dW;
// matmul_ogs.py, the ragged dw comment).  Both operands are MN-major tiles of
// reduction rows; dense operands come in by TMA and the rows past an expert's
// end are zeroed in shared memory before the MMA, gathered operands come in
// by cp.async with zero fill.  Given a workspace, gathered operands are first
// copied into expert order (one HBM-bound row gather each) and the reduction
// runs on the dense 2-CTA path: every reduction block of a gathered operand
// needs 64 newly gathered rows, which cp.async fetches far slower than TMA
// streams a dense tile.
#include "gemm_launch.cuh"

namespace gg {
int gather_rows_launch(const uint16_t* src, const int32_t* gather_idx, int div, int64_t src_rows,
                       int64_t R, int64_t cols, uint16_t* dst, int32_t* status, cudaStream_t stream);
}

using namespace gg;

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Workspace bytes of the expert-order copies: X rows (permute_x), then dY rows (permute_y).
size_t dw_workspace_bytes(int64_t R, int64_t N, int64_t K, int permute_x, int permute_y) {
    return (permute_x ? align256(static_cast<size_t>(R) * K * 2) : 0) +
           (permute_y ? align256(static_cast<size_t>(R) * N * 2) : 0);
}

int dw_launch(const gg_bf16* X, const gg_bf16* dY, const int32_t* m_sizes, const int32_t* gather_idx,
              int64_t T, int topk, int E, int64_t N, int64_t K, int permute_x, int permute_y,
              gg_bf16* dW, int32_t* status, cudaStream_t st) {
    const int64_t R = T * topk;
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

}  // namespace

namespace gg {
size_t backward_dw_workspace_bytes(int64_t T, int topk, int64_t N, int64_t K, int flags) {
    if (T < 0 || topk < 1 || N < 0 || K < 0) return 0;
    return dw_workspace_bytes(T * topk, N, K, flags & GG_PERMUTE_X, flags & GG_PERMUTE_Y);
}
}  // namespace gg

extern "C" int gg_backward_dW(const gg_bf16* X, const gg_bf16* dY, const int32_t* m_sizes,
                              const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N,
                              int64_t K, int permute_x, int permute_y, gg_bf16* dW, void* workspace,
                              size_t workspace_bytes, int32_t* status, void* stream) {
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
    if (R == 0) return cuda_result(cudaMemsetAsync(dW, 0, static_cast<size_t>(E) * N * K * 2, st));
    if (!X || !dY) return GG_ERR_INVALID_ARG;
    if (!al16(X) || !al16(dY)) return GG_ERR_UNSUPPORTED;
    if (workspace && (permute_x || permute_y)) {
        if (!al16(workspace) || workspace_bytes < dw_workspace_bytes(R, N, K, permute_x, permute_y))
            return GG_ERR_WORKSPACE;
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        const gg_bf16* Xd = X;
        const gg_bf16* dYd = dY;
        if (permute_x) {
            gg_bf16* Xg = reinterpret_cast<gg_bf16*>(ws);
            const int rc = gather_rows_launch(X, gather_idx, topk, T, R, K, Xg, status, st);
            if (rc != GG_OK) return rc;
            Xd = Xg;
            ws += align256(static_cast<size_t>(R) * K * 2);
        }
        if (permute_y) {
            gg_bf16* dYg = reinterpret_cast<gg_bf16*>(ws);
            const int rc = gather_rows_launch(dY, gather_idx, 1, R, R, N, dYg, status, st);
            if (rc != GG_OK) return rc;
            dYd = dYg;
        }
        return dw_launch(Xd, dYd, m_sizes, gather_idx, T, topk, E, N, K, 0, 0, dW, status, st);
    }
    return dw_launch(X, dY, m_sizes, gather_idx, T, topk, E, N, K, permute_x, permute_y, dW, status,
                     st);
}
