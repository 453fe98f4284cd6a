// gemm_ragged_m.cu -- entry points whose output rows are ragged per expert:
// the forward grouped GEMM (also with the fused SwiGLU of matmul_ogs.py's
// FusedActivation, or with the top-k combine fused into the epilogue as
// fp32 or bf16 atomic adds) and the backward dX (interface.py, grouped_gemm_forward
// and grouped_gemm_dX), also with the SwiGLU backward fused into its epilogue.  Both run the persistent tcgen05
// engine of gemm_engine.cuh over the expert-order row tiles.
#include "gemm_launch.cuh"

namespace gg {
int combine_launch(const uint16_t* Y, const int32_t* row_id_map, const float* topk_w, int64_t T,
                   int topk, int64_t N, uint16_t* out, int32_t* status, cudaStream_t stream);
int f32_to_bf16_launch(const float* src, int64_t n, uint16_t* dst, cudaStream_t stream);
}

using namespace gg;

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Upper bound on the expert-order row tiles (matmul_ogs.py, RoutingData.n_blocks).
int64_t row_tile_bound(int64_t R, int E) {
    if (R <= E) return R;
    return (R - E + 1 + kBM - 1) / kBM + E - 1;
}

GemmParams base_params(int E, int topk, int64_t R, const int32_t* m_sizes, const int32_t* gather_idx,
                       int32_t* status) {
    GemmParams p{};
    p.E = E;
    p.topk = topk;
    p.R = R;
    p.m_sizes = m_sizes;
    p.gather_idx = gather_idx;
    p.status = status;
    return p;
}

}  // namespace

extern "C" {

int gg_forward(const gg_bf16* X, const gg_bf16* W, const int32_t* m_sizes,
               const int32_t* gather_idx, const float* topk_w, int64_t T, int topk, int E,
               int64_t N, int64_t K, int permute_x, int permute_y, int fuse_mul_post, gg_bf16* Y,
               int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || N < 0 || K < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS || N % 8 || K % 8) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return GG_ERR_UNSUPPORTED;
    if ((permute_x || permute_y) && !gather_idx) return GG_ERR_INVALID_ARG;
    if (fuse_mul_post && (!permute_y || !topk_w)) return GG_ERR_INVALID_ARG;
    if (R == 0 || N == 0) return GG_OK;
    if (!m_sizes || !Y) return GG_ERR_INVALID_ARG;
    if (!al16(Y)) return GG_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {  // X and W have no elements (may be NULL)
        const cudaError_t e = cudaMemsetAsync(Y, 0, static_cast<size_t>(R * N) * 2, st);
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
        return GG_OK;
    }
    if (!X || !W) return GG_ERR_INVALID_ARG;
    if (!al16(X) || !al16(W)) return GG_ERR_UNSUPPORTED;
    GemmParams p = base_params(E, topk, R, m_sizes, gather_idx, status);
    p.N = static_cast<int>(N);
    p.Kred = static_cast<int>(K);
    p.out = Y;
    p.ld_out = N;
    p.scatter_out = permute_y ? 1 : 0;
    p.scale = fuse_mul_post ? topk_w : nullptr;
    CUtensorMap mA{}, mB{};
    const int64_t bound = row_tile_bound(R, E) * ((N + kBN - 1) / kBN);
    if (permute_x) {
        if (!encode_map_3d(&mB, W, K, N, E, K, N * K, kBK, kBN)) return GG_ERR_CUDA;
        p.ga = GatherSrc{X, K, T, K, ROW_TOKEN};
        return launch_gemm<KIND_RAGGED_M, false, false, true, false, false>(mB, mB, mB, mB, p, bound, st);
    }
    // 2-CTA tiles: each CTA loads half of the 256 W rows of an n-tile
    if (!encode_map_3d(&mB, W, K, N, E, K, N * K, kBK, kBN / 2)) return GG_ERR_CUDA;
    if (!encode_map_2d(&mA, X, K, R, K, kBK, kBM)) return GG_ERR_CUDA;
    return launch_gemm<KIND_RAGGED_M, false, false, false, false, true>(mA, mB, mA, mB, p, bound, st);
}

int gg_forward_swiglu(const gg_bf16* X, const gg_bf16* W, const int32_t* m_sizes,
                      const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N, int64_t K,
                      int permute_x, gg_bf16* Y, gg_bf16* A, int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || N < 0 || K < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS || N % 16 || K % 8) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return GG_ERR_UNSUPPORTED;
    if (permute_x && !gather_idx) return GG_ERR_INVALID_ARG;
    if (R == 0 || N == 0) return GG_OK;
    if (!m_sizes || !A) return GG_ERR_INVALID_ARG;
    if (!al16(A) || (Y && !al16(Y))) return GG_ERR_UNSUPPORTED;
    if (K > 0 && (!X || !W)) return GG_ERR_INVALID_ARG;  // with K == 0 they have no elements
    if (K > 0 && (!al16(X) || !al16(W))) return GG_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {  // y = 0, so silu(0) * 0 = 0
        cudaError_t e = cudaMemsetAsync(A, 0, static_cast<size_t>(R * (N / 2)) * 2, st);
        if (e == cudaSuccess && Y) e = cudaMemsetAsync(Y, 0, static_cast<size_t>(R * N) * 2, st);
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
        return GG_OK;
    }
    GemmParams p = base_params(E, topk, R, m_sizes, gather_idx, status);
    p.N = static_cast<int>(N);
    p.Kred = static_cast<int>(K);
    p.out = Y;  // may be null: activation only
    p.ld_out = N;
    p.act_out = A;
    p.ld_act = N / 2;
    CUtensorMap mA{}, mB{};
    const int64_t bound = row_tile_bound(R, E) * ((N + kBN - 1) / kBN);
    if (permute_x) {
        if (!encode_map_3d(&mB, W, K, N, E, K, N * K, kBK, kBN)) return GG_ERR_CUDA;
        p.ga = GatherSrc{X, K, T, K, ROW_TOKEN};
        return launch_gemm<KIND_RAGGED_M, false, false, true, false, false>(mB, mB, mB, mB, p, bound, st);
    }
    if (!encode_map_3d(&mB, W, K, N, E, K, N * K, kBK, kBN / 2)) return GG_ERR_CUDA;
    if (!encode_map_2d(&mA, X, K, R, K, kBK, kBM)) return GG_ERR_CUDA;
    return launch_gemm<KIND_RAGGED_M, false, false, false, false, true>(mA, mB, mA, mB, p, bound, st);
}

int gg_forward_combine(const gg_bf16* X, const gg_bf16* W, const int32_t* m_sizes,
                       const int32_t* gather_idx, const float* topk_w, int64_t T, int topk, int E,
                       int64_t N, int64_t K, int permute_x, gg_bf16* out, void* workspace,
                       size_t workspace_bytes, int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || N < 0 || K < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS || N % 8 || K % 8) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return GG_ERR_UNSUPPORTED;
    if (T == 0 || N == 0) return GG_OK;
    if (!m_sizes || !gather_idx || !out) return GG_ERR_INVALID_ARG;
    if (!al16(out)) return GG_ERR_UNSUPPORTED;
    if (K > 0 && (!X || !W)) return GG_ERR_INVALID_ARG;  // with K == 0 they have no elements
    if (K > 0 && (!al16(X) || !al16(W))) return GG_ERR_UNSUPPORTED;
    // fp32 sums in the caller's workspace, or (small topk only) bf16 adds into out
    const size_t acc_bytes = static_cast<size_t>(T) * static_cast<size_t>(N) * sizeof(float);
    const bool fp32 = workspace != nullptr;
    if (fp32 && (workspace_bytes < acc_bytes || !al16(workspace))) return GG_ERR_WORKSPACE;
    if (!fp32 && topk > GG_COMBINE_BF16_MAX_TOPK) return GG_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* acc = static_cast<float*>(workspace);
    // the adds accumulate into zeroed sums (every token row gets topk adds)
    int rc = fp32 ? cuda_result(cudaMemsetAsync(acc, 0, acc_bytes, st))
                  : cuda_result(cudaMemsetAsync(out, 0, static_cast<size_t>(T * N) * 2, st));
    if (rc != GG_OK) return rc;
    if (K > 0) {
        GemmParams p = base_params(E, topk, R, m_sizes, gather_idx, status);
        p.N = static_cast<int>(N);
        p.Kred = static_cast<int>(K);
        p.out = fp32 ? nullptr : out;
        p.acc_out = fp32 ? acc : nullptr;
        p.ld_out = N;
        p.combine_out = 1;
        p.scale = topk_w;
        CUtensorMap mA{}, mB{};
        const int64_t bound = row_tile_bound(R, E) * ((N + kBN - 1) / kBN);
        if (permute_x) {
            if (!encode_map_3d(&mB, W, K, N, E, K, N * K, kBK, kBN)) return GG_ERR_CUDA;
            p.ga = GatherSrc{X, K, T, K, ROW_TOKEN};
            rc = launch_gemm<KIND_RAGGED_M, false, false, true, false, false>(mB, mB, mB, mB, p, bound, st);
        } else {
            if (!encode_map_3d(&mB, W, K, N, E, K, N * K, kBK, kBN / 2)) return GG_ERR_CUDA;
            if (!encode_map_2d(&mA, X, K, R, K, kBK, kBM)) return GG_ERR_CUDA;
            rc = launch_gemm<KIND_RAGGED_M, false, false, false, false, true>(mA, mB, mA, mB, p, bound, st);
        }
        if (rc != GG_OK) return rc;
    }
    return fp32 ? f32_to_bf16_launch(acc, T * N, out, st) : GG_OK;
}

int gg_backward_dX(const gg_bf16* dY, const gg_bf16* W, const int32_t* m_sizes,
                   const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N, int64_t K,
                   int permute_x, int permute_y, gg_bf16* dX, gg_bf16* dX_tok, int32_t* status,
                   void* stream) {
    if (T < 0 || topk < 1 || E < 1 || N < 0 || K < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS || N % 8 || K % 8) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return GG_ERR_UNSUPPORTED;
    if ((permute_x || permute_y) && !gather_idx) return GG_ERR_INVALID_ARG;
    if (dX_tok && !permute_x) return GG_ERR_INVALID_ARG;
    if (R == 0 || K == 0) return GG_OK;
    if (!m_sizes || !dX) return GG_ERR_INVALID_ARG;
    if (!al16(dX) || (dX_tok && !al16(dX_tok))) return GG_ERR_UNSUPPORTED;
    if (N > 0 && (!dY || !W)) return GG_ERR_INVALID_ARG;  // with N == 0 they have no elements
    if (N > 0 && (!al16(dY) || !al16(W))) return GG_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = GG_OK;
    if (N == 0) {
        const cudaError_t e = cudaMemsetAsync(dX, 0, static_cast<size_t>(R * K) * 2, st);
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
    } else {
        GemmParams p = base_params(E, topk, R, m_sizes, gather_idx, status);
        p.N = static_cast<int>(K);      // output columns
        p.Kred = static_cast<int>(N);   // reduction over the forward's N
        p.out = dX;
        p.ld_out = K;
        p.scatter_out = permute_x ? 1 : 0;
        CUtensorMap mA{}, mB{};
        // B[k, n] = W[e][n, k]: MN-major, 64-wide k chunks over 64 rows of n.
        if (!encode_map_3d(&mB, W, K, N, E, K, N * K, 64, kBK)) return GG_ERR_CUDA;
        const int64_t bound = row_tile_bound(R, E) * ((K + kBN - 1) / kBN);
        if (permute_y) {
            p.ga = GatherSrc{dY, N, R, N, ROW_SLOT};
            rc = launch_gemm<KIND_RAGGED_M, false, true, true, false, false>(mB, mB, mB, mB, p, bound, st);
        } else {
            if (!encode_map_2d(&mA, dY, N, R, N, kBK, kBM)) return GG_ERR_CUDA;
            if (K % 64 == 0) {  // W's 128-column half tile as one box of two 64-column chunks
                if (!encode_map_mn_chunks_planes(&mB, W, K, N, E, K, N * K, kBK, (kBN / 2) / 64))
                    return GG_ERR_CUDA;
                p.mn_chunk_view = 1;
            }
            rc = launch_gemm<KIND_RAGGED_M, false, true, false, false, true>(mA, mB, mA, mB, p, bound, st);
        }
    }
    if (rc != GG_OK || !dX_tok) return rc;
    return combine_launch(dX, nullptr, nullptr, T, topk, K, dX_tok, status, st);
}

int gg_backward_dX_swiglu(const gg_bf16* dY, const gg_bf16* W, const int32_t* m_sizes, int64_t T,
                          int topk, int E, int64_t N, int64_t K, const gg_bf16* H, gg_bf16* dH,
                          int32_t* status, void* stream) {
    if (T < 0 || topk < 1 || E < 1 || N < 0 || K < 0) return GG_ERR_INVALID_ARG;
    if (topk > GG_MAX_TOPK || E > GG_MAX_EXPERTS || N % 8 || K % 8) return GG_ERR_UNSUPPORTED;
    const int64_t R = T * topk;
    if (R >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || 2 * K >= (int64_t(1) << 31))
        return GG_ERR_UNSUPPORTED;
    if (R == 0 || K == 0) return GG_OK;
    if (!m_sizes || !dH) return GG_ERR_INVALID_ARG;
    if (!al16(dH)) return GG_ERR_UNSUPPORTED;
    if (N > 0 && (!dY || !W || !H)) return GG_ERR_INVALID_ARG;  // N == 0: dH = 0, no inputs read
    if (N > 0 && (!al16(dY) || !al16(W) || !al16(H))) return GG_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) {  // dA = 0, so dH = 0
        const cudaError_t e = cudaMemsetAsync(dH, 0, static_cast<size_t>(R * 2 * K) * 2, st);
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
        return GG_OK;
    }
    GemmParams p = base_params(E, topk, R, m_sizes, nullptr, status);
    p.N = static_cast<int>(K);
    p.Kred = static_cast<int>(N);
    p.out = dH;
    p.ld_out = 2 * K;
    p.swiglu_h = H;
    p.ld_h = 2 * K;
    CUtensorMap mA{}, mB{};
    if (!encode_map_3d(&mB, W, K, N, E, K, N * K, 64, kBK)) return GG_ERR_CUDA;
    const int64_t bound = row_tile_bound(R, E) * ((K + kBN - 1) / kBN);
    if (!encode_map_2d(&mA, dY, N, R, N, kBK, kBM)) return GG_ERR_CUDA;
    if (K % 64 == 0) {
        if (!encode_map_mn_chunks_planes(&mB, W, K, N, E, K, N * K, kBK, (kBN / 2) / 64)) return GG_ERR_CUDA;
        p.mn_chunk_view = 1;
    }
    return launch_gemm<KIND_RAGGED_M, false, true, false, false, true>(mA, mB, mA, mB, p, bound, st);
}

}  // extern "C"
