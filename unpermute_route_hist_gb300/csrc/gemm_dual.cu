// gemm_dual.cu -- two experts' GEMMs with different row counts and output
// widths, one launch (backend.py, asym_dual_gmm_separated).  The two problems'
// tiles form one list for the persistent engine; each problem has its own pair
// of tensor maps.  trans_a stores the inputs (k, m); trans_b stores the
// weights (n, k) -- which decides whether each operand tile is K- or MN-major.
// When its 128 x 256 tiles fill more than one wave of SMs it runs on 2-CTA
// pairs like the other dense launches: a pair takes two adjacent 128-row
// m-tiles of one problem (the second a phantom past an odd m-tile count), each
// CTA loading its own rows and half of the 256 columns, so each SM's operand
// stream is a third smaller (8192 x 8192 rows: 1258 -> 1486 TFLOP/s).  A
// problem that fits one wave keeps single-CTA tiles, which start ~1 us sooner
// (the stated 512/256-row shape: 9.8 us against 10.8 us on pairs), and one that
// fits a wave even in 128 x 128 tiles runs those, over twice as many SMs.
#include "gemm_launch.cuh"

using namespace gg;

namespace {
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}

extern "C" int gg_dual_asym(const gg_bf16* X0, const gg_bf16* X1, const gg_bf16* W0,
                            const gg_bf16* W1, gg_bf16* Y0, gg_bf16* Y1, int64_t m0, int64_t m1,
                            int64_t k, int64_t n0, int64_t n1, int trans_a, int trans_b,
                            int32_t* status, void* stream) {
    if (m0 < 0 || m1 < 0 || k < 0 || n0 < 0 || n1 < 0) return GG_ERR_INVALID_ARG;
    if (m0 % 8 || m1 % 8 || k % 8 || n0 % 8 || n1 % 8) return GG_ERR_UNSUPPORTED;
    const int64_t lim = int64_t(1) << 31;
    if (m0 >= lim || m1 >= lim || k >= lim || n0 >= lim || n1 >= lim) return GG_ERR_UNSUPPORTED;
    const bool e0 = m0 == 0 || n0 == 0, e1 = m1 == 0 || n1 == 0;
    if (e0 && e1) return GG_OK;
    // with k == 0 the X and W operands have no elements (may be NULL)
    const bool kz = k == 0;
    if ((!e0 && (!Y0 || (!kz && (!X0 || !W0)))) || (!e1 && (!Y1 || (!kz && (!X1 || !W1)))))
        return GG_ERR_INVALID_ARG;
    if ((!e0 && (!al16(Y0) || (!kz && (!al16(X0) || !al16(W0))))) ||
        (!e1 && (!al16(Y1) || (!kz && (!al16(X1) || !al16(W1))))))
        return GG_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (k == 0) {
        cudaError_t e = cudaSuccess;
        if (!e0) e = cudaMemsetAsync(Y0, 0, static_cast<size_t>(m0 * n0) * 2, st);
        if (e == cudaSuccess && !e1) e = cudaMemsetAsync(Y1, 0, static_cast<size_t>(m1 * n1) * 2, st);
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
        return GG_OK;
    }
    GemmParams p{};
    p.E = 2;
    p.Kred = static_cast<int>(k);
    p.status = status;
    p.dual[0] = DualProblem{e0 ? 0 : static_cast<int>(m0), e0 ? 0 : static_cast<int>(n0), Y0, n0};
    p.dual[1] = DualProblem{e1 ? 0 : static_cast<int>(m1), e1 ? 0 : static_cast<int>(n1), Y1, n1};
    const int64_t single_tiles = ((m0 + kBM - 1) / kBM) * ((n0 + kBN - 1) / kBN) +
                                 ((m1 + kBM - 1) / kBM) * ((n1 + kBN - 1) / kBN);
    const int64_t narrow_tiles = ((m0 + kBM - 1) / kBM) * ((n0 + kBN / 2 - 1) / (kBN / 2)) +
                                 ((m1 + kBM - 1) / kBM) * ((n1 + kBN / 2 - 1) / (kBN / 2));
    const bool pair = single_tiles > num_sms();
    // one wave even in 128 x 128 tiles: those, so twice as many SMs share the work
    const bool narrow = !pair && narrow_tiles <= num_sms();
    p.narrow = narrow ? 1 : 0;
    CUtensorMap mA[2], mB[2];
    const gg_bf16* Xs[2] = {X0, X1};
    const gg_bf16* Ws[2] = {W0, W1};
    const int64_t ms[2] = {m0, m1}, ns[2] = {n0, n1};
    for (int q = 0; q < 2; ++q) {
        const int src = (q == 0 ? e0 : e1) ? 1 - q : q;  // an empty problem borrows the other's maps
        bool ok;
        if (trans_a) ok = encode_map_2d(&mA[q], Xs[src], ms[src], k, ms[src], 64, kBK);
        else ok = encode_map_2d(&mA[q], Xs[src], k, ms[src], k, kBK, kBM);
        if (!ok) return GG_ERR_CUDA;
        if (trans_b) ok = encode_map_2d(&mB[q], Ws[src], k, ns[src], k, kBK, (pair || narrow) ? kBN / 2 : kBN);
        else ok = encode_map_2d(&mB[q], Ws[src], ns[src], k, ns[src], 64, kBK);
        if (!ok) return GG_ERR_CUDA;
    }
    if (!pair) {
        const int64_t tiles = narrow ? narrow_tiles : single_tiles;
        if (trans_a && trans_b)
            return launch_gemm<KIND_DUAL, true, false, false, false, false>(mA[0], mB[0], mA[1], mB[1], p, tiles, st);
        if (trans_a)
            return launch_gemm<KIND_DUAL, true, true, false, false, false>(mA[0], mB[0], mA[1], mB[1], p, tiles, st);
        if (trans_b)
            return launch_gemm<KIND_DUAL, false, false, false, false, false>(mA[0], mB[0], mA[1], mB[1], p, tiles, st);
        return launch_gemm<KIND_DUAL, false, true, false, false, false>(mA[0], mB[0], mA[1], mB[1], p, tiles, st);
    }
    // pair units: two m-tiles of one problem and one n-tile
    const int64_t bound = ((m0 + 2 * kBM - 1) / (2 * kBM)) * ((n0 + kBN - 1) / kBN) +
                          ((m1 + 2 * kBM - 1) / (2 * kBM)) * ((n1 + kBN - 1) / kBN);
    if (trans_a && trans_b)
        return launch_gemm<KIND_DUAL, true, false, false, false, true>(mA[0], mB[0], mA[1], mB[1], p, bound, st);
    if (trans_a)
        return launch_gemm<KIND_DUAL, true, true, false, false, true>(mA[0], mB[0], mA[1], mB[1], p, bound, st);
    if (trans_b)
        return launch_gemm<KIND_DUAL, false, false, false, false, true>(mA[0], mB[0], mA[1], mB[1], p, bound, st);
    return launch_gemm<KIND_DUAL, false, true, false, false, true>(mA[0], mB[0], mA[1], mB[1], p, bound, st);
}
