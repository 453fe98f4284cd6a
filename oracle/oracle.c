/*
 * oracle.c -- plain, slow, obviously-correct CPU statement of the MoE grouped
 * (ragged) GEMM hot path.  TEST INFRASTRUCTURE ONLY: nothing in the product
 * library links, includes or calls this file.  Only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark load it (through oracle.py).
 *
 * Every floating-point result is accumulated in fp64 in the natural loop order
 * (reduction index ascending).  bf16 values are carried as raw uint16 bit
 * patterns and widened exactly.  Where the pages store a bf16 tensor that a
 * later step reads (the dX rows summed over top-k), the oracle rounds to bf16
 * at that point too, so it follows the same data path the pages describe.
 *
 * Sources (page title, then section):
 *   [U]  unslothai--unsloth  unsloth/kernels/moe/grouped_gemm/interface.py
 *        grouped_gemm_forward / grouped_gemm_dX / grouped_gemm_dW docstrings,
 *        GroupedGemm.backward
 *   [V]  vllm third_party/triton_kernels/matmul_ogs.py
 *        GatherIndx / ScatterIndx, RoutingData.n_blocks, the ragged-dw comment
 *        block with its worked example, matmul_ogs_torch
 *   [W]  VLA/wall_x/fusions/backend.py
 *        asym_dual_gmm_separated, permute, unpermute
 *
 * Parity pins for each function live in tests/test_oracle_*.py.  No function
 * here is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 -- */

/* bf16 -> double, exact: a bf16 is the top 16 bits of an IEEE fp32. */
static double bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16, round to nearest, ties to even, done in one rounding step
 * (no detour through fp32, which could round twice).  bf16 has 8 significant
 * bits and the fp32 exponent range (normal minimum 2^-126, subnormal quantum
 * 2^-133). */
static uint16_t double_to_bf16(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);               /* a = m * 2^e, m in [0.5, 1) */
        int q = e - 8;              /* quantum of an 8-significant-bit number */
        if (q < -133) q = -133;     /* subnormal bf16 quantum */
        double scaled = ldexp(a, -q);      /* exact: power-of-two scaling */
        double n = nearbyint(scaled);      /* default rounding mode: ties to even */
        r = ldexp(n, q);
    }
    float f = (float)r;             /* exact: r already has <= 8 significant bits */
    if (r > 3.3895313892515355e38) f = INFINITY; /* beyond the largest bf16 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t h = (uint16_t)(u >> 16);
    if (neg) h |= 0x8000u;
    return h;
}

void oracle_round_bf16(const double* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(in[i]);
}

void oracle_widen_bf16(const uint16_t* in, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_double(in[i]);
}

/* ----------------------------------------------------------------- route -- */

/* Routing metadata from the router's expert choices.
 *
 * ids[f], f = t*topk + j, is the expert chosen in slot j of token t.
 *   m_sizes[e]        = #{f : ids[f] == e}                 ([U] m_sizes, [V] expt_hist)
 *   offsets[e]        = sum_{e' < e} m_sizes[e'],  offsets[E] = R = T*topk
 *   padded_offsets    = the same prefix over ceil(m_e/b)*b  ([V] ragged-dw example, its padded case)
 *   gather_idx[i]     = the flat slot f held by expert-order row i.  Rows of
 *                       expert e are offsets[e] .. offsets[e+1]-1 and hold its
 *                       slots in ascending f (stable counting sort; the pages
 *                       give no tie rule, this is the reading taken).
 *                       ([U] gather_indices: slicing by cumsum(m_sizes) gives
 *                       each expert's slots; // topk gives the token.)
 *   row_id_map[f]     = the row i with gather_idx[i] == f, i.e. the inverse
 *                       ([V] GatherIndx: dst_indx[src_indx] = arange).
 * Returns 0, or -1 if some id lies outside [0, E) (outputs then undefined). */
int oracle_route(const int32_t* ids, int64_t T, int topk, int E, int pad_block,
                 int32_t* m_sizes, int32_t* offsets, int32_t* padded_offsets,
                 int32_t* gather_idx, int32_t* row_id_map) {
    int64_t R = T * (int64_t)topk;
    if (E <= 0 || T < 0 || topk <= 0) return -1;
    for (int e = 0; e < E; ++e) m_sizes[e] = 0;
    for (int64_t f = 0; f < R; ++f) {
        int32_t e = ids[f];
        if (e < 0 || e >= E) return -1;
        m_sizes[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + m_sizes[e];
    if (padded_offsets) {
        padded_offsets[0] = 0;
        for (int e = 0; e < E; ++e) {
            int32_t b = pad_block;
            int32_t padded = ((m_sizes[e] + b - 1) / b) * b;
            padded_offsets[e + 1] = padded_offsets[e] + padded;
        }
    }
    int32_t* cursor = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t f = 0; f < R; ++f) {
        int32_t e = ids[f];
        int32_t i = offsets[e] + cursor[e];
        cursor[e] += 1;
        gather_idx[i] = (int32_t)f;
        if (row_id_map) row_id_map[f] = i;
    }
    free(cursor);
    return 0;
}

/* Upper bound on the number of block_m-row tiles a ragged split of n_rows rows
 * over E experts can need ([V] RoutingData.n_blocks). */
int64_t oracle_n_blocks(int64_t n_rows, int E, int block_m) {
    if (n_rows <= E) return n_rows;
    int64_t rest = n_rows - E + 1;
    if (rest < 0) rest = 0;
    return (rest + block_m - 1) / block_m + E - 1;
}

/* Start of each expert's slice along a ragged reduction dimension
 * ([V] ragged-dw comment): unpadded slices follow each other; padded slices
 * each occupy a multiple of block_k.  starts[E] is the end of the last one. */
void oracle_ragged_k_starts(const int32_t* hist, int E, int block_k, int padded,
                            int32_t* starts) {
    starts[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t k = hist[e];
        int32_t width = padded ? ((k + block_k - 1) / block_k) * block_k : k;
        starts[e + 1] = starts[e] + width;
    }
}

/* --------------------------------------------------------------- permute -- */

/* Xp[i, :] = X[gather_idx[i] / topk, :]   (token rows into expert order;
 * [W] permute, [U] permute_x "// topk gives the token").  Pure copy. */
void oracle_permute(const uint16_t* X, const int32_t* gather_idx, int64_t R, int topk,
                    int64_t K, uint16_t* Xp) {
    for (int64_t i = 0; i < R; ++i) {
        int64_t t = gather_idx[i] / topk;
        for (int64_t c = 0; c < K; ++c) Xp[i * K + c] = X[t * K + c];
    }
}

/* out[t, :] = sum_j w[t*topk+j] * Y[row(t*topk+j), :], row = row_id_map or
 * identity, w = 1 when absent.  Summed in j order, rounded once to bf16.
 * ([W] unpermute: weighted combine of each token's expert outputs; [V]
 * matmul_ogs_torch: accumulate the rows of every slot of a token.) */
void oracle_unpermute_combine(const uint16_t* Y, const int32_t* row_id_map,
                              const float* topk_w, int64_t T, int topk, int64_t N,
                              double* out) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int j = 0; j < topk; ++j) {
                int64_t f = t * topk + j;
                int64_t row = row_id_map ? row_id_map[f] : f;
                double w = topk_w ? (double)topk_w[f] : 1.0;
                acc += w * bf16_to_double(Y[row * N + n]);
            }
            out[t * N + n] = acc;
        }
    }
}

/* Backward of the combine above ([W] unpermute_bwd: gradients of the
 * unpermute forward, which also takes the forward's input for the
 * probabilities' gradient; prob absent means unit weights).  With G = dL/d out:
 *   dY[row(f)] = w[f] * G[t]                      (every slot f = t*topk + j)
 *   dw[f]      = sum_n G[t, n] * Y[row(f), n]     (skipped when dw == NULL)
 * Y is needed only for dw. */
void oracle_unpermute_combine_bwd(const uint16_t* G, const uint16_t* Y, const int32_t* row_id_map,
                                  const float* topk_w, int64_t T, int topk, int64_t N, double* dY,
                                  double* dw) {
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < topk; ++j) {
            int64_t f = t * topk + j;
            int64_t row = row_id_map ? row_id_map[f] : f;
            double w = topk_w ? (double)topk_w[f] : 1.0;
            double dot = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double g = bf16_to_double(G[t * N + n]);
                dY[row * N + n] = w * g;
                if (dw) dot += g * bf16_to_double(Y[row * N + n]);
            }
            if (dw) dw[f] = dot;
        }
    }
}

/* ------------------------------------------------------- grouped GEMM fwd -- */

/* Expert that owns expert-order row i (offsets is the exclusive prefix). */
static int expert_of_row(const int32_t* offsets, int E, int64_t i) {
    for (int e = 0; e < E; ++e)
        if (i >= offsets[e] && i < offsets[e + 1]) return e;
    return -1;
}

static void prefix(const int32_t* m_sizes, int E, int32_t* offsets) {
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + m_sizes[e];
}

/* One output row of the forward grouped GEMM ([U] grouped_gemm_forward):
 *   A row  = X[gather_idx[i] / topk] if permute_x else X[i]
 *   y[n]   = sum_k A[k] * W[e, n, k]          (W is (E, N, K), K contiguous)
 *   y     *= topk_w[gather_idx[i]]  if fuse_mul_post
 *   stored at row gather_idx[i] (token-major) if permute_y else row i.
 * Returns the destination row. */
static int64_t forward_row(const uint16_t* X, const uint16_t* W, const int32_t* gather_idx,
                           const float* topk_w, int topk, int e, int64_t N, int64_t K,
                           int permute_x, int permute_y, int fuse_mul_post, int64_t i,
                           double* y) {
    int64_t src = permute_x ? (int64_t)(gather_idx[i] / topk) : i;
    const uint16_t* a = X + src * K;
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t* w = W + ((int64_t)e * N + n) * K;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += bf16_to_double(a[k]) * bf16_to_double(w[k]);
        if (fuse_mul_post) acc *= (double)topk_w[gather_idx[i]];
        y[n] = acc;
    }
    return permute_y ? (int64_t)gather_idx[i] : i;
}

/* Full forward: Y is [R, N]; rows not owned by any expert cannot exist
 * because sum(m_sizes) == R. */
void oracle_forward(const uint16_t* X, const uint16_t* W, const int32_t* m_sizes,
                    const int32_t* gather_idx, const float* topk_w, int64_t T, int topk,
                    int E, int64_t N, int64_t K, int permute_x, int permute_y,
                    int fuse_mul_post, double* Y) {
    int64_t R = T * (int64_t)topk;
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    prefix(m_sizes, E, offsets);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < R; ++i) {
        int e = expert_of_row(offsets, E, i);
        double* y = (double*)malloc(sizeof(double) * (size_t)N);
        int64_t dst = forward_row(X, W, gather_idx, topk_w, topk, e, N, K, permute_x,
                                  permute_y, fuse_mul_post, i, y);
        memcpy(Y + dst * N, y, sizeof(double) * (size_t)N);
        free(y);
    }
    free(offsets);
}

/* Sampled forward: the same rows computed one by one for a list of
 * expert-order rows; out is [nrows, N], dest[r] the row it is stored at. */
void oracle_forward_rows(const uint16_t* X, const uint16_t* W, const int32_t* m_sizes,
                         const int32_t* gather_idx, const float* topk_w, int topk, int E,
                         int64_t N, int64_t K, int permute_x, int permute_y,
                         int fuse_mul_post, const int64_t* rows, int64_t nrows,
                         double* out, int64_t* dest) {
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    prefix(m_sizes, E, offsets);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int e = expert_of_row(offsets, E, rows[r]);
        dest[r] = forward_row(X, W, gather_idx, topk_w, topk, e, N, K, permute_x, permute_y,
                              fuse_mul_post, rows[r], out + r * N);
    }
    free(offsets);
}

/* ---------------------------------------------------------------- SwiGLU -- */

/* Gated activation over interleaved gate/up columns ([V] FusedActivation with
 * reduction_n = 2: the activation reduces each pair of adjacent output columns
 * to one).  h is [rows, 2*I] (fp64, e.g. a forward's exact output), act is
 * [rows, I]:  act[r, c] = silu(g) * u,  g = h[r, 2c], u = h[r, 2c + 1],
 * silu(g) = g / (1 + exp(-g)). */
void oracle_swiglu(const double* h, int64_t rows, int64_t I, double* act) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < I; ++c) {
            double g = h[r * 2 * I + 2 * c], u = h[r * 2 * I + 2 * c + 1];
            act[r * I + c] = g / (1.0 + exp(-g)) * u;
        }
}

/* Its gradient: given the stored bf16 H [rows, 2I] and dA = dL/d act [rows, I],
 *   d gate = dA * u * s * (1 + g * (1 - s)),   s = 1 / (1 + exp(-g))
 *   d up   = dA * g * s
 * written interleaved into dH [rows, 2I]. */
void oracle_swiglu_bwd(const uint16_t* H, const uint16_t* dA, int64_t rows, int64_t I,
                       double* dH) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < I; ++c) {
            double g = bf16_to_double(H[r * 2 * I + 2 * c]);
            double u = bf16_to_double(H[r * 2 * I + 2 * c + 1]);
            double d = bf16_to_double(dA[r * I + c]);
            double s = 1.0 / (1.0 + exp(-g));
            dH[r * 2 * I + 2 * c] = d * u * s * (1.0 + g * (1.0 - s));
            dH[r * 2 * I + 2 * c + 1] = d * g * s;
        }
}

/* The same gradient with the upstream dA given exactly (fp64) instead of as
 * stored bf16 values: the form the dX pass reaches when the activation's
 * backward runs on its unrounded output. */
void oracle_swiglu_bwd_f64(const uint16_t* H, const double* dA, int64_t rows, int64_t I,
                           double* dH) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < I; ++c) {
            double g = bf16_to_double(H[r * 2 * I + 2 * c]);
            double u = bf16_to_double(H[r * 2 * I + 2 * c + 1]);
            double d = dA[r * I + c];
            double s = 1.0 / (1.0 + exp(-g));
            dH[r * 2 * I + 2 * c] = d * u * s * (1.0 + g * (1.0 - s));
            dH[r * 2 * I + 2 * c + 1] = d * g * s;
        }
}

/* ------------------------------------------------------------ backward dX -- */

/* One row of dX ([U] grouped_gemm_dX): reduce over N,
 *   dY row = dY[gather_idx[i]] if the forward had permute_y else dY[i]
 *   dx[k]  = sum_n dYrow[n] * W[e, n, k]
 *   stored at row gather_idx[i] (token-slot order) if the forward had
 *   permute_x, else at row i. Returns the destination row. */
static int64_t dX_row(const uint16_t* dY, const uint16_t* W, const int32_t* gather_idx, int e,
                      int64_t N, int64_t K, int permute_x, int permute_y, int64_t i,
                      double* dx) {
    int64_t src = permute_y ? (int64_t)gather_idx[i] : i;
    const uint16_t* g = dY + src * N;
    for (int64_t k = 0; k < K; ++k) dx[k] = 0.0;
    for (int64_t n = 0; n < N; ++n) {
        double gn = bf16_to_double(g[n]);
        const uint16_t* w = W + ((int64_t)e * N + n) * K;
        for (int64_t k = 0; k < K; ++k) dx[k] += gn * bf16_to_double(w[k]);
    }
    return permute_x ? (int64_t)gather_idx[i] : i;
}

void oracle_backward_dX(const uint16_t* dY, const uint16_t* W, const int32_t* m_sizes,
                        const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N,
                        int64_t K, int permute_x, int permute_y, double* dX) {
    int64_t R = T * (int64_t)topk;
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    prefix(m_sizes, E, offsets);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < R; ++i) {
        int e = expert_of_row(offsets, E, i);
        double* dx = (double*)malloc(sizeof(double) * (size_t)K);
        int64_t dst = dX_row(dY, W, gather_idx, e, N, K, permute_x, permute_y, i, dx);
        memcpy(dX + dst * K, dx, sizeof(double) * (size_t)K);
        free(dx);
    }
    free(offsets);
}

void oracle_backward_dX_rows(const uint16_t* dY, const uint16_t* W, const int32_t* m_sizes,
                             const int32_t* gather_idx, int E, int64_t N, int64_t K,
                             int permute_x, int permute_y, const int64_t* rows, int64_t nrows,
                             double* out, int64_t* dest) {
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    prefix(m_sizes, E, offsets);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int e = expert_of_row(offsets, E, rows[r]);
        dest[r] = dX_row(dY, W, gather_idx, e, N, K, permute_x, permute_y, rows[r],
                         out + r * K);
    }
    free(offsets);
}

/* Sum of a token's top-k dX rows ([U] GroupedGemm.backward: dX stored as a
 * bf16 tensor of shape (T*topk, K), then viewed (T, topk, K) and summed over
 * the topk axis).  dX_bf16 is that stored bf16 tensor. */
void oracle_topk_sum(const uint16_t* dX_bf16, int64_t T, int topk, int64_t K, double* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int j = 0; j < topk; ++j)
                acc += bf16_to_double(dX_bf16[(t * topk + j) * K + k]);
            out[t * K + k] = acc;
        }
}

/* ------------------------------------------------------------ backward dW -- */

/* One row dW[e, n, :] ([U] grouped_gemm_dW; [V] ragged-dw comment: the
 * reduction runs over the expert's own rows only):
 *   dW[e, n, k] = sum_{i in expert e} dYrow(i)[n] * Xrow(i)[k]
 *   Xrow(i)  = X[gather_idx[i] / topk] if permute_x else X[i]
 *   dYrow(i) = dY[gather_idx[i]]       if permute_y else dY[i]
 * An expert with no rows gets an all-zero dW[e]. */
static void dW_row(const uint16_t* X, const uint16_t* dY, const int32_t* offsets,
                   const int32_t* gather_idx, int topk, int e, int64_t n, int64_t N, int64_t K,
                   int permute_x, int permute_y, double* dw) {
    for (int64_t k = 0; k < K; ++k) dw[k] = 0.0;
    for (int64_t i = offsets[e]; i < offsets[e + 1]; ++i) {
        int64_t rx = permute_x ? (int64_t)(gather_idx[i] / topk) : i;
        int64_t ry = permute_y ? (int64_t)gather_idx[i] : i;
        double g = bf16_to_double(dY[ry * N + n]);
        const uint16_t* x = X + rx * K;
        for (int64_t k = 0; k < K; ++k) dw[k] += g * bf16_to_double(x[k]);
    }
}

void oracle_backward_dW(const uint16_t* X, const uint16_t* dY, const int32_t* m_sizes,
                        const int32_t* gather_idx, int64_t T, int topk, int E, int64_t N,
                        int64_t K, int permute_x, int permute_y, double* dW) {
    (void)T;
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    prefix(m_sizes, E, offsets);
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
    for (int e = 0; e < E; ++e)
        for (int64_t n = 0; n < N; ++n)
            dW_row(X, dY, offsets, gather_idx, topk, e, n, N, K, permute_x, permute_y,
                   dW + ((int64_t)e * N + n) * K);
    free(offsets);
}

/* Sampled dW: rows (e[r], n[r]) of dW, out is [nrows, K]. */
void oracle_backward_dW_rows(const uint16_t* X, const uint16_t* dY, const int32_t* m_sizes,
                             const int32_t* gather_idx, int topk, int E, int64_t N, int64_t K,
                             int permute_x, int permute_y, const int32_t* es,
                             const int64_t* ns, int64_t nrows, double* out) {
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    prefix(m_sizes, E, offsets);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r)
        dW_row(X, dY, offsets, gather_idx, topk, es[r], ns[r], N, K, permute_x, permute_y,
               out + r * K);
    free(offsets);
}

/* ------------------------------------------------------- dual asymmetric -- */

/* Y = op(Xs) @ op(Ws) for one expert of the dual GEMM ([W]
 * asym_dual_gmm_separated: out0 = in0 @ w0, out1 = in1 @ w1, shared k).
 * Reading of the flags: trans_a means the input is stored (k, m) instead of
 * (m, k); trans_b means the weight is stored (n, k) instead of (k, n). */
static void dense_op_gemm(const uint16_t* Xs, const uint16_t* Ws, int64_t m, int64_t k,
                          int64_t n, int trans_a, int trans_b, double* Y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; ++r)
        for (int64_t c = 0; c < n; ++c) {
            double acc = 0.0;
            for (int64_t q = 0; q < k; ++q) {
                double a = bf16_to_double(trans_a ? Xs[q * m + r] : Xs[r * k + q]);
                double b = bf16_to_double(trans_b ? Ws[c * k + q] : Ws[q * n + c]);
                acc += a * b;
            }
            Y[r * n + c] = acc;
        }
}

void oracle_dual_asym(const uint16_t* X0, const uint16_t* X1, const uint16_t* W0,
                      const uint16_t* W1, int64_t m0, int64_t m1, int64_t k, int64_t n0,
                      int64_t n1, int trans_a, int trans_b, double* Y0, double* Y1) {
    dense_op_gemm(X0, W0, m0, k, n0, trans_a, trans_b, Y0);
    dense_op_gemm(X1, W1, m1, k, n1, trans_a, trans_b, Y1);
}

/* Sampled dual: selected rows of output `which` (0 or 1); out is [nrows, n]. */
void oracle_dual_asym_rows(const uint16_t* Xs, const uint16_t* Ws, int64_t m, int64_t k,
                           int64_t n, int trans_a, int trans_b, const int64_t* rows,
                           int64_t nrows, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < nrows; ++s) {
        int64_t r = rows[s];
        for (int64_t c = 0; c < n; ++c) {
            double acc = 0.0;
            for (int64_t q = 0; q < k; ++q) {
                double a = bf16_to_double(trans_a ? Xs[q * m + r] : Xs[r * k + q]);
                double b = bf16_to_double(trans_b ? Ws[c * k + q] : Ws[q * n + c]);
                acc += a * b;
            }
            out[s * n + c] = acc;
        }
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
