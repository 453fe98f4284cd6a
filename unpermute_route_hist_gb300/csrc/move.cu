// move.cu -- the two HBM-bound row movers of the MoE path.
//
//  permute            token rows into expert order (wall_x backend.py, permute;
//                     interface.py, permute_x).  Token-stationary: each token
//                     row X[t] is read from HBM once and written to the topk
//                     rows row_id_map[t*topk + j] of Xp.
//  unpermute_combine  expert outputs back to token order with the weighted sum
//                     over a token's slots (backend.py, unpermute; matmul_ogs.py,
//                     matmul_ogs_torch's fp32 accumulation).  Output-stationary
//                     and deterministic: out[t] sums its slots in slot order.
//  swiglu backward    gradient of the gated activation over interleaved gate/up
//                     columns (matmul_ogs.py, FusedActivation, reduction_n = 2).
//  combine backward   its gradient (backend.py, unpermute_bwd): each slot's row
//                     gets the token's output gradient times the slot weight,
//                     and each weight gets <output gradient, forward row>.
//  gather rows        expert-order copies of gathered operands for dW
//                     (interface.py, grouped_gemm_dW with permute_x/permute_y),
//                     so its reduction reads dense tiles.
//  fp32 -> bf16       the final rounding of the fused combine's fp32 sums.
//
// They move whole rows as 16-byte vectors (row widths are multiples of 8
// bf16): permute and combine one warp per token row, the combine backward one
// CTA per token row, in grids of at most 8 CTAs per SM.
#include "common.cuh"

namespace gg {
namespace {

constexpr int kMoveThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

constexpr int kWarpsPerCta = kMoveThreads / 32;
constexpr int kVecsInFlight = 4;  // 16-byte loads each lane keeps in flight

// Slot j's entry of a per-token index held two per lane (j = lane, lane + 32);
// a full-warp shuffle, so every lane must call it with the same j.
__device__ __forceinline__ int32_t slot_entry(int32_t lo, int32_t hi, int j) {
    const int32_t a = __shfl_sync(0xffffffffu, lo, j & 31);
    const int32_t b = __shfl_sync(0xffffffffu, hi, j & 31);
    return j < 32 ? a : b;
}
__device__ __forceinline__ float slot_entry_f(float lo, float hi, int j) {
    const float a = __shfl_sync(0xffffffffu, lo, j & 31);
    const float b = __shfl_sync(0xffffffffu, hi, j & 31);
    return j < 32 ? a : b;
}

// Row index of slot f through the map (identity when NULL); -1 and a status
// code when it is out of range.
__device__ __forceinline__ int32_t mapped_row(const int32_t* map, int64_t f, int64_t R, int32_t* status) {
    int32_t r = map ? map[f] : static_cast<int32_t>(f);
    if (r < 0 || r >= R) {
        set_status(status, GG_DEV_BAD_ROW_INDEX);
        r = -1;
    }
    return r;
}

// One warp per token: its topk destination rows are held in lanes, the row is
// read in passes of 32 lanes x kVecsInFlight 16-byte vectors (all loads of a
// pass in flight together), and each pass is written to every destination.
__global__ void __launch_bounds__(kMoveThreads)
permute_kernel(const uint4* __restrict__ X, const int32_t* __restrict__ row_id_map, int64_t T,
               int topk, int64_t row_vecs, uint4* __restrict__ Xp, int64_t R, int32_t* status) {
    const int lane = lane_id();
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp_id(); t < T; t += nwarps) {
        const int32_t d_lo = lane < topk ? mapped_row(row_id_map, t * topk + lane, R, status) : -1;
        const int32_t d_hi = lane + 32 < topk ? mapped_row(row_id_map, t * topk + lane + 32, R, status) : -1;
        const uint4* src = X + t * row_vecs;
        for (int64_t c0 = 0; c0 < row_vecs; c0 += 32 * kVecsInFlight) {
            uint4 v[kVecsInFlight];
#pragma unroll
            for (int u = 0; u < kVecsInFlight; ++u) {
                const int64_t c = c0 + u * 32 + lane;
                if (c < row_vecs) v[u] = ld_stream(src + c);
            }
            for (int j = 0; j < topk; ++j) {
                const int32_t d = slot_entry(d_lo, d_hi, j);
                if (d < 0) continue;
                uint4* dst = Xp + static_cast<int64_t>(d) * row_vecs;
#pragma unroll
                for (int u = 0; u < kVecsInFlight; ++u) {
                    const int64_t c = c0 + u * 32 + lane;
                    if (c < row_vecs) dst[c] = v[u];
                }
            }
        }
    }
}

__device__ __forceinline__ void bf16x8_fma(float (&acc)[8], const uint4& v, float w) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        acc[2 * q] = fmaf(w, f.x, acc[2 * q]);
        acc[2 * q + 1] = fmaf(w, f.y, acc[2 * q + 1]);
    }
}

// One warp per token: out[t] = sum over slots j (in order) of w_j * Y[row_j],
// fp32, one rounding; passes of 32 lanes x kVecsInFlight vectors, the loads of
// one slot's pass in flight together.
__global__ void __launch_bounds__(kMoveThreads)
combine_kernel(const uint4* __restrict__ Y, const int32_t* __restrict__ row_id_map,
               const float* __restrict__ topk_w, int64_t T, int topk, int64_t row_vecs, int64_t R,
               uint4* __restrict__ out, int32_t* status) {
    const int lane = lane_id();
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp_id(); t < T; t += nwarps) {
        const int32_t s_lo = lane < topk ? mapped_row(row_id_map, t * topk + lane, R, status) : -1;
        const int32_t s_hi = lane + 32 < topk ? mapped_row(row_id_map, t * topk + lane + 32, R, status) : -1;
        const float w_lo = lane < topk ? (topk_w ? topk_w[t * topk + lane] : 1.0f) : 0.0f;
        const float w_hi = lane + 32 < topk ? (topk_w ? topk_w[t * topk + lane + 32] : 1.0f) : 0.0f;
        for (int64_t c0 = 0; c0 < row_vecs; c0 += 32 * kVecsInFlight) {
            float acc[kVecsInFlight][8];
#pragma unroll
            for (int u = 0; u < kVecsInFlight; ++u)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
            for (int j = 0; j < topk; ++j) {
                const int32_t sr = slot_entry(s_lo, s_hi, j);
                const float w = slot_entry_f(w_lo, w_hi, j);
                if (sr < 0) continue;
                const uint4* src = Y + static_cast<int64_t>(sr) * row_vecs;
                uint4 v[kVecsInFlight];
#pragma unroll
                for (int u = 0; u < kVecsInFlight; ++u) {
                    const int64_t c = c0 + u * 32 + lane;
                    if (c < row_vecs) v[u] = ld_stream(src + c);
                }
#pragma unroll
                for (int u = 0; u < kVecsInFlight; ++u)
                    if (c0 + u * 32 + lane < row_vecs) bf16x8_fma(acc[u], v[u], w);
            }
#pragma unroll
            for (int u = 0; u < kVecsInFlight; ++u) {
                const int64_t c = c0 + u * 32 + lane;
                if (c < row_vecs) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                    o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                    o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                    o.w = pack_bf16x2(acc[u][6], acc[u][7]);
                    out[t * row_vecs + c] = o;
                }
            }
        }
    }
}

// Backward of the combine: dY[row(f)] = bf16(w[f] * G[t]); dw[f] = <G[t], Y[row(f)]>.
// One CTA per token; G[t] is read from HBM once (its chunks stay in L1 across the
// token's slots); each slot's dot product is summed per thread, then per warp
// (shuffle tree), then over warps in warp order, so the result is deterministic.
__global__ void __launch_bounds__(kMoveThreads)
combine_bwd_kernel(const uint4* __restrict__ G, const uint4* __restrict__ Y,
                   const int32_t* __restrict__ row_id_map, const float* __restrict__ topk_w,
                   int64_t T, int topk, int64_t row_vecs, int64_t R, uint4* __restrict__ dY,
                   float* __restrict__ dw, int32_t* status) {
    constexpr int kWarps = kMoveThreads / 32;
    __shared__ int32_t row_s[GG_MAX_TOPK];
    __shared__ float w_s[GG_MAX_TOPK];
    __shared__ float part_s[kWarps][GG_MAX_TOPK];
    const int lane = lane_id(), warp = warp_id();
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();
        if (threadIdx.x < topk) {
            const int64_t f = t * topk + threadIdx.x;
            int32_t r = row_id_map ? row_id_map[f] : static_cast<int32_t>(f);
            if (r < 0 || r >= R) {
                set_status(status, GG_DEV_BAD_ROW_INDEX);
                r = -1;
            }
            row_s[threadIdx.x] = r;
            w_s[threadIdx.x] = topk_w ? topk_w[f] : 1.0f;
        }
        __syncthreads();
        const uint4* g_row = G + t * row_vecs;
        for (int j = 0; j < topk; ++j) {
            const int32_t r = row_s[j];
            const float w = w_s[j];
            float dot = 0.f;
            for (int64_t c = threadIdx.x; c < row_vecs; c += kMoveThreads) {
                const uint4 gv = __ldg(g_row + c);
                const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&gv);
                float gf[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f2 = __bfloat1622float2(gh[q]);
                    gf[2 * q] = f2.x;
                    gf[2 * q + 1] = f2.y;
                }
                if (r >= 0) {
                    uint4 o;
                    o.x = pack_bf16x2(w * gf[0], w * gf[1]);
                    o.y = pack_bf16x2(w * gf[2], w * gf[3]);
                    o.z = pack_bf16x2(w * gf[4], w * gf[5]);
                    o.w = pack_bf16x2(w * gf[6], w * gf[7]);
                    dY[static_cast<int64_t>(r) * row_vecs + c] = o;
                    if (dw) {
                        const uint4 yv = ld_stream(Y + static_cast<int64_t>(r) * row_vecs + c);
                        const __nv_bfloat162* yh = reinterpret_cast<const __nv_bfloat162*>(&yv);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 y2 = __bfloat1622float2(yh[q]);
                            dot = fmaf(gf[2 * q], y2.x, dot);
                            dot = fmaf(gf[2 * q + 1], y2.y, dot);
                        }
                    }
                }
            }
            if (dw) {
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, d);
                if (lane == 0) part_s[warp][j] = dot;
            }
        }
        if (dw) {
            __syncthreads();
            if (threadIdx.x < topk) {
                float sum = 0.f;
                for (int q = 0; q < kWarps; ++q) sum += part_s[q][threadIdx.x];
                dw[t * topk + threadIdx.x] = row_s[threadIdx.x] >= 0 ? sum : 0.f;
            }
        }
    }
}

// SwiGLU backward over interleaved gate/up columns: each thread takes 8
// activations (16 bytes of dA) and the 16 matching columns of H, and writes
// the 16 columns of dH.  Grid-stride over 8-activation groups.
__global__ void __launch_bounds__(kMoveThreads)
swiglu_bwd_kernel(const uint4* __restrict__ H, const uint4* __restrict__ dA, int64_t groups,
                  uint4* __restrict__ dH) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kMoveThreads + threadIdx.x; i < groups;
         i += static_cast<int64_t>(gridDim.x) * kMoveThreads) {
        const uint4 dv = ld_stream(dA + i);
        const uint4 h0 = ld_stream(H + 2 * i), h1 = ld_stream(H + 2 * i + 1);
        const __nv_bfloat162* dh = reinterpret_cast<const __nv_bfloat162*>(&dv);
        const __nv_bfloat162* hh[2] = {reinterpret_cast<const __nv_bfloat162*>(&h0),
                                       reinterpret_cast<const __nv_bfloat162*>(&h1)};
        uint32_t outw[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float2 gu = __bfloat1622float2(hh[q >> 2][q & 3]);  // (gate, up) of activation q
            const float2 d2 = __bfloat1622float2(dh[q >> 1]);
            const float d = (q & 1) ? d2.y : d2.x;
            const float s = 1.0f / (1.0f + __expf(-gu.x));
            outw[q] = pack_bf16x2(d * gu.y * s * (1.0f + gu.x * (1.0f - s)), d * gu.x * s);
        }
        dH[2 * i] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
        dH[2 * i + 1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
    }
}

// Row gather into expert order: dst[i] = src[gather_idx[i] / div] for every
// expert-order row i (div = topk: token rows; 1: token-slot rows).  One warp
// per destination row, kVecsInFlight 16-byte loads in flight per lane.  An
// index outside the source sets GG_DEV_BAD_ROW_INDEX and the row is zeroed.
__global__ void __launch_bounds__(kMoveThreads)
gather_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ gather_idx, int div,
                   int64_t src_rows, int64_t R, int64_t row_vecs, uint4* __restrict__ dst,
                   int32_t* status) {
    const int lane = lane_id();
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp_id(); i < R; i += nwarps) {
        const int32_t f = gather_idx[i];
        int64_t r = f < 0 ? -1 : static_cast<int64_t>(static_cast<uint32_t>(f) / static_cast<uint32_t>(div));
        if (r < 0 || r >= src_rows) {
            if (lane == 0) set_status(status, GG_DEV_BAD_ROW_INDEX);
            r = -1;
        }
        const uint4* s = src + r * row_vecs;
        uint4* d = dst + i * row_vecs;
        for (int64_t c0 = 0; c0 < row_vecs; c0 += 32 * kVecsInFlight) {
            uint4 v[kVecsInFlight];
#pragma unroll
            for (int u = 0; u < kVecsInFlight; ++u) {
                const int64_t c = c0 + u * 32 + lane;
                v[u] = (c < row_vecs && r >= 0) ? ld_stream(s + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kVecsInFlight; ++u) {
                const int64_t c = c0 + u * 32 + lane;
                if (c < row_vecs) d[c] = v[u];
            }
        }
    }
}

// fp32 -> bf16 (round to nearest even), 8 values per thread and step.
__global__ void __launch_bounds__(kMoveThreads)
f32_to_bf16_kernel(const float4* __restrict__ src, int64_t groups, uint4* __restrict__ dst) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kMoveThreads + threadIdx.x; i < groups;
         i += static_cast<int64_t>(gridDim.x) * kMoveThreads) {
        const float4 a = src[2 * i], b = src[2 * i + 1];
        dst[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                            pack_bf16x2(b.z, b.w));
    }
}

unsigned move_grid(int64_t rows) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t g = static_cast<int64_t>(sms) * 8;  // 8 resident 256-thread CTAs per SM
    return static_cast<unsigned>(rows < g ? rows : g);
}

}  // namespace

int permute_launch(const uint16_t* X, const int32_t* row_id_map, int64_t T, int topk, int64_t K,
                   uint16_t* Xp, int32_t* status, cudaStream_t stream) {
    const int64_t R = T * topk;
    clear_pending_launch_error();
    permute_kernel<<<move_grid((T + kWarpsPerCta - 1) / kWarpsPerCta), kMoveThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(X), row_id_map, T, topk, K / 8, reinterpret_cast<uint4*>(Xp),
        R, status);
    return launch_result();
}

int swiglu_bwd_launch(const uint16_t* H, const uint16_t* dA, int64_t rows, int64_t I, uint16_t* dH,
                      cudaStream_t stream) {
    const int64_t groups = rows * I / 8;
    int64_t blocks = (groups + kMoveThreads - 1) / kMoveThreads;
    const int64_t cap = static_cast<int64_t>(move_grid(INT64_MAX)) * 4;
    if (blocks > cap) blocks = cap;
    clear_pending_launch_error();
    swiglu_bwd_kernel<<<static_cast<unsigned>(blocks), kMoveThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(H), reinterpret_cast<const uint4*>(dA), groups,
        reinterpret_cast<uint4*>(dH));
    return launch_result();
}

int combine_bwd_launch(const uint16_t* G, const uint16_t* Y, const int32_t* row_id_map,
                       const float* topk_w, int64_t T, int topk, int64_t N, uint16_t* dY, float* dw,
                       int32_t* status, cudaStream_t stream) {
    const int64_t R = T * topk;
    clear_pending_launch_error();
    combine_bwd_kernel<<<move_grid(T), kMoveThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(G), reinterpret_cast<const uint4*>(Y), row_id_map, topk_w, T,
        topk, N / 8, R, reinterpret_cast<uint4*>(dY), dw, status);
    return launch_result();
}

int gather_rows_launch(const uint16_t* src, const int32_t* gather_idx, int div, int64_t src_rows,
                       int64_t R, int64_t cols, uint16_t* dst, int32_t* status, cudaStream_t stream) {
    clear_pending_launch_error();
    gather_rows_kernel<<<move_grid((R + kWarpsPerCta - 1) / kWarpsPerCta), kMoveThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(src), gather_idx, div, src_rows, R, cols / 8,
        reinterpret_cast<uint4*>(dst), status);
    return launch_result();
}

int f32_to_bf16_launch(const float* src, int64_t n, uint16_t* dst, cudaStream_t stream) {
    const int64_t groups = n / 8;
    int64_t blocks = (groups + kMoveThreads - 1) / kMoveThreads;
    const int64_t cap = static_cast<int64_t>(move_grid(INT64_MAX)) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return GG_OK;
    clear_pending_launch_error();
    f32_to_bf16_kernel<<<static_cast<unsigned>(blocks), kMoveThreads, 0, stream>>>(
        reinterpret_cast<const float4*>(src), groups, reinterpret_cast<uint4*>(dst));
    return launch_result();
}

int combine_launch(const uint16_t* Y, const int32_t* row_id_map, const float* topk_w, int64_t T,
                   int topk, int64_t N, uint16_t* out, int32_t* status, cudaStream_t stream) {
    const int64_t R = T * topk;
    clear_pending_launch_error();
    combine_kernel<<<move_grid((T + kWarpsPerCta - 1) / kWarpsPerCta), kMoveThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(Y), row_id_map, topk_w, T, topk, N / 8, R,
        reinterpret_cast<uint4*>(out), status);
    return launch_result();
}

}  // namespace gg
