// route.cu -- routing metadata on the GPU: per-expert histogram (m_sizes),
// exclusive offsets, padded offsets, the stable expert-order permutation
// (gather_idx) and its inverse (row_id_map).
//
// What is computed follows the grouped_gemm interface.py docstrings (m_sizes,
// gather_indices sliced by cumsum(m_sizes)) and matmul_ogs.py (expt_hist,
// GatherIndx/ScatterIndx, the padded ragged layout).  The design is a counting
// sort in four short passes over the R = T*topk slots, split into warp chunks
// of kChunk consecutive slots:
//   1. count     every warp histograms its chunk (warp match, no atomics)
//                into counts[e][chunk]
//   2. scan      one CTA per expert: exclusive scan of counts[e][*] over the
//                chunks, total -> m_sizes[e]
//   3. offsets   one CTA: exclusive scans of m_sizes (plain and padded)
//   4. scatter   every warp walks its chunk again in slot order; a slot's row
//                is offsets[e] + (expert e's count before this chunk) + (its
//                rank among equal ids earlier in the chunk).  Slots therefore
//                land in ascending order within each expert (stable).
// Integer work only: results are exact and independent of scheduling.
#include "common.cuh"

namespace gg {
namespace {

constexpr int kChunk = 256;          // slots per warp chunk (8 rounds of 32)
constexpr int kWarpsPerCta = 4;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Pass 1: counts[e * C + c] = #{slots of chunk c with id e}.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
route_count_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int64_t C,
                   int32_t* __restrict__ counts, int32_t* status) {
    extern __shared__ int32_t hist_all[];
    const int w = warp_id(), lane = lane_id();
    int32_t* hist = hist_all + w * E;
    const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + w;
    if (chunk >= C) return;
    for (int e = lane; e < E; e += 32) hist[e] = 0;
    __syncwarp();
    const int64_t base = chunk * kChunk;
    for (int r = 0; r < kChunk / 32; ++r) {
        const int64_t f = base + r * 32 + lane;
        int e = -1;
        if (f < R) {
            e = ids[f];
            if (e < 0 || e >= E) {
                set_status(status, GG_DEV_BAD_EXPERT_ID);
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int leader = __ffs(peers) - 1;
        if (lane == leader && e >= 0) hist[e] += __popc(peers);
        __syncwarp();
    }
    for (int e = lane; e < E; e += 32) counts[static_cast<int64_t>(e) * C + chunk] = hist[e];
}

// Pass 2: one CTA per expert.  counts[e][*] becomes its exclusive prefix over
// chunks; the total is m_sizes[e].
__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t* __restrict__ counts, int64_t C, int32_t* __restrict__ m_sizes) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry_s;
    const int e = blockIdx.x;
    int32_t* row = counts + static_cast<int64_t>(e) * C;
    const int t = threadIdx.x, lane = lane_id(), w = warp_id();
    const int nw = blockDim.x / 32;
    if (t == 0) carry_s = 0;
    __syncthreads();
    for (int64_t c0 = 0; c0 < C; c0 += blockDim.x) {
        const int64_t c = c0 + t;
        const int32_t v = c < C ? row[c] : 0;
        int32_t x = v;  // inclusive warp scan
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += y;
        }
        if (lane == 31) warp_tot[w] = x;
        __syncthreads();
        if (w == 0) {
            int32_t s = lane < nw ? warp_tot[lane] : 0;
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, s, d);
                if (lane >= d) s += y;
            }
            if (lane < nw) warp_tot[lane] = s;  // inclusive over warps
        }
        __syncthreads();
        const int32_t carry = carry_s;
        const int32_t before_warp = w > 0 ? warp_tot[w - 1] : 0;
        if (c < C) row[c] = carry + before_warp + x - v;
        __syncthreads();
        if (t == 0) carry_s = carry + warp_tot[nw - 1];
        __syncthreads();
    }
    if (t == 0) m_sizes[e] = carry_s;
}

// Pass 3: offsets (and padded offsets) from m_sizes; single CTA.
__global__ void __launch_bounds__(1024)
route_offsets_kernel(const int32_t* __restrict__ m_sizes, int E, int pad_block, int64_t R,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ padded,
                     int32_t* status) {
    __shared__ int32_t warp_tot[2][32];
    __shared__ int32_t carry_s[2];
    const int t = threadIdx.x, lane = lane_id(), w = warp_id();
    const int nw = blockDim.x / 32;
    if (t == 0) carry_s[0] = carry_s[1] = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + t;
        const int32_t v = e < E ? m_sizes[e] : 0;
        const int32_t pv = (e < E && pad_block > 0) ? ((v + pad_block - 1) / pad_block) * pad_block : 0;
        int32_t x = v, px = pv;
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, d);
            const int32_t py = __shfl_up_sync(0xffffffffu, px, d);
            if (lane >= d) { x += y; px += py; }
        }
        if (lane == 31) { warp_tot[0][w] = x; warp_tot[1][w] = px; }
        __syncthreads();
        if (w == 0) {
            int32_t s = lane < nw ? warp_tot[0][lane] : 0;
            int32_t ps = lane < nw ? warp_tot[1][lane] : 0;
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, s, d);
                const int32_t py = __shfl_up_sync(0xffffffffu, ps, d);
                if (lane >= d) { s += y; ps += py; }
            }
            if (lane < nw) { warp_tot[0][lane] = s; warp_tot[1][lane] = ps; }
        }
        __syncthreads();
        const int32_t c0 = carry_s[0], c1 = carry_s[1];
        if (e < E) {
            offsets[e] = c0 + (w > 0 ? warp_tot[0][w - 1] : 0) + x - v;
            if (padded) padded[e] = c1 + (w > 0 ? warp_tot[1][w - 1] : 0) + px - pv;
        }
        __syncthreads();
        if (t == 0) { carry_s[0] = c0 + warp_tot[0][nw - 1]; carry_s[1] = c1 + warp_tot[1][nw - 1]; }
        __syncthreads();
    }
    if (t == 0) {
        offsets[E] = carry_s[0];
        if (padded) padded[E] = carry_s[1];
        if (static_cast<int64_t>(carry_s[0]) != R) set_status(status, GG_DEV_SIZES_MISMATCH);
    }
}

// Pass 4: stable scatter.  run[e] = offsets[e] + counts[e][chunk] is the next
// free row of expert e for this warp; slots are visited in ascending order.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
route_scatter_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int64_t C,
                     const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                     int32_t* __restrict__ gather_idx, int32_t* __restrict__ row_id_map) {
    extern __shared__ int32_t run_all[];
    const int w = warp_id(), lane = lane_id();
    int32_t* run = run_all + w * E;
    const int64_t chunk = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + w;
    if (chunk >= C) return;
    for (int e = lane; e < E; e += 32) run[e] = offsets[e] + counts[static_cast<int64_t>(e) * C + chunk];
    __syncwarp();
    const int64_t base = chunk * kChunk;
    const unsigned lt = lanemask_lt();
    for (int r = 0; r < kChunk / 32; ++r) {
        const int64_t f = base + r * 32 + lane;
        int e = -1;
        if (f < R) {
            e = ids[f];
            if (e < 0 || e >= E) e = -1;  // reported by the count pass
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int32_t pos = 0;
        if (e >= 0) pos = run[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) run[e] += __popc(peers);
        __syncwarp();
        if (e >= 0 && pos >= 0 && pos < R) {
            gather_idx[pos] = static_cast<int32_t>(f);
            if (row_id_map) row_id_map[f] = pos;
        }
    }
}

int64_t num_chunks(int64_t R) { return (R + kChunk - 1) / kChunk; }

}  // namespace

int route_launch(const int32_t* ids, int64_t T, int topk, int E, int pad_block, int32_t* m_sizes,
                 int32_t* offsets, int32_t* padded, int32_t* gather_idx, int32_t* row_id_map,
                 int32_t* counts, int32_t* status, cudaStream_t stream) {
    const int64_t R = T * topk;
    const int64_t C = num_chunks(R);
    const size_t smem = static_cast<size_t>(kWarpsPerCta) * E * sizeof(int32_t);
    const unsigned grid_chunks = static_cast<unsigned>((C + kWarpsPerCta - 1) / kWarpsPerCta);
    clear_pending_launch_error();
    // kWarpsPerCta * E * 4 bytes <= 32 KB for E <= GG_MAX_EXPERTS: default limit.
    if (R > 0) {
        route_count_kernel<<<grid_chunks, kWarpsPerCta * 32, smem, stream>>>(ids, R, E, C, counts,
                                                                            status);
        route_scan_kernel<<<E, 256, 0, stream>>>(counts, C, m_sizes);
    } else {
        const int rc = cuda_result(cudaMemsetAsync(m_sizes, 0, sizeof(int32_t) * E, stream));
        if (rc != GG_OK) return rc;
    }
    route_offsets_kernel<<<1, 1024, 0, stream>>>(m_sizes, E, pad_block, R, offsets,
                                                 pad_block > 0 ? padded : nullptr, status);
    if (R > 0)
        route_scatter_kernel<<<grid_chunks, kWarpsPerCta * 32, smem, stream>>>(
            ids, R, E, C, counts, offsets, gather_idx, row_id_map);
    return launch_result();
}

size_t route_workspace_bytes(int64_t T, int topk, int E) {
    const int64_t R = T * topk;
    const size_t b = static_cast<size_t>(num_chunks(R)) * static_cast<size_t>(E) * sizeof(int32_t);
    return (b + 255) & ~static_cast<size_t>(255);
}

}  // namespace gg
