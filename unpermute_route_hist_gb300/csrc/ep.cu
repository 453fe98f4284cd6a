// ep.cu -- expert-parallel layout of the MoE layer across G ranks
// (matmul_ogs.py: FusedComm and post_matmul_comm_torch, the exchange of
// routed rows between the ranks that hold different experts).
//
// Rank r holds the E_loc = E / G experts [r * E_loc, (r + 1) * E_loc).  After
// its own routing, rank r's expert-order rows for the experts of rank d form
// one contiguous block (experts are sorted), so dispatch sends block d to rank
// d.  Rank r receives, from every source rank s, s's rows for r's experts,
// source after source and, within a source, expert after expert:
//     received block (s, e) holds recv_m[s][e] rows.
// The local grouped GEMMs want expert-contiguous rows, so received row j of
// block (s, e), q-th in its block, goes to local expert-order row
//     row_map[j] = local_off[e] + sum_{s' < s} recv_m[s'][e] + q,
// local_off being the exclusive prefix of local_m[e] = sum_s recv_m[s][e].
// Within an expert, rows thus stay in (source rank, source's own) order:
// the order a single routing of all ranks' tokens, numbered rank after
// rank, would give.
//
// gg_ep_plan is host code (the all-to-all splits are host integers anyway);
// gg_ep_recv_map computes the same row map on the device from the received
// count matrix, without a round trip of R_loc integers through the host.
#include <vector>

#include "common.cuh"

namespace gg {
namespace {

constexpr int kMapThreads = 256;
constexpr int kMaxBlocks = GG_MAX_EXPERTS;  // G * E_loc = E <= GG_MAX_EXPERTS

// In-CTA exclusive scan of n (<= kMaxBlocks) values v[idx(i)] taken in the
// order i = 0..n-1; writes out[idx(i)].  Each thread scans a contiguous run.
template <typename Idx>
__device__ void block_exclusive_scan(const int32_t* v, int32_t* out, int n, Idx idx, int32_t* warp_sums) {
    const int per = (n + kMapThreads - 1) / kMapThreads;
    const int lo = min(n, static_cast<int>(threadIdx.x) * per), hi = min(n, lo + per);
    int32_t sum = 0;
    for (int i = lo; i < hi; ++i) sum += v[idx(i)];
    // inclusive scan of the thread sums
    const int lane = lane_id(), w = warp_id();
    int32_t x = sum;
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int32_t s = lane < kMapThreads / 32 ? warp_sums[lane] : 0;
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += y;
        }
        if (lane < kMapThreads / 32) warp_sums[lane] = s;
    }
    __syncthreads();
    int32_t run = (w > 0 ? warp_sums[w - 1] : 0) + x - sum;
    for (int i = lo; i < hi; ++i) {
        out[idx(i)] = run;
        run += v[idx(i)];
    }
    __syncthreads();
}

// row_map[j] for every received row j < R_loc (see the file comment).  Every
// CTA builds the block tables in shared memory, then maps rows grid-stride.
__global__ void __launch_bounds__(kMapThreads)
ep_recv_map_kernel(const int32_t* __restrict__ recv_m, int G, int E_loc, int64_t R_loc,
                   int32_t* __restrict__ row_map, int32_t* status) {
    __shared__ int32_t cnt[kMaxBlocks];
    __shared__ int32_t src_start[kMaxBlocks];  // first received row of block (s, e), s-major
    __shared__ int32_t dst_start[kMaxBlocks];  // its first local row, e-major prefix
    __shared__ int32_t warp_sums[kMapThreads / 32];
    const int n = G * E_loc;
    bool bad = false;
    for (int i = threadIdx.x; i < n; i += kMapThreads) {
        int32_t c = recv_m[i];
        if (c < 0) { bad = true; c = 0; }
        cnt[i] = c;
    }
    __syncthreads();
    // s-major order is the storage order; e-major visits (e, s) as e * G + s
    block_exclusive_scan(cnt, src_start, n, [](int i) { return i; }, warp_sums);
    block_exclusive_scan(cnt, dst_start, n, [G, E_loc](int i) { return (i % G) * E_loc + i / G; }, warp_sums);
    const int64_t total = static_cast<int64_t>(src_start[n - 1]) + cnt[n - 1];
    if (blockIdx.x == 0 && threadIdx.x == 0 && (bad || total != R_loc)) set_status(status, GG_DEV_SIZES_MISMATCH);
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kMapThreads + threadIdx.x; j < R_loc;
         j += static_cast<int64_t>(gridDim.x) * kMapThreads) {
        if (j >= total) { row_map[j] = -1; continue; }
        // the last block whose start is <= j holds row j: an empty block shares
        // its start with the next one, and j < total rules out an empty last block
        int lo = 0, hi = n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (src_start[mid] <= j) lo = mid; else hi = mid - 1;
        }
        row_map[j] = dst_start[lo] + static_cast<int32_t>(j - src_start[lo]);
    }
}

}  // namespace
}  // namespace gg

using namespace gg;

extern "C" {

int gg_ep_plan(const int32_t* m_sizes, const int32_t* recv_m, int G, int E_loc, int64_t* send_counts,
               int64_t* recv_counts, int32_t* local_m_sizes, int32_t* row_map, int64_t row_map_len) {
    if (G < 1 || E_loc < 1 || !m_sizes || !recv_m || !send_counts || !recv_counts || !local_m_sizes)
        return GG_ERR_INVALID_ARG;
    if (static_cast<int64_t>(G) * E_loc > GG_MAX_EXPERTS) return GG_ERR_UNSUPPORTED;
    int64_t total = 0;
    for (int d = 0; d < G; ++d) {
        int64_t s = 0, r = 0;
        for (int e = 0; e < E_loc; ++e) {
            const int32_t a = m_sizes[d * E_loc + e], b = recv_m[d * E_loc + e];
            if (a < 0 || b < 0) return GG_ERR_INVALID_ARG;
            s += a;
            r += b;
        }
        send_counts[d] = s;
        recv_counts[d] = r;
        total += r;
    }
    if (total >= (int64_t(1) << 31)) return GG_ERR_UNSUPPORTED;
    for (int e = 0; e < E_loc; ++e) {
        int64_t c = 0;
        for (int s = 0; s < G; ++s) c += recv_m[s * E_loc + e];
        local_m_sizes[e] = static_cast<int32_t>(c);
    }
    if (!row_map) return GG_OK;
    if (row_map_len != total) return GG_ERR_INVALID_ARG;
    // block (s, e) -> first local row: e-major exclusive prefix
    std::vector<int64_t> dst(static_cast<size_t>(G) * E_loc);
    int64_t run = 0;
    for (int e = 0; e < E_loc; ++e)
        for (int s = 0; s < G; ++s) {
            dst[static_cast<size_t>(s) * E_loc + e] = run;
            run += recv_m[s * E_loc + e];
        }
    int64_t j = 0;  // received rows come block after block, s-major
    for (int s = 0; s < G; ++s)
        for (int e = 0; e < E_loc; ++e)
            for (int32_t q = 0; q < recv_m[s * E_loc + e]; ++q)
                row_map[j++] = static_cast<int32_t>(dst[static_cast<size_t>(s) * E_loc + e] + q);
    return GG_OK;
}

int gg_ep_recv_map(const int32_t* recv_m, int G, int E_loc, int64_t R_loc, int32_t* row_map,
                   int32_t* status, void* stream) {
    if (G < 1 || E_loc < 1 || R_loc < 0) return GG_ERR_INVALID_ARG;
    if (static_cast<int64_t>(G) * E_loc > GG_MAX_EXPERTS || R_loc >= (int64_t(1) << 31))
        return GG_ERR_UNSUPPORTED;
    if (R_loc == 0) return GG_OK;
    if (!recv_m || !row_map) return GG_ERR_INVALID_ARG;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (R_loc + kMapThreads - 1) / kMapThreads;
    if (blocks > 2 * sms) blocks = 2 * sms;
    clear_pending_launch_error();
    ep_recv_map_kernel<<<static_cast<unsigned>(blocks), kMapThreads, 0,
                         reinterpret_cast<cudaStream_t>(stream)>>>(recv_m, G, E_loc, R_loc, row_map,
                                                                   status);
    return launch_result();
}

}  // extern "C"
