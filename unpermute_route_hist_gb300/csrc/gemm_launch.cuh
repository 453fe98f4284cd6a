// gemm_launch.cuh -- host side of the grouped GEMM engine: tensor-map encoders
// (defined in abi.cu) and launch_gemm, which picks the kernel instantiation (tile
// schedule, dual tile width), sets the launch-time parameters and launches the
// persistent grid (one CTA per SM, or one 2-CTA cluster per SM pair).
#pragma once

#include "gemm_engine.cuh"

namespace gg {

// Process-wide tile schedule mode (GG_SCHEDULE_*), set by gg_set_gemm_schedule.
extern std::atomic<int> g_gemm_schedule;

// One device's tile counters for the dynamic schedule, two words a launch slot.
static __device__ uint32_t g_sched[2 * kSchedSlots];
// Next launch slot, per device index.
static std::atomic<uint32_t> g_sched_next[64];

// ------------------------------------------------------------------ host --

bool encode_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer);
bool encode_map_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_elems, uint64_t stride2_elems, uint32_t b0, uint32_t b1);
bool encode_map_mn_chunks(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                          uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_chunks);
bool encode_map_mn_chunks_planes(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                                 uint64_t planes, uint64_t row_stride_elems,
                                 uint64_t plane_stride_elems, uint32_t box_rows,
                                 uint32_t box_chunks);
int num_sms();

template <int KIND, bool A_MN, bool B_MN, bool A_GATHER, bool B_GATHER, bool PAIR>
int launch_gemm(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
                const CUtensorMap& b1, const GemmParams& p, int64_t tile_bound, cudaStream_t stream) {
    using Tr = GemmTraits<KIND, A_MN, B_MN, A_GATHER, B_GATHER, PAIR>;
    const size_t smem = gemm_smem_bytes<PAIR>(p.E);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
    if (dev < 0 || dev >= 64) dev = 0;
    const int64_t sms = num_sms();
    if (tile_bound < 1) tile_bound = 1;
    // 32-byte stores need every destination row 32-byte aligned: the base and the
    // row pitch (a multiple of 16 bf16)
    GemmParams q = p;
    auto rows32 = [](const void* base, int64_t ld) {
        return base != nullptr && (reinterpret_cast<uintptr_t>(base) & 31u) == 0 && ld % 16 == 0;
    };
    if (KIND == KIND_DUAL)
        q.st32 = (p.dual[0].m == 0 || rows32(p.dual[0].out, p.dual[0].ld_out)) &&
                 (p.dual[1].m == 0 || rows32(p.dual[1].out, p.dual[1].ld_out));
    else
        q.st32 = rows32(p.out, p.ld_out);
    q.act_st32 = rows32(p.act_out, p.ld_act);
    if (!PAIR) q.st32 = q.act_st32 = 0;
    // Dynamic schedule for long tiles: its hand-off costs a few hundred cycles a
    // tile, and lock-step co-readers of short tiles meet their DRAM misses all at
    // once, so short tiles keep the static round-robin (measured: dynamic wins
    // 1-4% at 64-448 reduction blocks a tile and loses 2-6% at 12-24).  RAGGED_K:
    // the mean expert's reduction length.  This launch's pair of tile counters is
    // taken in turn; tile numbers travel as 32-bit values.
    q.sched = nullptr;
    const int64_t mean_blocks = KIND == KIND_RAGGED_K ? p.R / (kBK * (p.E > 0 ? p.E : 1)) : p.Kred / kBK;
    const int mode = g_gemm_schedule.load(std::memory_order_relaxed);
    const bool dyn = mode == GG_SCHEDULE_DYNAMIC ||
                     (mode == GG_SCHEDULE_AUTO && mean_blocks >= (KIND == KIND_RAGGED_K ? kDynMinBlocksK : kDynMinBlocksM));
    // (past 2^30 tiles the static schedule, whose tile numbers are 64-bit)
    if (Tr::kDynSched && dyn && tile_bound <= (int64_t(1) << 30)) {
        static std::atomic<void*> sched_base[64];
        void* base = sched_base[dev].load(std::memory_order_acquire);
        if (!base) {
            e = cudaGetSymbolAddress(&base, g_sched);
            if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
            sched_base[dev].store(base, std::memory_order_release);
        }
        const uint32_t s = g_sched_next[dev].fetch_add(1u, std::memory_order_relaxed) % kSchedSlots;
        q.sched = static_cast<uint32_t*>(base) + 2 * s;
    }
    auto kern = grouped_gemm_kernel<KIND, A_MN, B_MN, A_GATHER, B_GATHER, PAIR, false, false>;
    int kid = 0;
    if constexpr (Tr::kDynSched)
        if (q.sched) { kern = grouped_gemm_kernel<KIND, A_MN, B_MN, A_GATHER, B_GATHER, PAIR, true, false>; kid = 1; }
    if constexpr (KIND == KIND_DUAL && !PAIR)
        if (p.narrow) { kern = grouped_gemm_kernel<KIND, A_MN, B_MN, A_GATHER, B_GATHER, PAIR, false, true>; kid = 2; }
    // the shared-memory opt-in is set once per kernel and device (host overhead
    // matters for small launches)
    static std::atomic<bool> smem_set[3][64];
    if (!smem_set[kid][dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(gemm_smem_bytes<PAIR>(GG_MAX_EXPERTS)));
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
        smem_set[kid][dev].store(true, std::memory_order_release);
    }
    clear_pending_launch_error();
    if (!PAIR) {
        const int64_t grid = tile_bound < sms ? tile_bound : sms;
        kern<<<static_cast<unsigned>(grid), Tr::kThreads, smem, stream>>>(a0, b0, a1, b1, q);
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(Tr::kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // as many 2-CTA clusters as can be resident at once (a GPC with an odd
        // SM count leaves an SM out), at most one per tile pair
        // (the same for both schedules' kernels: same block, registers and shared memory)
        static std::atomic<int> max_clusters[64];
        int mc = max_clusters[dev].load(std::memory_order_relaxed);
        if (mc == 0) {
            cfg.gridDim = dim3(static_cast<unsigned>(sms & ~int64_t(1)));
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            if (e != cudaSuccess || n < 1) {
                record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidConfiguration);
                return GG_ERR_CUDA;
            }
            max_clusters[dev].store(n, std::memory_order_relaxed);
            mc = n;
        }
        const int64_t clusters = tile_bound < mc ? tile_bound : mc;
        cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
        e = cudaLaunchKernelEx(&cfg, kern, a0, b0, a1, b1, q);
        if (e != cudaSuccess) { record_cuda_error(e); return GG_ERR_CUDA; }
    }
    return launch_result();
}

}  // namespace gg
