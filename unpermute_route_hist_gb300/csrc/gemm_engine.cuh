// gemm_engine.cuh -- persistent, warp-specialised grouped GEMM on tcgen05.
//
// One kernel template serves every grouped contraction of the MoE path:
//   forward  Y_e  = A_e  . W[e]^T    ragged M (each expert's rows), K-major A, B
//   dX       dX_e = dY_e . W[e]      ragged M, K-major A, MN-major B (W read along N)
//   dW       dW_e = dY_e^T . X_e     ragged reduction (each expert's rows),
//                                    MN-major A and B
//   dual     Y_p  = op(X_p) . op(W_p), p = 0, 1, one launch
// (interface.py: grouped_gemm_forward / _dX / _dW; matmul_ogs.py: the ragged
// dw comment; backend.py: asym_dual_gmm_separated.)
//
// Tile: 128 x 256 output, reduction blocks of kBK, a shared-memory ring of
// operand stages, fp32 accumulators in tensor memory (two 256-column buffers
// so the epilogue of one tile overlaps the main loop of the next).
// PAIR: 2-CTA clusters run the cta_group::2 MMA on a 256 x 256 tile made of two
// adjacent m-tiles of the same expert and n-tile.  Each CTA holds its own A
// rows and one half of the B columns (32 KB a stage instead of 48, so six
// stages fit), the even CTA issues the MMA for both, and each CTA's tensor
// memory holds the accumulator of its own 128 rows.  Warp roles:
//   warp 0      tile scheduler + TMA producer (lane 0) for dense operands
//   warp 1      TMEM allocation + MMA issue (lane 0 alone; single-CTA dW: the
//               whole warp joins at a ragged tail stage to zero it)
//   warps 2-5   epilogue: TMEM -> registers -> scale -> bf16 -> global rows
//   warps 6-9   (only with a gathered operand) cp.async row-gather producers;
//               each thread's copies arrive on the stage barrier as they land
//   warp 6      (PAIR dW) each tile's ragged tail block, loaded into its own
//               buffer: zeroes this CTA's rows past the expert's end and
//               signals the even CTA's issuer
// Every role walks the same tile list, decoded from m_sizes in shared memory:
// static (slot + j*nslot, per CTA or cluster), or, with the dynamic schedule of
// the pair kernels over experts, the tile numbers the even CTA's producer takes
// from a per-launch counter and passes to every role of both CTAs through a
// shared-memory queue.  The host side (tensor maps, launches) is gemm_launch.cuh.
//
// Shared-memory operand layouts are the tcgen05 canonical swizzled layouts:
// K-major tiles are rows of kBK bf16 with a swizzle as wide as the row (64-
// or 128-byte), 8-row atoms; MN-major tiles are 64-element MN chunks, each kBK
// reduction rows of 128 B with the 128-byte swizzle.  TMA with the matching
// swizzle writes exactly these; the gather producers write the same swizzle by
// hand (kmajor_chunk_offset, and chunk c of an MN row r at c ^ (r & 7)).
#pragma once

#include <atomic>

#include "common.cuh"

namespace gg {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;                  // reduction block (32 or 64)
constexpr int kMaxStages = 6;
// K-major tiles: rows of kBK bf16 (kKRowBytes), swizzled over the row width
constexpr int kKRowBytes = kBK * 2;
constexpr int kKChunks = kKRowBytes / 16;  // 16-byte chunks per K-major row
constexpr int kABytes = kBM * kBK * 2;
constexpr int kGroupM = 16;             // m-tiles per raster group (L2 reuse)
constexpr int kGatherWarps = 4;
constexpr int kTQ = 8;                  // tile-queue entries (dynamic schedule)
constexpr int kSchedSlots = 1024;       // device tile counters, taken in turn by launches
constexpr int kDynMinBlocksM = 48;      // dynamic schedule from this many reduction blocks a tile
constexpr int kDynMinBlocksK = 32;      // (RAGGED_K: of the mean expert)

enum GemmKind { KIND_RAGGED_M = 0, KIND_RAGGED_K = 1, KIND_DUAL = 2 };
// Row index of a gathered operand row for expert-order row i.
enum RowMode { ROW_DIRECT = 0, ROW_TOKEN = 1 /* gather_idx[i] / topk */, ROW_SLOT = 2 /* gather_idx[i] */ };

struct GatherSrc {
    const uint16_t* ptr;  // base of the source matrix
    int64_t ld;           // elements between consecutive source rows
    int64_t rows;         // number of source rows (bounds check)
    int64_t cols;         // number of valid columns (MN extent or reduction extent)
    int row_mode;
};

struct DualProblem {
    int m, n;
    uint16_t* out;
    int64_t ld_out;
};

struct GemmParams {
    int E, topk;
    int64_t R;
    int M;     // KIND_RAGGED_K: rows of each dW[e]
    int N;     // output columns (per problem for dual: see dual[])
    int Kred;  // reduction length (RAGGED_M, DUAL)
    const int32_t* m_sizes;
    const int32_t* gather_idx;
    GatherSrc ga, gb;        // gathered A / B sources (when gathered)
    uint16_t* out;
    int64_t ld_out;
    int scatter_out;         // RAGGED_M: store row gather_idx[i] instead of i
    const float* scale;      // RAGGED_M: multiply row i by scale[gather_idx[i]]
    // RAGGED_M: add row i (scaled) into token row gather_idx[i] / topk of a
    // zeroed [T, N] output with bf16 atomic adds (the top-k combine, fused)
    int combine_out;
    // RAGGED_M with combine_out: add the scaled fp32 rows into this zeroed
    // [T, N] fp32 buffer with fp32 atomic adds instead (out is then null)
    float* acc_out;
    // RAGGED_M: the output is the upstream gradient dA of a SwiGLU over
    // interleaved gate/up columns; instead of dA, store dH[i, 2c], dH[i, 2c+1]
    // into out (ld_out = 2N) from the stored pre-activation H[i, 2c], H[i, 2c+1]
    const uint16_t* swiglu_h;
    int64_t ld_h;
    // pair, dense: the MN-major maps are 64-column chunk views (one box per
    // operand and stage instead of one per chunk); RAGGED_K: A and B,
    // RAGGED_M: B, a view per expert plane
    int mn_chunk_view;
    // RAGGED_M: also (or only, when out is null) store the gated activation of
    // each pair of adjacent output columns, act[c] = silu(y[2c]) * y[2c+1]
    uint16_t* act_out;
    int64_t ld_act;
    DualProblem dual[2];
    // set at launch of a pair kernel: the output rows (act_out's rows) start 32-byte
    // aligned, so the epilogue stores 32 bytes of a row at a time (st32 also
    // replaces the shared-memory staging of the pair epilogue)
    int st32;
    int act_st32;
    // dynamic schedule (pair kernels with ragged rows or reductions): this launch's
    // counters {tiles handed out past the first wave, pairs finished}, zero at
    // launch and reset to zero by the last pair to finish
    uint32_t* sched;
    // dual problems that fit one wave of SMs in 128 x 128 tiles run them (single
    // CTAs): twice the tiles of 128 x 256, so more SMs share the work
    int narrow;
    int32_t* status;
};

struct TileInfo {
    int e;          // expert (problem index for dual)
    int64_t row0;   // first output row: expert-order row (RAGGED_M), dW row, dual row
    int rows;       // valid output rows in the tile
    int n0;         // first output column
    int64_t red0;   // first reduction row (RAGGED_K), else 0
    int red_len;    // reduction length of the tile
    int nkb;        // reduction blocks
};

// RAGGED_K: experts are scheduled longest first, bucketed by their reduction
// block count in quarter octaves (bucket 0: no rows)
constexpr int kOrdBuckets = 128;
__device__ __forceinline__ int expert_size_bucket(int nblocks) {
    if (nblocks <= 0) return 0;
    const int lg = 31 - __clz(nblocks);
    const int frac = lg >= 2 ? ((nblocks >> (lg - 2)) & 3) : (lg == 1 ? ((nblocks & 1) << 1) : 0);
    return min(kOrdBuckets - 1, 1 + 4 * lg + frac);
}

struct SharedCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull;   // PAIR dW: this CTA's copies of a tile's tail block have landed
    uint64_t pfull;   // PAIR dW, even CTA: both CTAs' tail halves are zeroed
    uint64_t tempty;  // PAIR dW: the tail buffer's MMAs have completed
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int bad_sizes;
    int64_t total_tiles;
    int32_t ord_start[kOrdBuckets];  // RAGGED_K: expert-order counting sort (prologue only)
    // dynamic schedule: the even CTA's producer writes tile numbers into tq of both
    // CTAs (tq_full: one arrival; in the odd CTA also the 4 bytes of an asynchronous
    // remote store); every reader of both CTAs acknowledges an entry on the even
    // CTA's tq_empty before it is rewritten
    int32_t tq[kTQ];
    uint64_t tq_full[kTQ];
    uint64_t tq_empty[kTQ];
};


// Tiles are scheduled in "units": one m-tile, or (PAIR) two adjacent m-tiles
// of the same expert / problem and n-tile that a 2-CTA cluster computes
// together, CTA rank r taking m-tile 2*unit + r.  A rank whose m-tile falls
// past the end gets rows <= 0 (a phantom tile: it still loads its operand
// boxes, its accumulator rows are computed and handed back, nothing is stored).
// TN: output columns of a tile (dual problems in narrow single-CTA tiles: kBN / 2)
template <int KIND, bool PAIR, int TN = kBN>
__device__ __forceinline__ TileInfo decode_tile(int64_t t, const GemmParams& p,
                                                const int32_t* s_off, const int32_t* s_tp,
                                                uint32_t rank) {
    constexpr int U = PAIR ? 2 : 1;
    constexpr int kGroupU = kGroupM / U;  // units per raster group
    TileInfo ti;
    if (KIND == KIND_RAGGED_M) {
        // Units of expert e occupy [s_tp[e]*nt_total, s_tp[e+1]*nt_total).  Inside
        // an expert its units are split into near-equal groups of at most
        // kGroupU; a group sweeps every n-tile with m fastest, so W[e]'s tiles
        // are shared by the group's CTAs in L2 and no group spans two experts.
        const int nt_total = (p.N + kBN - 1) / kBN;
        const int ut_glob = static_cast<int>(t / nt_total);
        int lo = 0, hi = p.E - 1;  // largest e with s_tp[e] <= ut_glob
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_tp[mid] <= ut_glob) lo = mid; else hi = mid - 1;
        }
        const int e = lo;
        const int ut_e = s_tp[e + 1] - s_tp[e];
        const int loc = static_cast<int>(t - static_cast<int64_t>(s_tp[e]) * nt_total);
        // group count rounded to nearest (at least 1): an expert a little taller
        // than kGroupU units stays one group, so W[e] is streamed once
        const int ngroups = max(1, (ut_e + kGroupU / 2) / kGroupU);
        const int gh = (ut_e + ngroups - 1) / ngroups;  // group height
        const int group = loc / (gh * nt_total);
        const int gsize = min(gh, ut_e - group * gh);
        const int gl = loc - group * gh * nt_total;
        const int lmt = (group * gh + gl % gsize) * U + static_cast<int>(rank);
        const int nt = gl / gsize;
        const int me = s_off[e + 1] - s_off[e];
        ti.e = e;
        ti.row0 = static_cast<int64_t>(s_off[e]) + static_cast<int64_t>(lmt) * kBM;
        ti.rows = min(kBM, me - lmt * kBM);
        ti.n0 = nt * kBN;
        ti.red0 = 0;
        ti.red_len = p.Kred;
    } else if (KIND == KIND_RAGGED_K) {
        const int mt_per = (p.M + kBM - 1) / kBM;
        const int ut_per = (mt_per + U - 1) / U;
        const int nt_per = (p.N + kBN - 1) / kBN;
        const int64_t per_e = static_cast<int64_t>(ut_per) * nt_per;
        // tiles come expert after expert in s_tp's order (longest reduction first,
        // written by the prologue in place of RAGGED_M's tile prefix)
        const int pos = static_cast<int>(t / per_e);
        const int e = s_tp[pos];
        const int loc = static_cast<int>(t - static_cast<int64_t>(pos) * per_e);
        // grouped raster inside the expert: kGroupU units x every n-tile, m
        // fastest, so concurrent CTAs share both A and B tiles in L2 and no
        // single tile is read by every SM at once
        const int per_group = kGroupU * nt_per;
        const int group = loc / per_group;
        const int first = group * kGroupU;
        const int gsize = min(ut_per - first, kGroupU);
        const int gl = loc - group * per_group;
        const int mt = (first + gl % gsize) * U + static_cast<int>(rank), nt = gl / gsize;
        ti.e = e;
        ti.row0 = static_cast<int64_t>(mt) * kBM;
        ti.rows = min(kBM, p.M - mt * kBM);
        ti.n0 = nt * kBN;
        ti.red0 = s_off[e];
        ti.red_len = s_off[e + 1] - s_off[e];
    } else {
        const int ut0 = ((p.dual[0].m + kBM - 1) / kBM + U - 1) / U;
        const int64_t tiles0 = static_cast<int64_t>(ut0) * ((p.dual[0].n + TN - 1) / TN);
        const int q = t < tiles0 ? 0 : 1;
        const int64_t lt = q == 0 ? t : t - tiles0;
        const int utq = ((p.dual[q].m + kBM - 1) / kBM + U - 1) / U;
        const int mt = static_cast<int>(lt % utq) * U + static_cast<int>(rank);
        const int nt = static_cast<int>(lt / utq);
        ti.e = q;
        ti.row0 = static_cast<int64_t>(mt) * kBM;
        ti.rows = min(kBM, p.dual[q].m - mt * kBM);
        ti.n0 = nt * TN;
        ti.red0 = 0;
        ti.red_len = p.Kred;
    }
    ti.nkb = (ti.red_len + kBK - 1) / kBK;
    return ti;
}

template <int KIND>
__device__ __forceinline__ int tile_cols(const GemmParams& p, int e) {
    return KIND == KIND_DUAL ? p.dual[e].n : p.N;
}

// Source row of a gathered operand for expert-order row i; -1 if out of range.
__device__ __forceinline__ int64_t gather_row(const GemmParams& p, const GatherSrc& g, int64_t i) {
    int64_t r;
    if (g.row_mode == ROW_DIRECT) {
        r = i;
    } else {
        const int32_t f = p.gather_idx[i];
        r = g.row_mode == ROW_TOKEN ? static_cast<int64_t>(f) / p.topk : static_cast<int64_t>(f);
    }
    if (r < 0 || r >= g.rows) {
        set_status(p.status, GG_DEV_BAD_ROW_INDEX);
        return -1;
    }
    return r;
}

// NARROW: single-CTA dual tiles of 128 x 128 (kBN / 2 output columns).
template <int KIND, bool A_MN, bool B_MN, bool A_GATHER, bool B_GATHER, bool PAIR, bool NARROW = false>
struct GemmTraits {
    static_assert(!(PAIR && (A_GATHER || B_GATHER)), "2-CTA tiles are loaded by TMA only");
    static_assert(!NARROW || (!PAIR && KIND == KIND_DUAL), "narrow tiles: single-CTA dual problems");
    static constexpr int kTileN = NARROW ? kBN / 2 : kBN;  // output columns of a tile
    static constexpr int kTmemCols = 2 * kTileN;           // two fp32 accumulators
    static constexpr bool kAnyGather = A_GATHER || B_GATHER;
    static constexpr bool kCpGatherFence = kAnyGather;  // cp.async-written stages
    static constexpr int kThreads = 32 * (6 + (kAnyGather ? kGatherWarps : 0) + (PAIR && KIND == KIND_RAGGED_K ? 1 : 0));
    // PAIR dW: a five-stage ring plus one buffer for each tile's ragged tail
    // block, which is loaded a few stages into the tile and consumed last
    // (its rows past the expert's end are zeroed meanwhile).
    static constexpr int kStages = PAIR ? (KIND == KIND_RAGGED_K ? 5 : 6) : (NARROW ? 6 : 4);
    static constexpr int kBufStages = kStages + (PAIR && KIND == KIND_RAGGED_K ? 1 : 0);
    static constexpr int kBRows = PAIR ? kBN / 2 : kTileN;  // B tile rows (n) held by one CTA
    static constexpr uint32_t kBBytes = kBRows * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(PAIR ? 2 * kBM : kBM, kTileN, A_MN ? 1 : 0, B_MN ? 1 : 0);
    static constexpr uint32_t kTmaBytes = (A_GATHER ? 0u : kABytes) + (B_GATHER ? 0u : kBBytes);
    static constexpr uint32_t kFullCount = 1 + (kAnyGather ? kGatherWarps * 32 : 0);
    // PAIR: both CTAs' TMA bytes of a stage complete on the even CTA's barrier,
    // except for a ragged reduction's tail block (dW): it goes to the tail
    // buffer, each CTA's copies complete on its own tail barrier (tfull), an
    // extra warp of each CTA zeroes the rows past the expert's end, and both
    // signal the even CTA (pfull).  The MMA issuer stays a single thread that
    // only waits.
    static constexpr bool kTailBuf = PAIR && KIND == KIND_RAGGED_K;
    // pair kernels with ragged rows stage each epilogue warp's rows in shared memory
    // (4 KB a warp) so that global stores go out as whole 128-byte row segments (dW's
    // tiles, long reductions sharing shared-memory bandwidth, measured faster without)
    static constexpr bool kEpiStage = PAIR && KIND == KIND_RAGGED_M;
    // Pair kernels over experts can take tiles from a device counter after the
    // first wave, in tile order, so the pairs that read the same operand tile read
    // it at about the same time (a static round-robin lets them drift apart, and
    // the tile is fetched from DRAM again).  The launch chooses (GemmParams.sched);
    // the dual GEMM keeps the static schedule.
    static constexpr bool kDynSched = PAIR && KIND != KIND_DUAL;
    // readers of a tile-queue entry: even CTA: MMA issuer, 4 epilogue warps (+ the
    // dW tail helper); odd CTA: producer, 4 epilogue warps (+ the tail helper)
    static constexpr int kTqReaders = 10 + (kTailBuf ? 2 : 0);
    static_assert(kStages <= kMaxStages, "stage ring");
    static_assert(kBufStages * kStageBytes <= (PAIR ? 6u : 4u) * (kABytes + (PAIR ? kBN / 2 : kBN) * kBK * 2),
                  "ring fits the shared-memory layout");
};

// per epilogue warp: 32 rows x 128 B of staged output, then the 32 rows' destination pointers
constexpr int kEpiWarpBytes = 4096 + 32 * 8;
constexpr int kEpiStageBytes = 4 * kEpiWarpBytes;

template <bool PAIR>
__host__ __device__ constexpr size_t gemm_smem_bytes(int E) {
    return 1024 /* alignment slack */ +
           static_cast<size_t>(PAIR ? 6 : 4) * (kABytes + (PAIR ? kBN / 2 : kBN) * kBK * 2) +
           (PAIR ? kEpiStageBytes : 0) + sizeof(SharedCtl) + 2 * static_cast<size_t>(E + 1) * sizeof(int32_t) + 16;
}
static_assert(gemm_smem_bytes<true>(GG_MAX_EXPERTS) <= 227 * 1024, "shared memory (pair)");
static_assert(gemm_smem_bytes<false>(GG_MAX_EXPERTS) <= 227 * 1024, "shared memory");

// Byte offset of 16-byte chunk c of row r in a K-major tile: the swizzle XORs
// the chunk index with address bits 7.. (128-byte rows: r & 7; 64-byte rows:
// (r >> 1) & 3), matching TMA's 128-/64-byte swizzle of the same tile.
__host__ __device__ constexpr uint32_t kmajor_chunk_offset(int r, int c) {
    return kKRowBytes == 128 ? static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4))
                             : static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// Shared-memory descriptor of k-step `ks` (16 reduction elements) of an operand tile.
template <bool MN_MAJOR>
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile_addr, int ks) {
    if (MN_MAJOR) {
        // MN chunks of 64 elements are kBK*128 bytes apart (leading offset);
        // 8-row reduction groups are 1 KB apart (stride offset); a k-step is
        // 16 reduction rows = 2 KB further.  128-byte swizzle.
        return smem_desc(tile_addr + ks * 2048, kBK * 128, 1024, kLayoutSw128);
    } else {
        // rows of kKRowBytes, 8-row atoms 8*kKRowBytes apart; a k-step is 32 B
        // along the row.  Swizzle span = row width.
        return smem_desc(tile_addr + ks * 32, 16, 8 * kKRowBytes,
                         kKRowBytes == 128 ? kLayoutSw128 : kLayoutSw64);
    }
}

// DYN: the dynamic tile schedule (a separate instantiation, so the static one
// carries none of its code).
template <int KIND, bool A_MN, bool B_MN, bool A_GATHER, bool B_GATHER, bool PAIR, bool DYN, bool NARROW>
__global__ void __launch_bounds__((GemmTraits<KIND, A_MN, B_MN, A_GATHER, B_GATHER, PAIR, NARROW>::kThreads), 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                    const GemmParams p) {
    using Tr = GemmTraits<KIND, A_MN, B_MN, A_GATHER, B_GATHER, PAIR, NARROW>;
    constexpr int TN = Tr::kTileN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* stage_base = smem;
    constexpr int kStages = Tr::kStages;
    constexpr uint32_t kStageBytes = Tr::kStageBytes;
    uint8_t* epi_stage = smem + Tr::kBufStages * kStageBytes;  // kEpiStageBytes when Tr::kEpiStage
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(epi_stage + (Tr::kEpiStage ? kEpiStageBytes : 0));
    int32_t* s_off = reinterpret_cast<int32_t*>(ctl + 1);
    int32_t* s_tp = s_off + (p.E + 1);

    const int warp = warp_id(), lane = lane_id();
    volatile int* abort_flag = &ctl->abort_flag;
    // persistent schedule: CTAs (or 2-CTA clusters) take units slot, slot + nslot, ...
    // (static), or slot and then units handed out by the launch's counter (DYN)
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;  // PAIR: the CTA that issues the MMAs
    const int64_t slot = PAIR ? static_cast<int64_t>(cluster_id_x()) : static_cast<int64_t>(blockIdx.x);
    const int64_t nslot = PAIR ? static_cast<int64_t>(nclusters_x()) : static_cast<int64_t>(gridDim.x);

    // ---------------------------------------------------------- prologue --
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], Tr::kFullCount);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tmem_full[b], 1);
            // PAIR: the even CTA's barrier also counts the odd CTA's epilogue warps
            mbar_init(&ctl->tmem_empty[b], PAIR ? 8 : 4);
        }
        mbar_init(&ctl->drain, 1);
        mbar_init(&ctl->tfull, 1);
        mbar_init(&ctl->pfull, 2);  // the two CTAs' tail helpers
        mbar_init(&ctl->tempty, 1);
        if (DYN) {
            for (int j = 0; j < kTQ; ++j) {
                mbar_init(&ctl->tq_full[j], 1);
                mbar_init(&ctl->tq_empty[j], Tr::kTqReaders);
            }
        }
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA0);
        tma_prefetch_desc(&tmB0);
        if (KIND == KIND_DUAL) {
            tma_prefetch_desc(&tmA1);
            tma_prefetch_desc(&tmB1);
        }
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(&ctl->tmem_base, Tr::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&ctl->tmem_base, Tr::kTmemCols);
            tmem_relinquish();
        }
    }
    if (warp == 2) {
        // Row offsets and (RAGGED_M) m-tile prefix of the experts: one warp,
        // each lane scans a contiguous segment, then a warp scan of the sums.
        int64_t total_tiles = 0;
        int bad = 0;
        if (KIND == KIND_DUAL) {
            constexpr int U = PAIR ? 2 : 1;
            const int64_t t0 = static_cast<int64_t>(((p.dual[0].m + kBM - 1) / kBM + U - 1) / U) * ((p.dual[0].n + TN - 1) / TN);
            const int64_t t1 = static_cast<int64_t>(((p.dual[1].m + kBM - 1) / kBM + U - 1) / U) * ((p.dual[1].n + TN - 1) / TN);
            total_tiles = t0 + t1;
        } else {
            const int seg = (p.E + 31) / 32;
            const int e_lo = min(p.E, lane * seg), e_hi = min(p.E, e_lo + seg);
            int64_t rsum = 0;
            int tsum = 0;
            for (int e = e_lo; e < e_hi; ++e) {
                const int m = p.m_sizes[e];
                if (m < 0) bad = 1;
                rsum += m > 0 ? m : 0;
                tsum += m > 0 ? ((m + kBM - 1) / kBM + (PAIR ? 1 : 0)) / (PAIR ? 2 : 1) : 0;
            }
            int64_t rx = rsum;
            int tx = tsum;
            for (int d = 1; d < 32; d <<= 1) {
                const int64_t ry = __shfl_up_sync(0xffffffffu, rx, d);
                const int ty = __shfl_up_sync(0xffffffffu, tx, d);
                if (lane >= d) { rx += ry; tx += ty; }
            }
            int64_t rrun = rx - rsum;
            int trun = tx - tsum;
            for (int e = e_lo; e < e_hi; ++e) {
                const int m = max(p.m_sizes[e], 0);
                s_off[e] = static_cast<int32_t>(rrun);
                s_tp[e] = trun;
                rrun += m;
                trun += ((m + kBM - 1) / kBM + (PAIR ? 1 : 0)) / (PAIR ? 2 : 1);
            }
            const int64_t rtot = __shfl_sync(0xffffffffu, rx, 31);
            const int ttot = __shfl_sync(0xffffffffu, tx, 31);
            bad = __any_sync(0xffffffffu, bad);
            if (rtot != p.R) bad = 1;
            if (lane == 0) {
                s_off[p.E] = static_cast<int32_t>(rtot);
                s_tp[p.E] = ttot;
            }
            if (KIND == KIND_RAGGED_M) {
                total_tiles = static_cast<int64_t>(ttot) * ((p.N + kBN - 1) / kBN);
            } else {
                total_tiles = static_cast<int64_t>(p.E) * (((p.M + kBM - 1) / kBM + (PAIR ? 1 : 0)) / (PAIR ? 2 : 1)) *
                              ((p.N + kBN - 1) / kBN);
            }
            if (KIND == KIND_RAGGED_K) {
                // Longest-first expert order into s_tp: a stable counting sort by size
                // bucket, descending.  Chunks of 32 experts are visited in order and
                // ranked within a chunk by lane, so every CTA computes the same order.
                // A dW tile's cost grows with its expert's rows; putting the longest
                // tiles first lets the short ones fill in at the end (of the static
                // round-robin, or of the dynamic hand-out, which then is greedy
                // longest-first) instead of a long tile landing last on one CTA.
                __syncwarp();
                int32_t* cnt = ctl->ord_start;
                for (int b = lane; b < kOrdBuckets; b += 32) cnt[b] = 0;
                __syncwarp();
                const unsigned lt = (1u << lane) - 1u;
                for (int e0 = 0; e0 < p.E; e0 += 32) {
                    const int e = e0 + lane;
                    const int b = e < p.E ? expert_size_bucket((s_off[e + 1] - s_off[e] + kBK - 1) / kBK) : -1;
                    const unsigned peers = __match_any_sync(0xffffffffu, b);
                    if (b >= 0 && (peers & lt) == 0) cnt[b] += __popc(peers);
                    __syncwarp();
                }
                // exclusive prefix in descending bucket order (4 buckets a lane)
                int c4[kOrdBuckets / 32], sum = 0;
#pragma unroll
                for (int q = 0; q < kOrdBuckets / 32; ++q) {
                    c4[q] = cnt[kOrdBuckets - 1 - (lane * (kOrdBuckets / 32) + q)];
                    sum += c4[q];
                }
                int incl = sum;
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += y;
                }
                int run = incl - sum;
                __syncwarp();
#pragma unroll
                for (int q = 0; q < kOrdBuckets / 32; ++q) {
                    cnt[kOrdBuckets - 1 - (lane * (kOrdBuckets / 32) + q)] = run;
                    run += c4[q];
                }
                __syncwarp();
                for (int e0 = 0; e0 < p.E; e0 += 32) {
                    const int e = e0 + lane;
                    const int b = e < p.E ? expert_size_bucket((s_off[e + 1] - s_off[e] + kBK - 1) / kBK) : -1;
                    const unsigned peers = __match_any_sync(0xffffffffu, b);
                    if (b >= 0) s_tp[cnt[b] + __popc(peers & lt)] = e;
                    __syncwarp();
                    if (b >= 0 && (peers & lt) == 0) cnt[b] += __popc(peers);
                    __syncwarp();
                }
            }
        }
        if (lane == 0) {
            ctl->bad_sizes = bad;
            ctl->total_tiles = bad ? 0 : total_tiles;
            if (bad && blockIdx.x == 0) set_status(p.status, GG_DEV_SIZES_MISMATCH);
        }
    }
    tc_fence_before();
    __syncthreads();
    // the partner CTA's barriers must be initialised before any multicast
    // copy or remote arrival reaches them
    if (PAIR) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int64_t total_tiles = ctl->total_tiles;
    const uint32_t stage0 = smem_u32(stage_base);

    // ---------------------------------------------------- tile sequence --
    // Tile k of this CTA's sequence, -1 past the end.  Static schedule: slot +
    // k * nslot.  Dynamic: entry k of the tile queue (one thread per reading role
    // calls it, for every k in turn); the entry is acknowledged on the even CTA's
    // tq_empty as soon as it is read.
    auto ack_entry = [&](int j, int32_t t) {
        if (leader) {
            mbar_arrive(&ctl->tq_empty[j]);
        } else {
            // the arrival's address depends on the value read, so the read has
            // completed before the even CTA can see the arrival and rewrite the entry
            uint32_t remote = mapa_u32(&ctl->tq_empty[j], 0);
            uint32_t z;
            asm volatile("and.b32 %0, %1, 0;" : "=r"(z) : "r"(t));
            mbar_arrive_remote_relaxed(remote + z);
        }
    };
    static_assert(!DYN || Tr::kDynSched, "dynamic schedule: pair kernels over experts");
    constexpr bool dyn = DYN;
    auto read_tile = [&](int k) -> int32_t {
        if (!dyn) {
            const int64_t t = slot + k * nslot;
            return t < total_tiles ? static_cast<int32_t>(t) : -1;
        } else {
            const int j = k % kTQ;
            const uint32_t par = static_cast<uint32_t>(k / kTQ) & 1u;
            // (odd CTA: a cluster-scope acquire, pairing with the release of the even
            // CTA's remote store completing on this barrier)
            if (!mbar_wait(&ctl->tq_full[j], par, abort_flag, p.status, 0, kWaitLimitNs, !leader)) return -1;
            const int32_t t = *reinterpret_cast<volatile int32_t*>(&ctl->tq[j]);
            ack_entry(j, t);
            return t;
        }
    };
    // As read_tile, but only if entry k is already there (the MMA issuer looks
    // ahead with it and must not block while its own tile is in flight).
    auto try_read_tile = [&](int k, int32_t& t) -> bool {
        if (!dyn) {
            const int64_t ts = slot + k * nslot;
            t = ts < total_tiles ? static_cast<int32_t>(ts) : -1;
            return true;
        } else {
            const int j = k % kTQ;
            const uint32_t par = static_cast<uint32_t>(k / kTQ) & 1u;
            if (!(leader ? mbar_try_wait(&ctl->tq_full[j], par) : mbar_try_wait_cluster(&ctl->tq_full[j], par)))
                return false;
            const int32_t v = *reinterpret_cast<volatile int32_t*>(&ctl->tq[j]);
            ack_entry(j, v);
            t = v;
            return true;
        }
    };
    // warp-uniform read_tile (lane 0 reads, every lane gets the tile)
    auto read_tile_warp = [&](int k) -> int32_t {
        if (!dyn) return read_tile(k);
        int32_t t = 0;
        if (lane == 0) t = read_tile(k);
        return __shfl_sync(0xffffffffu, t, 0);
    };

    // Rows [valid, zr_end) of a stage's dense operands hold the next expert's
    // reduction rows: overwrite them with zeros (both operands, so no 0 * inf).
    auto zero_tail = [&](int stage, int valid, int zr_end) {
        const int nz = zr_end - valid;
        if (nz <= 0) return;
        const uint4 z = make_uint4(0, 0, 0, 0);
        uint8_t* st = stage_base + stage * kStageBytes;
        if (!A_GATHER) {
            for (int idx = lane; idx < nz * (kBM / 64) * 8; idx += 32) {
                const int piece = idx & 7, rest = idx >> 3;
                const int cc = rest % (kBM / 64), r = valid + rest / (kBM / 64);
                *reinterpret_cast<uint4*>(st + cc * kBK * 128 + r * 128 + piece * 16) = z;
            }
        }
        if (!B_GATHER) {
            for (int idx = lane; idx < nz * (Tr::kBRows / 64) * 8; idx += 32) {
                const int piece = idx & 7, rest = idx >> 3;
                const int cc = rest % (Tr::kBRows / 64), r = valid + rest / (Tr::kBRows / 64);
                *reinterpret_cast<uint4*>(st + kABytes + cc * kBK * 128 + r * 128 + piece * 16) = z;
            }
        }
        fence_proxy_async_smem();
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            uint32_t tail_uses = 0;  // PAIR dW: tail blocks issued so far
            bool ok = true;
            // dynamic schedule: the even CTA's producer takes the tiles (its first
            // tile is its slot, later ones come from the launch's counter) and
            // writes each into the tile queue of both CTAs
            const bool writer = dyn && leader;
            bool pub_ok = true;
            auto publish = [&](int k, int32_t tv) -> bool {
                const int j = k % kTQ;
                const uint32_t par = static_cast<uint32_t>(k / kTQ) & 1u;
                if (!mbar_wait(&ctl->tq_empty[j], par ^ 1u, abort_flag, p.status)) return false;
                *reinterpret_cast<volatile int32_t*>(&ctl->tq[j]) = tv;
                mbar_arrive(&ctl->tq_full[j]);
                st_async_u32_signal(&ctl->tq[j], &ctl->tq_full[j], 1, static_cast<uint32_t>(tv));
                return true;
            };
            int32_t t = writer ? (slot < total_tiles ? static_cast<int32_t>(slot) : -1) : read_tile(0);
            int npub = 0;  // entries the writer has published
            if (writer) {
                if (publish(0, static_cast<int32_t>(t))) ++npub;
                else { ok = pub_ok = false; t = -1; }
            }
            // The writer asks the counter two tiles ahead (the reply for entry k+1 was
            // asked for as tile k-1 started) and publishes entry k+1 a few blocks into
            // tile k: the counter's latency stays hidden, and the readers (the odd
            // CTA's producer above all) find the entry well before they need it.
            uint32_t g = 0;
            if (writer && t >= 0) g = atomicAdd(p.sched, 1u);
            for (int k = 0; t >= 0; ++k) {
                int32_t t_next = -1;
                bool next_known = !writer;
                uint32_t g_after = 0;
                if (writer) g_after = atomicAdd(p.sched, 1u);
                auto publish_next = [&]() -> bool {
                    if (next_known) return true;
                    next_known = true;
                    const int64_t tn = nslot + static_cast<int64_t>(g);
                    t_next = tn < total_tiles ? static_cast<int32_t>(tn) : -1;
                    if (!publish(k + 1, static_cast<int32_t>(t_next))) { pub_ok = false; return false; }
                    ++npub;
                    return true;
                };
                const TileInfo ti = decode_tile<KIND, PAIR, TN>(t, p, s_off, s_tp, rank);
                const CUtensorMap* mA = (KIND == KIND_DUAL && ti.e == 1) ? &tmA1 : &tmA0;
                const CUtensorMap* mB = (KIND == KIND_DUAL && ti.e == 1) ? &tmB1 : &tmB0;
                // PAIR: one reduction block into (sA, sB), completing on barrier `bar`
                // (a shared::cluster address).  A: this CTA's own m-tile (an odd CTA
                // past the expert's last m-tile still loads its box: those rows are
                // never stored).  B: this CTA's half of the n-tile's columns.
                auto load_pair = [&](uint8_t* sA, uint8_t* sB, uint32_t bar, int32_t red) {
                    const int32_t nb = ti.n0 + static_cast<int32_t>(rank) * (kBN / 2);
                    const bool chunk_view = KIND != KIND_DUAL && p.mn_chunk_view;
                    if (!A_MN) {
                        tma_load_2d_pair(sA, mA, bar, red, static_cast<int32_t>(ti.row0));
                    } else if (chunk_view) {
                        tma_load_3d_pair(sA, mA, bar, 0, red, static_cast<int32_t>(ti.row0 / 64));
                    } else {
#pragma unroll
                        for (int cc = 0; cc < kBM / 64; ++cc)
                            tma_load_2d_pair(sA + cc * kBK * 128, mA, bar, static_cast<int32_t>(ti.row0) + cc * 64, red);
                    }
                    if (!B_MN) {
                        if (KIND == KIND_RAGGED_M) tma_load_3d_pair(sB, mB, bar, red, nb, ti.e);
                        else tma_load_2d_pair(sB, mB, bar, red, nb);
                    } else if (chunk_view) {
                        if (KIND == KIND_RAGGED_M) tma_load_4d_pair(sB, mB, bar, 0, red, nb / 64, ti.e);
                        else tma_load_3d_pair(sB, mB, bar, 0, red, nb / 64);
                    } else {
#pragma unroll
                        for (int cc = 0; cc < Tr::kBRows / 64; ++cc) {
                            if (KIND == KIND_RAGGED_M)
                                tma_load_3d_pair(sB + cc * kBK * 128, mB, bar, nb + cc * 64, red, ti.e);
                            else
                                tma_load_2d_pair(sB + cc * kBK * 128, mB, bar, nb + cc * 64, red);
                        }
                    }
                };
                // PAIR dW: whole reduction blocks go through the ring; the ragged tail
                // block (if any) goes to the tail buffer once kStages + 1 blocks of the
                // tile are issued (or after the last whole block), by when the previous
                // tile's tail has normally been consumed.
                const int nfull = Tr::kTailBuf ? ti.red_len / kBK : ti.nkb;
                const int tail_at = (Tr::kTailBuf && nfull < ti.nkb) ? min(nfull, kStages + 1) : -1;
                for (int kb = 0; kb <= nfull; ++kb) {
                    if (Tr::kTailBuf && kb == tail_at) {
                        if (!mbar_wait(&ctl->tempty, (tail_uses & 1u) ^ 1u, abort_flag, p.status)) { ok = false; break; }
                        uint8_t* tA = stage_base + kStages * kStageBytes;
                        mbar_arrive_expect_tx(&ctl->tfull, kStageBytes);
                        load_pair(tA, tA + kABytes, mapa_u32(&ctl->tfull, rank),
                                  static_cast<int32_t>(ti.red0 + static_cast<int64_t>(nfull) * kBK));
                        ++tail_uses;
                    }
                    if (kb == nfull) break;
                    if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    uint8_t* sA = stage_base + stage * kStageBytes;
                    uint8_t* sB = sA + kABytes;
                    const int32_t red = static_cast<int32_t>(ti.red0 + static_cast<int64_t>(kb) * kBK);
                    if (PAIR) {
                        if (leader) mbar_arrive_expect_tx(&ctl->full[stage], 2 * kStageBytes);
                        load_pair(sA, sB, mapa_u32(&ctl->full[stage], 0), red);
                    } else {
                        if (Tr::kTmaBytes) mbar_arrive_expect_tx(&ctl->full[stage], Tr::kTmaBytes);
                        else mbar_arrive(&ctl->full[stage]);
                        if (!A_GATHER) {
                            if (!A_MN) {
                                tma_load_2d(sA, mA, &ctl->full[stage], red, static_cast<int32_t>(ti.row0));
                            } else {
#pragma unroll
                                for (int cc = 0; cc < kBM / 64; ++cc)
                                    tma_load_2d(sA + cc * kBK * 128, mA, &ctl->full[stage],
                                                static_cast<int32_t>(ti.row0) + cc * 64, red);
                            }
                        }
                        if (!B_GATHER) {
                            if (!B_MN) {
                                if (KIND == KIND_RAGGED_M)
                                    tma_load_3d(sB, mB, &ctl->full[stage], red, ti.n0, ti.e);
                                else
                                    tma_load_2d(sB, mB, &ctl->full[stage], red, ti.n0);
                            } else {
#pragma unroll
                                for (int cc = 0; cc < Tr::kBRows / 64; ++cc) {
                                    if (KIND == KIND_RAGGED_M)
                                        tma_load_3d(sB + cc * kBK * 128, mB, &ctl->full[stage],
                                                    ti.n0 + cc * 64, red, ti.e);
                                    else
                                        tma_load_2d(sB + cc * kBK * 128, mB, &ctl->full[stage],
                                                    ti.n0 + cc * 64, red);
                                }
                            }
                        }
                    }
                    ++issued;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                    if (writer && kb == 2 && !publish_next()) { ok = false; break; }
                }
                if (!ok) break;
                if (writer) {
                    if (!publish_next()) { ok = false; break; }
                    t = t_next;
                    g = g_after;
                } else {
                    t = read_tile(k + 1);
                }
            }
            if (writer) {
                // a producer that gave up still ends its readers' sequences
                if (!ok && pub_ok) publish(npub, -1);
                // This pair takes no more tiles.  The last pair to get here has seen
                // every pair's last request (each precedes its pair's count), so it
                // can reset the counters for the next launch that uses them.
                uint32_t old;
                asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.sched + 1) : "memory");
                if (old == static_cast<uint32_t>(nslot) - 1u) {
                    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p.sched), "r"(0u) : "memory");
                    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p.sched + 1), "r"(0u) : "memory");
                }
            }
            // Let every TMA copy this thread issued land before the CTA can exit.
            // (PAIR, odd CTA: its copies complete on the even CTA's barriers, or
            // on its own tail barrier that its warp 6 waits for; the even CTA's
            // MMAs consume all of them before the teardown's cluster barrier.)
            if (!PAIR || leader) {
                const int64_t pend = issued < kStages ? issued : kStages;
                int dstage = stage;
                uint32_t dphase = phase;
                for (int64_t j = 0; j < pend; ++j) {
                    if (--dstage < 0) { dstage = kStages - 1; dphase ^= 1u; }
                    int dummy = 0;
                    mbar_wait(&ctl->full[dstage], dphase, reinterpret_cast<volatile int*>(&dummy), p.status);
                }
            }
        }
    } else if (warp == 1) {
        if ((!PAIR || leader) && (KIND != KIND_RAGGED_K || Tr::kTailBuf)) {
            // ------------------------------------ MMA issuer (lane 0 alone) --
            // No stage needs the warp (no ragged tails to zero here; a dW pair's
            // tails are zeroed by warp 6 of each CTA), so lane 0 runs the loop by
            // itself: no per-stage shuffle or warp barrier between one stage's
            // MMAs and the next.
            if (lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                uint32_t tail_uses = 0;  // PAIR dW: tail blocks consumed so far
                uint32_t acc_count = 0;
                bool ok = true, any_mma = false;
                // The next tile is decoded right after this tile's first MMAs are
                // issued, while the tensor core works on them, instead of at the
                // tile boundary, where the issuer may be the critical path.  (With
                // the dynamic schedule only if its number is already in the queue:
                // the entry may wait for this tile's loads, so the issuer blocks on
                // it only at the tile's end.)
                int32_t t = read_tile(0);
                TileInfo ti_next = t >= 0 ? decode_tile<KIND, PAIR, TN>(t, p, s_off, s_tp, rank) : TileInfo{};
                int32_t t_next = -1;
                for (int k = 0; t >= 0 && ok; ++k, t = t_next) {
                    const TileInfo ti = ti_next;
                    bool next_decoded = false;
                    auto decode_next = [&](bool block) {
                        if (next_decoded) return;
                        if (block) t_next = read_tile(k + 1);
                        else if (!try_read_tile(k + 1, t_next)) return;
                        next_decoded = true;
                        if (t_next >= 0) ti_next = decode_tile<KIND, PAIR, TN>(t_next, p, s_off, s_tp, rank);
                    };
                    if (ti.nkb == 0) { decode_next(true); continue; }
                    const uint32_t buf = acc_count & 1u;
                    const uint32_t acc_phase = (acc_count >> 1) & 1u;
                    if (!mbar_wait(&ctl->tmem_empty[buf], acc_phase ^ 1u, abort_flag, p.status, 0, kWaitLimitNs, PAIR)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * TN;
                    // a dW pair's ragged tail block (the last, partly filled one) comes
                    // from the tail buffer after the loop, so the per-stage path carries
                    // no tail test: the issue latency after a stage lands is the
                    // critical path
                    const int nfull = Tr::kTailBuf ? static_cast<int>(ti.red_len / kBK) : ti.nkb;
                    // one reduction block: wait for it, issue its MMAs, release its stage
                    auto issue_block = [&](int kb) -> bool {
                        if (!mbar_wait(&ctl->full[stage], phase, abort_flag, p.status)) return false;
                        tc_fence_after();
                        // cp.async writes are generic-proxy; order them before the
                        // tensor core's async-proxy reads of this stage
                        if (Tr::kCpGatherFence) fence_proxy_async_smem();
                        const uint32_t sA = stage0 + stage * kStageBytes;
                        const uint32_t sB = sA + kABytes;
#pragma unroll
                        for (int ks = 0; ks < kBK / 16; ++ks) {
                            const uint64_t ad = operand_desc<A_MN>(sA, ks), bd = operand_desc<B_MN>(sB, ks);
                            const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
                            if (PAIR) umma_bf16_pair(d_tmem, ad, bd, Tr::kIdesc, acc);
                            else umma_bf16(d_tmem, ad, bd, Tr::kIdesc, acc);
                        }
                        if (PAIR) umma_commit_pair(&ctl->empty[stage], 0x3);
                        else umma_commit(&ctl->empty[stage]);
                        any_mma = true;
                        if (++stage == kStages) { stage = 0; phase ^= 1u; }
                        return true;
                    };
                    // the first block is peeled off, so the per-block loop has no test
                    // for the decode
                    if (nfull > 0) {
                        if (!issue_block(0)) { ok = false; break; }
                        decode_next(false);
                    }
                    for (int kb = 1; kb < nfull; ++kb)
                        if (!issue_block(kb)) { ok = false; break; }
                    if (!ok) break;
                    if constexpr (Tr::kTailBuf) if (nfull < ti.nkb) {
                        // both CTAs' halves of the tail block have landed and were zeroed
                        const int valid = static_cast<int>(ti.red_len - static_cast<int64_t>(nfull) * kBK);
                        if (!mbar_wait(&ctl->pfull, tail_uses & 1u, abort_flag, p.status, 0, kWaitLimitNs, true)) {
                            ok = false;
                            break;
                        }
                        ++tail_uses;
                        tc_fence_after();
                        const uint32_t sA = stage0 + kStages * kStageBytes;
                        const uint32_t sB = sA + kABytes;
                        for (int ks = 0; ks < (valid + 15) / 16; ++ks) {
                            const uint64_t ad = operand_desc<A_MN>(sA, ks), bd = operand_desc<B_MN>(sB, ks);
                            umma_bf16_pair(d_tmem, ad, bd, Tr::kIdesc, (nfull > 0 || ks > 0) ? 1u : 0u);
                        }
                        umma_commit_pair(&ctl->tempty, 0x3);  // the tail buffer is free in both CTAs
                        any_mma = true;
                    }
                    decode_next(true);
                    if (PAIR) umma_commit_pair(&ctl->tmem_full[buf], 0x3);
                    else umma_commit(&ctl->tmem_full[buf]);
                    ++acc_count;
                }
                // All MMAs of this thread finish before TMEM is released.
                if (any_mma) {
                    if (PAIR) umma_commit_pair(&ctl->drain, 0x1);
                    else umma_commit(&ctl->drain);
                    int dummy = 0;
                    mbar_wait(&ctl->drain, 0, reinterpret_cast<volatile int*>(&dummy), p.status);
                }
            }
            __syncwarp();
        } else if (!PAIR) {
            // ------------- MMA issuer with ragged tails (single-CTA dW) --
            // Lane 0 waits and issues; the other lanes join it only at a tail
            // stage, to zero the rows past the expert's end.  Every lane walks the
            // same loop (no early exit), so the warp-wide steps at tail stages
            // always match up, also after lane 0 has given up on a wait.
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_count = 0;
            bool ok = true, any_mma = false;
            for (int64_t t = slot; t < total_tiles; t += nslot) {
                const TileInfo ti = decode_tile<KIND, PAIR, TN>(t, p, s_off, s_tp, rank);
                if (ti.nkb == 0) continue;
                const uint32_t buf = acc_count & 1u;
                const uint32_t acc_phase = (acc_count >> 1) & 1u;
                if (lane == 0 && ok) {
                    ok = mbar_wait(&ctl->tmem_empty[buf], acc_phase ^ 1u, abort_flag, p.status, 0, kWaitLimitNs, PAIR);
                    tc_fence_after();
                }
                const uint32_t d_tmem = tmem_base + buf * TN;
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    if (lane == 0 && ok) ok = mbar_wait(&ctl->full[stage], phase, abort_flag, p.status);
                    const uint32_t sA = stage0 + stage * kStageBytes;
                    const uint32_t sB = sA + kABytes;
                    int ksteps = kBK / 16;
                    const int valid = KIND == KIND_RAGGED_K ? min(kBK, ti.red_len - kb * kBK) : kBK;
                    if (valid < kBK) {  // the same for every lane
                        ksteps = (valid + 15) / 16;
                        // lane 0 has seen the stage land (or given up)
                        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) zero_tail(stage, valid, ksteps * 16);
                        __syncwarp();
                    }
                    if (lane == 0 && ok) {
                        tc_fence_after();
                        // cp.async writes are generic-proxy; order them before the
                        // tensor core's async-proxy reads of this stage
                        if (Tr::kAnyGather) fence_proxy_async_smem();
                        for (int ks = 0; ks < ksteps; ++ks) {
                            const uint64_t ad = operand_desc<A_MN>(sA, ks), bd = operand_desc<B_MN>(sB, ks);
                            umma_bf16(d_tmem, ad, bd, Tr::kIdesc, (kb > 0 || ks > 0) ? 1u : 0u);
                        }
                        umma_commit(&ctl->empty[stage]);
                        any_mma = true;
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (lane == 0 && ok) umma_commit(&ctl->tmem_full[buf]);
                ++acc_count;
            }
            // All MMAs of this thread finish before TMEM is released.
            if (lane == 0 && any_mma) {
                umma_commit(&ctl->drain);
                int dummy = 0;
                mbar_wait(&ctl->drain, 0, reinterpret_cast<volatile int*>(&dummy), p.status);
            }
            __syncwarp();
        }
    } else if (warp < 6) {
        // ----------------------------------------------------- epilogue --
        const int q = warp & 3;        // TMEM lane quarter this warp may access
        const uint64_t out_pol = l2_policy_evict_first();
        const int r = q * 32 + lane;   // tile row of this thread
        uint32_t acc_count = 0;
        int64_t t_static = slot;  // static schedule: this CTA's next tile
        for (int k = 0;; ++k) {
            int64_t t;
            if constexpr (DYN) {
                t = read_tile_warp(k);
                if (t < 0) break;
            } else {
                t = t_static;
                if (t >= total_tiles) break;
                t_static += nslot;
            }
            // (PAIR: an odd CTA past its expert's last m-tile has rows <= 0; it
            // still takes part in the accumulator hand-off but stores nothing.)
            const TileInfo ti = decode_tile<KIND, PAIR, TN>(t, p, s_off, s_tp, rank);
            const int ncols = tile_cols<KIND>(p, ti.e);
            // destination row, scale, output base
            uint16_t* out = p.out;
            int64_t ld = p.ld_out;
            int64_t dest = -1;
            float sc = 1.0f;
            if (r < ti.rows) {
                if (KIND == KIND_RAGGED_M) {
                    const int64_t i = ti.row0 + r;
                    dest = i;
                    if (p.scatter_out || p.scale || p.combine_out) {
                        const int32_t f = p.gather_idx[i];
                        if (f < 0 || f >= p.R) { set_status(p.status, GG_DEV_BAD_ROW_INDEX); dest = -1; }
                        else {
                            if (p.scatter_out) dest = f;
                            if (p.combine_out) dest = static_cast<int64_t>(static_cast<uint32_t>(f) / static_cast<uint32_t>(p.topk));
                            if (p.scale) sc = p.scale[f];
                        }
                    }
                } else if (KIND == KIND_RAGGED_K) {
                    dest = static_cast<int64_t>(ti.e) * p.M + ti.row0 + r;
                } else {
                    out = p.dual[ti.e].out;
                    ld = p.dual[ti.e].ld_out;
                    dest = ti.row0 + r;
                }
            }
            uint16_t* orow = (dest >= 0 && out) ? out + dest * ld : nullptr;
            float* frow = (KIND == KIND_RAGGED_M && dest >= 0 && p.acc_out) ? p.acc_out + dest * ld : nullptr;
            uint16_t* arow_out = (KIND == KIND_RAGGED_M && dest >= 0 && p.act_out) ? p.act_out + dest * p.ld_act : nullptr;
            if (ti.nkb == 0) {
                if (orow) {
                    for (int c = ti.n0; c < min(ti.n0 + TN, ncols); c += 8)
                        *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
                }
                continue;
            }
            // staged stores (below): every row's destination pointer goes to shared
            // memory before the wait (its index load completes meanwhile), where the
            // lanes storing that row read it; the work after the accumulator lands
            // is TMEM loads and stores only
            const bool staged = Tr::kEpiStage && out != nullptr && !p.st32;
            uint8_t* stg = epi_stage + q * kEpiWarpBytes;
            uint16_t** srow = reinterpret_cast<uint16_t**>(stg + 4096);
            if (staged) {
                srow[lane] = orow;
                __syncwarp();
            }
            // SwiGLU backward (dX with the stored H): this row's H values for the first
            // kHAhead 16-column steps are loaded before the accumulator lands; each
            // step then loads the step kHAhead further on, so the L2 latency of H is
            // hidden behind four steps of work
            constexpr int kHAhead = 4;
            static_assert((kBN / 16) % kHAhead == 0, "whole groups of steps");
            const uint16_t* hrow = nullptr;
            uint4 hq[kHAhead][4];
            auto load_h = [&](int col0, uint4 (&h)[4]) {
#pragma unroll
                for (int qd = 0; qd < 4; ++qd)
                    if (col0 + qd * 4 < ncols) h[qd] = __ldg(reinterpret_cast<const uint4*>(hrow + 2 * col0 + qd * 8));
            };
            if constexpr (KIND == KIND_RAGGED_M && !Tr::kAnyGather) {
                if (p.swiglu_h && orow) {
                    hrow = p.swiglu_h + dest * p.ld_h;
#pragma unroll
                    for (int j = 0; j < kHAhead; ++j) load_h(ti.n0 + j * 16, hq[j]);
                }
            }
            const uint32_t buf = acc_count & 1u;
            const uint32_t acc_phase = (acc_count >> 1) & 1u;
            if (!warp_wait(&ctl->tmem_full[buf], acc_phase, abort_flag, p.status, 64, PAIR)) break;
            tc_fence_after();
            // hand the accumulator back to the MMA issuer (the even CTA's, for a pair).
            // The TMEM loads have completed (tcgen05.wait::ld) before the arrive, so
            // it needs no cluster-scope release: that would wait for this thread's
            // global stores in flight.
            auto release_acc = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR && rank != 0) mbar_arrive_remote(&ctl->tmem_empty[buf], 0);
                    else mbar_arrive(&ctl->tmem_empty[buf]);
                }
            };
            if (ti.rows <= 0) {
                release_acc();
                ++acc_count;
                continue;
            }
            const uint32_t taddr0 = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * TN;
            // convert and store 32 accumulator columns starting at output column col0,
            // straight from registers (16 bytes of the thread's own row per store)
            auto store_out32 = [&](const uint32_t (&v)[32], int col0) {
                if (KIND == KIND_RAGGED_M && frow) {
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc) {
                        const int col = col0 + pc * 4;
                        if (col < ncols)
                            red_add_f32x4(frow + col, __uint_as_float(v[pc * 4 + 0]) * sc,
                                          __uint_as_float(v[pc * 4 + 1]) * sc,
                                          __uint_as_float(v[pc * 4 + 2]) * sc,
                                          __uint_as_float(v[pc * 4 + 3]) * sc);
                    }
                }
                if (orow) {
                    // eight bf16 of the row, scaled, as one 16-byte piece
                    auto piece = [&](int pc) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(v[pc * 8 + 0]) * sc, __uint_as_float(v[pc * 8 + 1]) * sc);
                        o.y = pack_bf16x2(__uint_as_float(v[pc * 8 + 2]) * sc, __uint_as_float(v[pc * 8 + 3]) * sc);
                        o.z = pack_bf16x2(__uint_as_float(v[pc * 8 + 4]) * sc, __uint_as_float(v[pc * 8 + 5]) * sc);
                        o.w = pack_bf16x2(__uint_as_float(v[pc * 8 + 6]) * sc, __uint_as_float(v[pc * 8 + 7]) * sc);
                        return o;
                    };
                    if constexpr (PAIR) {
                        // both pieces of a step formed first: one 32-byte store when the
                        // row is 32-byte aligned (st32) and both are in range
#pragma unroll
                        for (int pc = 0; pc < 4; pc += 2) {
                            const int col = col0 + pc * 8;
                            const uint4 o0 = piece(pc), o1 = piece(pc + 1);
                            if (KIND == KIND_RAGGED_M && p.combine_out) {
                                if (col < ncols) red_add_bf16x8(orow + col, o0);
                                if (col + 8 < ncols) red_add_bf16x8(orow + col + 8, o1);
                            } else if (p.st32 && col + 8 < ncols) {
                                st_global_32_policy(orow + col, o0, o1, out_pol);
                            } else {
                                if (col < ncols) st_global_16_policy(orow + col, o0, out_pol);
                                if (col + 8 < ncols) st_global_16_policy(orow + col + 8, o1, out_pol);
                            }
                        }
                    } else {
#pragma unroll
                        for (int pc = 0; pc < 4; ++pc) {
                            const int col = col0 + pc * 8;
                            if (col < ncols) {
                                if (KIND == KIND_RAGGED_M && p.combine_out) red_add_bf16x8(orow + col, piece(pc));
                                else st_global_16_policy(orow + col, piece(pc), out_pol);
                            }
                        }
                    }
                }
            };
            auto store_act32 = [&](const uint32_t (&v)[32], int col0) {
                if (arow_out) {
                    // 16 gate/up pairs of this chunk -> 16 activations (two 16-byte
                    // pieces; one 32-byte store when act_st32 and both are in range)
                    auto piece = [&](int pc) {
                        float a[8];
#pragma unroll
                        for (int qq = 0; qq < 8; ++qq) {
                            const float g = __uint_as_float(v[pc * 16 + 2 * qq]);
                            const float u = __uint_as_float(v[pc * 16 + 2 * qq + 1]);
                            a[qq] = g / (1.0f + __expf(-g)) * u;
                        }
                        uint4 o;
                        o.x = pack_bf16x2(a[0], a[1]);
                        o.y = pack_bf16x2(a[2], a[3]);
                        o.z = pack_bf16x2(a[4], a[5]);
                        o.w = pack_bf16x2(a[6], a[7]);
                        return o;
                    };
                    if constexpr (PAIR) {
                        const uint4 o0 = piece(0), o1 = piece(1);
                        if (p.act_st32 && col0 + 16 < ncols) {
                            st_global_32_policy(arow_out + col0 / 2, o0, o1, out_pol);
                        } else {
                            if (col0 < ncols) st_global_16_policy(arow_out + col0 / 2, o0, out_pol);
                            if (col0 + 16 < ncols) st_global_16_policy(arow_out + col0 / 2 + 8, o1, out_pol);
                        }
                    } else {
#pragma unroll
                        for (int pc = 0; pc < 2; ++pc)
                            if (col0 + pc * 16 < ncols) st_global_16_policy(arow_out + col0 / 2 + pc * 8, piece(pc), out_pol);
                    }
                }
            };
            // Staged store of 64 columns (va: col0.., vb: col0+32..): every lane writes
            // its row's 128 bytes to the warp's staging rows (16-byte pieces rotated by
            // row, so neither phase has bank conflicts), then eight lanes per row write
            // four whole 128-byte row segments per store instruction.  Every lane of
            // the warp takes part (shuffles and warp barriers).
            auto store_out64_staged = [&](const uint32_t (&va)[32], const uint32_t (&vb)[32], int col0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t* v = j < 4 ? va : vb;
                    const int b = (j & 3) * 8;
                    uint4 o;
                    o.x = pack_bf16x2(__uint_as_float(v[b + 0]) * sc, __uint_as_float(v[b + 1]) * sc);
                    o.y = pack_bf16x2(__uint_as_float(v[b + 2]) * sc, __uint_as_float(v[b + 3]) * sc);
                    o.z = pack_bf16x2(__uint_as_float(v[b + 4]) * sc, __uint_as_float(v[b + 5]) * sc);
                    o.w = pack_bf16x2(__uint_as_float(v[b + 6]) * sc, __uint_as_float(v[b + 7]) * sc);
                    *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
                }
                __syncwarp();
                const int j = lane & 7;
                const int col = col0 + j * 8;
                // all eight shared-memory reads are issued before the first global
                // store (the stores' memory clobber would otherwise serialise each
                // read's latency behind the previous store)
                uint4 o[8];
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int row = (lane >> 3) + 4 * it;
                    o[it] = *reinterpret_cast<const uint4*>(stg + row * 128 + ((j ^ (row & 7)) << 4));
                }
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    uint16_t* dr = srow[(lane >> 3) + 4 * it];
                    if (dr && col < ncols) {
                        if (KIND == KIND_RAGGED_M && p.combine_out) red_add_bf16x8(dr + col, o[it]);
                        else st_global_16_policy(dr + col, o[it], out_pol);
                    }
                }
                __syncwarp();
            };
            // (dense operands only: the 10-warp gather kernels have no registers to spare)
            if constexpr (KIND == KIND_RAGGED_M && !Tr::kAnyGather) if (p.swiglu_h) {
                // SwiGLU backward on the fp32 accumulator (dA), 16 columns a step;
                // each 8-H group gives 4 (gate, up) gradient pairs.  The H rows of
                // this CTA's next tile are prefetched into L2 now (that epilogue
                // runs a whole main loop later), and each step's 32 H values are
                // loaded kHAhead steps ahead (above), so the stores do not wait.
                {
                    const int64_t tn = t + nslot;
                    if (tn < total_tiles) {
                        const TileInfo tni = decode_tile<KIND, PAIR, TN>(tn, p, s_off, s_tp, rank);
                        if (r < tni.rows) {
                            const char* hn = reinterpret_cast<const char*>(p.swiglu_h + (tni.row0 + r) * p.ld_h + 2 * tni.n0);
                            const int nbytes = 4 * min(kBN, ncols - tni.n0);  // 2 H values per column
                            for (int b = 0; b < nbytes; b += 128) prefetch_l2(hn + b);
                        }
                    }
                }
                // groups of kHAhead steps: the ring slot is a compile-time index and
                // the loop body stays small (the whole 16-step loop unrolled ran
                // twice as slow)
#pragma unroll 1
                for (int cg = 0; cg < kBN / 16; cg += kHAhead)
#pragma unroll
                for (int j = 0; j < kHAhead; ++j) {
                    const int c = cg + j;
                    const int col0 = ti.n0 + c * 16;
                    uint4 (&hv)[4] = hq[j];
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(taddr0 + c * 16, v);
                    tmem_ld_wait();
                    if (c == kBN / 16 - 1) release_acc();
                    if (hrow) {
#pragma unroll
                        for (int qd = 0; qd < 4; ++qd) {
                            if (col0 + qd * 4 < ncols) {
                                const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&hv[qd]);
                                uint32_t o[4];
#pragma unroll
                                for (int a = 0; a < 4; ++a) {
                                    const float2 gu = __bfloat1622float2(hh[a]);  // (gate, up)
                                    const float d = __uint_as_float(v[qd * 4 + a]);
                                    const float sg = 1.0f / (1.0f + __expf(-gu.x));
                                    o[a] = pack_bf16x2(d * gu.y * sg * (1.0f + gu.x * (1.0f - sg)), d * gu.x * sg);
                                }
                                st_global_16_policy(orow + 2 * col0 + qd * 8, make_uint4(o[0], o[1], o[2], o[3]), out_pol);
                            }
                        }
                        // this slot's next use is kHAhead steps on
                        if (c + kHAhead < kBN / 16) load_h(col0 + kHAhead * 16, hq[j]);
                    }
                }
                ++acc_count;
                continue;
            }
            // Four 32-column TMEM loads per wait: the loads' latency is paid once per
            // 128 columns.  The accumulator is handed back to the MMA warp as soon as
            // the last load has landed in registers, before its columns are stored.
            constexpr int kColsPerWait = 128;
#pragma unroll 1
            for (int c = 0; c < TN / kColsPerWait; ++c) {
                uint32_t v0[32], v1[32], v2[32], v3[32];
                const uint32_t ta = taddr0 + c * kColsPerWait;
                tmem_ld_32x32b_x32(ta, v0);
                tmem_ld_32x32b_x32(ta + 32, v1);
                tmem_ld_32x32b_x32(ta + 64, v2);
                tmem_ld_32x32b_x32(ta + 96, v3);
                tmem_ld_wait();
                if (c == TN / kColsPerWait - 1) release_acc();
                const int col0 = ti.n0 + c * kColsPerWait;
                if (staged) {
                    store_act32(v0, col0);
                    store_act32(v1, col0 + 32);
                    store_out64_staged(v0, v1, col0);
                    store_act32(v2, col0 + 64);
                    store_act32(v3, col0 + 96);
                    store_out64_staged(v2, v3, col0 + 64);
                } else {
                    store_act32(v0, col0);
                    store_out32(v0, col0);
                    store_act32(v1, col0 + 32);
                    store_out32(v1, col0 + 32);
                    store_act32(v2, col0 + 64);
                    store_out32(v2, col0 + 64);
                    store_act32(v3, col0 + 96);
                    store_out32(v3, col0 + 96);
                }
            }
            ++acc_count;
        }
    } else if (Tr::kTailBuf) {
        // ----------------------------- warp 6 of a dW pair: ragged tail blocks --
        // For each tile with a tail block: wait for this CTA's copies of it (tfull,
        // one phase per tail block), zero the rows past the expert's end in this
        // CTA's operands, and signal the even CTA's issuer (pfull counts both
        // CTAs).  The odd CTA's signal is a cluster-scope release: its zeroed rows
        // are read by the pair's MMA issued from the even CTA.  The block was
        // loaded a few stages into the tile and is consumed at its end, so this
        // work overlaps the tile's main loop.
        uint32_t tail_uses = 0;
        for (int k = 0;; ++k) {
            const int32_t t = read_tile_warp(k);
            if (t < 0) break;
            const TileInfo ti = decode_tile<KIND, PAIR, TN>(t, p, s_off, s_tp, rank);
            const int nfull = ti.red_len / kBK;
            if (nfull == ti.nkb) continue;
            if (!warp_wait(&ctl->tfull, tail_uses & 1u, abort_flag, p.status)) break;
            ++tail_uses;
            zero_tail(kStages, ti.red_len - nfull * kBK, ((ti.red_len - nfull * kBK + 15) / 16) * 16);
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(&ctl->pfull);
                else mbar_arrive_cluster(&ctl->pfull, 0);
            }
            __syncwarp();
        }
    } else {
        // ---------------------------------------------- gather producers --
        // Index loads run one step ahead of the copies that need them: the slot
        // numbers for the next stage (MN-major, dW) or the next tile (K-major)
        // are loaded while the current copies are issued, so no cp.async waits
        // on a dependent index load.
        if (Tr::kAnyGather) {
            const int gt = threadIdx.x - 6 * 32;  // 0 .. 127
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // K-major gathered A: thread gt copies chunk gt % kKChunks of rows
            // gt / kKChunks + kARowStep * j (fixed over the tile).
            constexpr int kARowStep = 128 / kKChunks;
            constexpr int kARows = kBM / kARowStep;
            int32_t a_next[kARows];
            auto fetch_a_rows = [&](int64_t tt) {
#pragma unroll
                for (int j = 0; j < kARows; ++j) a_next[j] = -1;
                if (tt < total_tiles) {
                    const TileInfo tn = decode_tile<KIND, PAIR, TN>(tt, p, s_off, s_tp, rank);
#pragma unroll
                    for (int j = 0; j < kARows; ++j) {
                        const int rr = gt / kKChunks + kARowStep * j;
                        if (rr < tn.rows) a_next[j] = p.gather_idx[tn.row0 + rr];
                    }
                }
            };
            // MN-major gathered operands (dW): the kBK slot numbers of a stage are
            // loaded cooperatively (lane L holds rows kIPL*L .. kIPL*L+kIPL-1) three
            // stages before use, then handed to the copying threads by shuffle.
            constexpr int kIPL = kBK / 32;  // slot numbers per lane (1 or 2)
            const int glane = gt & 31;
            int32_t q_lo[4], q_hi[4];  // look-ahead ring: stage kb in entry kb % 4 (below)
            auto load_stage_idx = [&](const TileInfo& tn, int kb, int32_t& lo, int32_t& hi) {
                const int64_t k0 = static_cast<int64_t>(kb) * kBK + kIPL * glane;
                lo = (kb < tn.nkb && k0 < tn.red_len) ? p.gather_idx[tn.red0 + k0] : -1;
                hi = (kIPL == 2 && kb < tn.nkb && k0 + 1 < tn.red_len) ? p.gather_idx[tn.red0 + k0 + 1] : -1;
            };
            // slot number of reduction row rr of the current stage.  Full-warp
            // shuffles: every lane must call it, whatever its own row or column
            // validity (a lane that skipped it would leave the warp waiting).
            auto stage_slot = [&](int32_t lo, int32_t hi, int rr) -> int32_t {
                const int32_t l = __shfl_sync(0xffffffffu, lo, rr / kIPL);
                const int32_t h = __shfl_sync(0xffffffffu, hi, rr / kIPL);
                return (kIPL == 2 && (rr & 1)) ? h : l;
            };
            // slot number -> source row of a gathered operand, -1 if absent or out of range
            auto src_row = [&](const GatherSrc& g, int32_t f) -> int64_t {
                if (f < 0) return -1;
                // 32-bit division: slot numbers are below 2^31
                const int64_t r = g.row_mode == ROW_TOKEN ? static_cast<int64_t>(static_cast<uint32_t>(f) / static_cast<uint32_t>(p.topk))
                                                          : static_cast<int64_t>(f);
                if (r >= g.rows) { set_status(p.status, GG_DEV_BAD_ROW_INDEX); return -1; }
                return r;
            };
            if (A_GATHER && !A_MN) fetch_a_rows(slot);
            for (int64_t t = slot; t < total_tiles && ok; t += nslot) {
                const TileInfo ti = decode_tile<KIND, PAIR, TN>(t, p, s_off, s_tp, rank);
                const uint16_t* arow[kARows];
                if (A_GATHER && !A_MN) {
#pragma unroll
                    for (int j = 0; j < kARows; ++j) {
                        const int64_t sr = src_row(p.ga, a_next[j]);
                        arow[j] = sr >= 0 ? p.ga.ptr + sr * p.ga.ld : nullptr;
                    }
                    fetch_a_rows(t + nslot);
                }
                constexpr bool kRedGather = (A_GATHER && A_MN) || B_GATHER;
                if (kRedGather) {
                    load_stage_idx(ti, 0, q_lo[0], q_hi[0]);
                    load_stage_idx(ti, 1, q_lo[1], q_hi[1]);
                    load_stage_idx(ti, 2, q_lo[2], q_hi[2]);
                }
                // one reduction block: wait for its stage, gather its rows, arrive when they land
                auto do_stage = [&](int kb, int32_t cur_lo, int32_t cur_hi) -> bool {
                    if (!warp_wait(&ctl->empty[stage], phase ^ 1u, abort_flag, p.status, 32)) return false;
                    const uint32_t sA = stage0 + stage * kStageBytes;
                    const uint32_t sB = sA + kABytes;
                    // source rows of this lane's kIPL reduction rows, once a stage; the
                    // copies below take them by shuffle
                    int32_t ar_lo = -1, ar_hi = -1, br_lo = -1, br_hi = -1;
                    if (A_GATHER && A_MN) {
                        ar_lo = static_cast<int32_t>(src_row(p.ga, cur_lo));
                        ar_hi = kIPL == 2 ? static_cast<int32_t>(src_row(p.ga, cur_hi)) : -1;
                    }
                    if (B_GATHER) {
                        br_lo = static_cast<int32_t>(src_row(p.gb, cur_lo));
                        br_hi = kIPL == 2 ? static_cast<int32_t>(src_row(p.gb, cur_hi)) : -1;
                    }
                    if (A_GATHER) {
                        if (!A_MN) {
                            const int c = gt % kKChunks;
                            const int64_t col = static_cast<int64_t>(kb) * kBK + c * 8;
                            const bool cv = col < p.ga.cols;
#pragma unroll
                            for (int j = 0; j < kARows; ++j) {
                                const int rr = gt / kKChunks + kARowStep * j;
                                const uint32_t dst = sA + kmajor_chunk_offset(rr, c);
                                const bool v = cv && arow[j] != nullptr;
                                cp_async_16(dst, v ? static_cast<const void*>(arow[j] + col) : p.ga.ptr, v ? 16u : 0u);
                            }
                        } else {
                            // MN-major: reduction rows are gathered rows; 16 pieces of 8 elements per row.
                            const int pc = gt & 15;
                            const int64_t mn = ti.row0 + pc * 8;
                            const bool mv = mn < p.ga.cols;
#pragma unroll
                            for (int j = 0; j < kBK / 8; ++j) {
                                const int rr = (gt >> 4) + 8 * j;
                                const int32_t r = stage_slot(ar_lo, ar_hi, rr);  // every lane shuffles
                                const int64_t sr = mv ? r : -1;
                                const uint32_t dst = sA + (pc >> 3) * (kBK * 128) + rr * 128 + (((pc & 7) ^ (rr & 7)) << 4);
                                cp_async_16(dst, sr >= 0 ? static_cast<const void*>(p.ga.ptr + sr * p.ga.ld + mn) : p.ga.ptr,
                                            sr >= 0 ? 16u : 0u);
                            }
                        }
                    }
                    if (B_GATHER) {
                        // Only MN-major gathered B occurs (dW with the forward's token gather).
                        const int pc = gt & 31;
                        const int64_t mn = static_cast<int64_t>(ti.n0) + pc * 8;
                        const bool mv = mn < p.gb.cols;
#pragma unroll
                        for (int j = 0; j < kBK / 4; ++j) {
                            const int rr = (gt >> 5) + 4 * j;
                            const int32_t r = stage_slot(br_lo, br_hi, rr);  // every lane shuffles
                            const int64_t sr = mv ? r : -1;
                            const uint32_t dst = sB + (pc >> 3) * (kBK * 128) + rr * 128 + (((pc & 7) ^ (rr & 7)) << 4);
                            cp_async_16(dst, sr >= 0 ? static_cast<const void*>(p.gb.ptr + sr * p.gb.ld + mn) : p.gb.ptr,
                                        sr >= 0 ? 16u : 0u);
                        }
                    }
                    // the stage's barrier gets this thread's arrival when its copies land
                    cp_async_mbar_arrive(&ctl->full[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                    return true;
                };
                // The index look-ahead ring: stage kb's slot numbers sit in entry kb % 4,
                // loaded three stages before.  Four stages an outer step keep every entry
                // index a compile-time constant, so no register is moved while its load
                // is in flight (a rotating ring would wait for each new load at once).
                if constexpr (kRedGather) {
                    for (int kb0 = 0; kb0 < ti.nkb && ok; kb0 += 4) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int kb = kb0 + u;
                            if (kb >= ti.nkb) break;
                            load_stage_idx(ti, kb + 3, q_lo[(u + 3) & 3], q_hi[(u + 3) & 3]);
                            if (!do_stage(kb, q_lo[u], q_hi[u])) { ok = false; break; }
                        }
                    }
                } else {
                    for (int kb = 0; kb < ti.nkb; ++kb)
                        if (!do_stage(kb, 0, 0)) { ok = false; break; }
                }
            }
            // every copy lands before the CTA can exit
            cp_async_wait<0>();
        }
    }

    // ----------------------------------------------------------- teardown --
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves while the other may still signal it
    tc_fence_after();
    if (warp == 1) {
        if (PAIR) tmem_dealloc_pair(tmem_base, Tr::kTmemCols);
        else tmem_dealloc(tmem_base, Tr::kTmemCols);
    }
}

}  // namespace gg
