// kernel_params.h -- host/device shared description of one GEMM launch.
#pragma once

#include <cstdint>

namespace bwgemm {

// Device-side status bits (OR-ed into the plan's status word; 0 = fine).
enum : uint32_t {
    kStatusProducerTimeout = 1u << 0,
    kStatusMmaTimeout = 1u << 1,
    kStatusEpilogueTimeout = 1u << 2,
    kStatusSplitTimeout = 1u << 3,
    kStatusBadConfig = 1u << 4,
};

constexpr int kTileK = 64;             // K elements per pipeline stage (128 B rows: 128B swizzle)
constexpr int kMmaK = 16;              // K per tcgen05.mma of kind::f16 (32 bytes)
constexpr int kRowsPerCta = 128;       // accumulator rows per CTA (TMEM lanes)
constexpr int kEpiWarps = 8;           // two warps per 32-lane quarter of TMEM, half the columns each
constexpr int kThreads = 32 * (2 + kEpiWarps);  // producer, MMA, 8 epilogue warps
constexpr int kCountersPerWarp = 1;    // arrival counters per (tile, cta, epilogue warp)
constexpr int kClcSlots = 4;           // cluster-launch-control responses in flight
constexpr int kStoreCols = 32;         // columns per epilogue store box (64 B rows)

#ifdef __CUDACC__
#define BWGEMM_HD __host__ __device__
#else
#define BWGEMM_HD
#endif

// tcgen05 instruction descriptor of kind::f16 (PTX ISA, "Instruction
// descriptor"): D = f32 (bits 4-5 = 1); A and B = bf16 (1) or f16 (0) at bits
// 7-9 / 10-12; both K-major (bits 15, 16 = 0); N >> 3 at bits 17-22;
// M >> 4 at bits 24-28; dense, no negation, no saturation.
BWGEMM_HD constexpr uint32_t make_idesc(int dtype, int m, int n)
{
    return (1u << 4) | (uint32_t(dtype == 0 ? 1 : 0) << 7) | (uint32_t(dtype == 0 ? 1 : 0) << 10) |
           (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// Work decomposition of one launch.  Tiles are numbered in grouped raster
// order.  Tiles [0, dp_tiles) are "data-parallel": each is one unit, or
// split_k slices of its K range (split-K).  Tiles [dp_tiles, num_tiles) form
// the stream-K region: its sk_tiles * num_k_blocks K-block iterations are
// divided evenly among the workers (CTA pairs, or CTAs for the 1-SM form);
// a worker's range is cut at tile edges into pieces.  Every worker first
// walks its stream-K range, then its data-parallel units (round robin).
struct GemmParams {
    int32_t M, N, K;
    int32_t num_m_blocks;   // ceil(M / (CG * 128))
    int32_t num_n_blocks;   // ceil(N / BN)
    int32_t num_k_blocks;   // ceil(K / 64)
    int32_t num_tiles;      // num_m_blocks * num_n_blocks
    int32_t split_k;        // >= 1 slices per data-parallel tile
    int32_t dp_tiles;       // data-parallel tiles (ids [0, dp_tiles))
    int32_t dp_units;       // dp_tiles * split_k
    int32_t sk_tiles;       // stream-K tiles (ids [dp_tiles, num_tiles))
    int32_t raster_group;   // m-blocks per raster group (>= 1)
    int64_t sk_iters;       // sk_tiles * num_k_blocks
    int32_t dtype;          // 0 = bf16, 1 = fp16 (inputs and output)
    uint32_t idesc;         // tcgen05 instruction descriptor (MMA N = min(BN, 256))
    uint32_t idesc2;        // second MMA of a 320-column unit (N = 64), else 0
    uint64_t timeout_ns;    // bound on every device-side wait
    uint32_t* status;       // device status word
    float* partials;        // fp32 partial tiles of split-K slices / stream-K pieces
    uint32_t* tile_sems;    // per (tile, cta, warp) arrival counters, zero between calls
    int32_t stall_kblock;   // test hook: producer never fills this k-block of its first unit (< 0: off)
    int32_t split_scatter;  // split-K in one wave: the slices of a tile reduce-scatter (see epilogue)
    int32_t prefetch;       // K blocks of the streamed operand the producer prefetches
                            // into L2 ahead of its loads (0: off)
    int32_t prefetch_b;     // the streamed operand: 1 = B, 0 = A
    int32_t clc;            // 1: one cluster per tile, running clusters take over pending ones
                            //    through cluster launch control (whole tiles only)
    uint64_t* trace;        // optional timeline: kTraceSlots %globaltimer stamps per CTA (null: off)
    uint16_t* c;            // C itself, for the boxes a TMA store cannot clip exactly
    int64_t ldc;            // elements between rows of C
    int32_t k_chunks_a;     // whole 64-element K chunks the 3-D view of A covers
    int32_t k_chunks_b;     // (floor(K / 64)) and of B; 0: that view was not built
    int32_t pair_copies;    // 1: load two K blocks per copy where the 3-D views allow
    int32_t ks;             // K slices of a tile inside one cluster (1, or 2: split-K whose
                            // two slices exchange partials through distributed shared memory)
    int32_t c_pairs;        // 1: the second C map stores two 32-column chunks at once
    int32_t c_chunks;       // whole 32-column chunks of a C row the 3-D C view covers
};

// Timeline slots of one CTA (nanoseconds of %globaltimer, 0 = not reached).
enum : int {
    kTraceEntry = 0,          // kernel entry
    kTraceReady = 1,          // barriers, TMEM and the dependency wait done
    kTraceFirstLoad = 2,      // producer issues its first TMA load
    kTraceLastLoad = 3,       // producer issued its last TMA load
    kTraceEpiDone = 4,        // epilogue warp 2 finished (stores complete)
    kTraceExit = 5,           // teardown done
    kTraceSetup = 6,          // barriers, TMEM and the cluster barrier of the prologue done
    kTraceUnitKnown = 7,      // producer worked out its first unit (before the dependency wait)
    kTraceUnit0 = 8,          // then per unit u < kTraceUnits: MMA start, MMA end,
    kTraceUnits = 14,         //   epilogue start, epilogue end (4 slots each)
    kTraceSlots = kTraceUnit0 + 4 * kTraceUnits,
};

}  // namespace bwgemm
