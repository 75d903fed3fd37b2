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
constexpr int kEpiWarps = 4;           // one warp per 32-lane quarter of TMEM
constexpr int kThreads = 32 * (2 + kEpiWarps);  // producer, MMA, 4 epilogue warps
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

struct GemmParams {
    int32_t M, N, K;
    int32_t num_m_blocks;   // ceil(M / (CG * 128))
    int32_t num_n_blocks;   // ceil(N / BN)
    int32_t num_k_blocks;   // ceil(K / 64)
    int32_t num_tiles;      // num_m_blocks * num_n_blocks
    int32_t split_k;        // >= 1; units = num_tiles * split_k
    int32_t num_units;
    int32_t raster_group;   // m-blocks per raster group (>= 1)
    int32_t dtype;          // 0 = bf16, 1 = fp16 (inputs and output)
    uint32_t idesc;         // tcgen05 instruction descriptor
    uint64_t timeout_ns;    // bound on every device-side wait
    uint32_t* status;       // device status word
    float* partials;        // split-K fp32 partial tiles (split_k > 1)
    uint32_t* tile_sems;    // split-K per (tile, cta, warp) turn counters, zero between calls
    int32_t stall_kblock;   // test hook: producer never fills this k-block of unit 0 (< 0: off)
    int32_t pad_;
};

}  // namespace bwgemm
