// gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   C[M x N] = A[M x K] * B[N x K]^T, A and B K-major bf16/fp16, fp32
//   accumulation in TMEM, bf16/fp16 output.
//
// Structure (one CTA per SM, or one CTA pair per two SMs when CG == 2):
//   warp 0      TMA producer: fills a STAGES-deep ring of 64-wide K blocks of A
//               and B (128B-swizzled), guarded by full/empty mbarrier pairs.
//   warp 1      TMEM allocator; lane 0 (of the leader CTA) issues every
//               tcgen05.mma and commits stage release / accumulator-ready.
//   warps 2..5  epilogue: tcgen05.ld -> fp32 -> bf16/fp16 -> swizzled smem ->
//               TMA store, double-buffered per warp; with split-K, every
//               split writes an fp32 partial and the last to arrive sums
//               them in split order and stores C.
// Two fp32 accumulators live in TMEM (2 x BN columns), so the epilogue of one
// work unit overlaps the MMAs of the next.  Work units (tile, k-split) are
// handed out statically in a grouped raster order.
//
// Where the pages describe each part:
//   ring + phase tracking, producer/consumer warps, empty barriers passing on
//   the first lap: "Writing a Blackwell GEMM by hand", steps 2 and 3;
//   "Matrix Multiplication on NVIDIA's Blackwell", Kernel 6.
//   128B swizzle with 64-wide K tiles: CuTeDSL post step 4; deep dive Kernel 3
//   and the appendix on the Swizzle<3,4,3> functor.
//   first MMA overwrites, later ones accumulate; 4 MMAs of K=16 per 64-wide
//   block: CuTeDSL post step 1; deep dive Kernel 2.
//   TMEM accumulator and tcgen05.ld epilogue: CuTeDSL post, TMEM section.
//   TMA-store epilogue, double-buffered: deep dive Kernels 4 and 7.
//   2-SM MMA (cta_group::2, 256-row tiles, leader CTA issues): deep dive
//   Kernel 5.
//   TMEM accumulator ring (accum_full / accum_empty), persistent CTAs:
//   deep dive Kernel 8.  Grouped rasterisation for L2 reuse: Kernel 9.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernel_params.h"
#include "ptx.cuh"

namespace bwgemm {

template <int CG, int BN, int STAGES>
struct KernelConfig {
    static_assert(CG == 1 || CG == 2, "CTA group is 1 or 2");
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN in [64, 256], multiple of 32");
    static constexpr int kTileM = CG * kRowsPerCta;             // rows per work unit
    static constexpr int kBRows = (CG == 1) ? BN : BN / 2;      // B rows this CTA loads
    static constexpr int kABytes = kRowsPerCta * kTileK * 2;    // 16 KiB
    static constexpr int kBBytes = kBRows * kTileK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;       // per CTA
    static constexpr int kTxBytes = kStageBytes * CG;           // landing per stage on the leader
    static constexpr int kStoreBufBytes = 32 * kStoreCols * 2;  // one 32 x 32 output box
    static constexpr int kTmemCols = 2 * BN;                    // two fp32 accumulators
    static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                  "TMEM allocation is a power of two in [32, 512] columns");
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffStore = kOffB + STAGES * kBBytes;
    static constexpr int kOffBar = kOffStore + kEpiWarps * 2 * kStoreBufBytes;
    static constexpr int kNumBars = 2 * STAGES + 4;  // full[S], empty[S], acc_full[2], acc_empty[2]
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KiB
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms need 1 KiB alignment");
    static_assert(kSmemBytes <= 227 * 1024, "exceeds the 227 KiB shared memory of one CTA");
    // bytes of one CTA's fp32 partial tile (split-K)
    static constexpr int kPartialFloats = kRowsPerCta * BN;
};

// tcgen05 shared-memory descriptor of a K-major operand tile written by TMA
// with 128B swizzle: rows of 128 bytes (64 elements), 8-row swizzle atoms of
// 1 KiB stacked along M/N (stride byte offset = 1024).  The leading byte
// offset is not used by swizzled K-major layouts (set to 16 B).  Bits 46-48
// hold the fixed value 0b001; bits 61-63 the swizzle mode (2 = 128B).
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t smem)
{
    uint64_t d = 0;
    d |= uint64_t((smem & 0x3FFFFu) >> 4);
    d |= uint64_t(16 >> 4) << 16;
    d |= uint64_t(1024 >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

struct WorkUnit {
    int tile, split;
    int m_blk, n_blk;
    int kb0, kb1;  // K blocks [kb0, kb1)
};

__device__ __forceinline__ WorkUnit decode_unit(const GemmParams& p, int u)
{
    WorkUnit w;
    const int S = p.split_k;
    w.tile = u / S;
    w.split = u - w.tile * S;
    w.kb0 = int((long long)w.split * p.num_k_blocks / S);
    w.kb1 = int((long long)(w.split + 1) * p.num_k_blocks / S);
    // grouped raster: walk `raster_group` m-blocks down, then step along N
    const int G = p.raster_group;
    const int per_group = G * p.num_n_blocks;
    const int g = w.tile / per_group;
    const int first_m = g * G;
    const int gm = min(p.num_m_blocks - first_m, G);
    const int local = w.tile - g * per_group;
    w.m_blk = first_m + local % gm;
    w.n_blk = local / gm;
    return w;
}

// Bounded wait on an mbarrier phase.  Gives up after p.timeout_ns (recording
// `code` in the status word) or as soon as another role of this CTA gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const GemmParams& p,
                                           volatile uint32_t* abort_flag, uint32_t code)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::global_timer_ns();
#pragma unroll 1
    while (true) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (ptx::global_timer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.status, code);
            *abort_flag = 1u;
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi, int dtype)
{
    const float a = __uint_as_float(lo), b = __uint_as_float(hi);
    if (dtype == 0) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // .x (low half) = a
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Hand a fully read TMEM accumulator back to the MMA warp (of the leader CTA).
template <int CG>
__device__ __forceinline__ void release_accumulator(uint32_t bar, int lane)
{
    ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
        if constexpr (CG == 1)
            ptx::mbar_arrive(bar);
        else
            ptx::mbar_arrive_cluster(ptx::map_to_cta(bar, 0));
    }
}

// Convert one thread's 32 fp32 values (one row, 32 consecutive columns) and
// stage the warp's 32 x 32 box in shared memory with the 64-byte swizzle the
// C tensor map uses (16-byte chunk index XOR bits 7-8 of the offset), then
// TMA-store it.  Two staging buffers per warp alternate; a buffer is reused
// only after the bulk store issued from it two boxes earlier finished reading.
__device__ __forceinline__ void store_box(const uint32_t (&r)[32], const GemmParams& p,
                                          const CUtensorMap* tmap_c, uint32_t my_store,
                                          int& chunk_ctr, int lane, int col, int m_row)
{
    constexpr int kBufBytes = 32 * kStoreCols * 2;
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        packed[i] = pack2(r[2 * i], r[2 * i + 1], p.dtype);
    const uint32_t sb = my_store + uint32_t((chunk_ctr & 1) * kBufBytes);
    if (lane == 0)
        ptx::bulk_wait_group_read<1>();
    __syncwarp();
    const uint32_t row_addr = sb + uint32_t(lane * 64);
    const uint32_t swz = uint32_t((lane >> 1) & 3);
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        ptx::st_shared_v4(row_addr + ((uint32_t(ch) ^ swz) << 4), packed[4 * ch + 0],
                          packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (m_row < p.M && col < p.N)  // boxes wholly outside C are skipped
            ptx::tma_store_2d(tmap_c, sb, col, m_row);
        ptx::bulk_commit_group();
    }
    ++chunk_ctr;
}

template <int CG, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    using Cfg = KernelConfig<CG, BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;
    const int cluster_id = blockIdx.x / CG;
    const int num_clusters = gridDim.x / CG;

    const uint32_t sA = base + Cfg::kOffA;
    const uint32_t sB = base + Cfg::kOffB;
    const uint32_t sStore = base + Cfg::kOffStore;
    const uint32_t bar_full = base + Cfg::kOffBar;      // + 8 * stage
    const uint32_t bar_empty = bar_full + 8 * STAGES;   // + 8 * stage
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;  // + 8 * buffer
    const uint32_t bar_acc_empty = bar_acc_full + 16;      // + 8 * buffer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmemSlot);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffAbort);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);   // producer's arrive.expect_tx (+ bytes)
            ptx::mbar_init(bar_empty + 8 * s, 1);  // one tcgen05.commit
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_acc_full + 8 * b, 1);                 // one tcgen05.commit
            ptx::mbar_init(bar_acc_empty + 8 * b, kEpiWarps * CG);   // every epilogue warp of the pair
        }
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_a);
        ptx::prefetch_tensormap(&tmap_b);
        ptx::prefetch_tensormap(&tmap_c);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before_sync();
    if constexpr (CG == 2)
        ptx::cluster_sync();
    else
        __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
                const WorkUnit w = decode_unit(p, u);
                const int a_row = w.m_blk * Cfg::kTileM + int(rank) * kRowsPerCta;
                const int b_row = w.n_blk * BN + int(rank) * Cfg::kBRows;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_phase(bar_empty + 8 * stage, phase ^ 1u, p, abort_flag,
                                    kStatusProducerTimeout)) {
                        ok = false;
                        break;
                    }
                    const bool stall = p.stall_kblock >= 0 && blockIdx.x == 0 &&
                                       u == cluster_id && kb - w.kb0 == p.stall_kblock;
                    if (!stall) {
                        const uint32_t fb = bar_full + 8 * stage;
                        const uint32_t dA = sA + stage * Cfg::kABytes;
                        const uint32_t dB = sB + stage * Cfg::kBBytes;
                        if constexpr (CG == 1) {
                            ptx::mbar_arrive_expect_tx(fb, Cfg::kTxBytes);
                            ptx::tma_load_2d(dA, &tmap_a, fb, kb * kTileK, a_row);
                            ptx::tma_load_2d(dB, &tmap_b, fb, kb * kTileK, b_row);
                        } else {
                            // both CTAs' bytes are counted on the leader's barrier
                            const uint32_t leader_fb = ptx::map_to_cta(fb, 0);
                            if (rank == 0)
                                ptx::mbar_arrive_expect_tx(fb, Cfg::kTxBytes);
                            ptx::tma_load_2d_pair(dA, &tmap_a, leader_fb, kb * kTileK, a_row);
                            ptx::tma_load_2d_pair(dB, &tmap_b, leader_fb, kb * kTileK, b_row);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = p.idesc;
            const uint64_t a_desc0 = make_sdesc_sw128(sA);
            const uint64_t b_desc0 = make_sdesc_sw128(sB);
            int stage = 0;
            uint32_t phase = 0;
            int t = 0;
            bool ok = true;
            for (int u = cluster_id; ok && u < p.num_units; u += num_clusters, ++t) {
                const WorkUnit w = decode_unit(p, u);
                const int buf = t & 1;
                const uint32_t acc_phase = uint32_t(t >> 1) & 1u;
                if (!wait_phase(bar_acc_empty + 8 * buf, acc_phase ^ 1u, p, abort_flag,
                                kStatusMmaTimeout))
                    break;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + uint32_t(buf * BN);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_phase(bar_full + 8 * stage, phase, p, abort_flag, kStatusMmaTimeout)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint64_t ad = a_desc0 + uint64_t((stage * Cfg::kABytes) >> 4);
                    const uint64_t bd = b_desc0 + uint64_t((stage * Cfg::kBBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTileK / kMmaK; ++kk) {
                        // advance 16 elements = 32 bytes along K inside the swizzle atom
                        ptx::mma_f16<CG>(d_tmem, ad + uint64_t(kk * 2), bd + uint64_t(kk * 2), idesc,
                                         (kb > w.kb0 || kk > 0) ? 1u : 0u);
                    }
                    if constexpr (CG == 1)
                        ptx::mma_commit(bar_empty + 8 * stage);
                    else
                        ptx::mma_commit_pair(bar_empty + 8 * stage, 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                if constexpr (CG == 1)
                    ptx::mma_commit(bar_acc_full + 8 * buf);
                else
                    ptx::mma_commit_pair(bar_acc_full + 8 * buf, 0x3);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const uint32_t my_store = sStore + uint32_t((warp - 2) * 2 * Cfg::kStoreBufBytes);
        int chunk_ctr = 0;
        int t = 0;
        for (int u = cluster_id; u < p.num_units; u += num_clusters, ++t) {
            const WorkUnit w = decode_unit(p, u);
            const int buf = t & 1;
            const uint32_t acc_phase = uint32_t(t >> 1) & 1u;
            if (!wait_phase(bar_acc_full + 8 * buf, acc_phase, p, abort_flag,
                            kStatusEpilogueTimeout))
                break;
            ptx::tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * BN);
            const int m_row = w.m_blk * Cfg::kTileM + int(rank) * kRowsPerCta + q * 32;
            const int n_col = w.n_blk * BN;
            if (p.split_k == 1) {
                // ---- direct epilogue: TMEM -> registers -> bf16/fp16 -> smem -> TMA store
#pragma unroll 1
                for (int c = 0; c < BN / kStoreCols; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                    ptx::tmem_ld_wait();
                    if (c == BN / kStoreCols - 1)
                        release_accumulator<CG>(bar_acc_empty + 8 * buf, lane);
                    store_box(r, p, &tmap_c, my_store, chunk_ctr, lane, n_col + c * kStoreCols, m_row);
                }
            } else {
                // ---- split-K: every split stores its fp32 partial; the last of
                // the S splits to arrive (per warp quarter) sums all S partials in
                // split order 0..S-1 -- the same order whichever arrives last --
                // and writes C.  No split waits on another.
                const int S = p.split_k;
                const int ctile = w.tile * CG + int(rank);
                // partial slot layout per (tile, split, cta): [chunk][v = 0..7][row 0..127] float4
                float4* slot0 = reinterpret_cast<float4*>(p.partials) +
                                size_t(w.tile * S * CG + int(rank)) * (Cfg::kPartialFloats / 4);
                const size_t split_stride = size_t(CG) * (Cfg::kPartialFloats / 4);
                float4* mine = slot0 + size_t(w.split) * split_stride + row;
#pragma unroll 1
                for (int c = 0; c < BN / kStoreCols; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                    ptx::tmem_ld_wait();
                    if (c == BN / kStoreCols - 1)
                        release_accumulator<CG>(bar_acc_empty + 8 * buf, lane);
                    float4* pc = mine + size_t(c) * 8 * kRowsPerCta;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        __stcg(pc + v * kRowsPerCta,
                               make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                           __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
                }
                __threadfence();
                __syncwarp();
                uint32_t* counter = p.tile_sems + (ctile * kEpiWarps + q);
                uint32_t last = 0;
                if (lane == 0)
                    last = (atomicAdd(counter, 1u) == uint32_t(S - 1)) ? 1u : 0u;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
#pragma unroll 1
                    for (int c = 0; c < BN / kStoreCols; ++c) {
                        float acc[32];
                        const float4* pc = slot0 + size_t(c) * 8 * kRowsPerCta + row;
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const float4 x = __ldcg(pc + v * kRowsPerCta);
                            acc[4 * v + 0] = x.x;
                            acc[4 * v + 1] = x.y;
                            acc[4 * v + 2] = x.z;
                            acc[4 * v + 3] = x.w;
                        }
#pragma unroll 1
                        for (int j = 1; j < S; ++j) {
                            const float4* pj = pc + size_t(j) * split_stride;
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const float4 x = __ldcg(pj + v * kRowsPerCta);
                                acc[4 * v + 0] += x.x;
                                acc[4 * v + 1] += x.y;
                                acc[4 * v + 2] += x.z;
                                acc[4 * v + 3] += x.w;
                            }
                        }
                        uint32_t r[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(acc[i]);
                        store_box(r, p, &tmap_c, my_store, chunk_ctr, lane, n_col + c * kStoreCols,
                                  m_row);
                    }
                    __syncwarp();
                    if (lane == 0)
                        *counter = 0u;  // re-armed for the next launch
                }
            }
        }
        if (lane == 0)
            ptx::bulk_wait_group_all();
        __syncwarp();
    }

    // --------------------------------------------------------------- teardown
    __syncwarp();
    ptx::tc_fence_before_sync();
    if constexpr (CG == 2)
        ptx::cluster_sync();
    else
        __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace bwgemm
