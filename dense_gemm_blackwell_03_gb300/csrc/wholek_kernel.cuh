// wholek_kernel.cuh -- whole-K tcgen05 GEMM on CTA pairs for 129 to 256 rows
// of A: all rows of A on the MMA's M side, a narrow block of weight rows on
// its N side, no split of K.
//
// The decode linears of "Writing a Blackwell GEMM by hand" ("Two workloads,
// not one") and of "Matrix Multiplication on NVIDIA's Blackwell" stream a
// weight matrix B (N x K) past a few hundred rows of A.  With 256 x 256 pair
// tiles N = 8192 makes 32 tiles, too few for the SMs, so the main kernel
// splits K in two and exchanges partial sums after the last MMA.  Here one
// pair holds all of A's rows (M = 256 over the pair, tcgen05.mma
// cta_group::2, each CTA 128 of them) and BN weight rows (the MMA's N, each
// CTA copying BN / 2 of them), with BN chosen so that the tiles fill the pairs
// of the GPU once (N = 8192: 74 tiles of 112 on 148 SMs).  Every CTA walks the
// whole K range: no partial sums, and the accumulator is C itself.
//
// The ring holds stages of KPS K blocks (one 3-D TMA copy per operand) where
// K allows, one K block at a time for what is left.
//
//   warp 0      TMA producer of both operands (the whole warp walks the
//               stages; an elected lane issues); both CTAs' bytes are counted
//               on the even CTA's full barriers.
//   warp 1      TMEM allocator and, in the even CTA, MMA issuer: 4
//               tcgen05.mma of K = 16 per K block, the first of the launch
//               overwrites; the commit frees the stage in both CTAs.
//   warps 2..5  epilogue, one per TMEM lane quarter q: lane 32 q + i holds row
//               32 q + i of this CTA's 128 rows of C, TMEM columns = the BN
//               columns of C.  Each warp converts its 32 rows into a block of
//               32 x BN in shared memory (the idle ring) and writes it with one
//               TMA store (rows past M and columns past N clipped); the block
//               holding a row end off a 16-byte boundary is written with plain
//               stores instead.
//
// At entry, before the set-up and the dependency wait, the producer lane
// prefetches the CTA's first weight K blocks into L2 (a prefetch only warms
// L2, so it is safe even if the previous kernel on the stream writes the
// weights).  Every wait is bounded
// (the main kernel's wait_phase); after an abort the kernel drains its MMAs
// and loads before it releases TMEM and shared memory.
#pragma once

#include "gemm_kernel.cuh"

namespace bwgemm {

constexpr int kWkRowsA = 128;          // rows of A per CTA (M = 256 over the pair)
constexpr int kWkEpiWarps = 4;
constexpr int kWkThreads = 32 * (2 + kWkEpiWarps);
constexpr int kWkPrefetchBytes = 64 * 1024;  // weights prefetched into L2 before the dependency wait

template <int BN, int KPS, int STAGES>
struct WholeKConfig {
    static_assert(BN % 16 == 0 && BN >= 64 && BN <= 256, "the MMA's N (M = 256): a multiple of 16, 64..256");
    static_assert(KPS >= 1 && KPS <= 4, "K blocks per whole stage");
    static constexpr int kBRows = BN / 2;                    // weight rows this CTA copies
    static constexpr int kABlock = kWkRowsA * kTileK * 2;    // one K block of A's rows: 16 KiB
    static constexpr int kBBlock = kBRows * kTileK * 2;      // one K block of this CTA's weight rows
    static constexpr int kABytes = KPS * kABlock;
    static constexpr int kBBytes = KPS * kBBlock;
    static constexpr int kTmemCols = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
    static constexpr int kOutBytes = 32 * BN * 2;            // a warp's staging block: 32 rows x BN
    static constexpr int kOffA = 0;
    static constexpr int kOffB = STAGES * kABytes;
    static constexpr int kOffOut = 0;                        // staging reuses the idle ring
    static constexpr int kOffBar = kOffB + STAGES * kBBytes;  // full[S], empty[S], acc_full, drain
    static constexpr int kNumBars = 2 * STAGES + 2;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KiB
    static_assert(kABlock % 1024 == 0 && kBBlock % 1024 == 0,
                  "every K block of both operands starts on a 1 KiB swizzle-atom boundary");
    static_assert(kWkEpiWarps * kOutBytes <= kOffBar, "the epilogue's staging fits the ring");
    static_assert(kOutBytes % 1024 == 0, "staging blocks stay 1 KiB aligned");
    static_assert(kSmemBytes <= 227 * 1024, "exceeds the 227 KiB shared memory of one CTA");
};

// Kernel view of the problem (GemmParams, operands not swapped): M = rows of
// A (<= 256), N = weight rows, K; c / ldc = C (M x N).  tmap_a / tmap_a3:
// A in boxes of 128 rows (2-D, and the 3-D view of KPS K blocks);
// tmap_b / tmap_b3: B in boxes of BN / 2 rows; tmap_c: C in boxes of 32
// rows x BN columns, no swizzle.  k_chunks_a / k_chunks_b: whole 64-element K
// chunks the 3-D views cover (0: no 3-D view).  Launched in clusters of two
// consecutive CTAs; pair t computes columns [t BN, t BN + BN).
template <int BN, int KPS, int STAGES>
__global__ void __launch_bounds__(kWkThreads, 1)
    wholek_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                  const __grid_constant__ CUtensorMap tmap_a3, const __grid_constant__ CUtensorMap tmap_b3,
                  const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    using Cfg = WholeKConfig<BN, KPS, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();  // in the pair; 0 issues the MMAs
    const uint32_t sA = base + Cfg::kOffA;
    const uint32_t sB = base + Cfg::kOffB;
    const uint32_t bar_full = base + Cfg::kOffBar;         // + 8 * stage
    const uint32_t bar_empty = bar_full + 8 * STAGES;      // + 8 * stage
    const uint32_t bar_acc = bar_empty + 8 * STAGES;       // the accumulator is complete
    const uint32_t bar_drain = bar_acc + 8;                // after an abort: the issued MMAs completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmemSlot);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffAbort);
    const int tile = int(blockIdx.x) / 2;
    const int n0 = tile * BN;                            // first column of C (weight row) of the pair
    const int a_row0 = int(rank) * kWkRowsA;             // this CTA's rows of A and of C
    const int b_row0 = n0 + int(rank) * Cfg::kBRows;     // this CTA's weight rows

    // Stages walk the K blocks in order: KPS of them together when all are
    // whole chunks of both 3-D views, else one (the ragged last block, or whole
    // ones left over); producer and MMA warp step through the same sequence.
    const int KB = p.num_k_blocks;
    auto blocks_at = [&](int kb) {
        return (KPS > 1 && kb + KPS <= p.k_chunks_a && kb + KPS <= p.k_chunks_b) ? KPS : 1;
    };

    constexpr int kInitThread = 2 * 32;  // an epilogue warp, idle until the accumulator is ready
    if (threadIdx.x == kInitThread) {
        if (p.trace) {
            uint64_t* row = p.trace + size_t(blockIdx.x) * kTraceSlots;
#pragma unroll 1
            for (int i = 0; i < kTraceSlots; ++i)
                row[i] = 0ull;
        }
        trace_mark(p, kTraceEntry);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);   // the even CTA's producer's arrive.expect_tx (+ bytes)
            ptx::mbar_init(bar_empty + 8 * s, 1);  // one tcgen05.commit
        }
        ptx::mbar_init(bar_acc, 1);
        ptx::mbar_init(bar_drain, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_a);
        ptx::prefetch_tensormap(&tmap_b);
        if (KPS > 1 && p.k_chunks_a >= KPS) {
            ptx::prefetch_tensormap(&tmap_a3);
            ptx::prefetch_tensormap(&tmap_b3);
        }
        // the first weight blocks into L2 at once, ahead of the set-up and of
        // the dependency wait
        constexpr int kPf = kWkPrefetchBytes / Cfg::kBBlock;  // weight K blocks prefetched
#pragma unroll 1
        for (int kb = 0; kb < KB && kb < kPf; ++kb)
            ptx::tma_prefetch_2d(&tmap_b, kb * kTileK, b_row0);
    }
    if (warp == 2 && lane == 0)
        ptx::prefetch_tensormap(&tmap_c);
    if (warp == 1) {
        ptx::tmem_alloc<2>(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish<2>();
    }
    ptx::tc_fence_before_sync();
    ptx::cluster_sync();  // both CTAs' barriers exist before either copies or commits to them
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == kInitThread)
        trace_mark(p, kTraceSetup);
    // everything above may overlap the previous kernel on the stream; each role
    // waits for it just before its first access to global memory
    ptx::launch_dependents();
    uint32_t armed_mask = 0, armed_parity = 0;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        ptx::grid_dependency_wait();
        if (lane == 0)
            trace_mark(p, kTraceReady);
        const uint32_t leader_full = ptx::map_to_cta(bar_full, 0);
        int i = 0;  // stage count
#pragma unroll 1
        for (int kb = 0; kb < KB; ++i) {
            const int s = i % STAGES;
            const uint32_t phase = uint32_t(i / STAGES) & 1u;
            const int nkb = blocks_at(kb);
            if (!__all_sync(0xffffffffu, wait_phase(bar_empty + 8 * s, phase ^ 1u, p, abort_flag,
                                                    kStatusProducerTimeout)))
                break;
            // test hook: the producer of CTA 0 never fills this stage of the launch
            const bool stall = p.stall_kblock >= 0 && blockIdx.x == 0 && p.stall_kblock == i;
            if (!stall && rank == 0) {  // warp-uniform bookkeeping for the abort drain
                armed_mask |= 1u << (s & 31);
                armed_parity = (armed_parity & ~(1u << (s & 31))) | (phase << (s & 31));
            }
            if (!stall && ptx::elect_one()) {
                if (i == 0)
                    trace_mark(p, kTraceFirstLoad);
                const uint32_t fb = leader_full + 8 * s;
                const uint32_t dA = sA + uint32_t(s * Cfg::kABytes);
                const uint32_t dB = sB + uint32_t(s * Cfg::kBBytes);
                if (rank == 0)
                    ptx::mbar_arrive_expect_tx(fb, uint32_t(2 * nkb * (Cfg::kABlock + Cfg::kBBlock)));
                if (nkb == KPS && KPS > 1) {
                    ptx::tma_load_3d_pair(dA, &tmap_a3, fb, 0, a_row0, kb);
                    ptx::tma_load_3d_pair(dB, &tmap_b3, fb, 0, b_row0, kb);
                } else {
                    ptx::tma_load_2d_pair(dA, &tmap_a, fb, kb * kTileK, a_row0);
                    ptx::tma_load_2d_pair(dB, &tmap_b, fb, kb * kTileK, b_row0);
                }
            }
            __syncwarp();
            kb += nkb;
        }
        if (lane == 0)
            trace_mark(p, kTraceLastLoad);
    } else if (warp == 1 && rank == 0) {
        // ---------------------------------------------------------- MMA issue
        const uint64_t a_desc0 = make_sdesc_sw128(sA);
        const uint64_t b_desc0 = make_sdesc_sw128(sB);
        const uint32_t tmem0 = __shfl_sync(0xffffffffu, tmem_base, 0);
        bool ok = true;
        if (lane == 0)
            trace_unit(p, 0, 0);
        int i = 0;  // stage count
#pragma unroll 1
        for (int kb = 0; kb < KB; ++i) {
            const int s = i % STAGES;
            const uint32_t phase = uint32_t(i / STAGES) & 1u;
            ok = __all_sync(0xffffffffu, wait_phase(bar_full + 8 * s, phase, p, abort_flag, kStatusMmaTimeout));
            if (!ok)
                break;
            ptx::tc_fence_after_sync();
            const int nkb = blocks_at(kb);
            if (ptx::elect_one()) {
#pragma unroll 1
                for (int c = 0; c < nkb; ++c) {
                    // K block c of the stage: 128 rows of A / BN / 2 weight rows, 128 bytes each
                    const uint64_t ad = a_desc0 + uint64_t((s * Cfg::kABytes + c * Cfg::kABlock) >> 4);
                    const uint64_t bd = b_desc0 + uint64_t((s * Cfg::kBBytes + c * Cfg::kBBlock) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTileK / kMmaK; ++kk)
                        ptx::mma_f16<2>(tmem0, ad + uint64_t(kk * 2), bd + uint64_t(kk * 2), p.idesc,
                                        (kb > 0 || c > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit_pair(bar_empty + 8 * s, 0x3);
            }
            __syncwarp();
            kb += nkb;
        }
        if (ok) {
            if (ptx::elect_one())
                ptx::mma_commit_pair(bar_acc, 0x3);
            __syncwarp();
            if (lane == 0)
                trace_unit(p, 0, 1);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        // C may be read by the kernel before this one: write only after it completed
        ptx::grid_dependency_wait();
        const int q = warp & 3;  // the TMEM lane quarter this warp may access
        if (__all_sync(0xffffffffu, wait_phase(bar_acc, 0u, p, abort_flag, kStatusEpilogueTimeout))) {
            ptx::tc_fence_after_sync();
            if (warp == 2 && lane == 0)
                trace_unit(p, 0, 2);
            const int m0 = a_row0 + 32 * q;  // this warp's first row of C
            const int m = m0 + lane;         // this lane's row
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16);
            // A TMA store clips at the end of a row of C only in whole 16-byte
            // chunks: the tile holding a row end off one is written with plain
            // stores; rows past M are clipped by the store.
            const bool ragged = (p.N & 7) != 0 && n0 + BN > p.N;
            const uint32_t out = base + uint32_t(Cfg::kOffOut + q * Cfg::kOutBytes);
            const bool live = m0 < p.M && n0 < p.N;
            // the staging blocks reuse the ring, last written by TMA and read by
            // the MMAs that bar_acc saw complete
            ptx::fence_proxy_async_smem();
            // all of the lane's BN accumulator columns first (one wait), then
            // convert and place them 16 at a time
            uint32_t r[BN];
#pragma unroll
            for (int c = 0; c < BN; c += 16)
                ptx::tmem_ld_32x32b_x16(taddr + uint32_t(c), r + c);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < BN; c += 16) {
                uint32_t packed[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float lo = __uint_as_float(r[c + 2 * j]), hi = __uint_as_float(r[c + 2 * j + 1]);
                    const uint32_t blo = p.dtype == 0 ? __bfloat16_as_ushort(__float2bfloat16_rn(lo))
                                                      : __half_as_ushort(__float2half_rn(lo));
                    const uint32_t bhi = p.dtype == 0 ? __bfloat16_as_ushort(__float2bfloat16_rn(hi))
                                                      : __half_as_ushort(__float2half_rn(hi));
                    packed[j] = blo | (bhi << 16);
                }
                if (ragged) {
                    if (m < p.M) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (n0 + c + j < p.N)
                                p.c[size_t(m) * size_t(p.ldc) + size_t(n0 + c + j)] =
                                    uint16_t((j & 1) ? (packed[j >> 1] >> 16) : (packed[j >> 1] & 0xFFFFu));
                    }
                } else if (live) {
                    const uint32_t dst = out + uint32_t((lane * BN + c) * 2);
                    ptx::st_shared_v4(dst, packed[0], packed[1], packed[2], packed[3]);
                    ptx::st_shared_v4(dst + 16, packed[4], packed[5], packed[6], packed[7]);
                }
            }
            if (!ragged && live) {
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(&tmap_c, out, n0, m0);
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_all();
                }
            }
            __syncwarp();
            if (warp == 2 && lane == 0) {
                trace_unit(p, 0, 3);
                trace_mark(p, kTraceEpiDone);
            }
        }
    }

    // --------------------------------------------------------------- teardown
    // As in the main kernel: after an abort, drain the MMAs and the loads this
    // CTA armed (bounded) and settle before TMEM and shared memory are
    // released; the even CTA's barriers count both CTAs' loads and neither CTA
    // leaves before the other.
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
        if (warp == 1 && rank == 0) {
            if (ptx::elect_one())
                ptx::mma_commit_pair(bar_drain, 0x1);
            __syncwarp();
            drain_wait(bar_drain, 0u, kDrainNs);
        }
        if (warp == 0) {
#pragma unroll 1
            for (int s = 0; s < STAGES; ++s)
                if ((armed_mask >> s) & 1u)
                    drain_wait(bar_full + 8 * s, (armed_parity >> s) & 1u, kDrainNs);
            if (lane == 0)
                settle(kSettleNs);
        }
        __syncwarp();
        __syncthreads();
    }
    ptx::tc_fence_before_sync();
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc<2>(tmem_base, Cfg::kTmemCols);
        if (lane == 0)
            trace_mark(p, kTraceExit);
    }
}

}  // namespace bwgemm
