// skinny_kernel.cuh -- whole-K tcgen05 GEMM for decode batches of at most 64
// rows of A: 64 weight rows per CTA and no split of K.
//
// For M <= 64 the kernel computes C^T = B A^T ("Writing a Blackwell GEMM by
// hand", "Two workloads, not one": decode batches of 1 to 64 rows padded to
// the 128-row MMA take twice cuBLAS's time): the weight rows of B are the
// MMA's M side, 64 per CTA, and the few rows of A are its N (BN = 16, 32 or
// 64, zero-filled by TMA past M).  Each CTA walks the whole K range for its
// 64 weight rows, so no partial sums are exchanged; N = 8192 takes 128 CTAs.
//
// Two forms (CG):
//   CG = 1   one CTA, tcgen05.mma M = 64 (cta_group::1); the CTA copies all
//            BN rows of A for every K block.
//   CG = 2   a cluster of two CTAs on 128 weight rows, tcgen05.mma M = 128
//            (cta_group::2) issued by the even CTA: each CTA copies its own 64
//            weight rows and half of A's BN rows (the MMA's N is split across
//            the pair), so the copies of A from L2, as many bytes per stage
//            as the weights at BN = 64, are halved.
//
// The ring holds stages of KPS K blocks (one 3-D TMA copy per operand, KPS x
// 128 contiguous bytes of each row) where K allows, one K block at a time for
// what is left: a stage of four K blocks of 64 weight rows is one 32 KiB
// copy, which shared memory fills at about 1.6 times the rate it fills from
// 16 KiB copies.  A pair takes three K blocks per stage, so that six stages
// fit and more weight bytes are in flight.
//
//   warp 0      TMA producer (the whole warp walks the stages; an elected lane
//               issues); full/empty mbarrier pairs per stage.  In a pair both
//               CTAs' bytes are counted on the even CTA's full barrier.
//   warp 1      TMEM allocator and (in the even CTA of a pair) MMA issuer: 4
//               tcgen05.mma of K = 16 per K block, the first of the launch
//               overwrites; commit frees the stage (in both CTAs of a pair).
//   warps 2..5  epilogue, one per TMEM lane quarter q.  Accumulator layouts:
//               CG = 1 (M = 64): weight row 16 q + i in lane i of quarter q
//               (i < 16; lanes 16-31 are not written), columns = the MMA's N.
//               CG = 2 (M = 128, measured): in each CTA its weight row i < 64
//               sits in lane i for the MMA's columns [0, BN/2) and in lane
//               64 + i for [BN/2, BN), both at TMEM columns [0, BN/2).
//               Each warp reads its quarter with 32x32b loads, puts its
//               values into its own staging block (CG = 1: BN rows of A x 16
//               weight columns, CG = 2: BN/2 rows x 32 columns) and writes the
//               block with one TMA store (rows past M, columns past N
//               clipped; a block holding a row end off a 16-byte boundary is
//               written with plain stores).
//
// At entry, before the set-up and the dependency wait, the producer lane
// prefetches the CTA's first kSkPrefetchKBlocks K blocks of weights into L2:
// the previous kernel on the stream is still finishing, HBM would otherwise
// idle, and a prefetch only warms L2, so it is safe even if that kernel
// writes the weights.
//
// Every wait is bounded (the main kernel's wait_phase); after an abort the
// kernel drains its MMAs and loads before it releases TMEM and shared memory,
// as the main kernel does.
#pragma once

#include "gemm_kernel.cuh"

namespace bwgemm {

constexpr int kSkRows = 64;            // weight rows per CTA
constexpr int kSkEpiWarps = 4;         // one per TMEM lane quarter
constexpr int kSkThreads = 32 * (2 + kSkEpiWarps);
constexpr int kSkPrefetchKBlocks = 8;  // weights prefetched into L2 before the dependency wait

template <int BN, int KPS, int STAGES, int CG>
struct SkinnyConfig {
    static_assert(BN == 16 || BN == 32 || BN == 64, "the MMA's N: 16, 32 or 64 rows of A");
    static_assert(KPS >= 2 && KPS <= 8, "K blocks per whole stage");
    static_assert(CG == 1 || (CG == 2 && BN == 64), "one CTA, or a pair at BN = 64 (M = 128, N = 64)");
    static constexpr int kXRows = BN / CG;                    // rows of A this CTA copies
    static constexpr int kWBlock = kSkRows * kTileK * 2;      // one K block of 64 weight rows: 8 KiB
    static constexpr int kXBlock = kXRows * kTileK * 2;       // one K block of this CTA's rows of A
    static constexpr int kWBytes = KPS * kWBlock;
    static constexpr int kXBytes = KPS * kXBlock;
    static constexpr int kTmemCols = BN / CG < 32 ? 32 : BN / CG;  // a power of two, at least 32
    static constexpr int kOutCols = 16 * CG;                  // weight columns of a warp's block
    static constexpr int kOutRows = BN / CG;                  // rows of A of a warp's block
    static constexpr int kOutBytes = kOutCols * kOutRows * 2;
    static constexpr int kOffW = 0;
    static constexpr int kOffX = STAGES * kWBytes;
    static constexpr int kOffOut = kOffX + STAGES * kXBytes;  // kSkEpiWarps staging blocks
    static constexpr int kOffBar = kOffOut + kSkEpiWarps * kOutBytes;  // full[S], empty[S], acc_full, drain
    static constexpr int kNumBars = 2 * STAGES + 2;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KiB
    static_assert(kWBlock % 1024 == 0 && kXBlock % 1024 == 0,
                  "every K block of both operands starts on a 1 KiB swizzle-atom boundary");
    static_assert(kOutBytes % 128 == 0, "staging blocks stay 128-byte aligned");
    static_assert(kSmemBytes <= 227 * 1024, "exceeds the 227 KiB shared memory of one CTA");
};

// Kernel view of the problem (GemmParams): M = the weight rows (the caller's
// N), N = the rows of A (the caller's M, <= BN), K; c / ldc = the caller's C,
// M_caller x N_caller.  k_chunks_a / k_chunks_b: whole 64-element K chunks the
// 3-D views of the weights and of A cover (0: no 3-D view).  tmap_x / tmap_x3
// copy BN / CG rows of A; tmap_c stores boxes of kOutRows x kOutCols, no
// swizzle.  CG = 2 launches in clusters of two consecutive CTAs.
template <int BN, int KPS, int STAGES, int CG>
__global__ void __launch_bounds__(kSkThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                  const __grid_constant__ CUtensorMap tmap_w3, const __grid_constant__ CUtensorMap tmap_x3,
                  const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    using Cfg = SkinnyConfig<BN, KPS, STAGES, CG>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;  // in the pair; 0 issues the MMAs
    const uint32_t sW = base + Cfg::kOffW;
    const uint32_t sX = base + Cfg::kOffX;
    const uint32_t bar_full = base + Cfg::kOffBar;         // + 8 * stage
    const uint32_t bar_empty = bar_full + 8 * STAGES;      // + 8 * stage
    const uint32_t bar_acc = bar_empty + 8 * STAGES;       // the accumulator is complete
    const uint32_t bar_drain = bar_acc + 8;                // after an abort: the issued MMAs completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmemSlot);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffAbort);
    const int n0 = int(blockIdx.x) * kSkRows;    // first weight row of this CTA
    const int x_row0 = int(rank) * Cfg::kXRows;  // first row of A this CTA copies

    // Stages walk the K blocks in order: K blocks kb .. kb + KPS - 1 together when
    // all are whole 64-element chunks of the 3-D views, else K block kb alone
    // (the ragged last block, or whole ones left over); producer and MMA warp
    // step through the same sequence.  The 3-D views cover only whole chunks,
    // and there are at most KB of those.
    const int KB = p.num_k_blocks;
    auto blocks_at = [&](int kb) {
        return (kb + KPS <= p.k_chunks_a && kb + KPS <= p.k_chunks_b) ? KPS : 1;
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
            ptx::mbar_init(bar_full + 8 * s, 1);   // the (even CTA's) producer's arrive.expect_tx (+ bytes)
            ptx::mbar_init(bar_empty + 8 * s, 1);  // one tcgen05.commit
        }
        ptx::mbar_init(bar_acc, 1);
        ptx::mbar_init(bar_drain, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_w);
        ptx::prefetch_tensormap(&tmap_x);
        if (p.k_chunks_a >= KPS)
            ptx::prefetch_tensormap(&tmap_w3);
        if (p.k_chunks_b >= KPS)
            ptx::prefetch_tensormap(&tmap_x3);
        // the first weight blocks into L2 at once, ahead of the set-up and of
        // the dependency wait
        if (p.k_chunks_a >= KPS) {
#pragma unroll 1
            for (int kb = 0; kb + KPS <= p.k_chunks_a && kb < kSkPrefetchKBlocks; kb += KPS)
                ptx::tma_prefetch_3d(&tmap_w3, 0, n0, kb);
        }
    }
    if (warp == 2 && lane == 0)
        ptx::prefetch_tensormap(&tmap_c);
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before_sync();
    if constexpr (CG == 2)
        ptx::cluster_sync();  // both CTAs' barriers exist before either copies or commits to them
    else
        __syncthreads();
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
        const uint32_t leader_full = (CG == 2) ? ptx::map_to_cta(bar_full, 0) : bar_full;
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
                const uint32_t dW = sW + uint32_t(s * Cfg::kWBytes);
                const uint32_t dX = sX + uint32_t(s * Cfg::kXBytes);
                const uint32_t bytes = uint32_t(nkb * (Cfg::kWBlock + Cfg::kXBlock));
                if (rank == 0)
                    ptx::mbar_arrive_expect_tx(fb, uint32_t(CG) * bytes);
                if constexpr (CG == 1) {
                    if (nkb == KPS) {
                        ptx::tma_load_3d(dW, &tmap_w3, fb, 0, n0, kb);
                        ptx::tma_load_3d(dX, &tmap_x3, fb, 0, x_row0, kb);
                    } else {
                        ptx::tma_load_2d(dW, &tmap_w, fb, kb * kTileK, n0);
                        ptx::tma_load_2d(dX, &tmap_x, fb, kb * kTileK, x_row0);
                    }
                } else {
                    if (nkb == KPS) {
                        ptx::tma_load_3d_pair(dW, &tmap_w3, fb, 0, n0, kb);
                        ptx::tma_load_3d_pair(dX, &tmap_x3, fb, 0, x_row0, kb);
                    } else {
                        ptx::tma_load_2d_pair(dW, &tmap_w, fb, kb * kTileK, n0);
                        ptx::tma_load_2d_pair(dX, &tmap_x, fb, kb * kTileK, x_row0);
                    }
                }
            }
            __syncwarp();
            kb += nkb;
        }
        if (lane == 0)
            trace_mark(p, kTraceLastLoad);
    } else if (warp == 1 && rank == 0) {
        // ---------------------------------------------------------- MMA issue
        const uint64_t w_desc0 = make_sdesc_sw128(sW);
        const uint64_t x_desc0 = make_sdesc_sw128(sX);
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
                    // K block c of the stage: 64 weight rows / this CTA's rows of A, 128 bytes each
                    const uint64_t wd = w_desc0 + uint64_t((s * Cfg::kWBytes + c * Cfg::kWBlock) >> 4);
                    const uint64_t xd = x_desc0 + uint64_t((s * Cfg::kXBytes + c * Cfg::kXBlock) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTileK / kMmaK; ++kk)
                        ptx::mma_f16<CG>(tmem0, wd + uint64_t(kk * 2), xd + uint64_t(kk * 2), p.idesc,
                                         (kb > 0 || c > 0 || kk > 0) ? 1u : 0u);
                }
                if constexpr (CG == 1)
                    ptx::mma_commit(bar_empty + 8 * s);
                else
                    ptx::mma_commit_pair(bar_empty + 8 * s, 0x3);
            }
            __syncwarp();
            kb += nkb;
        }
        if (ok) {
            if (ptx::elect_one()) {
                if constexpr (CG == 1)
                    ptx::mma_commit(bar_acc);
                else
                    ptx::mma_commit_pair(bar_acc, 0x3);
            }
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
            constexpr int kVals = BN / CG;  // accumulator columns per lane
            uint32_t r[kVals];
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16);
#pragma unroll
            for (int c = 0; c < kVals; c += 16)
                ptx::tmem_ld_32x32b_x16(taddr + uint32_t(c), r + c);
            ptx::tmem_ld_wait();
            // This lane's weight row n (a column of C) and the rows of A its
            // values belong to: t0 + j for value j.
            constexpr int kLanes = CG == 1 ? 16 : 32;  // lanes holding a weight row
            const int x0 = n0 + (CG == 1 ? 16 * q : 32 * (q & 1));
            const int t0 = CG == 1 ? 0 : (q >> 1) * kVals;
            const int n = x0 + lane;
            auto to_bits = [&](uint32_t bits) -> uint16_t {
                const float v = __uint_as_float(bits);
                return p.dtype == 0 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                                    : __half_as_ushort(__float2half_rn(v));
            };
            // A TMA store clips at the end of a row of C only in whole 16-byte
            // chunks, so the block holding a row end that is not on one is
            // written with plain stores; rows past M are clipped by the store.
            const bool ragged = (p.M & 7) != 0 && x0 < p.M && x0 + Cfg::kOutCols > p.M;
            if (ragged) {
                if (lane < kLanes && n < p.M) {
#pragma unroll
                    for (int j = 0; j < kVals; ++j)
                        if (t0 + j < p.N)
                            p.c[size_t(t0 + j) * size_t(p.ldc) + size_t(n)] = to_bits(r[j]);
                }
            } else if (x0 < p.M && t0 < p.N) {
                const uint32_t out = base + uint32_t(Cfg::kOffOut + q * Cfg::kOutBytes);
                if (lane < kLanes) {
#pragma unroll
                    for (int j = 0; j < kVals; ++j)
                        ptx::st_shared_u16(out + uint32_t((j * Cfg::kOutCols + lane) * 2), to_bits(r[j]));
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(&tmap_c, out, x0, t0);
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
    // released; in a pair the even CTA's barriers count both CTAs' loads and
    // neither CTA leaves before the other.
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
        if (warp == 1 && rank == 0) {
            if (ptx::elect_one()) {
                if constexpr (CG == 1)
                    ptx::mma_commit(bar_drain);
                else
                    ptx::mma_commit_pair(bar_drain, 0x1);
            }
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
    if constexpr (CG == 2)
        ptx::cluster_sync();
    else
        __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
        if (lane == 0)
            trace_mark(p, kTraceExit);
    }
}

}  // namespace bwgemm
