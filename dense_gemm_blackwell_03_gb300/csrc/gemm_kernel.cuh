// gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   C[M x N] = A[M x K] * B[N x K]^T, A and B K-major bf16/fp16, fp32
//   accumulation in TMEM, bf16/fp16 output.
//
// Structure (one CTA per SM, or one CTA pair per two SMs when CG == 2):
//   warp 0      TMA producer: fills a STAGES-deep ring of 64-wide K blocks of A
//               and B (128B-swizzled), guarded by full/empty mbarrier pairs.
//   warp 1      TMEM allocator; in the leader CTA the whole warp walks the
//               K blocks and one elected lane issues every tcgen05.mma and
//               commits stage release / accumulator-ready.
//   warps 2..9  epilogue (two per TMEM lane quarter, half the columns each):
//               tcgen05.ld -> fp32 -> bf16/fp16 -> swizzled smem -> TMA store,
//               double-buffered per warp.  A unit that covers only part of a
//               tile's K range (split-K slice or stream-K piece) combines
//               with the tile's other pieces through fp32 partials in a
//               fixed order (see the epilogue), without waiting on them.
// Two fp32 accumulators live in TMEM (2 x BN columns), so the epilogue of one
// work unit overlaps the MMAs of the next.  Work is handed out statically:
// each worker (CTA or CTA pair) first walks its share of the stream-K
// iterations, then its data-parallel tiles, in grouped raster order.
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
//
// TR = true runs the same pipeline on swapped operands (C^T = B A^T: the
// N x K operand fills the 128-row MMA side, the few rows of a small-M
// problem become the MMA's N) and writes each accumulator box transposed.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernel_params.h"
#include "ptx.cuh"

namespace bwgemm {

// RING_STORE: the epilogue stages its output boxes in the (idle) B ring
// instead of a region of its own -- the clustered split-K kernels, whose one
// unit per CTA ends with idle rings; the freed region buys another stage.
template <int CG, int BN, int STAGES, bool RING_STORE = false>
struct KernelConfig {
    static_assert(CG == 1 || CG == 2, "CTA group is 1 or 2");
    static_assert(BN % 32 == 0 && BN >= 64 && (BN <= 256 || (CG == 2 && BN <= 384)),
                  "BN in [64, 256] (multiple of 32), or up to 384 for the CTA pair");
    // columns of the first and second MMA of a K step: one MMA up to 256
    // columns; a wider pair unit (320, 384) issues N = 256 and N = BN - 256
    // into one accumulator, the second reading B rows [128, BN / 2) of each
    // CTA's stage
    static constexpr int kMmaN1 = BN <= 256 ? BN : 256;
    static constexpr int kMmaN2 = BN - kMmaN1;
    static constexpr int kTileM = CG * kRowsPerCta;             // rows per work unit
    static constexpr int kBRows = (CG == 1) ? BN : BN / 2;      // B rows this CTA loads
    static constexpr int kABytes = kRowsPerCta * kTileK * 2;    // 16 KiB
    static constexpr int kBBytes = kBRows * kTileK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;       // per CTA
    static constexpr int kTxBytes = kStageBytes * CG;           // landing per stage on the leader
    static constexpr int kStoreBufBytes = 32 * kStoreCols * 2;  // one 32 x 32 output box
    // two fp32 accumulators of BN columns; the allocation is a power of two,
    // the second accumulator starts half-way (column 256 for BN = 224)
    // (two when both fit the 512 TMEM columns, else one: a 320-column unit)
    static constexpr int kAccBufs = (2 * BN <= 512) ? 2 : 1;
    static constexpr int kTmemCols = (kAccBufs * BN <= 128) ? 128 : (kAccBufs * BN <= 256) ? 256 : 512;
    static constexpr int kAccStride = kTmemCols / 2;
    static_assert(kAccBufs * BN <= kTmemCols && kTmemCols <= 512, "the accumulators fit the TMEM allocation");
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffStore = kOffB + STAGES * kBBytes;
    static constexpr int kOffBar = kOffStore + (RING_STORE ? 0 : kEpiWarps * 2 * kStoreBufBytes);
    // full[S], empty[S], acc_full[2], acc_empty[2], clc_full[4], clc_empty[4],
    // exchange_ready, exchange_full[2], exchange_staged[2], mma_drain
    static constexpr int kNumBars = 2 * STAGES + 10 + 2 * kClcSlots;
    // 16-byte responses on 16-byte boundaries (the barrier count may be odd)
    static constexpr int kOffClcResp = (kOffBar + kNumBars * 8 + 15) & ~15;
    static constexpr int kOffTmemSlot = kOffClcResp + 16 * kClcSlots;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KiB
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms need 1 KiB alignment");
    static_assert(kOffStore % 128 == 0 && kOffBar % 8 == 0 && kOffClcResp % 16 == 0,
                  "store boxes need 128-byte, mbarriers 8-byte, launch-control responses 16-byte alignment");
    static_assert(kSmemBytes <= 227 * 1024, "exceeds the 227 KiB shared memory of one CTA");
    // floats of one CTA's fp32 partial tile
    static constexpr int kPartialFloats = kRowsPerCta * BN;
};

// Column of the tile (relative to its first column) that accumulator chunk c
// (32 columns) holds.  Up to 256 columns the accumulator is the tile.  In a
// wider pair unit each CTA stages B rows [0, H) of its half, H = BN / 2: the
// first MMA (N = 256) reads rows [0, 128) of both halves (tile columns 0-127
// and H..H+127), the second (N = BN - 256) rows [128, H) (tile columns
// 128..H-1 and H+128..BN-1).  For 320: chunks 0-3, 4-7, 8, 9 hold columns
// 0, 160, 128, 288 onwards.
template <int BN>
__device__ __forceinline__ int chunk_col(int c)
{
    if constexpr (BN <= 256) {
        return c * kStoreCols;
    } else {
        constexpr int H = BN / 2;          // B rows per CTA
        constexpr int E = (H - 128) / 32;  // chunks of the second MMA per half
        return c < 4 ? c * 32
                     : (c < 8 ? H + (c - 4) * 32 : (c < 8 + E ? 128 + (c - 8) * 32 : H + 128 + (c - 8 - E) * 32));
    }
}

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

enum : int { kUnitWhole = 0, kUnitSplit = 1, kUnitStreamK = 2 };

struct WorkUnit {
    int tile;      // raster tile id
    int m_blk, n_blk;
    int kb0, kb1;  // K blocks [kb0, kb1)
    int kind;      // kUnitWhole / kUnitSplit / kUnitStreamK
    int split;     // split-K slice index
    int sk_tile;   // stream-K tile index within the stream-K region
    int slot;      // stream-K: 0 = first unit of this worker's range, 1 = its last
};

// Grouped raster: walk `raster_group` m-blocks down, then step along N.
__device__ __forceinline__ void raster(const GemmParams& p, int tile, int& m_blk, int& n_blk)
{
    const int G = p.raster_group;
    const int per_group = G * p.num_n_blocks;
    const int g = tile / per_group;
    const int first_m = g * G;
    const int gm = min(p.num_m_blocks - first_m, G);
    const int local = tile - g * per_group;
    m_blk = first_m + local % gm;
    n_blk = local / gm;
}

// First K block of slice i of S over kb K blocks, floor(i * kb / S): in 32-bit
// arithmetic when the product fits (a 64-bit division is a long subroutine,
// and the MMA thread works out each unit's range between two units, while the
// tensor pipe drains).
__device__ __forceinline__ int slice_begin(int i, int kb, int S)
{
    if ((long long)i * kb < (1ll << 31))
        return int(unsigned(i) * unsigned(kb) / unsigned(S));
    return int((long long)i * kb / S);
}

// First stream-K iteration of `worker` (of `workers`): in 32-bit arithmetic
// when the product fits (a 64-bit division is a long subroutine on the
// critical path of every CTA's start), none at all without stream-K.
__device__ __forceinline__ long long sk_begin(const GemmParams& p, int worker, int workers)
{
    if (p.sk_iters == 0)
        return 0;
    const long long prod = (long long)worker * p.sk_iters;
    if (prod < (1ll << 32))
        return (long long)(unsigned(prod) / unsigned(workers));
    return prod / workers;
}

// The worker whose stream-K range holds iteration `it`.
__device__ __forceinline__ int sk_owner(const GemmParams& p, long long it, int workers)
{
    return int(((it + 1) * workers - 1) / p.sk_iters);
}

// The sequence of work units of one worker; every role walks the same one.
struct UnitIter {
    long long it, it_begin, it_end;  // this worker's stream-K iterations
    int u, u_end, step;              // data-parallel units u, u + step, ...

    __device__ __forceinline__ void init(const GemmParams& p, int worker, int workers)
    {
        it_begin = sk_begin(p, worker, workers);
        it_end = sk_begin(p, worker + 1, workers);
        it = it_begin;
        u = worker;
        u_end = p.dp_units;
        step = workers;
    }

    __device__ __forceinline__ bool next(const GemmParams& p, WorkUnit& w)
    {
        if (it < it_end) {
            const int KB = p.num_k_blocks;
            const int t = (it < (1ll << 31)) ? int(unsigned(it) / unsigned(KB)) : int(it / KB);
            w.kb0 = int(it - (long long)t * KB);
            w.kb1 = int(min((long long)KB, (long long)w.kb0 + (it_end - it)));
            w.kind = (w.kb0 == 0 && w.kb1 == KB) ? kUnitWhole : kUnitStreamK;
            w.sk_tile = t;
            w.slot = (it == it_begin) ? 0 : 1;
            w.split = 0;
            w.tile = p.dp_tiles + t;
            it += w.kb1 - w.kb0;
        } else if (u < u_end) {
            // slices of a tile in reverse K order: slice 0, the one that waits
            // for the others, has the largest unit id of its tile, so every
            // slice it waits for comes earlier in every worker's sequence
            const int S = p.split_k;
            w.tile = u / S;
            w.split = S - 1 - (u - w.tile * S);
            w.kb0 = slice_begin(w.split, p.num_k_blocks, S);
            w.kb1 = slice_begin(w.split + 1, p.num_k_blocks, S);
            w.kind = (S > 1) ? kUnitSplit : kUnitWhole;
            w.sk_tile = 0;
            w.slot = 0;
            u += step;
        } else {
            return false;
        }
        raster(p, w.tile, w.m_blk, w.n_blk);
        return true;
    }
};

__device__ __forceinline__ void trace_mark(const GemmParams& p, int slot)
{
    if (p.trace)
        p.trace[size_t(blockIdx.x) * kTraceSlots + slot] = ptx::global_timer_ns();
}

__device__ __forceinline__ void trace_unit(const GemmParams& p, int unit, int which)
{
    if (p.trace && unit < kTraceUnits)
        p.trace[size_t(blockIdx.x) * kTraceSlots + kTraceUnit0 + 4 * unit + which] =
            ptx::global_timer_ns();
}

// Time spent in one bounded wait.  %globaltimer is not guaranteed to move
// forward smoothly (the driver may re-synchronise it with the host clock), and
// a plain `now - start` in unsigned arithmetic would turn a step backwards
// into an immediate timeout.  So only forward steps count, each capped at
// 1 ms, and every poll counts at least 16 ns: a jump of the timer neither ends
// a wait early nor stretches it, and the wait ends even if the timer stops.
struct WaitClock {
    uint64_t last;
    uint64_t spent = 0;
    __device__ __forceinline__ WaitClock() : last(ptx::global_timer_ns()) {}
    __device__ __forceinline__ bool expired(uint64_t limit)
    {
        const uint64_t now = ptx::global_timer_ns();
        const int64_t step = int64_t(now - last);
        last = now;
        spent += uint64_t(step < 16 ? 16 : (step > 1000000 ? 1000000 : step));
        return spent > limit;
    }
};

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const GemmParams& p,
                                           volatile uint32_t* abort_flag, uint32_t code);

// The tile sequence of one worker.  Static: the stream-K / data-parallel
// iteration above.  With cluster launch control (p.clc): the cluster starts
// on the tile of its own launch index; every later tile is a cluster whose
// launch the leader cancelled, announced through a ring of kClcSlots
// responses (clc_full: response landed; clc_empty, in the leader CTA: every
// reader of both CTAs has decoded it).
struct Sched {
    UnitIter st;
    bool clc, first;
    int r;                    // next response to read
    int cs, mc, pair;         // CTAs per cluster, pairs per cluster, this CTA's pair
    int ks;                   // K slices per tile inside the cluster (pair = slice)
    uint32_t resp, full, empty_leader;

    __device__ __forceinline__ void init(const GemmParams& p, int worker, int workers, int cs_,
                                         int mc_, int pair_, uint32_t resp0, uint32_t full0,
                                         uint32_t empty0_leader)
    {
        st.init(p, worker, workers);
        cs = cs_;
        mc = mc_;
        pair = pair_;
        ks = p.ks;
        clc = p.clc != 0;
        first = true;
        r = 0;
        resp = resp0;
        full = full0;
        empty_leader = empty0_leader;
    }

    // Next unit; `arrive`: this thread reports its reading of a response.
    // WARP: the whole warp calls and decodes; it reconverges before the
    // arriving lane releases the slot.  `code`: status bit of a timeout.
    // With mc pairs per cluster a tile is a group of mc column blocks, pair i
    // of the cluster computing block mc * n + i.
    template <int CG, bool WARP = false>
    __device__ __forceinline__ bool next(const GemmParams& p, WorkUnit& w, bool arrive,
                                         volatile uint32_t* abort_flag, uint32_t code)
    {
        if (!clc) {
            if (!st.next(p, w))
                return false;
            if (ks > 1) {
                // the cluster's pairs take the K slices of one tile, in K order
                w.split = pair;
                w.kb0 = slice_begin(pair, p.num_k_blocks, ks);
                w.kb1 = slice_begin(pair + 1, p.num_k_blocks, ks);
                w.kind = kUnitSplit;
            } else {
                w.n_blk = w.n_blk * mc + pair;
            }
            return true;
        }
        int tile;
        if (first) {
            first = false;
            tile = int(blockIdx.x) / cs;
        } else {
            const int slot = r % kClcSlots;
            const uint32_t parity = uint32_t(r / kClcSlots) & 1u;
            bool landed = wait_phase(full + 8 * slot, parity, p, abort_flag, code);
            if constexpr (WARP)
                landed = __all_sync(0xffffffffu, landed);
            if (!landed)
                return false;
            uint32_t x = 0;
            const bool ok = ptx::clc_query(resp + 16 * slot, x);
            if constexpr (WARP)
                __syncwarp();
            if (arrive) {
                if constexpr (CG == 1)
                    ptx::mbar_arrive(empty_leader + 8 * slot);
                else
                    ptx::mbar_arrive_cluster(empty_leader + 8 * slot);
            }
            ++r;
            tile = ok ? int(x) / cs : -1;
        }
        if (tile < 0 || tile >= p.num_tiles)
            return false;
        w.tile = tile;
        w.kb0 = 0;
        w.kb1 = p.num_k_blocks;
        w.kind = kUnitWhole;
        w.split = 0;
        w.sk_tile = 0;
        w.slot = 0;
        raster(p, w.tile, w.m_blk, w.n_blk);
        w.n_blk = w.n_blk * mc + pair;
        return true;
    }
};

// Bounded wait on an mbarrier phase.  Gives up after p.timeout_ns (recording
// `code` in the status word) or as soon as another role of this CTA gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const GemmParams& p,
                                           volatile uint32_t* abort_flag, uint32_t code)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    WaitClock clock;
#pragma unroll 1
    while (true) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (clock.expired(p.timeout_ns)) {
            atomicOr(p.status, code);
            *abort_flag = 1u;
            return false;
        }
    }
}

// Bounded wait until a global counter reaches `want` (written by other CTAs
// with release semantics).  Gives up like wait_phase.
__device__ __forceinline__ bool wait_counter(const uint32_t* ctr, uint32_t want, const GemmParams& p,
                                             volatile uint32_t* abort_flag)
{
    if (ptx::ld_acquire_gpu(ctr) == want)
        return true;
    WaitClock clock;
#pragma unroll 1
    while (true) {
        __nanosleep(64);
        if (ptx::ld_acquire_gpu(ctr) == want)
            return true;
        if (*abort_flag)
            return false;
        if (clock.expired(p.timeout_ns)) {
            atomicOr(p.status, kStatusSplitTimeout);
            *abort_flag = 1u;
            return false;
        }
    }
}

// Bounded wait until a global counter reaches at least `want`.
__device__ __forceinline__ bool wait_counter_at_least(const uint32_t* ctr, uint32_t want,
                                                      const GemmParams& p,
                                                      volatile uint32_t* abort_flag)
{
    if (ptx::ld_acquire_gpu(ctr) >= want)
        return true;
    WaitClock clock;
#pragma unroll 1
    while (true) {
        __nanosleep(32);
        if (ptx::ld_acquire_gpu(ctr) >= want)
            return true;
        if (*abort_flag)
            return false;
        if (clock.expired(p.timeout_ns)) {
            atomicOr(p.status, kStatusSplitTimeout);
            *abort_flag = 1u;
            return false;
        }
    }
}

// After an abort: wait, bounded by `limit_ns` alone (the abort flag is
// already set), until the phase of `bar` with `parity` completed.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    WaitClock clock;
#pragma unroll 1
    while (!ptx::mbar_try_wait(bar, parity))
        if (clock.expired(limit_ns))
            return false;
    return true;
}

// After an abort: let `ns` of %globaltimer pass (bounded by polls too, should
// the timer stop), so that copies whose completion this CTA cannot observe --
// a pair follower's loads, counted on the leader's barriers; multicast loads
// from the other pair; an exchange copy in flight to or from the partner --
// land before the cluster's shared memory is released.
static __device__ __noinline__ void settle(uint64_t ns)
{
    WaitClock clock;
#pragma unroll 1
    while (!clock.expired(ns)) {
    }
}

// Bounds of the abort drain: ample for any copy or MMA in flight (they take
// microseconds), and short beside the wait limit that caused the abort.
constexpr uint64_t kDrainNs = 2000000;  // per drained barrier
constexpr uint64_t kSettleNs = 50000;

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

// Hand a fully read TMEM accumulator back to the MMA warp (of the pair's
// leader CTA, cluster rank `leader`).
template <int CG>
__device__ __forceinline__ void release_accumulator(uint32_t bar, int lane, uint32_t leader)
{
    ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
        if constexpr (CG == 1)
            ptx::mbar_arrive(bar);
        else
            ptx::mbar_arrive_cluster(ptx::map_to_cta(bar, leader));
    }
}

// Convert one thread's 32 fp32 values (one accumulator row, 32 consecutive
// columns) and stage the warp's 32 x 32 box in shared memory with the 64-byte
// swizzle the C tensor map uses (16-byte chunk index XOR bits 7-8 of the
// offset), then TMA-store it.  `m_row` is the accumulator row of lane 0,
// `col` the accumulator column of value 0.  With TR (swapped operands, the
// accumulator holds C transposed) the box is written transposed: accumulator
// rows are C columns and accumulator columns are C rows.  Two staging buffers
// per warp alternate; a buffer is reused only after the bulk store issued
// from it two boxes earlier finished reading.
//
// A TMA store clips at the end of a row of C only in whole 16-byte chunks: a
// box holding the end of a row whose length is not a multiple of 8 elements
// would also write the chunk's elements past the end, which belong to the
// caller.  That box is written with plain stores, element by element.
template <bool TR>
__device__ __noinline__ void store_box_ragged(const uint32_t (&packed)[16], const GemmParams& p,
                                              int lane, int col, int m_row)
{
    if constexpr (!TR) {
        // lane = row m_row + lane; values = columns col .. col + 31
        const int row = m_row + lane;
        if (row >= p.M)
            return;
        uint16_t* dst = p.c + size_t(row) * size_t(p.ldc);
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (col + i < p.N)
                dst[col + i] = uint16_t((i & 1) ? (packed[i >> 1] >> 16) : (packed[i >> 1] & 0xFFFFu));
    } else {
        // lane = column m_row + lane of C; values = rows col .. col + 31
        const int c_col = m_row + lane;
        if (c_col >= p.M)
            return;
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (col + i < p.N)
                p.c[size_t(col + i) * size_t(p.ldc) + size_t(c_col)] =
                    uint16_t((i & 1) ? (packed[i >> 1] >> 16) : (packed[i >> 1] & 0xFFFFu));
    }
}

// A warp's two staging buffers and the TMA stores reading them.  Single
// boxes alternate between the buffers; a paired store (two 32-column chunks
// in one instruction) reads both.
struct StoreQueue {
    uint32_t buf;       // shared address of the first 2 KiB buffer
    int ctr;            // single boxes staged so far
    bool pair_pending;  // the most recent store read both buffers
};

// The row end of C lies inside the 32-wide box at box_x and is not on a
// 16-byte boundary (a TMA store would write past it).
template <bool TR>
__device__ __forceinline__ bool box_is_ragged(const GemmParams& p, int col, int m_row)
{
    const int row_len = TR ? p.M : p.N;
    const int box_x = TR ? m_row : col;
    return (row_len & 7) != 0 && box_x < row_len && box_x + 32 > row_len;
}

// Convert and write one thread's 32 values into staging buffer sb (64-byte
// swizzle of the C tensor maps: 16-byte chunk index XOR bits 7-8 of the offset).
template <bool TR>
__device__ __forceinline__ void stage_box(const uint32_t (&r)[32], const GemmParams& p, uint32_t sb, int lane)
{
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        packed[i] = pack2(r[2 * i], r[2 * i + 1], p.dtype);
    if constexpr (!TR) {
        const uint32_t row_addr = sb + uint32_t(lane * 64);
        const uint32_t swz = uint32_t((lane >> 1) & 3);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
            ptx::st_shared_v4(row_addr + ((uint32_t(ch) ^ swz) << 4), packed[4 * ch + 0],
                              packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
    } else {
        // box row i = C row (col + i), box column lane = C column (m_row + lane)
        const uint32_t in_chunk = uint32_t((lane & 7) * 2);
        const uint32_t chunk = uint32_t(lane >> 3);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t addr = sb + uint32_t(i * 64) + ((chunk ^ uint32_t((i >> 1) & 3)) << 4) + in_chunk;
            const uint32_t h = (i & 1) ? (packed[i >> 1] >> 16) : (packed[i >> 1] & 0xFFFFu);
            ptx::st_shared_u16(addr, uint16_t(h));
        }
    }
}

template <bool TR>
__device__ __forceinline__ void store_box(const uint32_t (&r)[32], const GemmParams& p,
                                          const CUtensorMap* tmap_c, StoreQueue& sq, int lane, int col,
                                          int m_row)
{
    constexpr int kBufBytes = 32 * kStoreCols * 2;
    if (box_is_ragged<TR>(p, col, m_row)) {
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            packed[i] = pack2(r[2 * i], r[2 * i + 1], p.dtype);
        if ((TR ? col : m_row) < (TR ? p.N : p.M))
            store_box_ragged<TR>(packed, p, lane, col, m_row);
        return;
    }
    const uint32_t sb = sq.buf + uint32_t((sq.ctr & 1) * kBufBytes);
    if (lane == 0) {
        if (sq.pair_pending)
            ptx::bulk_wait_group_read<0>();
        else
            ptx::bulk_wait_group_read<1>();
    }
    sq.pair_pending = false;
    __syncwarp();
    stage_box<TR>(r, p, sb, lane);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (m_row < p.M && col < p.N) {  // boxes wholly outside C are skipped
            if constexpr (!TR)
                ptx::tma_store_2d(tmap_c, sb, col, m_row);
            else
                ptx::tma_store_2d(tmap_c, sb, m_row, col);
        }
        ptx::bulk_commit_group();
    }
    ++sq.ctr;
}

// Two adjacent 32-column chunks (accumulator columns col .. col + 63) as one
// TMA store: each SM's TMA unit spends about as long on a store as on an
// operand load, whatever its size, so halving the stores leaves it more time
// for the loads.  The chunks are staged one after the other into the warp's
// two buffers (pair_stage), then pair_store issues one store of both: through
// the 3-D view of C (32 columns x rows x whole 32-column chunks) for the
// operands in order, through a 64-row box when the accumulator holds C
// transposed.  Only whole, unragged chunks pair up (pair_ok).
template <bool TR>
__device__ __forceinline__ bool pair_ok(const GemmParams& p, int col, int m_row)
{
    if (!p.c_pairs || box_is_ragged<TR>(p, col, m_row) || box_is_ragged<TR>(p, col + 32, m_row))
        return false;
    return TR || (col / 32 + 1 < p.c_chunks);
}

__device__ __forceinline__ void pair_begin(StoreQueue& sq, int lane)
{
    if (lane == 0)
        ptx::bulk_wait_group_read<0>();  // no store reads either buffer any more
    __syncwarp();
}

template <bool TR>
__device__ __forceinline__ void pair_stage(const uint32_t (&r)[32], const GemmParams& p, const StoreQueue& sq,
                                           int half, int lane)
{
    stage_box<TR>(r, p, sq.buf + uint32_t(half * 32 * kStoreCols * 2), lane);
}

template <bool TR>
__device__ __forceinline__ void pair_store(const GemmParams& p, const CUtensorMap* tmap_c2, StoreQueue& sq,
                                           int lane, int col, int m_row)
{
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (m_row < p.M && col < p.N) {
            if constexpr (!TR)
                ptx::tma_store_3d(tmap_c2, sq.buf, 0, m_row, col / 32);
            else
                ptx::tma_store_2d(tmap_c2, sq.buf, m_row, col);
        }
        ptx::bulk_commit_group();
    }
    sq.pair_pending = true;
    sq.ctr = 0;
}

// MC: CTA pairs per cluster that share each A tile.  Pair i of the cluster
// computes column block MC * n + i of the tile group (m, n); the CTAs with the
// same rank in their pair need the same 128 A rows, so each loads 128 / MC of
// them once from L2 and multicasts them to all MC.
template <int CG, int BN, int STAGES, bool TR, int MC, int KS, bool RS = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_a2,
                const __grid_constant__ CUtensorMap tmap_b2, const __grid_constant__ CUtensorMap tmap_c2,
                const GemmParams p)
{
    // RS: one whole tile per CTA (a one-wave schedule), so the rings are idle
    // when the epilogue stores and hold its output boxes
    using Cfg = KernelConfig<CG, BN, STAGES, (KS > 1) || RS>;
    static_assert(MC == 1 || (MC == 2 && CG == 2), "A multicast pairs CTA pairs");
    static_assert(!RS || (KS == 1 && MC == 1), "ring-staged output: plain whole-tile kernels only");
    static_assert(KS == 1 || (KS == 2 && MC == 1), "a cluster holds column groups or K slices");
    constexpr int CS = CG * MC * KS;  // CTAs per cluster
    // K-slice exchange: each slice sends the other the 32-column chunks it owns,
    // one [128 rows][32 fp32] block per chunk, into the other's idle A ring
    // Ownership of a tile's 32-column chunks by the two K slices of a cluster:
    // pairs of adjacent chunks alternate between the slices (so each warp
    // stores its own pair with one paired store) up to the last multiple of
    // four chunks, single chunks after that.  The chunks a CTA does not own go
    // to consecutive slots of its staging block.  With an odd number of chunks
    // (BN = 224) the two slices own different numbers of them.
    constexpr int kTileChunks = BN / kStoreCols;
    constexpr int kPairedChunks = kTileChunks - kTileChunks % 4;  // chunks owned in pairs
    constexpr int kXchgSlots = (kTileChunks + 1) / 2;
    constexpr uint32_t kXchgSlotBytes = uint32_t(kRowsPerCta) * kStoreCols * 4;
    constexpr uint32_t kXchgBytes = uint32_t(kXchgSlots) * kXchgSlotBytes;
    auto chunk_owner = [](int c) { return c < kPairedChunks ? ((c >> 1) & 1) : (c & 1); };
    // index of c among the chunks of its owner: two per group of four in the
    // paired region, then every other chunk
    auto chunk_slot = [](int c) {
        return c < kPairedChunks ? ((c >> 2) * 2 + (c & 1)) : (kPairedChunks / 2 + ((c - kPairedChunks) >> 1));
    };
    static_assert(KS == 1 || int(kXchgBytes) <= STAGES * Cfg::kABytes, "exchange fits the A ring");
    static_assert(KS == 1 || int(kXchgBytes) + kEpiWarps * 2 * Cfg::kStoreBufBytes <= STAGES * Cfg::kBBytes,
                  "the exchange staging and the output boxes fit the B ring");
    static_assert(!RS || kEpiWarps * 2 * Cfg::kStoreBufBytes <= STAGES * Cfg::kBBytes,
                  "the output boxes fit the B ring");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CS > 1) ? ptx::cluster_ctarank() : 0u;  // in the cluster
    const uint32_t prank = (CG == 2) ? (rank & 1u) : 0u;            // in the CTA pair
    const uint32_t pair = rank / CG;                                // pair of the cluster
    const uint32_t leader = rank - prank;                           // the pair's MMA CTA
    const int worker = blockIdx.x / CS;
    const int workers = gridDim.x / CS;

    const uint32_t sA = base + Cfg::kOffA;
    const uint32_t sB = base + Cfg::kOffB;
    const uint32_t sStore = base + Cfg::kOffStore;
    const uint32_t bar_full = base + Cfg::kOffBar;         // + 8 * stage
    const uint32_t bar_empty = bar_full + 8 * STAGES;      // + 8 * stage
    const uint32_t bar_acc_full = bar_empty + 8 * STAGES;  // + 8 * buffer
    const uint32_t bar_acc_empty = bar_acc_full + 16;      // + 8 * buffer
    const uint32_t bar_clc_full = bar_acc_empty + 16;      // + 8 * slot
    const uint32_t bar_clc_empty = bar_clc_full + 8 * kClcSlots;  // + 8 * slot (leader's counts)
    const uint32_t bar_xready = bar_clc_empty + 8 * kClcSlots;    // the other slice's ring is free
    const uint32_t bar_xfull = bar_xready + 8;      // + 8 * half: the other slice's chunks landed
    const uint32_t bar_xstaged = bar_xfull + 16;    // + 8 * half: the half's four warps staged their rows
    const uint32_t bar_drain = bar_xstaged + 16;    // after an abort: the issued MMAs completed
    const uint32_t clc_resp = base + Cfg::kOffClcResp;     // + 16 * slot
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmemSlot);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + Cfg::kOffAbort);

    // Set-up runs in three warps at once: warp 3 (an epilogue warp, idle until
    // the first accumulator is ready) initialises the barriers, warp 1
    // allocates TMEM, warp 0 prefetches the tensor maps; meanwhile every role
    // works out its first work unit (below), which used to follow the set-up
    // and delayed the first loads of the CTAs that start last.
    constexpr int kInitThread = 3 * 32;
    if (threadIdx.x == kInitThread) {
        if (p.trace) {
            // this CTA's row of the timeline starts empty (cleared here rather than
            // by a memset on the stream, which would serialise back-to-back launches)
            uint64_t* row = p.trace + size_t(blockIdx.x) * kTraceSlots;
#pragma unroll 1
            for (int i = 0; i < kTraceSlots; ++i)
                row[i] = 0ull;
        }
        trace_mark(p, kTraceEntry);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);   // producer's arrive.expect_tx (+ bytes)
            ptx::mbar_init(bar_empty + 8 * s, MC);  // one tcgen05.commit per pair reading the stage
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_acc_full + 8 * b, 1);                // one tcgen05.commit
            ptx::mbar_init(bar_acc_empty + 8 * b, kEpiWarps * CG);  // every epilogue warp of the pair
        }
        for (int s = 0; s < kClcSlots; ++s) {
            ptx::mbar_init(bar_clc_full + 8 * s, 1);  // local producer's arrive.expect_tx(16)
            // readers of a response: producers and epilogue warps of every CTA, the MMA threads
            ptx::mbar_init(bar_clc_empty + 8 * s, CS * (1 + kEpiWarps) + CS / CG);
        }
        ptx::mbar_init(bar_xready, 1);  // the partner's arrival
        for (int h = 0; h < 2; ++h) {
            ptx::mbar_init(bar_xfull + 8 * h, 1);  // own arrive.expect_tx; the partner's bulk-copy bytes
            ptx::mbar_init(bar_xstaged + 8 * h, kEpiWarps / 2);
        }
        ptx::mbar_init(bar_drain, 1);  // one tcgen05.commit
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_a);
        ptx::prefetch_tensormap(&tmap_b);
        ptx::prefetch_tensormap(&tmap_c);
        if (p.c_pairs)
            ptx::prefetch_tensormap(&tmap_c2);
        if (p.k_chunks_a > 1)
            ptx::prefetch_tensormap(&tmap_a2);
        if (p.k_chunks_b > 1)
            ptx::prefetch_tensormap(&tmap_b2);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    // Every role walks the same unit sequence; the first unit is pure
    // arithmetic on the launch parameters (or, with cluster launch control, the
    // cluster's own index).  The producer and the MMA warp work theirs out now,
    // each into its own scheduler (dead in the other roles' code, so it costs
    // the epilogue no registers); the epilogue has until the first
    // accumulator is ready and works its out after the set-up.
    const uint32_t clc_empty_leader = (CS > 1) ? ptx::map_to_cta(bar_clc_empty, 0) : bar_clc_empty;
    Sched iter_p, iter_m;
    WorkUnit w0_p{}, w0_m{};
    bool have0_p = false, have0_m = false;
    if (warp == 0) {
        iter_p.init(p, worker, workers, CS, MC, int(pair), clc_resp, bar_clc_full, clc_empty_leader);
        have0_p = iter_p.next<CG, true>(p, w0_p, false, abort_flag, 0u);
    } else if (warp == 1 && prank == 0) {
        iter_m.init(p, worker, workers, CS, MC, int(pair), clc_resp, bar_clc_full, clc_empty_leader);
        have0_m = iter_m.next<CG, true>(p, w0_m, false, abort_flag, 0u);
    }
    ptx::tc_fence_before_sync();
    if constexpr (CS > 1)
        ptx::cluster_sync();
    else
        __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == kInitThread)
        trace_mark(p, kTraceSetup);

    // Everything above may overlap the previous kernel on the stream
    // (programmatic dependent launch), and so may each role's set-up below:
    // every role waits for that kernel to complete (griddepcontrol.wait) just
    // before its first access to global memory.  The next kernel may be
    // scheduled from here on.
    ptx::launch_dependents();
    // producer (warp 0) of a CTA whose full barriers count its loads (one CTA,
    // or a pair leader): stages armed with a load, and the parity of the phase
    // each last armed fill completes -- what the abort drain waits for
    uint32_t armed_mask = 0, armed_parity = 0;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The whole warp walks the unit and K-block sequence, so the loop state
        // is warp-uniform, and one elected lane issues the copies and barrier
        // updates.
        // (Run by lane 0 alone, every TMA instruction first moved its
        // per-thread operands into uniform registers; that bookkeeping cost
        // more than a K block's MMAs and left the tensor pipe waiting.)
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        bool first_unit = true;
        int requested = 0;
        Sched iter = iter_p;
        WorkUnit w = w0_p;
        // both CTAs' bytes of a pair are counted on the pair leader's barrier
        const uint32_t leader_full = (CG == 2) ? ptx::map_to_cta(bar_full, leader) : bar_full;
        for (bool have = have0_p; ok && have;
             have = ok && iter.next<CG, true>(p, w, lane == 0, abort_flag, kStatusProducerTimeout)) {
            if constexpr (RS) {
                // a ring-staged kernel runs one unit per CTA: a second one would
                // refill the ring its epilogue stages in -- a planning error
                if (!first_unit) {
                    if (lane == 0)
                        atomicOr(p.status, kStatusBadConfig);
                    break;
                }
            }
            const int a_row = w.m_blk * Cfg::kTileM + int(prank) * kRowsPerCta;
            const int b_row = w.n_blk * BN + int(prank) * Cfg::kBRows;
            if (first_unit) {
                // the first unit is known; now wait for the previous kernel
                if (lane == 0)
                    trace_mark(p, kTraceUnitKnown);
                ptx::grid_dependency_wait();
                if (lane == 0)
                    trace_mark(p, kTraceReady);
            }
            if (p.clc) {
                // ask for the tile after this one now, a whole tile ahead of need
                const int rq = requested++;
                const int slot = rq % kClcSlots;
                if (rank == 0) {
                    ok = __all_sync(0xffffffffu,
                                    wait_phase(bar_clc_empty + 8 * slot, (uint32_t(rq / kClcSlots) & 1u) ^ 1u,
                                               p, abort_flag, kStatusProducerTimeout));
                    if (!ok)
                        break;
                }
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar_clc_full + 8 * slot, 16);
                    if (rank == 0) {
                        if constexpr (CS == 1)
                            ptx::clc_try_cancel(clc_resp + 16 * slot, bar_clc_full + 8 * slot);
                        else
                            ptx::clc_try_cancel_all(clc_resp + 16 * slot, bar_clc_full + 8 * slot);
                    }
                }
                __syncwarp();
            }
            // L2 prefetch of the streamed operand (the one read from DRAM, not
            // shared by the tiles running at the same time) `prefetch` K
            // blocks ahead of the loads: the DRAM reads in flight are then not
            // bounded by the ring, and the ring's loads hit L2.  Two K blocks
            // per prefetch where the 3-D maps describe them (each TMA
            // instruction costs its unit the same time whatever its size).
            const int pf = p.prefetch;
            const CUtensorMap* pf_map2 = p.prefetch_b ? &tmap_b2 : &tmap_a2;
            const CUtensorMap* pf_map = p.prefetch_b ? &tmap_b : &tmap_a;
            const int pf_row = p.prefetch_b ? b_row : a_row;
            const int pf_chunks = p.prefetch_b ? p.k_chunks_b : p.k_chunks_a;
            int pf_next = w.kb0;  // first K block not yet prefetched
            auto prefetch_to = [&](int end) {
                end = min(end, w.kb1);
                while (pf_next < end) {
                    if (pf_next + 1 < end && pf_next + 1 < pf_chunks) {
                        ptx::tma_prefetch_3d(pf_map2, 0, pf_row, pf_next);
                        pf_next += 2;
                    } else {
                        ptx::tma_prefetch_2d(pf_map, pf_next * kTileK, pf_row);
                        pf_next += 1;
                    }
                }
            };
            if (pf > 0 && lane == 0)
                prefetch_to(w.kb0 + pf);
            for (int kb = w.kb0; kb < w.kb1;) {
                // Two K blocks in one copy per operand (3-D maps) when both are
                // whole 64-element chunks and the next ring stage follows this
                // one: a TMA copy costs about as much as 140 ns of its unit's
                // time whatever its size, so one copy per K block of 16 KiB
                // cannot keep up with the MMAs.  Both stages' bytes complete on
                // this stage's full barrier; the next stage's barrier only gets
                // an arrival (the MMA warp always consumes this stage first).
                const bool dbl = (stage % 2 == 0) && (stage + 1 < STAGES) && (kb + 1 < w.kb1) &&
                                 p.pair_copies && (kb + 1 < p.k_chunks_b) &&
                                 (MC > 1 || kb + 1 < p.k_chunks_a);
                const int nkb = dbl ? 2 : 1;
                if (pf > 0 && lane == 0)
                    prefetch_to(kb + nkb + pf);
                ok = __all_sync(0xffffffffu, wait_phase(bar_empty + 8 * stage, phase ^ 1u, p, abort_flag,
                                                        kStatusProducerTimeout));
                if (ok && dbl)
                    ok = __all_sync(0xffffffffu, wait_phase(bar_empty + 8 * (stage + 1), phase ^ 1u, p,
                                                            abort_flag, kStatusProducerTimeout));
                if (!ok)
                    break;
                const int rel = kb - w.kb0;
                const bool stall = p.stall_kblock >= 0 && blockIdx.x == 0 && first_unit &&
                                   p.stall_kblock >= rel && p.stall_kblock < rel + nkb;
                if (!stall && (CG == 1 || prank == 0)) {  // warp-uniform bookkeeping
                    armed_mask |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                }
                if (!stall && ptx::elect_one()) {
                    if (first_unit && kb == w.kb0)
                        trace_mark(p, kTraceFirstLoad);
                    const uint32_t fb = bar_full + 8 * stage;
                    const uint32_t dA = sA + stage * Cfg::kABytes;
                    const uint32_t dB = sB + stage * Cfg::kBBytes;
                    const uint32_t tx = Cfg::kTxBytes * uint32_t(nkb);
                    if constexpr (CG == 1) {
                        ptx::mbar_arrive_expect_tx(fb, tx);
                        if (dbl) {
                            ptx::mbar_arrive(fb + 8);
                            ptx::tma_load_3d(dA, &tmap_a2, fb, 0, a_row, kb);
                            ptx::tma_load_3d(dB, &tmap_b2, fb, 0, b_row, kb);
                        } else {
                            ptx::tma_load_2d(dA, &tmap_a, fb, kb * kTileK, a_row);
                            ptx::tma_load_2d(dB, &tmap_b, fb, kb * kTileK, b_row);
                        }
                    } else {
                        const uint32_t lfb = leader_full + 8 * stage;
                        if (prank == 0) {
                            ptx::mbar_arrive_expect_tx(fb, tx);
                            if (dbl)
                                ptx::mbar_arrive(fb + 8);
                        }
                        if constexpr (MC == 1) {
                            if (dbl)
                                ptx::tma_load_3d_pair(dA, &tmap_a2, lfb, 0, a_row, kb);
                            else
                                ptx::tma_load_2d_pair(dA, &tmap_a, lfb, kb * kTileK, a_row);
                        } else {
                            // rows [pair * 128 / MC, +128 / MC) of this CTA's 128, into
                            // the same place in every CTA of the cluster with this
                            // prank (one copy per K block: the part is not a whole
                            // ring stage, so two of them are not contiguous)
                            constexpr int kPart = kRowsPerCta / MC;
                            uint16_t mask = 0;
#pragma unroll
                            for (int i = 0; i < MC; ++i)
                                mask |= uint16_t(1u << (int(prank) + CG * i));
                            for (int j = 0; j < nkb; ++j)
                                ptx::tma_load_2d_pair_multicast(
                                    dA + uint32_t(j * Cfg::kABytes) + uint32_t(pair) * uint32_t(kPart * kTileK * 2),
                                    &tmap_a, lfb, (kb + j) * kTileK, a_row + int(pair) * kPart, mask);
                        }
                        if (dbl)
                            ptx::tma_load_3d_pair(dB, &tmap_b2, lfb, 0, b_row, kb);
                        else
                            ptx::tma_load_2d_pair(dB, &tmap_b, lfb, kb * kTileK, b_row);
                    }
                }
                __syncwarp();
                kb += nkb;
                stage += nkb;
                if (stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            first_unit = false;
        }
        if (lane == 0)
            trace_mark(p, kTraceLastLoad);
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue
        // The whole warp of the pair leader walks the unit and K-block
        // sequence (warp-uniform state) and one elected lane issues the MMAs
        // and commits.  Issued by `lane == 0` inside a one-thread branch, each
        // tcgen05.mma cost ~40 ns of issue (160-190 ns per K block of four),
        // which paced the tensor pipe below its rate; elected, ~15 ns.
        if (prank == 0) {
            ptx::grid_dependency_wait();
            const uint32_t idesc = p.idesc;
            const uint32_t idesc2 = p.idesc2;  // second MMA of a 320/384-column unit
            const uint64_t a_desc0 = make_sdesc_sw128(sA);
            const uint64_t b_desc0 = make_sdesc_sw128(sB);
            const uint32_t tmem0 = __shfl_sync(0xffffffffu, tmem_base, 0);
            int stage = 0;
            uint32_t phase = 0;
            int t = 0;
            bool ok = true;
            Sched iter = iter_m;
            WorkUnit w = w0_m;
            // Without launch control the unit sequence is pure arithmetic (a few
            // dependent integer divisions, ~0.5 us): the next unit is worked out
            // right after the current unit's first K block is issued, while the
            // tensor pipe is busy, instead of between units, where it left the
            // pipe idle.  With launch control it waits for a response and stays
            // between units.
            const bool ahead = !p.clc;
            bool have = have0_m;
            WorkUnit w_next;
            bool have_next = false;
            while (ok && have) {
                const int buf = Cfg::kAccBufs == 2 ? (t & 1) : 0;
                const uint32_t acc_phase = uint32_t(Cfg::kAccBufs == 2 ? (t >> 1) : t) & 1u;
                ++t;
                ok = __all_sync(0xffffffffu, wait_phase(bar_acc_empty + 8 * buf, acc_phase ^ 1u, p, abort_flag,
                                                        kStatusMmaTimeout));
                if (!ok)
                    break;
                ptx::tc_fence_after_sync();
                if (lane == 0)
                    trace_unit(p, t - 1, 0);
                const uint32_t d_tmem = tmem0 + uint32_t(buf * Cfg::kAccStride);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    ok = __all_sync(0xffffffffu, wait_phase(bar_full + 8 * stage, phase, p, abort_flag,
                                                            kStatusMmaTimeout));
                    if (!ok)
                        break;
                    ptx::tc_fence_after_sync();
                    const uint64_t ad = a_desc0 + uint64_t((stage * Cfg::kABytes) >> 4);
                    const uint64_t bd = b_desc0 + uint64_t((stage * Cfg::kBBytes) >> 4);
                    if (ptx::elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kTileK / kMmaK; ++kk) {
                            // advance 16 elements = 32 bytes along K inside the swizzle atom
                            ptx::mma_f16<CG>(d_tmem, ad + uint64_t(kk * 2), bd + uint64_t(kk * 2), idesc,
                                             (kb > w.kb0 || kk > 0) ? 1u : 0u);
                            if constexpr (Cfg::kMmaN2 > 0)
                                ptx::mma_f16<CG>(d_tmem + uint32_t(Cfg::kMmaN1), ad + uint64_t(kk * 2),
                                                 bd + uint64_t(((Cfg::kMmaN1 / 2) * 128) >> 4) +
                                                     uint64_t(kk * 2),
                                                 idesc2, (kb > w.kb0 || kk > 0) ? 1u : 0u);
                        }
                        // the stage is free once every pair sharing it has read it (with
                        // A multicast both pairs of the cluster, else this pair)
                        if constexpr (CG == 1)
                            ptx::mma_commit(bar_empty + 8 * stage);
                        else if constexpr (MC > 1)
                            ptx::mma_commit_pair(bar_empty + 8 * stage, uint16_t((1u << CS) - 1u));
                        else
                            ptx::mma_commit_pair(bar_empty + 8 * stage, uint16_t(0x3u << (CG * pair)));
                    }
                    __syncwarp();
                    if (ahead && kb == w.kb0)
                        have_next = iter.next<CG, true>(p, w_next, lane == 0, abort_flag, kStatusMmaTimeout);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                // the same elected lane: a commit tracks the MMAs its own thread issued
                if (ptx::elect_one()) {
                    if constexpr (CG == 1)
                        ptx::mma_commit(bar_acc_full + 8 * buf);
                    else
                        ptx::mma_commit_pair(bar_acc_full + 8 * buf, uint16_t(0x3u << (CG * pair)));
                }
                __syncwarp();
                if (lane == 0)
                    trace_unit(p, t - 1, 1);
                if (!ahead || w.kb0 >= w.kb1)  // (a unit without K blocks did not work it out)
                    have_next = iter.next<CG, true>(p, w_next, lane == 0, abort_flag, kStatusMmaTimeout);
                w = w_next;
                have = have_next;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Warps 2..9: two per TMEM lane quarter q (= warp % 4, the quarter a
        // warp may access); h selects the half of the columns it handles.
        ptx::grid_dependency_wait();
        const int ew = warp - 2;
        const int q = warp & 3;
        const int h = ew >> 2;
        // 32-column chunks of a tile: the first half (rounded up) for h = 0
        constexpr int kHalfChunks = (BN / kStoreCols + 1) / 2;
        const int c_begin = h * kHalfChunks;
        const int c_end = h ? BN / kStoreCols : kHalfChunks;
        const int row = q * 32 + lane;
        // the clustered split stages its output boxes in the B ring after the
        // exchange block (its one unit ends with the rings idle)
        const uint32_t store_base = (KS > 1) ? sB + kXchgBytes : (RS ? sB : sStore);
        StoreQueue sq{store_base + uint32_t(ew * 2 * Cfg::kStoreBufBytes), 0, false};
        constexpr size_t kSlotF4 = size_t(Cfg::kPartialFloats) / 4;  // float4s per CTA partial
        float4* const parts = reinterpret_cast<float4*>(p.partials);
        int t = 0;
        int xchg_count = 0;  // K-slice exchanges done (parity of the exchange barriers)
        Sched iter;
        iter.init(p, worker, workers, CS, MC, int(pair), clc_resp, bar_clc_full, clc_empty_leader);
        WorkUnit w;
        while (iter.next<CG, true>(p, w, lane == 0, abort_flag, kStatusEpilogueTimeout)) {
            if (t > 0 && warp == 2 && lane == 0)
                trace_unit(p, t - 1, 3);  // previous unit's epilogue finished
            const int buf = Cfg::kAccBufs == 2 ? (t & 1) : 0;
            const uint32_t acc_phase = uint32_t(Cfg::kAccBufs == 2 ? (t >> 1) : t) & 1u;
            ++t;
            // the warp leaves together: a lane that timed out just as the phase
            // completed must not strand the others in the aligned TMEM loads
            if (!__all_sync(0xffffffffu, wait_phase(bar_acc_full + 8 * buf, acc_phase, p, abort_flag,
                                                    kStatusEpilogueTimeout)))
                break;
            ptx::tc_fence_after_sync();
            if (warp == 2 && lane == 0)
                trace_unit(p, t - 1, 2);
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * Cfg::kAccStride);
            const int cta_row0 = w.m_blk * Cfg::kTileM + int(prank) * kRowsPerCta;
            const int m_row = cta_row0 + q * 32;  // first row of this warp's boxes
            const int n_col = w.n_blk * BN;
            if (KS > 1 && w.kind == kUnitSplit) {
                // ---- split-K inside the cluster: the two K slices of this tile
                // run on the two pairs (or CTAs) of the cluster.  Chunk c belongs
                // to slice chunk_owner(c).  Each CTA stages the chunks its partner (same
                // rank in the other slice) owns in its own idle B ring; the
                // exchange runs in two halves, one per column half of the epilogue
                // warps (h), whose staged chunks are contiguous in the block.  As
                // soon as the unit's MMAs are done (the rings are idle) one thread
                // tells the partner that this CTA's A ring may be written; once a
                // half's four warps have staged their rows and the partner's ring is
                // free, the half's first warp copies that half into it with one bulk
                // copy, counted on the partner's barrier of that half.  Each warp
                // then waits only for its half of the partner's chunks and stores
                // own + partner's in C.  One tile per cluster (the planner's one-wave rule), so no
                // later unit refills the rings.  Warps whose rows are all past M
                // take part too (the byte counts cover every row); their rows are
                // clipped.  (Per-thread st.async remote stores measured ~3 GB/s
                // per warp; a bulk copy per warp and chunk was fast but each copy
                // occupies the SM's TMA unit about as long as an operand load.)
                const int j = w.split;
                const uint32_t partner = rank ^ uint32_t(CG);
                const uint32_t xparity = uint32_t(xchg_count & 1);
                ++xchg_count;
                const uint32_t swz = uint32_t(row & 7);
                auto xoff = [&](int c, int v) -> uint32_t {  // [slot][row][16-byte v ^ row % 8]
                    return uint32_t(chunk_slot(c) * (kRowsPerCta * kStoreCols * 4) + row * (kStoreCols * 4)) +
                           ((uint32_t(v) ^ swz) << 4);
                };
                // chunks of half hh that slice jj owns, and the slot of the first one
                auto half_owned = [&](int jj, int hh) {
                    int n = 0;
                    for (int c = hh * kHalfChunks; c < (hh ? kTileChunks : kHalfChunks); ++c)
                        n += (chunk_owner(c) == jj) ? 1 : 0;
                    return n;
                };
                auto half_first_slot = [&](int jj, int hh) {
                    for (int c = hh * kHalfChunks; c < (hh ? kTileChunks : kHalfChunks); ++c)
                        if (chunk_owner(c) == jj)
                            return chunk_slot(c);
                    return 0;
                };
                if (warp == 2 && lane == 0) {
                    // the bytes each half receives, then: this CTA's A ring is free
                    ptx::mbar_arrive_expect_tx(bar_xfull, uint32_t(half_owned(j, 0)) * kXchgSlotBytes);
                    ptx::mbar_arrive_expect_tx(bar_xfull + 8, uint32_t(half_owned(j, 1)) * kXchgSlotBytes);
                    ptx::mbar_arrive_cluster(ptx::map_to_cta(bar_xready, partner));
                }
                int first_owned = c_end, last_owned = c_begin;
#pragma unroll 1
                for (int c = c_begin; c < c_end; ++c) {
                    if (chunk_owner(c) == j) {
                        first_owned = min(first_owned, c);
                        last_owned = c;
                        continue;
                    }
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        ptx::st_shared_v4(sB + xoff(c, v), r[4 * v + 0], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
                }
                ptx::fence_proxy_async_smem();  // the staged rows, visible to the bulk copy
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(bar_xstaged + 8 * h);
                if (first_owned >= c_end)
                    release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                if (ew == 4 * h) {
                    // the half's first warp sends the half
                    if (!__all_sync(0xffffffffu, wait_phase(bar_xstaged + 8 * h, xparity, p, abort_flag,
                                                            kStatusSplitTimeout)))
                        break;
                    if (!__all_sync(0xffffffffu, wait_phase(bar_xready, xparity, p, abort_flag,
                                                            kStatusSplitTimeout)))
                        break;
                    const int n_send = half_owned(1 - j, h);
                    if (lane == 0 && n_send > 0) {
                        const uint32_t off = uint32_t(half_first_slot(1 - j, h)) * kXchgSlotBytes;
                        ptx::bulk_copy_to_cluster(ptx::map_to_cta(sA + off, partner), sB + off,
                                                  uint32_t(n_send) * kXchgSlotBytes,
                                                  ptx::map_to_cta(bar_xfull + 8 * h, partner));
                    }
                }
                if (!__all_sync(0xffffffffu, wait_phase(bar_xfull + 8 * h, xparity, p, abort_flag,
                                                        kStatusSplitTimeout)))
                    break;
                // own chunk c: this slice's partial from TMEM + the partner's
                // from the A ring (two terms: the sum is the same whichever
                // slice adds)
                auto sum_chunk = [&](int c, uint32_t (&r)[32]) {
                    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                    uint32_t x[32];
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        ptx::ld_shared_v4(sA + xoff(c, v), x[4 * v + 0], x[4 * v + 1], x[4 * v + 2],
                                          x[4 * v + 3]);
                    ptx::tmem_ld_wait();
                    if (c == last_owned)
                        release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(x[i]));
                };
#pragma unroll 1
                for (int c = first_owned; c < c_end;) {
                    if (chunk_owner(c) != j) {
                        ++c;
                        continue;
                    }
                    const int col = n_col + chunk_col<BN>(c);
                    uint32_t r[32];
                    if (c + 1 < c_end && chunk_owner(c + 1) == j && chunk_col<BN>(c + 1) == chunk_col<BN>(c) + 32 &&
                        pair_ok<TR>(p, col, m_row)) {
                        pair_begin(sq, lane);
                        sum_chunk(c, r);
                        pair_stage<TR>(r, p, sq, 0, lane);
                        sum_chunk(c + 1, r);
                        pair_stage<TR>(r, p, sq, 1, lane);
                        pair_store<TR>(p, &tmap_c2, sq, lane, col, m_row);
                        c += 2;
                    } else {
                        sum_chunk(c, r);
                        store_box<TR>(r, p, &tmap_c, sq, lane, col, m_row);
                        ++c;
                    }
                }
                continue;
            }
            if constexpr (KS > 1) {
                // a clustered split-K kernel runs split units only (its output
                // boxes live in the B ring, which a unit without the exchange
                // would still be loading): anything else is a planning error
                if (lane == 0)
                    atomicOr(p.status, kStatusBadConfig);
                release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                continue;
            }

            if (m_row >= p.M) {
                // every row of this warp is padding past M: nothing to load or store
                // (the same holds for every piece of the tile, so no counter is used)
                release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                continue;
            }
            if (w.kind == kUnitWhole) {
                // ---- whole tile: TMEM -> registers -> bf16/fp16 -> smem -> TMA
                // store, two chunks per store where they pair up
#pragma unroll 1
                for (int c = c_begin; c < c_end;) {
                    const int col = n_col + chunk_col<BN>(c);
                    uint32_t r[32];
                    if (c + 1 < c_end && chunk_col<BN>(c + 1) == chunk_col<BN>(c) + 32 && pair_ok<TR>(p, col, m_row)) {
                        pair_begin(sq, lane);
                        ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                        ptx::tmem_ld_wait();
                        pair_stage<TR>(r, p, sq, 0, lane);
                        ptx::tmem_ld_32x32b_x32(taddr + uint32_t((c + 1) * kStoreCols), r);
                        ptx::tmem_ld_wait();
                        if (c + 1 == c_end - 1)
                            release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                        pair_stage<TR>(r, p, sq, 1, lane);
                        pair_store<TR>(p, &tmap_c2, sq, lane, col, m_row);
                        c += 2;
                    } else {
                        ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                        ptx::tmem_ld_wait();
                        if (c == c_end - 1)
                            release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                        store_box<TR>(r, p, &tmap_c, sq, lane, col, m_row);
                        ++c;
                    }
                }
                continue;
            }

            if (w.kind == kUnitSplit && p.split_scatter) {
                // ---- split-K, one wave: all S slices of the tile run at once, one
                // per worker.  Chunk c of the tile belongs to slice c % S.  Each
                // slice stores the chunks it does not own, counts itself, waits
                // for the other S - 1 (bounded: they never wait on anything
                // before storing), then sums its own chunks over slices 0..S-1 in
                // order -- its own share straight from TMEM -- and stores C.
                const int S = p.split_k;
                const int j = w.split;
                const int ctile = w.tile * CS + int(rank);
                uint32_t* const cnt = p.tile_sems + size_t(ctile * kEpiWarps + ew) * kCountersPerWarp;
                const bool row_ok = (cta_row0 + row) < p.M;
                auto chunk_ptr = [&](int slice, int c) -> float4* {
                    const size_t slot = size_t(w.tile * S + slice) * CS + rank;
                    return parts + slot * kSlotF4 + size_t(c) * 8 * kRowsPerCta + row;
                };
                // store the chunks other slices own
                bool owns_any = false;
                int last_owned = c_begin;
#pragma unroll 1
                for (int c = c_begin; c < c_end; ++c) {
                    if (c % S == j) {
                        owns_any = true;
                        last_owned = c;
                        continue;
                    }
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                    ptx::tmem_ld_wait();
                    if (row_ok) {
                        float4* dst = chunk_ptr(j, c);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            __stcg(dst + v * kRowsPerCta,
                                   make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                               __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
                    }
                }
                if (!owns_any)
                    release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                // publish: the warp barrier orders every lane's stores before lane
                // 0's release-add; the slice that arrives last need not poll
                __syncwarp();
                bool ready = true;
                if (lane == 0) {
                    const uint32_t old = ptx::atom_add_release_gpu(cnt, 1u);
                    if (old + 1u < uint32_t(S))
                        ready = wait_counter_at_least(cnt, uint32_t(S), p, abort_flag);
                }
                ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                __threadfence();
                if (owns_any) {
#pragma unroll 1
                    for (int c = c_begin; c < c_end; ++c) {
                        if (c % S != j)
                            continue;
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                        float4 acc[8];
                        float4 x[8];
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                        for (int i = 0; i < S; ++i) {
                            if (i == j) {
                                ptx::tmem_ld_wait();
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    x[v] = make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                                       __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                            } else {
                                const float4* src = chunk_ptr(i, c);
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    x[v] = (row_ok && ready) ? __ldcg(src + v * kRowsPerCta)
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                            if (i == 0) {
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    acc[v] = x[v];
                            } else {
#pragma unroll
                                for (int v = 0; v < 8; ++v) {
                                    acc[v].x += x[v].x;
                                    acc[v].y += x[v].y;
                                    acc[v].z += x[v].z;
                                    acc[v].w += x[v].w;
                                }
                            }
                        }
                        ptx::tmem_ld_wait();
                        if (c == last_owned)
                            release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            r[4 * v + 0] = __float_as_uint(acc[v].x);
                            r[4 * v + 1] = __float_as_uint(acc[v].y);
                            r[4 * v + 2] = __float_as_uint(acc[v].z);
                            r[4 * v + 3] = __float_as_uint(acc[v].w);
                        }
                        store_box<TR>(r, p, &tmap_c, sq, lane, n_col + chunk_col<BN>(c), m_row);
                    }
                }
                // second arrival: the slice that completes 2S has seen every other
                // slice pass its wait, so it re-arms the counter for the next launch
                __syncwarp();
                if (lane == 0 && atomicAdd(cnt, 1u) == uint32_t(2 * S - 1))
                    *cnt = 0u;
                continue;
            }

            // ---- one piece of a tile's K range (split-K slice or stream-K piece).
            // Pieces j = 0 .. P-1 in K order.  Pieces 1 .. P-1 store fp32 partials
            // and count themselves in T; piece 0 -- under stream-K the last unit of
            // its worker, so usually the last to finish -- waits until T = P - 1,
            // then forms C = p_0 + ((p_1 + p_2) + ... + p_{P-1}) with p_0 straight
            // from TMEM.  The order of the additions is fixed, so C is the same on
            // every run; pieces 1.. never wait, so piece 0's wait always ends.
            int pieces, j, first_worker = 0;
            long long tile_it0 = 0;
            int ctile;
            if (w.kind == kUnitSplit) {
                pieces = p.split_k;
                j = w.split;
                ctile = w.tile * CS + int(rank);
            } else {
                tile_it0 = (long long)w.sk_tile * p.num_k_blocks;
                first_worker = sk_owner(p, tile_it0, workers);
                pieces = sk_owner(p, tile_it0 + p.num_k_blocks - 1, workers) - first_worker + 1;
                j = worker - first_worker;
                ctile = w.sk_tile * CS + int(rank);
            }
            auto slot_of = [&](int i) -> size_t {  // CTA partial slot of piece i
                if (w.kind == kUnitSplit)
                    return size_t(w.tile * p.split_k + i) * CS + rank;
                const int wi = first_worker + i;
                const int si = (sk_begin(p, wi, workers) >= tile_it0) ? 0 : 1;
                return size_t(wi * 2 + si) * CS + rank;
            };
            uint32_t* const cnt = p.tile_sems + size_t(ctile * kEpiWarps + ew) * kCountersPerWarp;
            const bool row_ok = (cta_row0 + row) < p.M;  // padding rows move no bytes
            // partial layout per CTA slot: [chunk][v = 0..7][row 0..127] float4
            auto chunk_ptr = [&](size_t slot, int c) -> float4* {
                return parts + slot * kSlotF4 + size_t(c) * 8 * kRowsPerCta + row;
            };
            auto load_chunk = [&](size_t slot, int c, float4 (&x)[8]) {
                const float4* src = chunk_ptr(slot, c);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    x[v] = row_ok ? __ldcg(src + v * kRowsPerCta) : make_float4(0.f, 0.f, 0.f, 0.f);
            };
            auto add4 = [](float4& a, const float4& b) {
                a.x += b.x;
                a.y += b.y;
                a.z += b.z;
                a.w += b.w;
            };

            if (j == 0) {
                bool ready = true;
                if (lane == 0)
                    ready = wait_counter(cnt, uint32_t(pieces - 1), p, abort_flag);
                ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                if (!ready) {
                    release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                    continue;
                }
                __threadfence();
#pragma unroll 1
                for (int c = c_begin; c < c_end; ++c) {
                    // S' = p_1 + ... + p_{P-1}, two pieces' loads in flight at a time
                    float4 sp[8], x1[8];
                    load_chunk(slot_of(1), c, sp);
                    if (pieces > 2)
                        load_chunk(slot_of(2), c, x1);
                    if (pieces > 2) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            add4(sp[v], x1[v]);
                    }
#pragma unroll 1
                    for (int i = 3; i < pieces; i += 2) {
                        float4 y0[8], y1[8];
                        load_chunk(slot_of(i), c, y0);
                        if (i + 1 < pieces)
                            load_chunk(slot_of(i + 1), c, y1);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            add4(sp[v], y0[v]);
                        if (i + 1 < pieces) {
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                add4(sp[v], y1[v]);
                        }
                    }
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                    ptx::tmem_ld_wait();
                    if (c == c_end - 1)
                        release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + sp[v].x);
                        r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + sp[v].y);
                        r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + sp[v].z);
                        r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + sp[v].w);
                    }
                    store_box<TR>(r, p, &tmap_c, sq, lane, n_col + chunk_col<BN>(c), m_row);
                }
                __syncwarp();
                if (lane == 0)
                    *cnt = 0u;  // every piece has arrived: re-armed for the next launch
                continue;
            }

            // tail piece j >= 1: store this piece's partial, then count it
            const size_t mine = slot_of(j);
#pragma unroll 1
            for (int c = c_begin; c < c_end; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c * kStoreCols), r);
                ptx::tmem_ld_wait();
                if (c == c_end - 1)
                    release_accumulator<CG>(bar_acc_empty + 8 * buf, lane, leader);
                if (row_ok) {
                    float4* dst = chunk_ptr(mine, c);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        __stcg(dst + v * kRowsPerCta,
                               make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                           __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
                }
            }
            __threadfence();
            __syncwarp();
            if (lane == 0)
                atomicAdd(cnt, 1u);
        }
        if (t > 0 && warp == 2 && lane == 0)
            trace_unit(p, t - 1, 3);
        if (lane == 0)
            ptx::bulk_wait_group_all();
        if (warp == 2 && lane == 0)
            trace_mark(p, kTraceEpiDone);
        __syncwarp();
    }

    // --------------------------------------------------------------- teardown
    // Every role of this CTA has left its loop, so the abort flag is final.
    // After an abort, asynchronous work may still be in flight: drain it
    // (bounded) before the CTA's shared memory and TMEM are released.  The
    // MMA thread commits once more and waits, so every MMA it issued has
    // completed; the producer waits for each stage it armed to land; then the
    // CTA settles for copies it cannot observe.  Without an abort none of
    // this runs (every load was consumed, every MMA committed and waited for
    // by the epilogue, every store waited for above).
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
        if (warp == 1 && prank == 0) {
            if (ptx::elect_one()) {  // the lane that issued the MMAs
                if constexpr (CG == 1)
                    ptx::mma_commit(bar_drain);
                else
                    ptx::mma_commit_pair(bar_drain, uint16_t(1u << rank));
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
    if constexpr (CS > 1)
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
