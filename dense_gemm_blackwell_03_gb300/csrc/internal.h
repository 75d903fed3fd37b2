// internal.h -- declarations shared by the library's host-side translation units.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/bwgemm.h"
#include "kernel_params.h"

namespace bwgemm {

// Compiled kernel variants: (CTA group, BN, ring stages, swapped operands,
// pairs per cluster sharing A, K slices per cluster).  Every variant keeps the
// ring at <= 192 KiB of shared memory plus 32 KiB of epilogue staging.  The
// swapped variants compute C^T = B A^T for small M; the mc = 2 variants run
// clusters of two CTA pairs on adjacent column blocks that multicast their
// common A tile; the ks = 2 variants run the two K slices of a split-K tile
// in one cluster and exchange partials through distributed shared memory.
// The BN = 224 pair variants cut N = 8192 into 37 column tiles, so that one
// row block (x 2 K slices, or two row blocks) fills 74 of 76 CTA pairs; the
// BN = 320 ones (two MMAs per K step, one 320-column accumulator) cut
// N = 10240 into 32 tiles, whose 2 K slices fit 32 clusters of four; BN = 384
// cuts N = 28672 into 75 tiles, one wave of whole tiles.
struct Variant {
    int cg;      // 1: cta_group::1, 128-row units; 2: CTA pair, 256-row units
    int bn;      // columns of the MMA per unit (= MMA N)
    int stages;  // shared-memory ring depth
    bool trans;  // operands swapped, accumulator holds C transposed
    int mc;      // CTA pairs per cluster sharing each A tile (1 = no multicast)
    int ks;      // K slices of a tile per cluster (1, or 2 for the clustered split-K)
    bool rs = false;  // one whole tile per CTA: output boxes staged in the idle B ring,
                      // whose freed room holds one more stage (the clustered split-K
                      // variants do the same)
};

constexpr Variant kVariants[] = {
    {1, 256, 4, false, 1, 1}, {1, 128, 6, false, 1, 1}, {2, 256, 6, false, 1, 1},
    {2, 128, 8, false, 1, 1}, {2, 128, 8, true, 1, 1},  {2, 64, 9, true, 1, 1},
    {1, 128, 6, true, 1, 1},  {1, 64, 8, true, 1, 1},   {2, 256, 6, false, 2, 1},
    {2, 128, 8, false, 2, 1}, {2, 256, 7, false, 1, 2}, {1, 64, 9, true, 1, 2},
    {2, 224, 6, false, 1, 1}, {2, 224, 7, false, 1, 2},
    {2, 320, 5, false, 1, 1}, {2, 320, 6, false, 1, 2}, {2, 384, 4, false, 1, 1},
    {2, 224, 7, false, 1, 1, true}, {2, 384, 5, false, 1, 1, true},
};
constexpr int kNumVariants = int(sizeof(kVariants) / sizeof(kVariants[0]));

// Index into kVariants, or -1.
int find_variant(int cg, int bn, bool trans, int mc = 1, int ks = 1, bool rs = false);

// Dynamic shared memory bytes of a variant.
int variant_smem_bytes(int idx);

// Launch variant `idx` with `grid` CTAs (a multiple of its cluster size);
// with `pdl`, as a programmatic dependent launch (its prologue may overlap the
// previous kernel on the stream).  a2 / b2: 3-D views of the operands that
// copy two K blocks at once (used only when p.k_chunks > 1); c2: the view of
// C that stores two 32-column chunks at once (used only when p.c_pairs).
cudaError_t launch_variant(int idx, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                           const CUtensorMap& a2, const CUtensorMap& b2, const CUtensorMap& c2,
                           const GemmParams& p, int grid, cudaStream_t stream, bool pdl);

// Co-resident clusters (of cg * mc CTAs; single CTAs for cg * mc == 1) of
// variant `idx` on the current device.
cudaError_t variant_max_active(int idx, int* out);

// bwgemm_run_host: the row blocks of A and C of its copy/compute pipeline.
// Calls that move >= 16 MiB with M >= 1024 are split into blocks of whole
// 256-row tiles, 1024 rows from M = 2048 (512 below), at most
// kHostChunksMax of them, the last one halved so that the GEMM and the copy of
// C that nothing overlaps at the end are short.  host_row_blocks writes the
// first row of each block and M after the last into starts[] (room for
// kHostChunksMax + 1) and returns the number of blocks (1: no pipeline).
constexpr int kHostChunksMax = 12;
int host_row_blocks(int64_t M, int64_t N, int64_t K, int64_t* starts);
// ... and its columns of C (rows of B) per block when the rows are split:
// N in kHostColBlocksMax blocks of whole 256-column tiles once N >= 2048 and
// a block of C still holds 64 tiles of 256 x 256 (0: one block), so that the
// first GEMM waits for half of B instead of all of it and the copies of C
// start that much earlier.
constexpr int kHostColBlocksMax = 2;
int64_t host_block_cols(int64_t M, int64_t N, int64_t K);
// events of the pipeline: A blocks in, B blocks in, GEMMs done, start, end
constexpr int kHostEvents = kHostChunksMax + kHostColBlocksMax + kHostChunksMax * kHostColBlocksMax + 2;

// BWGEMM_OK when every operand a call reads or writes (A and B only when
// K > 0) is device or managed memory of `device`; BWGEMM_ERR_INVALID_ARG
// otherwise (host memory, memory of another GPU, an address the driver does
// not know).  Tensor maps, plain or multicast, are then only ever encoded on
// this GPU's own memory.
bwgemm_status_t check_operands_resident(const void* A, const void* B, const void* C, int64_t K, int device);

// The whole-K kernel for decode batches of at most 64 rows of A
// (skinny_kernel.cuh): 64 weight rows per CTA, the rows of A as the MMA's N
// (bn = 16, 32 or 64), no split of K.  skinny_cg(bn) CTAs per MMA: at bn =
// 64 a cluster of two (M = 128, cta_group::2), each CTA copying half of A's
// rows; one CTA (M = 64) below.  `skinny_stages(bn)` ring stages of
// `skinny_kblocks(bn)` K blocks in about 216 KiB of shared memory: four K
// blocks per stage (one 32 KiB copy of the weights) for one CTA; three for a
// pair, whose six stages of 36 KiB keep more weight bytes in flight than four
// of 48 KiB (measured 2 % faster at 64 rows).
constexpr int kSkinnyRows = 64;
constexpr int skinny_cg(int bn) { return bn == 64 ? 2 : 1; }
constexpr int skinny_kblocks(int bn) { return skinny_cg(bn) == 2 ? 3 : 4; }
constexpr int skinny_stages(int bn)
{
    return (216 * 1024) / (skinny_kblocks(bn) * (kSkinnyRows + bn / skinny_cg(bn)) * 128);
}
cudaError_t launch_skinny(int bn, const CUtensorMap& w, const CUtensorMap& x, const CUtensorMap& w3,
                          const CUtensorMap& x3, const CUtensorMap& c, const GemmParams& p, int grid,
                          cudaStream_t stream, bool pdl);

// The whole-K pair kernel for 129 to 256 rows of A (wholek_kernel.cuh): all
// rows of A on the MMA's M side (256 over a CTA pair), bn weight rows per
// pair (the MMA's N, a multiple of 16), no split of K.  Stages of
// wholek_kblocks() K blocks in about 224 KiB; the output staging reuses the
// ring.  The widths the library is built for, narrowest first:
constexpr int kWholeKWidths[] = {96, 112, 128, 144, 160, 192};
constexpr int wholek_kblocks(int /*bn*/) { return 2; }
constexpr int wholek_stages(int bn) { return (224 * 1024) / (wholek_kblocks(bn) * (128 + bn / 2) * 128); }
cudaError_t launch_wholek(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a3,
                          const CUtensorMap& b3, const CUtensorMap& c, const GemmParams& p, int grid,
                          cudaStream_t stream, bool pdl);

// Sizes of the split-K workspace regions.
constexpr uint64_t kCounterRegionBytes = 1ull << 20;  // per-(tile, cta, warp) arrival counters

struct Selection {
    bwgemm_config_t cfg;
    int variant_idx;  // into kVariants; -1 for the whole-K kernel of skinny_bn > 0
    int skinny_bn;    // > 0: the whole-K kernel for a few rows of A, MMA N = skinny_bn
    int wholek_bn;    // > 0: the whole-K pair kernel, wholek_bn weight rows per pair
    bool swap;  // the kernel sees the problem N x M (A and B exchanged)
    int num_m_blocks, num_n_blocks, num_k_blocks;
    int64_t sk_iters;
};

// The launch description of a selection (pointers, timeout and the test hook
// are left for the caller).
GemmParams make_params(const Selection& sel, int64_t M, int64_t N, int64_t K, bwgemm_dtype_t dtype);

// Host-only configuration choice (also behind bwgemm_select_config).
// max_pairs / max_quads: co-resident clusters of 2 and of 4 CTAs.
bwgemm_status_t select_config(int num_sms, int max_pairs, int max_quads, int64_t M, int64_t N, int64_t K,
                              const bwgemm_plan_options_t& opts, uint64_t workspace_bytes,
                              Selection* out);

}  // namespace bwgemm
