// api.cpp -- plans, tensor maps and launches behind the C ABI of bwgemm.h.
//
// TMA descriptors are built on the host (shape, strides, box, 128B swizzle,
// zero fill outside the tensor), the way both pages create them before the
// launch ("Writing a Blackwell GEMM by hand", TMA section: bounds and strides
// live in the descriptor; "Matrix Multiplication on NVIDIA's Blackwell",
// Kernel 2: host-side create_tma_tile).
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

using namespace bwgemm;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

struct TmapSlot {
    const void* ptr = nullptr;
    int64_t inner = 0, outer = 0, ld = 0;
    int64_t chunks = 0;  // 3-D K-chunk views: number of whole 64-element chunks (0: 2-D map)
    int dtype = -1;
    uint32_t box_inner = 0, box_outer = 0, box_depth = 0;
    int swizzle = -1;
    bool valid = false;
    CUtensorMap map;
};

// Build (or reuse) a 2-D tensor map of a row-major matrix: `outer` rows of
// `inner` elements, `ld` elements apart.
bwgemm_status_t get_tmap(TmapSlot& s, const void* ptr, int dtype, int64_t inner, int64_t outer,
                         int64_t ld, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz)
{
    if (s.valid && s.chunks == 0 && s.ptr == ptr && s.inner == inner && s.outer == outer && s.ld == ld &&
        s.dtype == dtype && s.box_inner == box_inner && s.box_outer == box_outer &&
        s.swizzle == int(swz))
        return BWGEMM_OK;
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return BWGEMM_ERR_NO_DEVICE;
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    const cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    s.valid = false;
    const CUresult r = enc(&s.map,
                           dtype == BWGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           2, const_cast<void*>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return BWGEMM_ERR_CUDA;
    s.ptr = ptr;
    s.inner = inner;
    s.outer = outer;
    s.ld = ld;
    s.chunks = 0;
    s.dtype = dtype;
    s.box_inner = box_inner;
    s.box_outer = box_outer;
    s.swizzle = int(swz);
    s.valid = true;
    return BWGEMM_OK;
}

// Build (or reuse) a 3-D view of a K-major operand for copies of several K
// blocks at once: dimension 0 = the 64 elements of one K chunk, 1 = rows (ld
// apart), 2 = whole K chunks (128 bytes apart).  A box {64, box_rows, depth}
// lands as `depth` consecutive 128-byte-swizzled [box_rows x 64] blocks (for
// the main kernel depth 2: two adjacent ring stages).  Only whole chunks are
// described, so no copy reads past K.
bwgemm_status_t get_tmap3(TmapSlot& s, const void* ptr, int dtype, int64_t chunks, int64_t rows,
                          int64_t ld, uint32_t box_rows, uint32_t depth = 2)
{
    if (s.valid && s.chunks == chunks && s.ptr == ptr && s.outer == rows && s.ld == ld &&
        s.dtype == dtype && s.box_outer == box_rows && s.box_depth == depth)
        return BWGEMM_OK;
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return BWGEMM_ERR_NO_DEVICE;
    const cuuint64_t dims[3] = {cuuint64_t(kTileK), cuuint64_t(rows), cuuint64_t(chunks)};
    const cuuint64_t strides[2] = {cuuint64_t(ld) * 2, cuuint64_t(kTileK) * 2};
    const cuuint32_t box[3] = {uint32_t(kTileK), box_rows, depth};
    const cuuint32_t estr[3] = {1, 1, 1};
    s.valid = false;
    const CUresult r = enc(&s.map,
                           dtype == BWGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           3, const_cast<void*>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return BWGEMM_ERR_CUDA;
    s.ptr = ptr;
    s.inner = kTileK;
    s.outer = rows;
    s.ld = ld;
    s.chunks = chunks;
    s.dtype = dtype;
    s.box_inner = kTileK;
    s.box_outer = box_rows;
    s.box_depth = depth;
    s.swizzle = int(CU_TENSOR_MAP_SWIZZLE_128B);
    s.valid = true;
    return BWGEMM_OK;
}

// Build (or reuse) the 3-D view of C for paired stores: dimension 0 = 32
// columns of one chunk, 1 = rows (ldc apart), 2 = whole 32-column chunks (64
// bytes apart).  A box {32, 32, 2} is two consecutive 64B-swizzled 32 x 32
// staging buffers.  Only whole chunks are described, so no store reaches past
// column 32 * chunks.
bwgemm_status_t get_tmap_cpairs(TmapSlot& s, void* C, int dtype, int64_t rows, int64_t chunks, int64_t ldc)
{
    if (s.valid && s.chunks == chunks && s.ptr == C && s.outer == rows && s.ld == ldc && s.dtype == dtype)
        return BWGEMM_OK;
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return BWGEMM_ERR_NO_DEVICE;
    const cuuint64_t dims[3] = {cuuint64_t(kStoreCols), cuuint64_t(rows), cuuint64_t(chunks)};
    const cuuint64_t strides[2] = {cuuint64_t(ldc) * 2, cuuint64_t(kStoreCols) * 2};
    const cuuint32_t box[3] = {uint32_t(kStoreCols), 32, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    s.valid = false;
    const CUresult r = enc(&s.map,
                           dtype == BWGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           3, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return BWGEMM_ERR_CUDA;
    s.ptr = C;
    s.inner = kStoreCols;
    s.outer = rows;
    s.ld = ldc;
    s.chunks = chunks;
    s.dtype = dtype;
    s.box_inner = kStoreCols;
    s.box_outer = 32;
    s.swizzle = int(CU_TENSOR_MAP_SWIZZLE_64B);
    s.valid = true;
    return BWGEMM_OK;
}

// Makes the plan's device current for the lifetime of the guard.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess)
            prev = -1;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard()
    {
        if (ok && prev >= 0)
            cudaSetDevice(prev);
    }
};

}  // namespace

namespace bwgemm {

bwgemm_status_t check_operands_resident(const void* A, const void* B, const void* C, int64_t K, int device)
{
    const void* ptrs[3] = {C, A, B};
    for (int i = 0; i < (K > 0 ? 3 : 1); ++i) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
            cudaGetLastError();  // an address the driver does not know: not this GPU's memory
            return BWGEMM_ERR_INVALID_ARG;
        }
        if ((a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) || a.device != device)
            return BWGEMM_ERR_INVALID_ARG;
    }
    return BWGEMM_OK;
}

}  // namespace bwgemm

struct bwgemm_plan_s {
    int device = 0;
    int num_sms = 0;
    int max_active[kNumVariants] = {};
    bwgemm_plan_options_t opts;
    uint32_t* d_status = nullptr;
    uint8_t* d_workspace = nullptr;
    uint64_t workspace_bytes = 0;
    TmapSlot tmaps[6];  // A, B, C, the 3-D two-K-block views of A and B, C for paired stores
    bwgemm_config_t last;
    uint64_t launches = 0;
    uint32_t last_status_bits = 0;
    // device staging buffers of bwgemm_run_host
    void* h2d[3] = {nullptr, nullptr, nullptr};
    size_t h2d_cap[3] = {0, 0, 0};
    // bwgemm_run_host's pipeline over row blocks: copy-in, GEMM and copy-out
    // streams and their events (created on first use)
    cudaStream_t side[3] = {nullptr, nullptr, nullptr};
    cudaEvent_t events[kHostEvents] = {};
    bool side_ready = false;
    // optional timeline (opts.trace): kTraceSlots stamps per CTA of the last launch
    uint64_t* d_trace = nullptr;
    int trace_ctas = 0;
    int last_grid = 0;
    // options chosen by bwgemm_tune, per shape; bwgemm_run uses them for that shape
    struct Tuned {
        int64_t M, N, K;
        int dtype;
        bwgemm_plan_options_t opts;
    };
    std::vector<Tuned> tuned;
};

namespace {

// The options bwgemm_run uses for a shape: the tuned ones if bwgemm_tune
// recorded some, else the plan's.
const bwgemm_plan_options_t& options_for(bwgemm_plan_t plan, int64_t M, int64_t N, int64_t K,
                                         bwgemm_dtype_t dtype)
{
    for (const auto& t : plan->tuned)
        if (t.M == M && t.N == N && t.K == K && t.dtype == int(dtype))
            return t.opts;
    return plan->opts;
}

// The whole-K kernel for a few rows of A: the weights (B, N x K) are the MMA's
// A operand in 64-row boxes, A's rows its B operand in boxes of skinny_bn /
// skinny_cg rows (zero-filled past M: each CTA of a pair copies its half);
// 3-D views copy skinny_kblocks(bn) whole K chunks at once.  C is stored in
// boxes of bn / cg rows x 16 cg columns (clipped at M and N).
bwgemm_status_t enqueue_skinny(bwgemm_plan_t plan, const bwgemm_plan_options_t& opts, const Selection& sel,
                               const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc, bwgemm_dtype_t dtype, cudaStream_t stream)
{
    bwgemm_status_t st;
    const uint32_t bn = uint32_t(sel.skinny_bn);
    const uint32_t cg = uint32_t(skinny_cg(int(bn)));
    const uint32_t x_rows = bn / cg;
    if ((st = get_tmap(plan->tmaps[0], B, dtype, K, N, ldb, kTileK, uint32_t(kSkinnyRows),
                       CU_TENSOR_MAP_SWIZZLE_128B)) != BWGEMM_OK ||
        (st = get_tmap(plan->tmaps[1], A, dtype, K, M, lda, kTileK, x_rows, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            BWGEMM_OK)
        return st;
    if ((st = get_tmap(plan->tmaps[2], C, dtype, N, M, ldc, 16 * cg, x_rows, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
        BWGEMM_OK)
        return st;
    GemmParams p = make_params(sel, M, N, K, dtype);
    const int64_t chunks = K / kTileK;
    const int kps = skinny_kblocks(int(bn));
    const bool views = chunks >= kps;
    const uint32_t depth = uint32_t(kps);
    if (views &&
        ((st = get_tmap3(plan->tmaps[3], B, dtype, chunks, N, ldb, uint32_t(kSkinnyRows), depth)) != BWGEMM_OK ||
         (st = get_tmap3(plan->tmaps[4], A, dtype, chunks, M, lda, x_rows, depth)) != BWGEMM_OK))
        return st;
    p.k_chunks_a = views ? int32_t(chunks) : 0;
    p.k_chunks_b = views ? int32_t(chunks) : 0;
    p.timeout_ns = opts.timeout_ns ? opts.timeout_ns : 4000000000ull;
    p.status = plan->d_status;
    p.c = static_cast<uint16_t*>(C);
    p.ldc = ldc;
    p.stall_kblock = opts.stall_kblock;
    if (plan->d_trace) {
        if (sel.cfg.grid > plan->trace_ctas)
            return BWGEMM_ERR_UNSUPPORTED;
        p.trace = plan->d_trace;
    }
    const CUtensorMap& w3 = views ? plan->tmaps[3].map : plan->tmaps[0].map;
    const CUtensorMap& x3 = views ? plan->tmaps[4].map : plan->tmaps[1].map;
    if (launch_skinny(int(bn), plan->tmaps[0].map, plan->tmaps[1].map, w3, x3, plan->tmaps[2].map, p,
                      sel.cfg.grid, stream, opts.pdl_off == 0) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    plan->last = sel.cfg;
    plan->last_grid = sel.cfg.grid;
    plan->launches += 1;
    return BWGEMM_OK;
}

// The whole-K pair kernel for 129 to 256 rows of A: A in boxes of 128 rows
// (each CTA of a pair its half, zero-filled past M), B in boxes of
// wholek_bn / 2 weight rows, 3-D views of wholek_kblocks() K chunks, C in
// boxes of 32 rows x wholek_bn columns (clipped at M and N).
bwgemm_status_t enqueue_wholek(bwgemm_plan_t plan, const bwgemm_plan_options_t& opts, const Selection& sel,
                               const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc, bwgemm_dtype_t dtype, cudaStream_t stream)
{
    bwgemm_status_t st;
    const uint32_t bn = uint32_t(sel.wholek_bn);
    if ((st = get_tmap(plan->tmaps[0], A, dtype, K, M, lda, kTileK, 128u, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            BWGEMM_OK ||
        (st = get_tmap(plan->tmaps[1], B, dtype, K, N, ldb, kTileK, bn / 2, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            BWGEMM_OK ||
        (st = get_tmap(plan->tmaps[2], C, dtype, N, M, ldc, bn, 32u, CU_TENSOR_MAP_SWIZZLE_NONE)) != BWGEMM_OK)
        return st;
    GemmParams p = make_params(sel, M, N, K, dtype);
    const int64_t chunks = K / kTileK;
    const int kps = wholek_kblocks(int(bn));
    const bool views = kps > 1 && chunks >= kps;
    if (views && ((st = get_tmap3(plan->tmaps[3], A, dtype, chunks, M, lda, 128u, uint32_t(kps))) != BWGEMM_OK ||
                  (st = get_tmap3(plan->tmaps[4], B, dtype, chunks, N, ldb, bn / 2, uint32_t(kps))) != BWGEMM_OK))
        return st;
    p.k_chunks_a = views ? int32_t(chunks) : 0;
    p.k_chunks_b = views ? int32_t(chunks) : 0;
    p.timeout_ns = opts.timeout_ns ? opts.timeout_ns : 4000000000ull;
    p.status = plan->d_status;
    p.c = static_cast<uint16_t*>(C);
    p.ldc = ldc;
    p.stall_kblock = opts.stall_kblock;
    if (plan->d_trace) {
        if (sel.cfg.grid > plan->trace_ctas)
            return BWGEMM_ERR_UNSUPPORTED;
        p.trace = plan->d_trace;
    }
    const CUtensorMap& a3 = views ? plan->tmaps[3].map : plan->tmaps[0].map;
    const CUtensorMap& b3 = views ? plan->tmaps[4].map : plan->tmaps[1].map;
    if (launch_wholek(int(bn), plan->tmaps[0].map, plan->tmaps[1].map, a3, b3, plan->tmaps[2].map, p,
                      sel.cfg.grid, stream, opts.pdl_off == 0) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    plan->last = sel.cfg;
    plan->last_grid = sel.cfg.grid;
    plan->launches += 1;
    return BWGEMM_OK;
}

bwgemm_status_t enqueue(bwgemm_plan_t plan, const bwgemm_plan_options_t& opts, const void* A,
                        const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                        int64_t ldb, int64_t ldc, bwgemm_dtype_t dtype, cudaStream_t stream)
{
    bwgemm_status_t st = bwgemm_check_args(A, B, C, M, N, K, lda, ldb, ldc, dtype);
    if (st != BWGEMM_OK)
        return st;
    if (M == 0 || N == 0)
        return BWGEMM_OK;
    // operands on another GPU or in host memory are refused before any tensor
    // map is encoded on them
    if ((st = check_operands_resident(A, B, C, K, plan->device)) != BWGEMM_OK)
        return st;
    if (K == 0) {  // empty sum: C = 0
        if (cudaMemset2DAsync(C, size_t(ldc) * 2, 0, size_t(N) * 2, size_t(M), stream) != cudaSuccess)
            return BWGEMM_ERR_CUDA;
        return BWGEMM_OK;
    }
    Selection sel;
    st = select_config(plan->num_sms, plan->max_active[find_variant(2, 256, false, 1)],
                       plan->max_active[find_variant(2, 256, false, 2)], M, N, K, opts,
                       plan->workspace_bytes, &sel);
    if (st != BWGEMM_OK)
        return st;
    if (sel.skinny_bn > 0)
        return enqueue_skinny(plan, opts, sel, A, B, C, M, N, K, lda, ldb, ldc, dtype, stream);
    if (sel.wholek_bn > 0)
        return enqueue_wholek(plan, opts, sel, A, B, C, M, N, K, lda, ldb, ldc, dtype, stream);
    const Variant& v = kVariants[sel.variant_idx];
    const uint32_t b_rows = uint32_t(v.cg == 1 ? v.bn : v.bn / 2);
    // the MMA's A operand (128-row side) and B operand; exchanged when swapped
    const void* opA = sel.swap ? B : A;
    const void* opB = sel.swap ? A : B;
    const int64_t rowsA = sel.swap ? N : M, rowsB = sel.swap ? M : N;
    const int64_t ldA = sel.swap ? ldb : lda, ldB = sel.swap ? lda : ldb;
    // with A multicast each CTA loads 128 / mc of its rows for all mc pairs
    if ((st = get_tmap(plan->tmaps[0], opA, dtype, K, rowsA, ldA, kTileK, uint32_t(kRowsPerCta / v.mc),
                       CU_TENSOR_MAP_SWIZZLE_128B)) != BWGEMM_OK)
        return st;
    if ((st = get_tmap(plan->tmaps[1], opB, dtype, K, rowsB, ldB, kTileK, b_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != BWGEMM_OK)
        return st;
    if ((st = get_tmap(plan->tmaps[2], C, dtype, N, M, ldc, kStoreCols, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B)) != BWGEMM_OK)
        return st;

    GemmParams p = make_params(sel, M, N, K, dtype);
    // 3-D views (two K blocks per copy or prefetch) need at least two whole K
    // chunks; with A multicast each CTA copies part of a stage of A, which a
    // 3-D view of whole stages does not describe
    const int64_t chunks = K / kTileK;
    const bool pair_copies = sel.cfg.copy_kblocks == 2 && chunks >= 2;
    const bool view_a = chunks >= 2 && v.mc == 1 && (pair_copies || (p.prefetch > 0 && !p.prefetch_b));
    const bool view_b = chunks >= 2 && (pair_copies || (p.prefetch > 0 && p.prefetch_b));
    if (view_a &&
        (st = get_tmap3(plan->tmaps[3], opA, dtype, chunks, rowsA, ldA, uint32_t(kRowsPerCta))) != BWGEMM_OK)
        return st;
    if (view_b && (st = get_tmap3(plan->tmaps[4], opB, dtype, chunks, rowsB, ldB, b_rows)) != BWGEMM_OK)
        return st;
    p.k_chunks_a = view_a ? int32_t(chunks) : 0;
    p.k_chunks_b = view_b ? int32_t(chunks) : 0;
    p.pair_copies = pair_copies ? 1 : 0;
    p.timeout_ns = opts.timeout_ns ? opts.timeout_ns : 4000000000ull;
    p.status = plan->d_status;
    p.c = static_cast<uint16_t*>(C);
    p.ldc = ldc;
    p.tile_sems = reinterpret_cast<uint32_t*>(plan->d_workspace);
    p.partials = reinterpret_cast<float*>(plan->d_workspace + kCounterRegionBytes);
    p.stall_kblock = opts.stall_kblock;
    if (plan->d_trace) {
        if (sel.cfg.grid > plan->trace_ctas)
            return BWGEMM_ERR_UNSUPPORTED;
        p.trace = plan->d_trace;  // each CTA clears its own row at entry
    }

    // C for stores of two 32-column chunks: a 3-D view of whole chunks with
    // the operands in order, a 64-row box of the 2-D layout when swapped
    // (the accumulator's columns are then rows of C)
    const int64_t c_chunks = N / kStoreCols;
    bool c_pairs = false;
    if (sel.swap) {
        if ((st = get_tmap(plan->tmaps[5], C, dtype, N, M, ldc, kStoreCols, 64, CU_TENSOR_MAP_SWIZZLE_64B)) !=
            BWGEMM_OK)
            return st;
        c_pairs = true;
    } else if (c_chunks >= 2) {
        if ((st = get_tmap_cpairs(plan->tmaps[5], C, dtype, M, c_chunks, ldc)) != BWGEMM_OK)
            return st;
        c_pairs = true;
    }
    p.c_pairs = c_pairs ? 1 : 0;
    p.c_chunks = int32_t(c_chunks);
    const CUtensorMap& c2 = c_pairs ? plan->tmaps[5].map : plan->tmaps[2].map;
    const CUtensorMap& a2 = view_a ? plan->tmaps[3].map : plan->tmaps[0].map;
    const CUtensorMap& b2 = view_b ? plan->tmaps[4].map : plan->tmaps[1].map;
    const cudaError_t err = launch_variant(sel.variant_idx, plan->tmaps[0].map, plan->tmaps[1].map,
                                           plan->tmaps[2].map, a2, b2, c2, p, sel.cfg.grid, stream,
                                           opts.pdl_off == 0);
    if (err != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    plan->last = sel.cfg;
    plan->last_grid = sel.cfg.grid;
    plan->launches += 1;
    return BWGEMM_OK;
}

bwgemm_status_t grow(void*& buf, size_t& cap, size_t need)
{
    if (cap >= need)
        return BWGEMM_OK;
    if (buf) {
        cudaFree(buf);
        buf = nullptr;
        cap = 0;
    }
    if (cudaMalloc(&buf, need) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    cap = need;
    return BWGEMM_OK;
}

}  // namespace

extern "C" {

bwgemm_status_t bwgemm_create_plan(bwgemm_plan_t* out, int device,
                                   const bwgemm_plan_options_t* opts)
{
    if (!out)
        return BWGEMM_ERR_INVALID_ARG;
    *out = nullptr;
    bwgemm_plan_options_t o;
    if (opts)
        o = *opts;
    else
        bwgemm_default_options(&o);
    for (int32_t r : o.reserved)
        if (r != 0)
            return BWGEMM_ERR_INVALID_ARG;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
        cudaGetLastError();
        return BWGEMM_ERR_NO_DEVICE;
    }
    if (device < 0 || device >= count)
        return BWGEMM_ERR_INVALID_ARG;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    if (major != 10 || minor != 3)
        return BWGEMM_ERR_UNSUPPORTED;  // sm_103 only: no other code path exists
    if (!encode_fn())
        return BWGEMM_ERR_NO_DEVICE;

    DeviceGuard guard(device);
    if (!guard.ok)
        return BWGEMM_ERR_CUDA;
    bwgemm_plan_s* plan = new (std::nothrow) bwgemm_plan_s();
    if (!plan)
        return BWGEMM_ERR_CUDA;
    plan->device = device;
    plan->num_sms = sms;
    plan->opts = o;
    plan->workspace_bytes = o.workspace_bytes ? o.workspace_bytes : (64ull << 20);
    std::memset(&plan->last, 0, sizeof(plan->last));
    for (int i = 0; i < kNumVariants; ++i) {
        if (variant_max_active(i, &plan->max_active[i]) != cudaSuccess || plan->max_active[i] <= 0) {
            cudaGetLastError();
            delete plan;
            return BWGEMM_ERR_UNSUPPORTED;  // kernel image does not load or does not fit
        }
    }
    if (cudaMalloc(&plan->d_status, 256) != cudaSuccess ||
        cudaMalloc(&plan->d_workspace, plan->workspace_bytes) != cudaSuccess ||
        cudaMemset(plan->d_status, 0, 256) != cudaSuccess ||
        cudaMemset(plan->d_workspace, 0, kCounterRegionBytes) != cudaSuccess) {
        cudaFree(plan->d_status);
        cudaFree(plan->d_workspace);
        delete plan;
        return BWGEMM_ERR_CUDA;
    }
    if (o.trace) {
        plan->trace_ctas = sms;
        if (cudaMalloc(&plan->d_trace, size_t(sms) * kTraceSlots * sizeof(uint64_t)) != cudaSuccess) {
            cudaFree(plan->d_status);
            cudaFree(plan->d_workspace);
            delete plan;
            return BWGEMM_ERR_CUDA;
        }
    }
    *out = plan;
    return BWGEMM_OK;
}

bwgemm_status_t bwgemm_destroy(bwgemm_plan_t plan)
{
    if (!plan)
        return BWGEMM_OK;
    DeviceGuard guard(plan->device);
    cudaDeviceSynchronize();
    cudaFree(plan->d_status);
    cudaFree(plan->d_workspace);
    if (plan->d_trace)
        cudaFree(plan->d_trace);
    for (cudaStream_t x : plan->side)
        if (x)
            cudaStreamDestroy(x);
    for (cudaEvent_t e : plan->events)
        if (e)
            cudaEventDestroy(e);
    for (void* b : plan->h2d)
        if (b)
            cudaFree(b);
    delete plan;
    return BWGEMM_OK;
}

bwgemm_status_t bwgemm_run(bwgemm_plan_t plan, const void* A, const void* B, void* C, int64_t M,
                           int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                           bwgemm_dtype_t dtype, void* stream)
{
    if (!plan)
        return BWGEMM_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok)
        return BWGEMM_ERR_CUDA;
    return enqueue(plan, options_for(plan, M, N, K, dtype), A, B, C, M, N, K, lda, ldb, ldc, dtype,
                   static_cast<cudaStream_t>(stream));
}

bwgemm_status_t bwgemm_get_status(bwgemm_plan_t plan, void* stream)
{
    if (!plan)
        return BWGEMM_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok)
        return BWGEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    uint32_t bits = 0;
    if (cudaMemcpy(&bits, plan->d_status, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    plan->last_status_bits = bits;
    if (bits == 0)
        return BWGEMM_OK;
    // clear the word and re-arm the split-K arrival counters an aborted launch may have left
    if (cudaMemset(plan->d_status, 0, sizeof(bits)) != cudaSuccess ||
        cudaMemset(plan->d_workspace, 0, kCounterRegionBytes) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    return BWGEMM_ERR_TIMEOUT;
}

uint32_t bwgemm_last_device_status(bwgemm_plan_t plan) { return plan ? plan->last_status_bits : 0u; }

bwgemm_status_t bwgemm_run_host(bwgemm_plan_t plan, const void* A_host, const void* B_host,
                                void* C_host, int64_t M, int64_t N, int64_t K, int64_t lda,
                                int64_t ldb, int64_t ldc, bwgemm_dtype_t dtype, void* stream)
{
    if (!plan)
        return BWGEMM_ERR_INVALID_ARG;
    // host operands need no alignment; the device copies are packed with
    // leading dimensions rounded up to 8 elements
    if (dtype != BWGEMM_BF16 && dtype != BWGEMM_FP16)
        return BWGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || ldc < N)
        return BWGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return BWGEMM_OK;
    if (!C_host || (K > 0 && (!A_host || !B_host)))
        return BWGEMM_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok)
        return BWGEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t dlda = std::max<int64_t>((K + 7) / 8 * 8, 8);
    const int64_t dldc = (N + 7) / 8 * 8;
    bwgemm_status_t st;
    if ((st = grow(plan->h2d[0], plan->h2d_cap[0], size_t(M) * dlda * 2)) != BWGEMM_OK ||
        (st = grow(plan->h2d[1], plan->h2d_cap[1], size_t(N) * dlda * 2)) != BWGEMM_OK ||
        (st = grow(plan->h2d[2], plan->h2d_cap[2], size_t(M) * dldc * 2)) != BWGEMM_OK)
        return st;
    // one linear copy when the host rows are already packed like the device copy
    auto copy_rows = [&](void* dst, int64_t dld, const void* src, int64_t sld, int64_t cols,
                         int64_t rows, cudaMemcpyKind kind, cudaStream_t cs) {
        if (sld == dld && dld == cols)
            return cudaMemcpyAsync(dst, src, size_t(rows) * size_t(cols) * 2, kind, cs);
        return cudaMemcpy2DAsync(dst, size_t(dld) * 2, src, size_t(sld) * 2, size_t(cols) * 2,
                                 size_t(rows), kind, cs);
    };
    const bwgemm_plan_options_t& opts = options_for(plan, M, N, K, dtype);
    int64_t starts[kHostChunksMax + 1];
    const int chunks = host_row_blocks(M, N, K, starts);
    if (chunks > 1) {
        // Pipeline over blocks of C: row block i of A and column block j of B
        // (rows of B) come over on the copy-in stream in the order B0, A0, B1,
        // ..., A1, A2, ...; GEMM (i, j) runs on the compute stream once both
        // have landed, and row block i of C goes back on the copy-out stream
        // after its last GEMM, so that the GEMMs and the copies of C overlap
        // the copies still coming in (the link to host memory, not the GPU,
        // bounds a call of this size).  The GEMMs run one after another on one
        // stream: they share the plan's workspace.
        const int64_t cols = host_block_cols(M, N, K);
        const int cblocks = cols > 0 ? int((N + cols - 1) / cols) : 1;
        const int64_t cw = cols > 0 ? cols : N;
        if (!plan->side_ready) {
            for (cudaStream_t& x : plan->side)
                if (cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking) != cudaSuccess)
                    return BWGEMM_ERR_CUDA;
            for (cudaEvent_t& e : plan->events)
                if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                    return BWGEMM_ERR_CUDA;
            plan->side_ready = true;
        }
        cudaStream_t s_in = plan->side[0], s_mm = plan->side[1], s_out = plan->side[2];
        cudaEvent_t* ev_a = plan->events;                              // [kHostChunksMax]
        cudaEvent_t* ev_b = ev_a + kHostChunksMax;                     // [kHostColBlocksMax]
        cudaEvent_t* ev_mm = ev_b + kHostColBlocksMax;                 // [kHostChunksMax][kHostColBlocksMax]
        cudaEvent_t ev_start = ev_mm[kHostChunksMax * kHostColBlocksMax];
        cudaEvent_t ev_end = ev_mm[kHostChunksMax * kHostColBlocksMax + 1];
        uint8_t* dA = static_cast<uint8_t*>(plan->h2d[0]);
        uint8_t* dB = static_cast<uint8_t*>(plan->h2d[1]);
        uint8_t* dC = static_cast<uint8_t*>(plan->h2d[2]);
        auto copy_a = [&](int i) {
            const int64_t r0 = starts[i], r = starts[i + 1] - starts[i];
            const uint8_t* hA = static_cast<const uint8_t*>(A_host) + size_t(r0) * size_t(lda) * 2;
            if (copy_rows(dA + size_t(r0) * dlda * 2, dlda, hA, lda, K, r, cudaMemcpyHostToDevice, s_in) !=
                    cudaSuccess ||
                cudaEventRecord(ev_a[i], s_in) != cudaSuccess)
                return false;
            return true;
        };
        auto copy_b = [&](int j) {
            const int64_t c0 = j * cw, c = std::min<int64_t>(cw, N - c0);
            const uint8_t* hB = static_cast<const uint8_t*>(B_host) + size_t(c0) * size_t(ldb) * 2;
            if (copy_rows(dB + size_t(c0) * dlda * 2, dlda, hB, ldb, K, c, cudaMemcpyHostToDevice, s_in) !=
                    cudaSuccess ||
                cudaEventRecord(ev_b[j], s_in) != cudaSuccess)
                return false;
            return true;
        };
        if (cudaEventRecord(ev_start, s) != cudaSuccess || cudaStreamWaitEvent(s_in, ev_start, 0) != cudaSuccess ||
            cudaStreamWaitEvent(s_mm, ev_start, 0) != cudaSuccess ||
            cudaStreamWaitEvent(s_out, ev_start, 0) != cudaSuccess)
            return BWGEMM_ERR_CUDA;
        // copy-in order: B0, A0, the other B blocks, then A1, A2, ...
        if (!copy_b(0) || !copy_a(0))
            return BWGEMM_ERR_CUDA;
        for (int j = 1; j < cblocks; ++j)
            if (!copy_b(j))
                return BWGEMM_ERR_CUDA;
        for (int i = 1; i < chunks; ++i)
            if (!copy_a(i))
                return BWGEMM_ERR_CUDA;
        for (int i = 0; i < chunks; ++i) {
            const int64_t r0 = starts[i], r = starts[i + 1] - starts[i];
            if (cudaStreamWaitEvent(s_mm, ev_a[i], 0) != cudaSuccess)
                return BWGEMM_ERR_CUDA;
            for (int j = 0; j < cblocks; ++j) {
                const int64_t c0 = j * cw, c = std::min<int64_t>(cw, N - c0);
                if (cudaStreamWaitEvent(s_mm, ev_b[j], 0) != cudaSuccess)
                    return BWGEMM_ERR_CUDA;
                if ((st = enqueue(plan, opts, dA + size_t(r0) * dlda * 2, dB + size_t(c0) * dlda * 2,
                                  dC + (size_t(r0) * dldc + size_t(c0)) * 2, r, c, K, dlda, dlda, dldc, dtype,
                                  s_mm)) != BWGEMM_OK)
                    return st;
            }
            // the row block of C goes back whole (whole rows: one linear copy
            // when the host rows are packed)
            cudaEvent_t done = ev_mm[i * kHostColBlocksMax];
            uint8_t* hC = static_cast<uint8_t*>(C_host) + size_t(r0) * size_t(ldc) * 2;
            if (cudaEventRecord(done, s_mm) != cudaSuccess || cudaStreamWaitEvent(s_out, done, 0) != cudaSuccess ||
                copy_rows(hC, ldc, dC + size_t(r0) * dldc * 2, dldc, N, r, cudaMemcpyDeviceToHost, s_out) !=
                    cudaSuccess)
                return BWGEMM_ERR_CUDA;
        }
        if (cudaEventRecord(ev_end, s_out) != cudaSuccess || cudaStreamWaitEvent(s, ev_end, 0) != cudaSuccess)
            return BWGEMM_ERR_CUDA;
        return bwgemm_get_status(plan, stream);
    }
    if (K > 0) {
        if (copy_rows(plan->h2d[0], dlda, A_host, lda, K, M, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            copy_rows(plan->h2d[1], dlda, B_host, ldb, K, N, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return BWGEMM_ERR_CUDA;
    }
    st = enqueue(plan, opts, plan->h2d[0], plan->h2d[1], plan->h2d[2], M, N, K, dlda, dlda, dldc, dtype, s);
    if (st != BWGEMM_OK)
        return st;
    if (copy_rows(C_host, ldc, plan->h2d[2], dldc, N, M, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return BWGEMM_ERR_CUDA;
    return bwgemm_get_status(plan, stream);
}

bwgemm_status_t bwgemm_plan_last_config(bwgemm_plan_t plan, bwgemm_config_t* out)
{
    if (!plan || !out)
        return BWGEMM_ERR_INVALID_ARG;
    *out = plan->last;
    return BWGEMM_OK;
}

bwgemm_status_t bwgemm_tune(bwgemm_plan_t plan, const void* A, const void* B, void* C, int64_t M,
                            int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                            bwgemm_dtype_t dtype, void* stream, int32_t iters, bwgemm_config_t* best)
{
    if (!plan || iters <= 0 || iters > 10000)
        return BWGEMM_ERR_INVALID_ARG;
    bwgemm_status_t st = bwgemm_check_args(A, B, C, M, N, K, lda, ldb, ldc, dtype);
    if (st != BWGEMM_OK)
        return st;
    DeviceGuard guard(plan->device);
    if (!guard.ok)
        return BWGEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // Candidates: the plan's options with one to three choices overridden
    // (-1 = keep).  Each is planned on the host first; ones that fail to plan
    // or plan to a configuration already seen are skipped.
    struct Override {
        int32_t variant, tile_n, split_k, schedule, copy_kblocks, cluster_split, raster_group, swap_ab,
            multicast;
    };
    constexpr int32_t X = -1;
    const Override kCandidates[] = {
        {X, X, X, X, X, X, X, X, X},  // the plan's own choice
        // schedule and split
        {X, X, 1, BWGEMM_SCHEDULE_TILES, X, X, X, X, X},
        {X, X, X, BWGEMM_SCHEDULE_STREAM_K, X, X, X, X, X},
        {X, X, 2, BWGEMM_SCHEDULE_TILES, X, X, X, X, X},
        {X, X, 3, BWGEMM_SCHEDULE_TILES, X, X, X, X, X},
        {X, X, 4, BWGEMM_SCHEDULE_TILES, X, X, X, X, X},
        {X, X, X, BWGEMM_SCHEDULE_CLC, X, X, X, X, X},
        {X, X, X, X, X, 1, X, X, X},  // split-K through L2 instead of in a cluster
        // copies per K block
        {X, X, X, X, 1, X, X, X, X},
        {X, X, X, X, 2, X, X, X, X},
        // tile shape: one CTA, narrower or wider pair tiles (the planner's own
        // widths 224 / 320 / 384 and the plain 256 in either direction)
        {X, 128, X, X, X, X, X, X, X},
        {BWGEMM_VARIANT_1SM, X, X, X, X, X, X, X, X},
        {BWGEMM_VARIANT_1SM, 128, X, X, X, X, X, X, X},
        {BWGEMM_VARIANT_2SM, 224, X, X, X, X, X, 1, X},
        {BWGEMM_VARIANT_2SM, 224, 2, BWGEMM_SCHEDULE_TILES, X, X, X, 1, X},
        {BWGEMM_VARIANT_2SM, 256, X, X, X, X, X, 1, X},
        {BWGEMM_VARIANT_2SM, 320, X, X, X, X, X, 1, X},
        {BWGEMM_VARIANT_2SM, 384, X, X, X, X, X, 1, X},
        // A multicast across two CTA pairs
        {BWGEMM_VARIANT_2SM, 256, X, X, X, X, X, 1, 2},
        {BWGEMM_VARIANT_2SM, 128, X, X, X, X, X, 1, 2},
        // raster group and operand order
        {X, X, X, X, X, X, 2, X, X},
        {X, X, X, X, X, X, 4, X, X},
        {X, X, X, X, X, X, 16, X, X},
        {X, X, X, X, X, X, X, 1, X},
        {X, X, X, X, X, X, X, 2, X},
    };
    const int pairs = plan->max_active[find_variant(2, 256, false, 1)];
    const int quads = plan->max_active[find_variant(2, 256, false, 2)];
    std::vector<bwgemm_plan_options_t> cands;
    std::vector<bwgemm_config_t> cfgs;
    for (const Override& o : kCandidates) {
        bwgemm_plan_options_t opts = plan->opts;
        opts.trace = 0;
        opts.stall_kblock = -1;
        opts.tuned_table = 1;  // the candidates are the rules' choices and their variations
        if (o.variant >= 0) opts.variant = o.variant;
        if (o.tile_n >= 0) opts.tile_n = o.tile_n;
        if (o.split_k >= 0) opts.split_k = o.split_k;
        if (o.schedule >= 0) opts.schedule = o.schedule;
        if (o.copy_kblocks >= 0) opts.copy_kblocks = o.copy_kblocks;
        if (o.cluster_split >= 0) opts.cluster_split = o.cluster_split;
        if (o.raster_group >= 0) opts.raster_group = o.raster_group;
        if (o.swap_ab >= 0) opts.swap_ab = o.swap_ab;
        if (o.multicast >= 0) opts.multicast = o.multicast;
        Selection sel;
        if (select_config(plan->num_sms, pairs, quads, M, N, K, opts, plan->workspace_bytes, &sel) != BWGEMM_OK)
            continue;
        bool seen = false;
        for (const auto& c : cfgs)
            seen = seen || std::memcmp(&c, &sel.cfg, sizeof(c)) == 0;
        if (seen)
            continue;
        cands.push_back(opts);
        cfgs.push_back(sel.cfg);
    }
    if (cands.empty())
        return BWGEMM_ERR_UNSUPPORTED;

    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0)
            cudaEventDestroy(e0);
        return BWGEMM_ERR_CUDA;
    }
    int best_i = -1;
    float best_ms = 0.f;
    for (size_t i = 0; i < cands.size(); ++i) {
        bool ok = true;
        for (int w = 0; w < 2 && ok; ++w)
            ok = enqueue(plan, cands[i], A, B, C, M, N, K, lda, ldb, ldc, dtype, s) == BWGEMM_OK;
        ok = ok && cudaEventRecord(e0, s) == cudaSuccess;
        for (int w = 0; w < iters && ok; ++w)
            ok = enqueue(plan, cands[i], A, B, C, M, N, K, lda, ldb, ldc, dtype, s) == BWGEMM_OK;
        ok = ok && cudaEventRecord(e1, s) == cudaSuccess;
        // a candidate whose launches reported a device-side error is not kept
        ok = ok && bwgemm_get_status(plan, stream) == BWGEMM_OK;
        float ms = 0.f;
        if (ok && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess && (best_i < 0 || ms < best_ms)) {
            best_i = int(i);
            best_ms = ms;
        }
        cudaGetLastError();
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (best_i < 0)
        return BWGEMM_ERR_CUDA;

    bool replaced = false;
    for (auto& t : plan->tuned)
        if (t.M == M && t.N == N && t.K == K && t.dtype == int(dtype)) {
            t.opts = cands[best_i];
            replaced = true;
        }
    if (!replaced)
        plan->tuned.push_back({M, N, K, int(dtype), cands[best_i]});
    // leave C holding the chosen configuration's result
    if ((st = enqueue(plan, cands[best_i], A, B, C, M, N, K, lda, ldb, ldc, dtype, s)) != BWGEMM_OK)
        return st;
    if (best)
        *best = cfgs[best_i];
    return BWGEMM_OK;
}

int32_t bwgemm_plan_tuned_count(bwgemm_plan_t plan) { return plan ? int32_t(plan->tuned.size()) : 0; }

uint64_t bwgemm_plan_launch_count(bwgemm_plan_t plan) { return plan ? plan->launches : 0u; }

bwgemm_status_t bwgemm_plan_read_trace(bwgemm_plan_t plan, uint64_t* out, int64_t capacity,
                                       int32_t* ctas, int32_t* slots)
{
    if (!plan || !plan->d_trace || !out || !ctas || !slots)
        return BWGEMM_ERR_INVALID_ARG;
    const int64_t n = int64_t(plan->last_grid) * kTraceSlots;
    if (capacity < n)
        return BWGEMM_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(out, plan->d_trace, size_t(n) * sizeof(uint64_t), cudaMemcpyDeviceToHost) !=
            cudaSuccess)
        return BWGEMM_ERR_CUDA;
    *ctas = plan->last_grid;
    *slots = kTraceSlots;
    return BWGEMM_OK;
}

}  // extern "C"
