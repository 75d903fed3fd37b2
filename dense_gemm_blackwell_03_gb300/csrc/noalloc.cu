// noalloc.cu -- split-K GEMM entry point that performs no device allocation.
//
// Some callers cannot call cudaMalloc: code that runs under a memory manager
// which has already reserved the device's memory for itself (a framework's
// caching allocator holding most of HBM), code whose device footprint must
// stay fixed after start-up, and latency-critical loops that must not risk
// the device-wide synchronisation cudaMalloc / cudaFree can cause.  The plan
// API cannot serve them, because bwgemm_create_plan allocates the plan's
// status word and split-K workspace.  bwgemm_run_splitk_noalloc runs the
// same split-K kernel with its scratch (fp32 partial tiles, arrival counters
// and a status word) in a fixed, file-scope device array instead.
//
// The array costs kNoAllocScratchBytes of device memory on every GPU that
// loads this library, held until the process exits.  Every call shares it,
// so calls whose kernels overlap on the GPU (different streams, or different
// host threads) race on it and give undefined results; serialise them.
#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

using namespace bwgemm;

constexpr size_t kNoAllocPartialBytes = BWGEMM_NOALLOC_PARTIAL_BYTES;  // fp32 partial tiles
constexpr size_t kNoAllocCounterBytes = BWGEMM_NOALLOC_COUNTER_BYTES;  // per (tile, cta, warp) counters
constexpr size_t kNoAllocCounters = kNoAllocCounterBytes / sizeof(uint32_t);
constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocScratchBytes = kNoAllocPartialBytes + kNoAllocCounterBytes + kNoAllocStatusBytes;
static_assert(kNoAllocCounters * sizeof(uint32_t) == kNoAllocCounterBytes, "whole counters");
static_assert(kNoAllocPartialBytes % 256 == 0 && kNoAllocCounterBytes % 256 == 0,
              "the counter region and the status word stay 256-byte aligned");

// layout: [partials 8 MiB][counters 64 KiB][status word (+ pad)]
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
    int num_sms = 0;
    int max_pairs = 0;
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn noalloc_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int dtype, int64_t inner,
            int64_t outer, int64_t ld, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz)
{
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    const cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dtype == BWGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
               2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The plan of an allocation-free call and the scratch it uses: split-K over
// whole tiles with the operands in the order given, one CTA pair (or CTA) per
// cluster, slices reducing through the array.  Host only.  When the planner
// cuts the split to one slice (K of one 64-wide block) no partials or
// counters are used, and the counters of the call are not touched.
bwgemm_status_t noalloc_select(int num_sms, int max_pairs, int64_t M, int64_t N, int64_t K, int32_t split_k,
                               Selection* sel, size_t* partial_bytes, size_t* counters)
{
    if (split_k < 2 || split_k > 16)
        return BWGEMM_ERR_INVALID_ARG;
    bwgemm_plan_options_t opts;
    bwgemm_default_options(&opts);
    opts.split_k = split_k;
    opts.swap_ab = 1;        // operands in the order given
    opts.multicast = 1;      // one CTA pair per cluster: the scratch below is sized for it
    opts.cluster_split = 1;  // slices reduce through the scratch array, not in a cluster
    opts.skinny = 1;         // the split-K kernel, also for a few rows of A
    opts.wholek = 1;         // and for up to 256 rows
    // plan as if the workspace were unbounded, then hold the need against the array
    const bwgemm_status_t st = select_config(num_sms, max_pairs, 0, M, N, K, opts, ~uint64_t(0), sel);
    if (st != BWGEMM_OK)
        return st;
    const Variant& v = kVariants[sel->variant_idx];
    const bool split = sel->cfg.split_k > 1;
    const size_t tiles = size_t(sel->cfg.num_tiles);
    *partial_bytes = split ? tiles * size_t(sel->cfg.split_k) * size_t(v.cg) * kRowsPerCta * size_t(v.bn) * 4 : 0;
    *counters = split ? tiles * size_t(v.cg) * kEpiWarps * kCountersPerWarp : 0;
    if (*partial_bytes > kNoAllocPartialBytes || *counters > kNoAllocCounters)
        return BWGEMM_ERR_WORKSPACE;  // this shape's split-K scratch exceeds the fixed array
    return BWGEMM_OK;
}

// Once per device, with that device current: resolve the array's device
// address (a host-side use of the symbol name is only a stand-in) and the
// occupancy figures the planner needs.  Allocates nothing.
bwgemm_status_t setup_device(int dev, DeviceSetup** out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return BWGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BWGEMM_ERR_CUDA;
        if (major != 10 || minor != 3)
            return BWGEMM_ERR_UNSUPPORTED;
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) {
            cudaGetLastError();
            return BWGEMM_ERR_CUDA;
        }
        int pairs = 0;
        if (variant_max_active(find_variant(2, 256, false, 1), &pairs) != cudaSuccess || pairs <= 0) {
            cudaGetLastError();
            return BWGEMM_ERR_UNSUPPORTED;
        }
        s.scratch = static_cast<unsigned char*>(addr);
        s.num_sms = sms;
        s.max_pairs = pairs;
        s.ready = true;
    }
    *out = &s;
    return BWGEMM_OK;
}

}  // namespace

extern "C" bwgemm_status_t bwgemm_run_splitk_noalloc(const void* A, const void* B, void* C,
                                                     int64_t M, int64_t N, int64_t K, int64_t lda,
                                                     int64_t ldb, int64_t ldc, bwgemm_dtype_t dtype,
                                                     int32_t split_k, void* stream)
{
    bwgemm_status_t st = bwgemm_check_args(A, B, C, M, N, K, lda, ldb, ldc, dtype);
    if (st != BWGEMM_OK)
        return st;
    if (split_k < 2 || split_k > 16)
        return BWGEMM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0)
        return BWGEMM_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return BWGEMM_ERR_NO_DEVICE;
    // the operands must be memory of the current device (no tensor map is
    // encoded on another GPU's or on host memory)
    if ((st = check_operands_resident(A, B, C, K, dev)) != BWGEMM_OK)
        return st;
    if (K == 0)  // empty sum: C = 0
        return cudaMemset2DAsync(C, size_t(ldc) * 2, 0, size_t(N) * 2, size_t(M), s) == cudaSuccess
                   ? BWGEMM_OK
                   : BWGEMM_ERR_CUDA;

    DeviceSetup* ds = nullptr;
    if ((st = setup_device(dev, &ds)) != BWGEMM_OK)
        return st;
    EncodeTiledFn enc = noalloc_encode_fn();
    if (!enc)
        return BWGEMM_ERR_NO_DEVICE;

    Selection sel;
    size_t partial_bytes = 0, counters = 0;  // used regions of the array
    if ((st = noalloc_select(ds->num_sms, ds->max_pairs, M, N, K, split_k, &sel, &partial_bytes, &counters)) !=
        BWGEMM_OK)
        return st;
    const Variant& v = kVariants[sel.variant_idx];

    unsigned char* partials = ds->scratch;
    uint32_t* ctr = reinterpret_cast<uint32_t*>(ds->scratch + kNoAllocPartialBytes);
    uint32_t* status = reinterpret_cast<uint32_t*>(ds->scratch + kNoAllocPartialBytes + kNoAllocCounterBytes);
    // the array keeps the previous call's contents: the arrival counters this
    // call uses (none without a split) and the status word must start at zero
    if ((counters > 0 && cudaMemsetAsync(ctr, 0, counters * sizeof(uint32_t), s) != cudaSuccess) ||
        cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess)
        return BWGEMM_ERR_CUDA;

    CUtensorMap ta, tb, tc;
    const uint32_t b_rows = uint32_t(v.cg == 1 ? v.bn : v.bn / 2);
    if (!encode(enc, &ta, A, dtype, K, M, lda, kTileK, kRowsPerCta, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(enc, &tb, B, dtype, K, N, ldb, kTileK, b_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(enc, &tc, C, dtype, N, M, ldc, kStoreCols, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return BWGEMM_ERR_CUDA;

    GemmParams p = make_params(sel, M, N, K, dtype);
    p.timeout_ns = 4000000000ull;
    p.status = status;
    p.c = static_cast<uint16_t*>(C);
    p.ldc = ldc;
    p.tile_sems = ctr;
    p.partials = reinterpret_cast<float*>(partials);
    // one copy per K block and no prefetch: the 3-D operand views are not built here
    p.k_chunks_a = p.k_chunks_b = 0;
    p.pair_copies = 0;
    p.prefetch = 0;
    // one 32-column chunk per C store (p.c_pairs = 0): no second C view is built
    return launch_variant(sel.variant_idx, ta, tb, tc, ta, tb, tc, p, sel.cfg.grid, s, false) == cudaSuccess
               ? BWGEMM_OK
               : BWGEMM_ERR_CUDA;
}

extern "C" bwgemm_status_t bwgemm_noalloc_scratch(int32_t num_sms, int32_t max_pairs, int64_t M, int64_t N,
                                                  int64_t K, int32_t split_k, uint64_t* partial_bytes,
                                                  uint64_t* counter_bytes)
{
    if (!partial_bytes || !counter_bytes || num_sms <= 0 || M < 0 || N < 0 || K < 0)
        return BWGEMM_ERR_INVALID_ARG;
    *partial_bytes = 0;
    *counter_bytes = 0;
    if (split_k < 2 || split_k > 16)
        return BWGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0 || K == 0)
        return BWGEMM_OK;  // no kernel: nothing of the array is used
    Selection sel;
    size_t parts = 0, counters = 0;
    const bwgemm_status_t st = noalloc_select(num_sms, max_pairs, M, N, K, split_k, &sel, &parts, &counters);
    if (st == BWGEMM_OK || st == BWGEMM_ERR_WORKSPACE) {
        *partial_bytes = parts;
        *counter_bytes = counters * sizeof(uint32_t);
    }
    return st;
}
