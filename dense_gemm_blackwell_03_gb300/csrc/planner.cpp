// planner.cpp -- host-only argument checks and launch-configuration choice.
//
// Nothing here touches the device, so all of it is testable without a GPU
// through bwgemm_check_args / bwgemm_select_config.
#include <algorithm>
#include <cstring>

#include "internal.h"

namespace bwgemm {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bwgemm_status_t select_config(int num_sms, int max_pairs, int64_t M, int64_t N, int64_t K,
                              const bwgemm_plan_options_t& opts, uint64_t workspace_bytes,
                              Selection* out)
{
    if (!out || num_sms <= 0 || M < 0 || N < 0 || K < 0)
        return BWGEMM_ERR_INVALID_ARG;
    if (max_pairs <= 0)
        max_pairs = num_sms / 2;
    for (int32_t r : opts.reserved)
        if (r != 0)
            return BWGEMM_ERR_INVALID_ARG;

    // Variant: the CTA-pair form (256-row units, each CTA streaming half of the
    // B tile) whenever there are more than 128 rows; one CTA per unit otherwise.
    int cg;
    switch (opts.variant) {
    case BWGEMM_VARIANT_AUTO: cg = (M > 128) ? 2 : 1; break;
    case BWGEMM_VARIANT_1SM: cg = 1; break;
    case BWGEMM_VARIANT_2SM: cg = 2; break;
    default: return BWGEMM_ERR_INVALID_ARG;
    }
    int bn;
    switch (opts.tile_n) {
    case 0: bn = (N <= 128) ? 128 : 256; break;
    case 128:
    case 256: bn = opts.tile_n; break;
    default: return BWGEMM_ERR_INVALID_ARG;
    }
    const int idx = find_variant(cg, bn);
    if (idx < 0)
        return BWGEMM_ERR_UNSUPPORTED;
    if (opts.split_k < 0 || opts.raster_group < 0 || opts.max_ctas < 0)
        return BWGEMM_ERR_INVALID_ARG;

    const int tile_m = kRowsPerCta * cg;
    const int64_t num_m = ceil_div(M, tile_m);
    const int64_t num_n = ceil_div(N, bn);
    const int64_t num_kb = ceil_div(K, kTileK);
    const int64_t tiles = num_m * num_n;
    if (num_m > (1 << 30) || num_n > (1 << 30) || tiles > (int64_t(1) << 30))
        return BWGEMM_ERR_UNSUPPORTED;

    // Concurrent work units the persistent grid holds.
    int64_t slots = (cg == 2) ? max_pairs : num_sms;
    if (opts.max_ctas > 0)
        slots = std::max<int64_t>(1, std::min<int64_t>(slots, opts.max_ctas / cg));

    // Split-K: when the tiles alone leave most of the GPU idle (decode-sized
    // M), cut each tile's K range into s slices so that tiles * s fills the
    // grid; keep at least 4 K blocks of 64 per slice.
    int64_t s = 1;
    if (opts.split_k > 0) {
        s = std::min<int64_t>(opts.split_k, std::max<int64_t>(num_kb, 1));
    } else if (tiles > 0 && tiles < slots && num_kb >= 8) {
        s = std::min<int64_t>({slots / tiles, num_kb / 4, 8});
        s = std::max<int64_t>(s, 1);
    }
    int64_t ws = 0;
    if (s > 1) {
        const int64_t counters = tiles * cg * kEpiWarps * 4;
        ws = int64_t(kCounterRegionBytes) + tiles * s * cg * int64_t(kRowsPerCta) * bn * 4;
        if (counters > int64_t(kCounterRegionBytes) || uint64_t(ws) > workspace_bytes) {
            if (opts.split_k > 1)
                return BWGEMM_ERR_WORKSPACE;
            s = 1;
            ws = 0;
        }
    }
    const int64_t units = tiles * s;
    const int64_t clusters = std::min<int64_t>(units, slots);

    int64_t group = opts.raster_group > 0 ? opts.raster_group : 8;
    group = std::max<int64_t>(1, std::min<int64_t>(group, std::max<int64_t>(num_m, 1)));

    Selection sel;
    std::memset(&sel, 0, sizeof(sel));
    sel.variant_idx = idx;
    sel.num_m_blocks = int(num_m);
    sel.num_n_blocks = int(num_n);
    sel.num_k_blocks = int(num_kb);
    sel.cfg.variant = (cg == 2) ? BWGEMM_VARIANT_2SM : BWGEMM_VARIANT_1SM;
    sel.cfg.tile_m = tile_m;
    sel.cfg.tile_n = bn;
    sel.cfg.tile_k = kTileK;
    sel.cfg.stages = kVariants[idx].stages;
    sel.cfg.split_k = int32_t(s);
    sel.cfg.raster_group = int32_t(group);
    sel.cfg.num_tiles = int32_t(tiles);
    sel.cfg.num_units = int32_t(units);
    sel.cfg.grid = int32_t(clusters * cg);
    sel.cfg.workspace_bytes = ws;
    *out = sel;
    return BWGEMM_OK;
}

}  // namespace bwgemm

using namespace bwgemm;

extern "C" {

void bwgemm_default_options(bwgemm_plan_options_t* opts)
{
    if (!opts)
        return;
    std::memset(opts, 0, sizeof(*opts));
    opts->stall_kblock = -1;
}

bwgemm_status_t bwgemm_check_args(const void* A, const void* B, const void* C, int64_t M,
                                  int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                  bwgemm_dtype_t dtype)
{
    if (dtype != BWGEMM_BF16 && dtype != BWGEMM_FP16)
        return BWGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0)
        return BWGEMM_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldc < N)
        return BWGEMM_ERR_INVALID_ARG;
    const int64_t kMaxDim = (int64_t(1) << 31) - 1;  // TMA coordinates are 32-bit
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return BWGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return BWGEMM_OK;
    if (!C)
        return BWGEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B))
        return BWGEMM_ERR_INVALID_ARG;
    if (!aligned16(C) || (ldc % 8) != 0)
        return BWGEMM_ERR_ALIGNMENT;
    if (K > 0 && (!aligned16(A) || !aligned16(B) || (lda % 8) != 0 || (ldb % 8) != 0))
        return BWGEMM_ERR_ALIGNMENT;
    if (lda > (int64_t(1) << 36) || ldb > (int64_t(1) << 36) || ldc > (int64_t(1) << 36))
        return BWGEMM_ERR_UNSUPPORTED;  // tensor-map strides stay below 2^40 bytes
    return BWGEMM_OK;
}

bwgemm_status_t bwgemm_select_config(int32_t num_sms, int32_t max_pairs, int64_t M, int64_t N,
                                     int64_t K, bwgemm_dtype_t dtype,
                                     const bwgemm_plan_options_t* opts, bwgemm_config_t* out)
{
    if (!out || (dtype != BWGEMM_BF16 && dtype != BWGEMM_FP16))
        return BWGEMM_ERR_INVALID_ARG;
    bwgemm_plan_options_t o;
    if (opts)
        o = *opts;
    else
        bwgemm_default_options(&o);
    const uint64_t ws = o.workspace_bytes ? o.workspace_bytes : (64ull << 20);
    Selection sel;
    const bwgemm_status_t st = select_config(num_sms, max_pairs, M, N, K, o, ws, &sel);
    if (st == BWGEMM_OK)
        *out = sel.cfg;
    return st;
}

const char* bwgemm_status_string(bwgemm_status_t status)
{
    switch (status) {
    case BWGEMM_OK: return "ok";
    case BWGEMM_ERR_INVALID_ARG: return "invalid argument";
    case BWGEMM_ERR_ALIGNMENT: return "pointer or leading dimension misaligned (16 B / 8 elements)";
    case BWGEMM_ERR_UNSUPPORTED: return "unsupported device or size";
    case BWGEMM_ERR_NO_DEVICE: return "no CUDA device";
    case BWGEMM_ERR_CUDA: return "CUDA error";
    case BWGEMM_ERR_TIMEOUT: return "device-side wait timed out";
    case BWGEMM_ERR_WORKSPACE: return "split-K workspace too small";
    }
    return "unknown status";
}

int32_t bwgemm_version(void) { return (BWGEMM_VERSION_MAJOR << 16) | BWGEMM_VERSION_MINOR; }

}  // extern "C"
