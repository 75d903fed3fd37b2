// planner.cpp -- host-only argument checks and launch-configuration choice.
//
// Nothing here touches the device, so all of it is testable without a GPU
// through bwgemm_check_args / bwgemm_select_config.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "tuned_table.h"

namespace bwgemm {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The entry of the tuned-options table for this shape, applied to `opts` when
// the caller allows it and left automatic every option the entry sets.
bool apply_tuned_table(bwgemm_plan_options_t& opts, int64_t M, int64_t N, int64_t K)
{
    if (opts.tuned_table != 0)
        return false;
    for (const TunedEntry& e : kTunedTable) {
        if (e.M == 0)
            break;
        if (e.M != M || e.N != N || e.K != K)
            continue;
        const int32_t set[] = {e.variant, e.tile_n, e.split_k, e.schedule, e.copy_kblocks,
                               e.cluster_split, e.raster_group, e.swap_ab, e.multicast, e.skinny};
        const int32_t mine[] = {opts.variant, opts.tile_n, opts.split_k, opts.schedule, opts.copy_kblocks,
                                opts.cluster_split, opts.raster_group, opts.swap_ab, opts.multicast, opts.skinny};
        for (int i = 0; i < 10; ++i)
            if (set[i] != 0 && mine[i] != 0)
                return false;  // the caller chose this option itself
        opts.variant = e.variant ? e.variant : opts.variant;
        opts.tile_n = e.tile_n ? e.tile_n : opts.tile_n;
        opts.split_k = e.split_k ? e.split_k : opts.split_k;
        opts.schedule = e.schedule ? e.schedule : opts.schedule;
        opts.copy_kblocks = e.copy_kblocks ? e.copy_kblocks : opts.copy_kblocks;
        opts.cluster_split = e.cluster_split ? e.cluster_split : opts.cluster_split;
        opts.raster_group = e.raster_group ? e.raster_group : opts.raster_group;
        opts.swap_ab = e.swap_ab ? e.swap_ab : opts.swap_ab;
        opts.multicast = e.multicast ? e.multicast : opts.multicast;
        opts.skinny = e.skinny ? e.skinny : opts.skinny;
        return true;
    }
    return false;
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int find_variant(int cg, int bn, bool trans, int mc, int ks, bool rs)
{
    for (int i = 0; i < kNumVariants; ++i)
        if (kVariants[i].cg == cg && kVariants[i].bn == bn && kVariants[i].trans == trans &&
            kVariants[i].mc == mc && kVariants[i].ks == ks && kVariants[i].rs == rs)
            return i;
    return -1;
}

bwgemm_status_t select_config(int num_sms, int max_pairs, int max_quads, int64_t M, int64_t N,
                              int64_t K, const bwgemm_plan_options_t& opts_in,
                              uint64_t workspace_bytes, Selection* out)
{
    if (!out || num_sms <= 0 || M < 0 || N < 0 || K < 0)
        return BWGEMM_ERR_INVALID_ARG;
    if (opts_in.tuned_table < 0 || opts_in.tuned_table > 1)
        return BWGEMM_ERR_INVALID_ARG;
    bwgemm_plan_options_t opts = opts_in;
    const bool tuned = apply_tuned_table(opts, M, N, K);
    if (max_pairs <= 0)
        max_pairs = num_sms / 2;
    if (max_quads <= 0)
        max_quads = std::max(1, max_pairs / 2);
    for (int32_t r : opts.reserved)
        if (r != 0)
            return BWGEMM_ERR_INVALID_ARG;

    // Operand order.  For a small-M, wide-N problem (decode batches of <= 64
    // rows) the kernel computes C^T = B A^T: B's N rows fill the 128-row MMA
    // side and A's few rows become a 64-wide MMA N, so a pipeline stage is
    // two thirds weights instead of padding.  (At M = 256 swapping doubles
    // the weight traffic into the SMs and measured slower.)
    bool swap;
    switch (opts.swap_ab) {
    case 0: swap = (M <= 64 && N >= 1024); break;
    case 1: swap = false; break;
    case 2: swap = true; break;
    default: return BWGEMM_ERR_INVALID_ARG;
    }
    const int64_t Mk = swap ? N : M;  // the kernel's M and N
    const int64_t Nk = swap ? M : N;

    // Variant: the CTA-pair form (256-row units, each CTA streaming half of the
    // B tile) whenever there are more than 128 rows; one CTA per unit otherwise.
    int cg;
    switch (opts.variant) {
    case BWGEMM_VARIANT_AUTO: cg = (Mk > 128 && !swap) ? 2 : 1; break;
    case BWGEMM_VARIANT_1SM: cg = 1; break;
    case BWGEMM_VARIANT_2SM: cg = 2; break;
    default: return BWGEMM_ERR_INVALID_ARG;
    }
    int bn;
    if (opts.tile_n == 0)
        bn = swap ? (Nk <= 64 ? 64 : 128) : (Nk <= 128 ? 128 : 256);
    else if (opts.tile_n == 64 || opts.tile_n == 128 || opts.tile_n == 224 || opts.tile_n == 256 ||
             opts.tile_n == 320 || opts.tile_n == 384)
        bn = opts.tile_n;
    else
        return BWGEMM_ERR_INVALID_ARG;
    // A multicast: clusters of two CTA pairs on adjacent column blocks, each
    // A tile read from L2 once for both pairs.  Off unless asked for: only 36
    // clusters of 4 CTAs fit on the 152 SMs at once (144 SMs), and the ~4 %
    // it gains per SM (8192^3) does not make up for the 8 idle SMs.
    int mc;
    switch (opts.multicast) {
    case 0: mc = 1; break;
    case 1: mc = 1; break;
    case 2: mc = 2; break;
    default: return BWGEMM_ERR_INVALID_ARG;
    }
    if (mc > 1 && (cg != 2 || swap))
        return BWGEMM_ERR_UNSUPPORTED;
    if (opts.split_k < 0 || opts.raster_group < 0 || opts.max_ctas < 0 || opts.prefetch < -1 ||
        opts.prefetch > 64 || opts.copy_kblocks < 0 || opts.copy_kblocks > 2)
        return BWGEMM_ERR_INVALID_ARG;

    const int tile_m = kRowsPerCta * cg;
    const int64_t num_m = ceil_div(Mk, tile_m);
    const int64_t num_kb = ceil_div(K, kTileK);

    // Workers (clusters of cs CTAs: pairs, pairs of pairs, or single CTAs)
    // the persistent grid holds at once.
    const int cs = cg * mc;
    int64_t slots = (cs == 4) ? max_quads : (cs == 2) ? max_pairs : num_sms;
    if (opts.max_ctas > 0)
        slots = std::max<int64_t>(1, std::min<int64_t>(slots, opts.max_ctas / cs));
    if (opts.schedule < BWGEMM_SCHEDULE_AUTO || opts.schedule > BWGEMM_SCHEDULE_CLC)
        return BWGEMM_ERR_INVALID_ARG;
    const bool clc = opts.schedule == BWGEMM_SCHEDULE_CLC;

    // Decode batches of at most 64 rows: the whole-K kernel with 64 weight rows
    // per CTA and the rows of A as the MMA's N, when its CTAs fit one wave: no
    // split of K, so no partial sums to exchange after the last MMA, which is
    // what split-K on 128-row tiles pays (N = 8192: 128 CTAs).  More than 32
    // rows: CTA pairs (M = 128 across the pair), each CTA copying half of A's
    // rows.  Taken unless an option asks for something only the main kernel
    // does.
    if (opts.skinny < 0 || opts.skinny > 2)
        return BWGEMM_ERR_INVALID_ARG;
    {
        const int sbn = Nk <= 16 ? 16 : (Nk <= 32 ? 32 : 64);
        const int scg = skinny_cg(sbn);
        const int64_t sk_units = ceil_div(Mk, int64_t(kSkinnyRows) * scg);  // CTAs or pairs
        const int64_t sk_ctas = sk_units * scg;
        const bool forced_other = opts.variant != BWGEMM_VARIANT_AUTO || opts.tile_n != 0 || opts.split_k > 1 ||
                                  clc || opts.schedule == BWGEMM_SCHEDULE_STREAM_K || mc != 1 ||
                                  opts.cluster_split == 2 || opts.prefetch > 0 || opts.copy_kblocks != 0 ||
                                  opts.raster_group > 0;
        const bool fits = swap && Nk <= 64 && sk_units >= 1 && sk_ctas <= num_sms &&
                          (scg == 1 || sk_units <= max_pairs) && (opts.max_ctas == 0 || sk_ctas <= opts.max_ctas);
        if (opts.skinny == 2 && !fits)
            return BWGEMM_ERR_UNSUPPORTED;
        if (fits && (opts.skinny == 2 || (opts.skinny == 0 && !forced_other))) {
            Selection sel;
            std::memset(&sel, 0, sizeof(sel));
            sel.variant_idx = -1;
            sel.skinny_bn = sbn;
            sel.swap = true;
            sel.num_m_blocks = int(sk_units);
            sel.num_n_blocks = 1;
            sel.num_k_blocks = int(num_kb);
            sel.cfg.variant = scg == 2 ? BWGEMM_VARIANT_2SM : BWGEMM_VARIANT_1SM;
            sel.cfg.tile_m = kSkinnyRows * scg;
            sel.cfg.tile_n = sbn;
            sel.cfg.tile_k = kTileK;
            sel.cfg.stages = skinny_stages(sbn);
            sel.cfg.split_k = 1;
            sel.cfg.raster_group = 1;
            sel.cfg.num_tiles = int32_t(sk_units);
            sel.cfg.num_units = int32_t(sk_units);
            sel.cfg.grid = int32_t(sk_ctas);
            sel.cfg.schedule = BWGEMM_SCHEDULE_TILES;
            sel.cfg.dp_tiles = int32_t(sk_units);
            sel.cfg.workers = int32_t(sk_units);
            sel.cfg.swap_ab = 1;
            sel.cfg.multicast = 1;
            sel.cfg.copy_kblocks = K / kTileK >= skinny_kblocks(sbn) ? skinny_kblocks(sbn) : 1;
            sel.cfg.tuned = tuned ? 1 : 0;
            sel.cfg.skinny = 1;
            *out = sel;
            return BWGEMM_OK;
        }
    }

    // 129 to 256 rows of A, operands in order: the whole-K pair kernel with all
    // rows of A on the MMA's M side (256 over the pair) and the narrowest block
    // of weight rows whose blocks fit the co-resident pairs once (N = 10240:
    // 72 blocks of 144), so that no K split and no exchange of partials is
    // needed.  Automatic only where the main kernel would take a pair tile
    // wider than 256 columns (two MMAs per K step into a single-buffered
    // accumulator, split in clusters): there it measured ~2 % faster (decode
    // QKV), while against 256-wide tiles split in clusters it was 2-10 %
    // slower (N = 8192, K = 8192 and 28672).  wholek = 2 requires it.
    if (opts.wholek < 0 || opts.wholek > 2)
        return BWGEMM_ERR_INVALID_ARG;
    int wbn = 0;
    for (int w : kWholeKWidths)
        if (wbn == 0 && ceil_div(N, int64_t(w)) <= max_pairs && 2 * ceil_div(N, int64_t(w)) <= num_sms)
            wbn = w;
    const int64_t wk_units = wbn ? ceil_div(N, int64_t(wbn)) : 0;  // pairs
    const bool wk_fits = !swap && M > 128 && M <= 256 && wbn > 0 &&
                         (opts.max_ctas == 0 || 2 * wk_units <= opts.max_ctas);
    const bool wk_forced_other = opts.variant != BWGEMM_VARIANT_AUTO || opts.tile_n != 0 || opts.split_k > 1 ||
                                 clc || opts.schedule == BWGEMM_SCHEDULE_STREAM_K || mc != 1 ||
                                 opts.cluster_split == 2 || opts.prefetch > 0 || opts.copy_kblocks != 0 ||
                                 opts.raster_group > 0 || opts.swap_ab == 2;
    if (opts.wholek == 2 && !wk_fits)
        return BWGEMM_ERR_UNSUPPORTED;
    auto wholek_selection = [&]() {
        Selection sel;
        std::memset(&sel, 0, sizeof(sel));
        sel.variant_idx = -1;
        sel.wholek_bn = wbn;
        sel.swap = false;
        sel.num_m_blocks = 1;
        sel.num_n_blocks = int(wk_units);
        sel.num_k_blocks = int(num_kb);
        sel.cfg.variant = BWGEMM_VARIANT_2SM;
        sel.cfg.tile_m = 256;
        sel.cfg.tile_n = wbn;
        sel.cfg.tile_k = kTileK;
        sel.cfg.stages = wholek_stages(wbn);
        sel.cfg.split_k = 1;
        sel.cfg.raster_group = 1;
        sel.cfg.num_tiles = int32_t(wk_units);
        sel.cfg.num_units = int32_t(wk_units);
        sel.cfg.grid = int32_t(2 * wk_units);
        sel.cfg.schedule = BWGEMM_SCHEDULE_TILES;
        sel.cfg.dp_tiles = int32_t(wk_units);
        sel.cfg.workers = int32_t(wk_units);
        sel.cfg.swap_ab = 0;
        sel.cfg.multicast = 1;
        sel.cfg.copy_kblocks = K / kTileK >= wholek_kblocks(wbn) ? wholek_kblocks(wbn) : 1;
        sel.cfg.tuned = tuned ? 1 : 0;
        sel.cfg.wholek = 1;
        return sel;
    };
    if (wk_fits && opts.wholek == 2) {
        *out = wholek_selection();
        return BWGEMM_OK;
    }

    // Tile width of the pair form: 224, 320 or 384 instead of 256 columns
    // when the problem then fits one wave clearly better.  N = 8192 makes 32
    // tiles of 256 (x 2 K slices, or x 2 row blocks: 64 of 76 pairs) but 37
    // of 224 (74 of 76); N = 10240 makes 40 tiles of 256 (too many for two
    // slices each: left to stream-K) but 32 of 320, whose two slices fill 64
    // pairs; N = 28672 makes 112 tiles of 256 (1.5 waves) but 75 of 384.
    // (The occupancy follows the one-wave split rule of the schedule below.)
    if (opts.tile_n == 0 && cg == 2 && !swap && mc == 1 && bn == 256 && opts.split_k == 0 && !clc &&
        opts.schedule != BWGEMM_SCHEDULE_STREAM_K) {
        // tiles, K slices per tile and the share of the workers busy in a
        // one-wave launch of whole tiles or split-K slices; 0 slices when the
        // launch would take more than one wave or be left to stream-K
        struct Wave {
            int64_t tiles, slices;
            double occupancy;
        };
        auto one_wave = [&](int64_t b) -> Wave {
            const int64_t t = num_m * ceil_div(Nk, b);
            if (t == 0 || t > slots)
                return {t, 0, 0.0};
            int64_t S = 1;
            if (num_kb >= 4 && double(t) < 0.8 * double(slots)) {
                S = std::min<int64_t>({slots / t, num_kb / 4, 4});
                if (S < 2 || double(t * S) < 0.75 * double(slots))
                    return {t, 0, 0.0};
            }
            return {t, S, double(t * S) / double(slots)};
        };
        // Two slices run in one cluster per tile (exchanging partials through
        // distributed shared memory) only while the tiles fit the co-resident
        // clusters of four CTAs; trading that exchange for the one through L2
        // measured slower than the 24 SMs it gains (decode M = 256, N = 8192:
        // 36 clusters of four fit on GB300, 37 tiles of 224 do not).
        // So a narrower or wider tile is taken only as whole tiles, or with
        // its two slices in clusters (where that width has a clustered form).
        auto clustered = [&](const Wave& w, int b) {
            return opts.cluster_split != 1 && w.slices == 2 && w.tiles <= max_quads &&
                   find_variant(2, b, false, 1, 2) >= 0;
        };
        const Wave w256 = one_wave(256);
        Wave best = w256;
        for (int b : {224, 320, 384}) {
            const Wave w = one_wave(b);
            if (w.occupancy > best.occupancy + 0.05 && (w.slices < 2 || clustered(w, b))) {
                best = w;
                bn = b;
            }
        }
    }
    const int idx = find_variant(cg, bn, swap, mc);
    if (idx < 0)
        return BWGEMM_ERR_UNSUPPORTED;
    const int64_t num_n = ceil_div(Nk, int64_t(bn) * mc);  // column groups of mc blocks
    const int64_t tiles = num_m * num_n;
    if (num_m > (1 << 30) || num_n > (1 << 30) || tiles > (int64_t(1) << 30))
        return BWGEMM_ERR_UNSUPPORTED;
    if (clc && opts.split_k > 1)
        return BWGEMM_ERR_INVALID_ARG;  // cluster launch control hands out whole tiles only

    // Schedule.  Whole tiles when they fill the workers evenly.  With fewer
    // tiles than workers: whole tiles when they still occupy >= 80 % of the
    // workers; else split-K in one wave (S slices per tile, all running at
    // once, reduce-scattering their partials) when S >= 2 fills >= 75 %;
    // else stream-K.  With more tiles than workers but a ragged last wave
    // (< 90 % full): stream-K -- the whole waves but the last one stay whole
    // tiles and the K iterations of the remaining tiles are divided evenly.
    bool stream_k = false;
    int64_t auto_split = 1;
    if (opts.split_k > 1 || opts.schedule == BWGEMM_SCHEDULE_TILES || clc || tiles == 0) {
        stream_k = false;
    } else if (opts.schedule == BWGEMM_SCHEDULE_STREAM_K) {
        stream_k = true;
    } else if (num_kb >= 4 && tiles % slots != 0) {
        if (tiles > slots) {
            const int64_t waves = (tiles + slots - 1) / slots;
            stream_k = double(tiles) / double(waves * slots) < 0.9;
        } else if (double(tiles) < 0.8 * double(slots)) {
            const int64_t S = std::min<int64_t>({slots / tiles, num_kb / 4, 4});
            if (S >= 2 && double(tiles * S) >= 0.75 * double(slots))
                auto_split = S;
            else
                stream_k = true;
        }
    }

    int64_t s = 1, dp_tiles = tiles, sk_tiles = 0, workers = 0, ws = 0;
    const int64_t slot_bytes = int64_t(cs) * kRowsPerCta * bn * 4;  // one piece's fp32 partial
    if (stream_k) {
        dp_tiles = (tiles >= 2 * slots) ? (tiles / slots - 1) * slots : 0;
        sk_tiles = tiles - dp_tiles;
        const int64_t iters = sk_tiles * num_kb;
        // at least 4 K blocks per worker; all workers when there are whole tiles too
        workers = dp_tiles > 0 ? slots : std::max<int64_t>(1, std::min<int64_t>(slots, iters / 4));
        ws = int64_t(kCounterRegionBytes) + workers * 2 * slot_bytes;
        const int64_t counters = sk_tiles * cs * kEpiWarps * kCountersPerWarp * 4;
        if (counters > int64_t(kCounterRegionBytes) || uint64_t(ws) > workspace_bytes) {
            if (opts.schedule == BWGEMM_SCHEDULE_STREAM_K)
                return BWGEMM_ERR_WORKSPACE;
            stream_k = false;
            dp_tiles = tiles;
            sk_tiles = 0;
            ws = 0;
        }
    }
    if (!stream_k) {
        // split-K over whole tiles: forced, chosen above, or (schedule = tiles)
        // when the tiles alone leave most workers idle; >= 4 K blocks per slice
        if (opts.split_k > 0) {
            s = std::min<int64_t>(opts.split_k, std::max<int64_t>(num_kb, 1));
        } else if (clc) {
            s = 1;
        } else if (auto_split > 1) {
            s = auto_split;
        } else if (opts.schedule == BWGEMM_SCHEDULE_TILES && tiles > 0 && tiles < slots &&
                   num_kb >= 8) {
            s = std::min<int64_t>({slots / tiles, num_kb / 4, 8});
            s = std::max<int64_t>(s, 1);
        }
        if (s > 1) {
            const int64_t counters = tiles * cs * kEpiWarps * kCountersPerWarp * 4;
            ws = int64_t(kCounterRegionBytes) + tiles * s * slot_bytes;
            if (counters > int64_t(kCounterRegionBytes) || uint64_t(ws) > workspace_bytes) {
                if (opts.split_k > 1)
                    return BWGEMM_ERR_WORKSPACE;
                s = 1;
                ws = 0;
            }
        }
        // with cluster launch control the grid holds one cluster per tile
        workers = clc ? tiles : std::min<int64_t>(tiles * s, slots);
    }
    // all slices of every tile in one wave: they may wait for one another
    const bool scatter = !stream_k && s > 1 && tiles * s <= slots;

    // Two K slices of a tile inside one cluster (two pairs, or two CTAs),
    // exchanging partials through distributed shared memory instead of L2:
    // one-wave split-K with two slices, when a cluster per tile fits at once.
    int idx_run = idx;
    bool cluster_split = false;
    if (opts.cluster_split < 0 || opts.cluster_split > 2)
        return BWGEMM_ERR_INVALID_ARG;
    if (opts.cluster_split != 1 && mc == 1 && scatter && s == 2 && !clc) {
        const int ks_idx = find_variant(cg, bn, swap, 1, 2);
        const int64_t ks_slots = (cg == 2) ? max_quads : max_pairs;  // clusters of 2 * cg CTAs
        if (ks_idx >= 0 && tiles <= ks_slots && (opts.max_ctas == 0 || tiles * cg * 2 <= opts.max_ctas)) {
            idx_run = ks_idx;
            cluster_split = true;
            workers = tiles;
            ws = 0;  // no partials or counters in global memory
        }
    }
    if (opts.cluster_split == 2 && !cluster_split)
        return BWGEMM_ERR_UNSUPPORTED;
    // One whole tile per worker (every CTA's only unit): the variant that
    // stages its output in the then idle operand ring and uses the room it
    // saves for one more stage, where there is one.
    if (!cluster_split && !stream_k && !clc && s == 1 && mc == 1 && tiles <= workers) {
        const int rs_idx = find_variant(cg, bn, swap, 1, 1, true);
        if (rs_idx >= 0)
            idx_run = rs_idx;
    }
    const int cs_run = cluster_split ? cg * 2 : cs;

    // Grouped raster ("Matrix Multiplication on NVIDIA's Blackwell", Kernel 9):
    // groups of 8 row blocks, walked down before stepping along N, keep the
    // operand tiles of one wave in L2 when the operands are larger than it
    // (8192^3: groups of 16 or 32 measured 1-7 % slower).  When both operands
    // fit in half the L2 (4096^3: 64 MiB), every row block of a column is
    // walked first instead (measured +1.1 % at the top clock, +1.5 % under
    // the power cap).
    constexpr int64_t kL2HalfBytes = int64_t(64) << 20;
    const int64_t operand_bytes = 2 * (Mk + Nk) * K;
    int64_t group = opts.raster_group > 0 ? opts.raster_group : (operand_bytes <= kL2HalfBytes ? num_m : 8);
    group = std::max<int64_t>(1, std::min<int64_t>(group, std::max<int64_t>(num_m, 1)));

    Selection sel;
    std::memset(&sel, 0, sizeof(sel));
    sel.variant_idx = idx_run;
    sel.swap = swap;
    sel.num_m_blocks = int(num_m);
    sel.num_n_blocks = int(num_n);
    sel.num_k_blocks = int(num_kb);
    sel.sk_iters = sk_tiles * num_kb;
    sel.cfg.variant = (cg == 2) ? BWGEMM_VARIANT_2SM : BWGEMM_VARIANT_1SM;
    sel.cfg.tile_m = tile_m;
    sel.cfg.tile_n = bn;
    sel.cfg.tile_k = kTileK;
    sel.cfg.stages = kVariants[idx_run].stages;  // the variant that runs
    sel.cfg.split_k = int32_t(s);
    sel.cfg.raster_group = int32_t(group);
    sel.cfg.num_tiles = int32_t(tiles);
    sel.cfg.num_units = int32_t(dp_tiles * s);
    sel.cfg.grid = int32_t(workers * cs_run);
    sel.cfg.workspace_bytes = ws;
    sel.cfg.schedule = clc ? BWGEMM_SCHEDULE_CLC
                           : (stream_k ? BWGEMM_SCHEDULE_STREAM_K : BWGEMM_SCHEDULE_TILES);
    sel.cfg.dp_tiles = int32_t(dp_tiles);
    sel.cfg.sk_tiles = int32_t(sk_tiles);
    sel.cfg.workers = int32_t(workers);
    sel.cfg.split_scatter = scatter ? 1 : 0;
    sel.cfg.swap_ab = swap ? 1 : 0;
    sel.cfg.multicast = mc;
    sel.cfg.cluster_split = cluster_split ? 1 : 0;
    sel.cfg.tuned = tuned ? 1 : 0;
    // K blocks per operand copy.  Two (3-D copies) when the kernel is compute
    // bound: one TMA copy occupies its unit for ~140 ns whatever its size, and
    // two 16 KiB copies per K block take longer than the K block's MMAs.  In
    // a memory-bound decode shape (a side of at most 256 rows) the coarser
    // stages cost more than the copies they save, so one.
    if (opts.copy_kblocks == 0)
        sel.cfg.copy_kblocks = (std::min(Mk, Nk) > 256 && num_kb >= 2) ? 2 : 1;
    else
        sel.cfg.copy_kblocks = opts.copy_kblocks;
    // L2 prefetch of the streamed operand (the one with more rows: read from
    // DRAM once, while the other stays in L2 for every tile): off unless
    // asked for.  Measured on the decode and tail shapes at distances 4 to 32
    // K blocks (one or two K blocks per prefetch) it was slower every time.
    sel.cfg.prefetch_kblocks = opts.prefetch > 0 ? opts.prefetch : 0;
    sel.cfg.prefetch_b = (Nk >= Mk) ? 1 : 0;

    if (wk_fits && opts.wholek == 0 && !wk_forced_other && sel.cfg.tile_n > 256) {
        *out = wholek_selection();
        return BWGEMM_OK;
    }
    *out = sel;
    return BWGEMM_OK;
}

namespace {

// rows of a full block of bwgemm_run_host's pipeline (0: no pipeline)
int64_t host_base_rows(int64_t M, int64_t N, int64_t K)
{
    const int64_t bytes = 2 * (M * K + N * K + M * N);
    if (K <= 0 || N <= 0 || M < 1024 || bytes < (int64_t(16) << 20))
        return 0;
    int64_t rows = M >= 2048 ? 1024 : 512;
    // at most kHostChunksMax - 1 full blocks (the last one is halved)
    rows = std::max<int64_t>(rows, ceil_div(ceil_div(M, int64_t(kHostChunksMax - 1)), 256) * 256);
    return rows < M ? rows : 0;
}

}  // namespace

int host_row_blocks(int64_t M, int64_t N, int64_t K, int64_t* starts)
{
    const int64_t rows = host_base_rows(M, N, K);
    starts[0] = 0;
    if (rows == 0) {
        starts[1] = M;
        return 1;
    }
    int n = 0;
    while (starts[n] + rows < M) {
        starts[n + 1] = starts[n] + rows;
        ++n;
    }
    // the last block: M - starts[n] rows, halved (whole 256-row tiles) when it
    // holds at least two tiles
    const int64_t last = M - starts[n];
    if (last >= 512) {
        starts[n + 1] = starts[n] + ceil_div(last / 2, int64_t(256)) * 256;
        ++n;
    }
    starts[n + 1] = M;
    return n + 1;
}

int64_t host_block_cols(int64_t M, int64_t N, int64_t K)
{
    const int64_t rows = host_base_rows(M, N, K);
    if (rows == 0 || N < 2048)
        return 0;
    const int64_t cols = ceil_div(ceil_div(N, int64_t(kHostColBlocksMax)), 256) * 256;
    // only blocks that still fill the GPU (64 tiles of 256 x 256): smaller
    // GEMMs run too far below the peak for the earlier start to pay
    if (cols >= N || rows * cols < int64_t(64) * 256 * 256)
        return 0;
    return cols;
}

GemmParams make_params(const Selection& sel, int64_t M, int64_t N, int64_t K, bwgemm_dtype_t dtype)
{
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (sel.wholek_bn > 0) {
        // the whole-K pair kernel: the caller's problem, all of M in one pair
        p.M = int32_t(M);
        p.N = int32_t(N);
        p.K = int32_t(K);
        p.num_m_blocks = 1;
        p.num_n_blocks = sel.num_n_blocks;
        p.num_k_blocks = sel.num_k_blocks;
        p.num_tiles = sel.cfg.num_tiles;
        p.split_k = 1;
        p.dp_tiles = sel.cfg.num_tiles;
        p.dp_units = sel.cfg.num_tiles;
        p.raster_group = 1;
        p.dtype = int32_t(dtype);
        p.idesc = make_idesc(int(dtype), 256, sel.wholek_bn);
        p.stall_kblock = -1;
        p.ks = 1;
        return p;
    }
    if (sel.skinny_bn > 0) {
        // the whole-K kernel: the weight rows (the caller's N) are its M
        p.M = int32_t(N);
        p.N = int32_t(M);
        p.K = int32_t(K);
        p.num_m_blocks = sel.num_m_blocks;
        p.num_n_blocks = 1;
        p.num_k_blocks = sel.num_k_blocks;
        p.num_tiles = sel.cfg.num_tiles;
        p.split_k = 1;
        p.dp_tiles = sel.cfg.num_tiles;
        p.dp_units = sel.cfg.num_tiles;
        p.raster_group = 1;
        p.dtype = int32_t(dtype);
        p.idesc = make_idesc(int(dtype), kSkinnyRows * skinny_cg(sel.skinny_bn), sel.skinny_bn);
        p.stall_kblock = -1;
        p.ks = 1;
        return p;
    }
    const Variant& v = kVariants[sel.variant_idx];
    p.M = int32_t(sel.swap ? N : M);  // the kernel's problem
    p.N = int32_t(sel.swap ? M : N);
    p.K = int32_t(K);
    p.num_m_blocks = sel.num_m_blocks;
    p.num_n_blocks = sel.num_n_blocks;
    p.num_k_blocks = sel.num_k_blocks;
    p.num_tiles = sel.cfg.num_tiles;
    p.split_k = sel.cfg.split_k;
    p.dp_tiles = sel.cfg.dp_tiles;
    p.dp_units = sel.cfg.num_units;
    p.sk_tiles = sel.cfg.sk_tiles;
    p.sk_iters = sel.sk_iters;
    p.raster_group = sel.cfg.raster_group;
    p.dtype = int32_t(dtype);
    p.idesc = make_idesc(int(dtype), kRowsPerCta * v.cg, std::min(v.bn, 256));
    p.idesc2 = v.bn > 256 ? make_idesc(int(dtype), kRowsPerCta * v.cg, v.bn - 256) : 0u;
    p.stall_kblock = -1;
    p.split_scatter = sel.cfg.split_scatter;
    p.prefetch = sel.cfg.prefetch_kblocks;
    p.prefetch_b = sel.cfg.prefetch_b;
    p.clc = sel.cfg.schedule == BWGEMM_SCHEDULE_CLC ? 1 : 0;
    p.ks = 1;
    if (sel.cfg.cluster_split) {
        // the cluster walks whole tiles; its pairs take the K slices
        p.ks = sel.cfg.split_k;
        p.split_k = 1;
        p.dp_units = sel.cfg.num_tiles;
        p.split_scatter = 0;
    }
    return p;
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

bwgemm_status_t bwgemm_select_config(int32_t num_sms, int32_t max_pairs, int32_t max_quads,
                                     int64_t M, int64_t N, int64_t K, bwgemm_dtype_t dtype,
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
    const bwgemm_status_t st = select_config(num_sms, max_pairs, max_quads, M, N, K, o, ws, &sel);
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
