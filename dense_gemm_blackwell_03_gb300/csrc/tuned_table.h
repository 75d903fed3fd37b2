// tuned_table.h -- written by `python -m dense_gemm_blackwell_03_gb300.tune_table
// --header`: plan options that the offline sweep over the pages' shapes measured
// faster than the planner's own choice (steady-state CUDA-event timing on
// GB300, alternating order).  select_config applies an entry when the shape
// matches exactly and the caller left every option it sets on automatic.
#pragma once

#include <cstdint>

namespace bwgemm {

struct TunedEntry {
    int64_t M, N, K;
    // the options the entry sets (0 = automatic, as in bwgemm_plan_options_t)
    int32_t variant, tile_n, split_k, schedule, copy_kblocks, cluster_split, raster_group, swap_ab,
        multicast, skinny;
};

// the last entry (M = 0) ends the table
constexpr TunedEntry kTunedTable[] = {
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0},
};

}  // namespace bwgemm
