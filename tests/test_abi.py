"""Host-only checks of the C ABI (no GPU): the library loads, exports every
symbol include/bwgemm.h declares, its structs match the header's layout, and
the host logic (argument checks, configuration choice) behaves as documented.
"""
from __future__ import annotations

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from dense_gemm_blackwell_03_gb300 import binding
from dense_gemm_blackwell_03_gb300.binding import BF16, FP16, Config, PlanOptions

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bwgemm.h")

OK, INVALID, ALIGN, UNSUP, NODEV, CUDA, TIMEOUT, WORKSPACE = range(8)


@pytest.fixture(scope="module")
def lib():
    return binding.load_library(build_if_missing=True)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bwgemm_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations parsed from bwgemm.h"
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert sorted(binding.EXPORTED) == names


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "bwgemm.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(bwgemm_plan_options_t), '
        "offsetof(bwgemm_plan_options_t, timeout_ns), offsetof(bwgemm_plan_options_t, pdl_off), "
        "sizeof(bwgemm_config_t), offsetof(bwgemm_config_t, workspace_bytes), "
        "offsetof(bwgemm_config_t, swap_ab));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got == [ctypes.sizeof(PlanOptions), PlanOptions.timeout_ns.offset,
                   PlanOptions.pdl_off.offset, ctypes.sizeof(Config), Config.workspace_bytes.offset,
                   Config.swap_ab.offset]


def test_version_and_status_strings(lib):
    assert lib.bwgemm_version() == (0 << 16) | 2
    for code in range(8):
        assert lib.bwgemm_status_string(code)
    assert lib.bwgemm_status_string(99) == b"unknown status"


def test_probe_tensor_rate_rejects_null_outputs(lib):
    # argument check before any device access (no GPU needed)
    assert lib.bwgemm_probe_tensor_rate(0, None, None) == 1  # BWGEMM_ERR_INVALID_ARG


def test_default_options(lib):
    o = PlanOptions()
    lib.bwgemm_default_options(ctypes.byref(o))
    assert o.variant == 0 and o.split_k == 0 and o.stall_kblock == -1 and o.timeout_ns == 0
    lib.bwgemm_default_options(None)  # tolerated


A0, B0, C0 = 0x10000, 0x20000, 0x30000  # 16-byte aligned fake addresses (never dereferenced)


@pytest.mark.parametrize("args,want", [
    ((A0, B0, C0, 128, 256, 64, 64, 64, 256, BF16), OK),
    ((A0, B0, C0, 128, 256, 64, 64, 64, 256, FP16), OK),
    ((A0, B0, C0, 128, 256, 64, 64, 64, 256, 2), INVALID),        # dtype
    ((A0, B0, C0, -1, 256, 64, 64, 64, 256, BF16), INVALID),      # negative size
    ((A0, B0, C0, 128, 256, 64, 56, 64, 256, BF16), INVALID),     # lda < K
    ((A0, B0, C0, 128, 256, 64, 64, 64, 248, BF16), INVALID),     # ldc < N
    ((A0, B0, 0, 128, 256, 64, 64, 64, 256, BF16), INVALID),      # NULL C
    ((0, B0, C0, 128, 256, 64, 64, 64, 256, BF16), INVALID),      # NULL A with K > 0
    ((0, 0, C0, 128, 256, 0, 0, 0, 256, BF16), OK),               # K = 0: A, B unused
    ((0, 0, 0, 0, 256, 64, 64, 64, 256, BF16), OK),               # M = 0: nothing to do
    ((0, 0, 0, 128, 0, 64, 64, 64, 0, BF16), OK),                 # N = 0
    ((A0 + 8, B0, C0, 128, 256, 64, 64, 64, 256, BF16), ALIGN),   # A not 16 B aligned
    ((A0, B0 + 2, C0, 128, 256, 64, 64, 64, 256, BF16), ALIGN),
    ((A0, B0, C0 + 4, 128, 256, 64, 64, 64, 256, BF16), ALIGN),
    ((A0, B0, C0, 128, 256, 60, 60, 64, 256, BF16), ALIGN),       # lda not a multiple of 8
    ((A0, B0, C0, 128, 250, 64, 64, 64, 250, BF16), ALIGN),       # ldc not a multiple of 8
    ((A0, B0, C0, 128, 256, 60, 64, 64, 256, BF16), OK),          # ragged K, aligned ld
    ((A0, B0, C0, 1 << 31, 256, 64, 64, 64, 256, BF16), UNSUP),   # beyond 32-bit coordinates
])
def test_check_args(lib, args, want):
    assert binding.check_args(*args) == want


def cfg(M, N, K, sms=148, pairs=0, quads=0, **opts):
    return binding.select_config(sms, M, N, K, max_pairs=pairs, max_quads=quads, **opts)


def test_select_square_uses_cta_pairs_and_stream_k():
    # 4096^3: 256 tiles of 256 x 256 over 76 pairs = 3.37 waves.  Two whole
    # waves stay whole tiles; the K iterations of the other 104 tiles are
    # divided evenly among the 76 pairs.
    c = cfg(4096, 4096, 4096, sms=152, pairs=76)
    assert c["variant"] == 2 and c["tile_m"] == 256 and c["tile_n"] == 256
    assert c["num_tiles"] == 16 * 16 and c["split_k"] == 1 and c["stages"] == 6
    assert c["schedule"] == binding.SCHEDULE_STREAM_K
    assert c["dp_tiles"] == 152 and c["sk_tiles"] == 104 and c["workers"] == 76
    assert c["grid"] == 152 and c["num_units"] == 152
    assert c["workspace_bytes"] == (1 << 20) + 76 * 2 * 2 * 128 * 256 * 4


def test_select_even_waves_stay_whole_tiles():
    # 8192 x 8192: 1024 tiles over 76 pairs = 13.5 waves (96 % full): whole tiles
    c = cfg(8192, 8192, 8192, sms=152, pairs=76)
    assert c["schedule"] == binding.SCHEDULE_TILES and c["dp_tiles"] == 1024
    assert c["sk_tiles"] == 0 and c["workspace_bytes"] == 0 and c["grid"] == 152
    # tiles that fill the workers exactly
    c = cfg(4096, 4096, 4096, sms=152, pairs=64)
    assert c["schedule"] == binding.SCHEDULE_TILES


def test_select_small_m_splits_k_in_one_wave():
    c = cfg(64, 8192, 8192, sms=152, pairs=76, swap_ab=1)
    assert c["variant"] == 1 and c["tile_m"] == 128 and c["num_tiles"] == 32
    # fewer tiles than SMs: 4 K slices per tile, all 128 slices in one wave,
    # reduce-scattering their partials
    assert c["schedule"] == binding.SCHEDULE_TILES and c["split_k"] == 4
    assert c["split_scatter"] == 1 and c["grid"] == 128


def test_select_decode_shapes():
    # attention out / MLP down on GB300 (76 pairs, 36 clusters of four): 32
    # tiles of 256 x 2 K slices, each tile's slices in one cluster.  224-wide
    # tiles (37 x 2 = 74 pairs) would need 37 clusters: their slices would
    # reduce through L2, which measured slower -> 256
    for N, K in ((8192, 8192), (8192, 28672)):
        c = cfg(256, N, K, sms=152, pairs=76, quads=36, swap_ab=1)
        assert c["variant"] == 2 and c["tile_n"] == 256 and c["num_tiles"] == 32
        assert c["split_k"] == 2 and c["cluster_split"] == 1 and c["grid"] == 128
        # the clustered kernel stages its output in the idle ring: seven stages
        assert c["stages"] == 7
        # with room for 37 clusters of four the 224-wide tiles keep the cluster
        c = cfg(256, N, K, sms=152, pairs=76, quads=38, swap_ab=1)
        assert c["tile_n"] == 224 and c["num_tiles"] == 37 and c["cluster_split"] == 1
        assert c["grid"] == 148
    # fused QKV: 40 tiles of 256 -- 2 slices would not fit one wave (stream-K);
    # 32 tiles of 320 (two MMAs per K step) x 2 slices in 32 clusters of four,
    # where the whole-K pair kernel (72 blocks of 144 weight rows) is taken
    c = cfg(256, 10240, 8192, sms=152, pairs=76, quads=36, swap_ab=1, wholek=1)
    assert c["tile_n"] == 320 and c["num_tiles"] == 32 and c["split_k"] == 2
    assert c["cluster_split"] == 1 and c["grid"] == 128 and c["stages"] == 6
    c = cfg(256, 10240, 8192, sms=152, pairs=76, quads=36, swap_ab=1)
    assert c["wholek"] == 1 and c["tile_n"] == 144 and c["num_tiles"] == 72 and c["grid"] == 144
    c = cfg(256, 10240, 8192, sms=152, pairs=76, quads=36, swap_ab=1, tile_n=256)
    assert c["schedule"] == binding.SCHEDULE_STREAM_K and c["workers"] == 76 and c["grid"] == 152
    # MLP up: 112 tiles of 256 = 1.47 waves (stream-K); 75 tiles of 384 (two
    # MMAs per K step) = one wave of whole tiles
    c = cfg(256, 28672, 8192, sms=152, pairs=76, swap_ab=1)
    assert c["tile_n"] == 384 and c["num_tiles"] == 75 and c["split_k"] == 1
    assert c["schedule"] == binding.SCHEDULE_TILES and c["grid"] == 150 and c["stages"] == 5
    c = cfg(256, 28672, 8192, sms=152, pairs=76, swap_ab=1, tile_n=256)
    assert c["schedule"] == binding.SCHEDULE_STREAM_K and c["dp_tiles"] == 0
    # a wider tile whose split would reduce through L2 is not taken: 32 tiles
    # of 384 x 2 slices (no clustered form of 384) -> 256 and stream-K
    assert cfg(256, 12288, 8192, sms=152, pairs=76, quads=36)["tile_n"] == 256
    # Gemma-like 512 x 8192 x 5376: 2 x 37 tiles of 224 fill 74 of 76 pairs
    # (2 x 32 of 256 would fill 64) -> whole tiles of 224
    c = cfg(512, 8192, 5376, sms=152, pairs=76)
    assert c["schedule"] == binding.SCHEDULE_TILES and c["split_k"] == 1 and c["grid"] == 148
    assert c["tile_n"] == 224 and c["num_tiles"] == 74
    # one tile per pair: the variant staging its output in the idle ring (7 stages);
    # 224-wide tiles on a multi-wave shape keep the plain variant (6)
    assert c["stages"] == 7
    assert cfg(4096, 4096, 4096, sms=152, pairs=76, tile_n=224)["stages"] == 6
    # the width rule stays out of multi-wave, stream-K, forced and 1-SM cases
    assert cfg(4096, 4096, 4096, sms=152, pairs=76)["tile_n"] == 256
    assert cfg(8192, 28672, 8192, sms=152, pairs=76)["tile_n"] == 256
    assert cfg(256, 10240, 8192, sms=152, pairs=76, schedule=binding.SCHEDULE_STREAM_K)["tile_n"] == 256
    assert cfg(256, 8192, 8192, sms=152, pairs=76, split_k=2)["tile_n"] == 256
    assert cfg(256, 8192, 8192, sms=152, pairs=76, multicast=2)["tile_n"] == 256
    assert cfg(128, 8192, 8192, sms=152, pairs=76)["tile_n"] == 256
    # explicit 224 and 320 exist only in the pair form with the operands in order
    for tn in (224, 320, 384):
        assert cfg(1000, 2000, 512, tile_n=tn, variant=2)["tile_n"] == tn
        for bad in (dict(variant=1), dict(swap_ab=2), dict(multicast=2)):
            with pytest.raises(binding.BwgemmError):
                cfg(1000, 2000, 512, tile_n=tn, **bad)
    with pytest.raises(binding.BwgemmError):
        cfg(1000, 2000, 512, tile_n=288)


def test_select_swapped_operands_for_small_m():
    # M <= 64 decode: C^T = B A^T, 128 rows of B per CTA, A's rows as a 64-wide
    # MMA N; 64 tiles, two K slices each, all in one wave
    for M in (1, 16, 64):
        c = cfg(M, 8192, 8192, sms=152, pairs=76, skinny=1)
        assert c["swap_ab"] == 1 and c["variant"] == 1 and (c["tile_m"], c["tile_n"]) == (128, 64)
        assert c["num_tiles"] == 64 and c["split_k"] == 2 and c["split_scatter"] == 1
        assert c["grid"] == 128
    # larger M or narrow N keep the operand order
    assert cfg(256, 8192, 8192)["swap_ab"] == 0
    assert cfg(512, 8192, 5376)["swap_ab"] == 0
    assert cfg(64, 512, 4096)["swap_ab"] == 0
    # forced either way; 256-wide units do not exist in swapped form
    c = cfg(256, 8192, 8192, swap_ab=2)
    assert c["swap_ab"] == 1 and c["tile_n"] == 128
    with pytest.raises(binding.BwgemmError):
        cfg(256, 8192, 8192, swap_ab=2, tile_n=256)
    with pytest.raises(binding.BwgemmError):
        cfg(256, 8192, 8192, swap_ab=3)


def test_select_cluster_launch_control():
    # one cluster per tile in the grid; running clusters cancel pending ones
    c = cfg(4096, 4096, 4096, sms=152, pairs=76, schedule=binding.SCHEDULE_CLC)
    assert c["schedule"] == binding.SCHEDULE_CLC and c["split_k"] == 1 and c["sk_tiles"] == 0
    assert c["num_tiles"] == 256 and c["workers"] == 256 and c["grid"] == 512
    c = cfg(64, 8192, 8192, sms=152, pairs=76, schedule=binding.SCHEDULE_CLC)
    assert c["swap_ab"] == 1 and c["grid"] == c["num_tiles"] == 64
    with pytest.raises(binding.BwgemmError):
        cfg(4096, 4096, 4096, schedule=binding.SCHEDULE_CLC, split_k=2)
    with pytest.raises(binding.BwgemmError):
        cfg(4096, 4096, 4096, schedule=4)


def test_select_multicast_pairs_of_pairs():
    # two CTA pairs per cluster on adjacent column blocks: a tile is 256 x 512
    c = cfg(4096, 4096, 4096, sms=152, pairs=76, multicast=2, schedule=binding.SCHEDULE_TILES)
    assert c["multicast"] == 2 and c["variant"] == 2 and c["tile_n"] == 256
    assert c["num_tiles"] == 16 * 8 and c["workers"] == 38 and c["grid"] == 152
    # an odd number of column blocks: the last group's second block is padding
    c = cfg(1024, 768, 512, sms=152, pairs=76, multicast=2)
    assert c["num_tiles"] == 4 * 2
    c = cfg(4096, 4096, 4096, sms=152, pairs=76, multicast=2, schedule=binding.SCHEDULE_STREAM_K)
    assert c["schedule"] == binding.SCHEDULE_STREAM_K and c["grid"] == 152
    assert c["dp_tiles"] + c["sk_tiles"] == 128 and c["dp_tiles"] % 38 == 0
    c = cfg(4096, 4096, 4096, sms=152, pairs=76, multicast=2, schedule=binding.SCHEDULE_CLC)
    assert c["grid"] == 4 * 128
    c = cfg(4096, 4096, 4096, sms=152, pairs=76, multicast=2, tile_n=128, schedule=1)
    assert c["num_tiles"] == 16 * 16 and c["tile_n"] == 128
    assert cfg(4096, 4096, 4096, sms=152, pairs=76)["multicast"] == 1
    assert cfg(4096, 4096, 4096, sms=152, pairs=76, multicast=1)["multicast"] == 1
    with pytest.raises(binding.BwgemmError):
        cfg(4096, 4096, 4096, multicast=2, variant=1)  # multicast joins CTA pairs
    with pytest.raises(binding.BwgemmError):
        cfg(32, 4096, 4096, multicast=2, swap_ab=2)
    with pytest.raises(binding.BwgemmError):
        cfg(4096, 4096, 4096, multicast=3)
    with pytest.raises(binding.BwgemmError):
        cfg(4096, 4096, 4096, copy_kblocks=3)
    assert cfg(4096, 4096, 4096, copy_kblocks=1)["copy_kblocks"] == 1


def test_select_cluster_split():
    # one-wave split-K with two slices: the slices of a tile share a cluster
    c = cfg(256, 8192, 8192, sms=152, pairs=76, tile_n=256)
    assert c["cluster_split"] == 1 and c["split_k"] == 2 and c["grid"] == 32 * 4
    assert c["workspace_bytes"] == 0
    c = cfg(256, 8192, 8192, sms=152, pairs=76)  # 37 tiles of 224 (38 clusters of four fit)
    assert c["tile_n"] == 224 and c["cluster_split"] == 1 and c["grid"] == 37 * 4
    c = cfg(16, 8192, 8192, sms=152, pairs=76, skinny=1)  # swapped: clusters of two single CTAs
    assert c["swap_ab"] == 1 and c["cluster_split"] == 1 and c["grid"] == 64 * 2
    c = cfg(256, 8192, 8192, sms=152, pairs=76, cluster_split=1)
    assert c["cluster_split"] == 0 and c["split_scatter"] == 1 and c["workspace_bytes"] > 0
    # 40 tiles of 256 need 40 clusters of four CTAs: more than fit at once
    c = cfg(256, 10240, 8192, sms=152, pairs=76, tile_n=256)
    assert c["cluster_split"] == 0
    with pytest.raises(binding.BwgemmError):
        cfg(256, 10240, 8192, sms=152, pairs=76, cluster_split=2, tile_n=256)
    # 32 tiles of 320 fit (the whole-K pair kernel, taken there by default, off)
    c = cfg(256, 10240, 8192, sms=152, pairs=76, wholek=1)
    assert c["tile_n"] == 320 and c["cluster_split"] == 1
    with pytest.raises(binding.BwgemmError):
        cfg(256, 8192, 8192, cluster_split=3)


def test_select_prefetch():
    c = cfg(256, 8192, 8192, sms=152, pairs=76)
    assert c["prefetch_kblocks"] == 0 and c["prefetch_b"] == 1  # off unless asked for
    c = cfg(256, 8192, 8192, sms=152, pairs=76, prefetch=8)
    assert c["prefetch_kblocks"] == 8 and c["prefetch_b"] == 1
    c = cfg(16, 8192, 8192, sms=152, pairs=76, prefetch=8)
    assert c["swap_ab"] == 1 and c["prefetch_b"] == 0  # swapped: the weights are the kernel's A
    assert cfg(256, 8192, 8192, prefetch=-1)["prefetch_kblocks"] == 0
    with pytest.raises(binding.BwgemmError):
        cfg(256, 8192, 8192, prefetch=65)


def test_select_kblocks_per_copy():
    # two K blocks per operand copy for compute-bound shapes, one for decode
    assert cfg(4096, 4096, 4096, sms=152, pairs=76)["copy_kblocks"] == 2
    assert cfg(512, 8192, 5376, sms=152, pairs=76)["copy_kblocks"] == 2
    assert cfg(256, 28672, 8192, sms=152, pairs=76)["copy_kblocks"] == 1
    assert cfg(32, 8192, 8192, sms=152, pairs=76, skinny=1)["copy_kblocks"] == 1  # swapped: N' = 32
    assert cfg(256, 28672, 8192, sms=152, pairs=76, copy_kblocks=2)["copy_kblocks"] == 2
    assert cfg(4096, 4096, 64, sms=152, pairs=76)["copy_kblocks"] == 1  # one K block


def test_select_tiles_schedule_splits_k():
    c = cfg(256, 8192, 8192, sms=152, pairs=76, schedule=binding.SCHEDULE_TILES, swap_ab=1,
            cluster_split=1, tile_n=256)
    assert c["schedule"] == binding.SCHEDULE_TILES and c["split_k"] == 2
    assert c["num_units"] == 64 and c["grid"] == 128 and c["split_scatter"] == 1
    assert c["workspace_bytes"] == (1 << 20) + 32 * 2 * 2 * 128 * 256 * 4  # partials through L2
    # more slices than one wave holds: no reduce-scatter (slices may not wait)
    c = cfg(256, 8192, 8192, sms=152, pairs=76, split_k=3, swap_ab=1)
    assert c["split_k"] == 3 and c["split_scatter"] == 0


def test_select_small_problems_use_few_workers():
    # 512^3: 4 tiles x 8 K blocks = 32 iterations, at least 4 per worker
    c = cfg(512, 512, 512, sms=152, pairs=76)
    assert c["schedule"] == binding.SCHEDULE_STREAM_K and c["workers"] == 8 and c["grid"] == 16
    # fewer than 4 K blocks: nothing to spread
    c = cfg(512, 512, 128, sms=152, pairs=76)
    assert c["schedule"] == binding.SCHEDULE_TILES and c["grid"] == 8


def test_select_forced_options():
    c = cfg(1024, 1024, 4096, variant=1, tile_n=128, split_k=3, raster_group=4, max_ctas=64)
    assert (c["variant"], c["tile_m"], c["tile_n"], c["stages"]) == (1, 128, 128, 6)
    assert c["split_k"] == 3 and c["raster_group"] == 4 and c["grid"] == 64
    assert c["schedule"] == binding.SCHEDULE_TILES
    assert c["num_tiles"] == 64 and c["num_units"] == 192
    # a forced split whose partials do not fit the workspace is refused
    with pytest.raises(binding.BwgemmError) as e:
        cfg(4096, 4096, 4096, variant=1, tile_n=128, split_k=3)
    assert e.value.status == WORKSPACE
    # split never exceeds the number of K blocks
    assert cfg(512, 512, 128, split_k=16)["split_k"] == 2


def test_select_rejects_bad_options():
    with pytest.raises(binding.BwgemmError):
        cfg(512, 512, 512, tile_n=96)
    with pytest.raises(binding.BwgemmError):
        cfg(512, 512, 512, variant=7)
    with pytest.raises(binding.BwgemmError) as e:
        cfg(256, 8192, 8192, split_k=4, workspace_bytes=1 << 20, swap_ab=1)
    assert e.value.status == WORKSPACE
    with pytest.raises(binding.BwgemmError) as e:
        cfg(4096, 4096, 4096, schedule=binding.SCHEDULE_STREAM_K, workspace_bytes=1 << 20)
    assert e.value.status == WORKSPACE
    with pytest.raises(binding.BwgemmError):
        cfg(512, 512, 512, schedule=5)
    # automatic stream-K falls back to whole tiles when the workspace is too small
    assert cfg(4096, 4096, 4096, workspace_bytes=1 << 20)["schedule"] == binding.SCHEDULE_TILES


def test_select_degenerate_shapes():
    assert cfg(0, 128, 128)["num_units"] == 0
    assert cfg(128, 0, 128)["grid"] == 0
    c = cfg(1, 1, 1)
    assert c["num_tiles"] == 1 and c["split_k"] == 1 and c["grid"] == 1


def test_plan_creation_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = lib.bwgemm_create_plan(ctypes.byref(h), 0, None)
    assert rc in (NODEV, CUDA) and not h.value
    assert lib.bwgemm_destroy(None) == OK
    assert lib.bwgemm_run(None, A0, B0, C0, 1, 1, 1, 8, 8, 8, BF16, None) == INVALID
    assert lib.bwgemm_get_status(None, None) == INVALID


@pytest.mark.parametrize("M", [1, 64, 200, 256, 512, 1024, 4096, 8192])
@pytest.mark.parametrize("N", [1024, 5376, 8192, 10240, 28672])
def test_one_unit_variants_get_one_unit_per_worker(M, N):
    """The ring-staged whole-tile variants (224 with 7 stages, 384 with 5) and
    the clustered split-K ones stage their output in the operand rings, which
    is only safe when each worker (CTA pair, or cluster for the split) runs a
    single unit: the planner must never hand them more (the kernels refuse a
    second unit with a status bit)."""
    for K in (5376, 8192):
        for opts in ({}, {"tile_n": 224}, {"tile_n": 384}, {"schedule": binding.SCHEDULE_TILES}):
            try:
                c = cfg(M, N, K, sms=152, pairs=76, quads=36, **opts)
            except binding.BwgemmError:
                continue
            ring_staged = c["split_k"] == 1 and c["variant"] == 2 and (
                (c["tile_n"] == 224 and c["stages"] == 7) or (c["tile_n"] == 384 and c["stages"] == 5))
            if ring_staged:
                assert c["schedule"] == binding.SCHEDULE_TILES and c["sk_tiles"] == 0
                assert c["num_units"] <= c["workers"], (M, N, K, opts, c)
            if c["cluster_split"] == 1:
                # one tile per cluster, one K slice per pair (or CTA) of it
                assert c["split_k"] == 2 and c["workers"] == c["num_tiles"], (M, N, K, opts, c)


def test_noalloc_scratch_stays_inside_the_array(lib):
    """The allocation-free entry point's use of its fixed array, on the host:
    a split cut to one slice writes no counters or partials, every accepted
    call fits both regions, and shapes that do not fit are refused."""
    PART, CTRS = 8 << 20, 64 << 10
    p, c = ctypes.c_uint64(), ctypes.c_uint64()

    def need(M, N, K, S, sms=148, pairs=74):
        rc = lib.bwgemm_noalloc_scratch(sms, pairs, M, N, K, S, ctypes.byref(p), ctypes.byref(c))
        return rc, p.value, c.value

    # K of one 64-wide block: the split is cut to one slice, nothing is cleared
    # (before, this cleared 256 KiB of counters for 4096 tiles into a 64 KiB region)
    assert need(16384, 16384, 64, 2) == (OK, 0, 0)
    assert need(256, 512, 64, 4) == (OK, 0, 0)
    # two K blocks: the same tiles now need partials and counters beyond the array
    rc, parts, ctrs = need(16384, 16384, 128, 2)
    assert rc == WORKSPACE and parts > PART and ctrs > CTRS
    # 2 pair tiles x 3 slices x 2 CTAs x 128 x 256 fp32; 2 tiles x 2 CTAs x 8 warps counters
    assert need(256, 512, 1600, 3) == (OK, 2 * 3 * 2 * 128 * 256 * 4, 2 * 2 * 8 * 4)
    assert need(0, 512, 1600, 3) == (OK, 0, 0) and need(256, 512, 0, 3) == (OK, 0, 0)
    for M in (1, 100, 256, 300, 1000, 4096):
        for N in (64, 264, 1024, 8192):
            for K in (16, 64, 65, 1000, 8192):
                for S in (2, 3, 8, 16):
                    rc, parts, ctrs = need(M, N, K, S)
                    assert rc in (OK, WORKSPACE), (M, N, K, S, rc)
                    if rc == OK:
                        assert parts <= PART and ctrs <= CTRS, (M, N, K, S, parts, ctrs)
                    if K <= 64:
                        assert (parts, ctrs) == (0, 0), (M, N, K, S)
    assert lib.bwgemm_noalloc_scratch(148, 74, 256, 512, 1600, 1, ctypes.byref(p), ctypes.byref(c)) == INVALID
    assert lib.bwgemm_noalloc_scratch(148, 74, 256, 512, 1600, 17, ctypes.byref(p), ctypes.byref(c)) == INVALID
    assert lib.bwgemm_noalloc_scratch(148, 74, 256, 512, 1600, 2, None, ctypes.byref(c)) == INVALID


def test_bench_load_path_rejects_bad_arguments(lib):
    # argument checks come before any device access (no GPU needed)
    gbs, ms = ctypes.c_double(), ctypes.c_double()
    for layout, source, ctas, stages, kblocks in ((8, 0, 0, 6, 64), (6, 0, 0, 4, 64), (-1, 0, 0, 6, 64), (0, 2, 0, 6, 64),
                                                  (0, -1, 0, 6, 64), (0, 0, -1, 6, 64), (0, 0, 0, 0, 64),
                                                  (0, 0, 0, 7, 64), (0, 0, 0, 6, 0)):
        assert lib.bwgemm_bench_load_path(0, layout, source, ctas, stages, kblocks, ctypes.byref(gbs),
                                          ctypes.byref(ms)) == INVALID
    assert lib.bwgemm_bench_load_path(0, 0, 0, 0, 6, 64, None, ctypes.byref(ms)) == INVALID


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_tuned_table_entries_apply(tmp_path):
    """The planner's table lookup (csrc/planner.cpp) compiled on the host with a
    substitute table of one entry: the entry applies to its exact shape when
    the options it sets are automatic, not when the caller set one of them,
    not with tuned_table = 1, and not to other shapes."""
    csrc = os.path.join(ROOT, "dense_gemm_blackwell_03_gb300", "csrc")
    cuda_inc = "/usr/local/cuda/include"
    if not os.path.exists(os.path.join(cuda_inc, "cuda.h")):
        pytest.skip("needs the CUDA headers")
    table = tmp_path / "tuned_table.h"
    table.write_text(
        "#pragma once\n#include <cstdint>\nnamespace bwgemm {\n"
        "struct TunedEntry { int64_t M, N, K; int32_t variant, tile_n, split_k, schedule, copy_kblocks,"
        " cluster_split, raster_group, swap_ab, multicast, skinny; };\n"
        "constexpr TunedEntry kTunedTable[] = {\n"
        "  {4096, 4096, 4096, 2, 224, 0, 0, 0, 0, 4, 1, 0, 0},\n"
        "  {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0},\n};\n}\n")
    main = tmp_path / "main.cpp"
    main.write_text(
        '#include <cstdio>\n#include "bwgemm.h"\n'
        "static void show(int64_t M, int table, int tile) {\n"
        "  bwgemm_plan_options_t o; bwgemm_default_options(&o); o.tuned_table = table; o.tile_n = tile;\n"
        "  bwgemm_config_t c; int st = bwgemm_select_config(148, 74, 36, M, 4096, 4096, BWGEMM_BF16, &o, &c);\n"
        '  printf("%d %d %d %d\\n", st, c.tile_n, c.raster_group, c.tuned);\n}\n'
        "int main() { show(4096, 0, 0); show(4096, 1, 0); show(4096, 0, 256); show(4000, 0, 0); return 0; }\n")
    # a copy of planner.cpp beside the substitute table (a quoted include looks
    # in the including file's own directory first)
    shutil.copy(os.path.join(csrc, "planner.cpp"), tmp_path / "planner.cpp")
    exe = tmp_path / "planner_test"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", csrc, "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, str(tmp_path / "planner.cpp"), str(main), "-o", str(exe)],
                   check=True, capture_output=True)
    got = [tuple(int(x) for x in line.split())
           for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()]
    assert got[0] == (0, 224, 4, 1)     # the entry: tile 224, raster group 4
    assert got[1][1:] == (256, 16, 0)   # rules only (4096^3: every row block of a column first)
    assert got[2][1:] == (256, 16, 0)   # the caller set tile_n: the entry does not apply
    assert got[3][3] == 0               # another shape


def test_tune_table_header_and_options():
    from dense_gemm_blackwell_03_gb300 import tune_table
    rows = [
        {"shape": "a", "M": 256, "N": 8192, "K": 8192, "gain": 1.03, "rules_us": 32.0, "tuned_us": 31.07,
         "options": {"variant": 2, "tile_n": 224, "split_k": 2, "schedule": 1, "copy_kblocks": 1,
                     "cluster_split": 1, "raster_group": 1, "swap_ab": 1, "multicast": 1, "skinny": 0}},
        {"shape": "b", "M": 1, "N": 8192, "K": 8192, "gain": 1.005, "rules_us": 27.0, "tuned_us": 26.9,
         "options": {"variant": 1, "tile_n": 64, "split_k": 2, "schedule": 1, "copy_kblocks": 1,
                     "cluster_split": 2, "raster_group": 4, "swap_ab": 2, "multicast": 1, "skinny": 0}},
        {"shape": "c", "M": 4096, "N": 4096, "K": 4096, "gain": 1.0, "same": True, "options": None},
    ]
    text = tune_table.header_text(rows)
    assert "{256, 8192, 8192, 2, 224, 2, 1, 1, 1, 1, 1, 1, 0},  // a:" in text
    assert "{1, 8192, 8192" not in text and "{4096" not in text  # below the gain bar / same
    assert text.rstrip().endswith("}  // namespace bwgemm")
    # the options that reproduce a configuration, checked through the host planner
    for M, N, K in ((256, 8192, 8192), (16, 8192, 8192), (4096, 4096, 4096), (512, 8192, 5376)):
        cfg = binding.select_config(148, M, N, K, max_pairs=74, max_quads=36)
        again = binding.select_config(148, M, N, K, max_pairs=74, max_quads=36, tuned_table=1,
                                      **tune_table.options_of(cfg))
        assert tune_table.same_config(cfg, again), (M, N, K)


def test_select_raster_group_by_operand_size():
    # operands within half the L2: walk every row block of a column first;
    # larger ones: groups of 8 row blocks
    assert binding.select_config(148, 4096, 4096, 4096, max_pairs=74)["raster_group"] == 16
    assert binding.select_config(148, 8192, 8192, 8192, max_pairs=74)["raster_group"] == 8
    assert binding.select_config(148, 8192, 28672, 8192, max_pairs=74)["raster_group"] == 8
    assert binding.select_config(148, 2048, 2048, 2048, max_pairs=74)["raster_group"] == 8  # 8 row blocks
    assert binding.select_config(148, 4096, 4096, 4096, max_pairs=74, raster_group=4)["raster_group"] == 4


def test_select_whole_k_kernel_for_a_few_rows():
    # M <= 64 rows of A (operands swapped): 64 weight rows per CTA (MMA M = 64),
    # the rows of A as the MMA's N rounded up to 16 / 32 / 64, whole K, one wave
    # (more than 32 rows: CTA pairs, M = 128 across the pair, each CTA copying
    # half of A's rows)
    for M, bn in ((1, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64)):
        cg = 2 if bn == 64 else 1
        c = cfg(M, 8192, 8192, sms=152, pairs=76)
        assert c["skinny"] == 1 and c["swap_ab"] == 1 and c["variant"] == cg
        assert (c["tile_m"], c["tile_n"], c["split_k"]) == (64 * cg, bn, 1)
        assert c["grid"] == 128 and c["num_tiles"] == 128 // cg and c["workspace_bytes"] == 0
        # stages of four K blocks (three for a pair) in about 216 KiB: 40, 48
        # or 36 KiB per CTA
        assert (c["stages"], c["copy_kblocks"]) == {16: (5, 4), 32: (4, 4), 64: (6, 3)}[bn]
    # pairs: 76 fit on 152 SMs (N = 9728), 77 do not
    assert cfg(64, 9728, 8192, sms=152, pairs=76)["skinny"] == 1
    assert cfg(64, 9856, 8192, sms=152, pairs=76)["skinny"] == 0
    assert cfg(64, 9728, 8192, sms=152, pairs=70)["skinny"] == 0
    # ragged N: the last CTA's weight rows past N are zero-filled and not stored
    assert cfg(16, 1100, 4096, sms=152, pairs=76)["grid"] == 18
    # fewer whole K chunks than a stage holds: one K block per stage
    assert cfg(16, 1100, 200, sms=152, pairs=76)["copy_kblocks"] == 1
    assert cfg(64, 1100, 200, sms=152, pairs=76)["copy_kblocks"] == 3
    assert cfg(64, 1100, 128, sms=152, pairs=76)["copy_kblocks"] == 1
    # more tiles than SMs, or more than 64 rows: the main kernel
    assert cfg(16, 28672, 8192, sms=152, pairs=76)["skinny"] == 0
    assert cfg(200, 8192, 8192, sms=152, pairs=76)["skinny"] == 0
    # an option only the main kernel has keeps it; skinny = 2 requires the whole-K form
    assert cfg(16, 8192, 8192, sms=152, pairs=76, split_k=2)["skinny"] == 0
    assert cfg(16, 8192, 8192, sms=152, pairs=76, skinny=1)["skinny"] == 0
    assert cfg(16, 8192, 8192, sms=152, pairs=76, skinny=2, split_k=2)["skinny"] == 1
    with pytest.raises(binding.BwgemmError):
        cfg(200, 8192, 8192, sms=152, pairs=76, skinny=2)
    with pytest.raises(binding.BwgemmError):
        cfg(16, 8192, 8192, skinny=3)



def test_select_whole_k_pair_kernel():
    # 129..256 rows of A, operands in order: all rows on the MMA's M side (256
    # over a pair), the narrowest block of weight rows (96, 112, ... 192) whose
    # blocks fit the 76 pairs once; stages of two K blocks in about 224 KiB
    for M in (129, 200, 256):
        c = cfg(M, 8192, 8192, sms=152, pairs=76, wholek=2)
        assert c["wholek"] == 1 and c["variant"] == 2 and (c["tile_m"], c["tile_n"]) == (256, 112)
        assert c["num_tiles"] == 74 and c["grid"] == 148 and c["split_k"] == 1
        assert c["stages"] == 4 and c["copy_kblocks"] == 2 and c["workspace_bytes"] == 0
    assert cfg(256, 6144, 4096, sms=152, pairs=76, wholek=2)["tile_n"] == 96   # 64 blocks
    assert cfg(256, 12288, 4096, sms=152, pairs=76, wholek=2)["tile_n"] == 192  # 64 blocks
    with pytest.raises(binding.BwgemmError):  # 74 pairs do not fit 140 CTAs
        cfg(256, 8192, 4096, sms=152, pairs=76, wholek=2, max_ctas=140)
    assert cfg(256, 8192, 100, sms=152, pairs=76, wholek=2)["copy_kblocks"] == 1  # one whole chunk
    # automatic only where the main kernel would take a tile wider than 256
    assert cfg(256, 8192, 8192, sms=152, pairs=76, quads=36)["wholek"] == 0
    assert cfg(200, 10240, 8192, sms=152, pairs=76, quads=36)["wholek"] == 1
    assert cfg(256, 12288, 8192, sms=152, pairs=76, quads=36)["wholek"] == 0  # 256-wide main tiles
    # an option only the main kernel has keeps it; wholek = 1 turns it off
    assert cfg(256, 10240, 8192, sms=152, pairs=76, quads=36, tile_n=320)["wholek"] == 0
    assert cfg(256, 10240, 8192, sms=152, pairs=76, quads=36, wholek=1)["wholek"] == 0
    # outside its range wholek = 2 is refused
    for M, N in ((128, 8192), (257, 8192), (256, 28672)):
        with pytest.raises(binding.BwgemmError):
            cfg(M, N, 8192, sms=152, pairs=76, wholek=2)
    with pytest.raises(binding.BwgemmError):
        cfg(256, 8192, 8192, sms=152, pairs=76, wholek=3)
