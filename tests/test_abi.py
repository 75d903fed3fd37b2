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
        '  printf("%zu %zu %zu %zu\\n", sizeof(bwgemm_plan_options_t), '
        "offsetof(bwgemm_plan_options_t, timeout_ns), sizeof(bwgemm_config_t), "
        "offsetof(bwgemm_config_t, workspace_bytes));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got == [ctypes.sizeof(PlanOptions), PlanOptions.timeout_ns.offset,
                   ctypes.sizeof(Config), Config.workspace_bytes.offset]


def test_version_and_status_strings(lib):
    assert lib.bwgemm_version() == (0 << 16) | 1
    for code in range(8):
        assert lib.bwgemm_status_string(code)
    assert lib.bwgemm_status_string(99) == b"unknown status"


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


def cfg(M, N, K, sms=148, pairs=0, **opts):
    return binding.select_config(sms, M, N, K, max_pairs=pairs, **opts)


def test_select_square_uses_cta_pairs():
    c = cfg(4096, 4096, 4096, sms=152, pairs=76)
    assert c["variant"] == 2 and c["tile_m"] == 256 and c["tile_n"] == 256
    assert c["num_tiles"] == 16 * 16 and c["split_k"] == 1
    assert c["grid"] == 2 * 76 and c["tile_k"] == 64 and c["stages"] == 6


def test_select_small_m_uses_single_cta_tiles():
    c = cfg(64, 8192, 8192, sms=152, pairs=76)
    assert c["variant"] == 1 and c["tile_m"] == 128
    assert c["num_tiles"] == 32
    # few tiles: K is split so that tiles x splits fills the GPU
    assert c["split_k"] == 4 and c["num_units"] == 128 and c["grid"] == 128


def test_select_decode_splits_k():
    c = cfg(256, 8192, 8192, sms=152, pairs=76)
    assert c["variant"] == 2 and c["num_tiles"] == 32 and c["split_k"] == 2
    assert c["num_units"] == 64 and c["grid"] == 128
    assert c["workspace_bytes"] == (1 << 20) + 32 * 2 * 2 * 128 * 256 * 4


def test_select_forced_options():
    c = cfg(1024, 1024, 4096, variant=1, tile_n=128, split_k=3, raster_group=4, max_ctas=64)
    assert (c["variant"], c["tile_m"], c["tile_n"], c["stages"]) == (1, 128, 128, 6)
    assert c["split_k"] == 3 and c["raster_group"] == 4 and c["grid"] == 64
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
        cfg(256, 8192, 8192, split_k=4, workspace_bytes=1 << 20)
    assert e.value.status == WORKSPACE


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
