"""GPU parity: the sm_103a kernels through the C ABI against the CPU oracle.

Small shapes are compared element by element over the whole output; the
pages' full-size shapes (4096^3, Llama-3-70B prefill and decode linears,
Gemma-3-27B-like and small-M tails) are compared on a seeded sample of 64
full rows and 64 full columns of C, in the configuration the benchmark times.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_blackwell_03_gb300 import binding
from dense_gemm_blackwell_03_gb300.workloads import SHAPES, bits_of, make_inputs, make_matrix
from parity import compare, sample_indices

pytestmark = pytest.mark.gpu

TORCH16 = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module")
def plan():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load_library(build_if_missing=True)
    p = binding.Plan(0)
    yield p
    assert p.status() == 0
    p.close()


def run_full(plan, A, B, dtype, exact=False, out=None):
    C = plan.gemm(A, B, out=out)
    assert plan.status() == 0
    ref = oracle.gemm(bits_of(A), bits_of(B), dtype)
    return compare(bits_of(C), ref, dtype, A.shape[1], exact=exact), C


# ---------------------------------------------------------------- small shapes
@pytest.mark.parametrize("variant", [1, 2])
def test_square512_integers_bit_exact(variant):
    s = SHAPES["square512_int"]
    A, B = make_inputs(s, device="cuda")
    with binding.Plan(0, variant=variant) as p:
        run_full(p, A, B, "bf16", exact=True)
        assert p.last_config()["variant"] == variant


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_square512_normal(plan, dtype):
    s = SHAPES["square512"].with_dtype(dtype)
    A, B = make_inputs(s, device="cuda")
    run_full(plan, A, B, dtype)


@pytest.mark.parametrize("K", [16, 32, 48, 64, 80, 200, 1000])
def test_k_steps_and_k_tails(plan, K):
    # the first MMA overwrites the accumulator, later ones add (K = 16: one
    # instruction); K not a multiple of 64 reads zeros past the end
    A = make_matrix(256, K, "int2", seed=100 + K, device="cuda")
    B = make_matrix(192, K, "int2", seed=200 + K, device="cuda")
    run_full(plan, A, B, "bf16", exact=True)


@pytest.mark.parametrize("M", [1, 16, 64, 127, 129, 200, 255, 257, 300])
def test_m_tails(plan, M):
    A = make_matrix(M, 512, "int2", seed=300 + M, device="cuda")
    B = make_matrix(320, 512, "int2", seed=400 + M, device="cuda")
    run_full(plan, A, B, "bf16", exact=True)


@pytest.mark.parametrize("N", [8, 40, 136, 264, 1000])
def test_n_tails(plan, N):
    A = make_matrix(384, 256, "normal", seed=500 + N, device="cuda")
    B = make_matrix(N, 256, "normal", seed=600 + N, device="cuda")
    run_full(plan, A, B, "bf16")


def test_strided_operands_and_output(plan):
    M, N, K = 300, 200, 328
    A = make_matrix(M, K, "int2", seed=701, device="cuda", ld=K + 24)
    B = make_matrix(N, K, "int2", seed=702, device="cuda", ld=K + 8)
    Cbuf = torch.full((M, N + 40), 7.0, dtype=torch.bfloat16, device="cuda")
    C = Cbuf[:, :N]
    run_full(plan, A, B, "bf16", exact=True, out=C)
    assert torch.all(Cbuf[:, N:] == 7.0), "wrote outside the output view"


@pytest.mark.parametrize("variant,tile_n", [(1, 128), (1, 256), (2, 128), (2, 224), (2, 256), (2, 320),
                                            (2, 384)])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_every_variant(variant, tile_n, dtype):
    A = make_matrix(520, 640, "normal", dtype, seed=800, device="cuda")
    B = make_matrix(600, 640, "normal", dtype, seed=801, device="cuda")
    with binding.Plan(0, variant=variant, tile_n=tile_n) as p:
        run_full(p, A, B, dtype)
        c = p.last_config()
        assert (c["variant"], c["tile_n"]) == (variant, tile_n)


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("split", [2, 3, 5])
def test_split_k_exact_and_deterministic(variant, split):
    A = make_matrix(256, 1600, "int2", seed=900, device="cuda")
    B = make_matrix(512, 1600, "int2", seed=901, device="cuda")
    with binding.Plan(0, variant=variant, split_k=split) as p:
        _, C1 = run_full(p, A, B, "bf16", exact=True)
        assert p.last_config()["split_k"] == split
        C2 = p.gemm(A, B)
        assert p.status() == 0
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("split,max_ctas", [(2, 0), (3, 0), (4, 0), (3, 4), (4, 6)])
def test_split_k_reduce_scatter_and_multi_wave(variant, split, max_ctas):
    # max_ctas = 0: every slice of every tile in one wave (reduce-scatter);
    # a small grid forces several waves, where slices may not wait on each other
    A = make_matrix(300, 2048, "int2", seed=950 + split, device="cuda")
    B = make_matrix(520, 2048, "int2", seed=960 + split, device="cuda")
    with binding.Plan(0, variant=variant, split_k=split, max_ctas=max_ctas) as p:
        _, C1 = run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["split_k"] == split
        assert c["split_scatter"] == (1 if max_ctas == 0 else 0)
        C2 = p.gemm(A, B)
        assert p.status() == 0
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


@pytest.mark.parametrize("variant,tile_n", [(1, 64), (1, 128), (2, 64), (2, 128)])
@pytest.mark.parametrize("M,N,K,opts", [
    (1, 1000, 520, {}),                          # one row of A, ragged N and K
    (37, 2056, 1040, {}),                         # ragged everything
    (200, 1536, 2048, {"split_k": 2}),            # one-wave split-K on swapped tiles
    (64, 4096, 4096, {"schedule": 2}),            # stream-K on swapped tiles
    (130, 3072, 1024, {"split_k": 3, "max_ctas": 4}),  # multi-wave split-K
])
def test_swapped_operands_exact(variant, tile_n, M, N, K, opts):
    # C^T = B A^T on the tensor cores, each accumulator box stored transposed
    A = make_matrix(M, K, "int2", seed=1900 + M, device="cuda")
    B = make_matrix(N, K, "int2", seed=2000 + N, device="cuda")
    with binding.Plan(0, variant=variant, tile_n=tile_n, swap_ab=2, **opts) as p:
        run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["swap_ab"] == 1 and c["tile_n"] == tile_n


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_swapped_operands_normal_inputs(dtype):
    A = make_matrix(96, 4096, "normal", dtype, seed=2100, device="cuda")
    B = make_matrix(3000, 4096, "weight", dtype, seed=2101, device="cuda")
    Cbuf = torch.full((96, 3008), 3.0, dtype=TORCH16[dtype], device="cuda")
    with binding.Plan(0, swap_ab=2) as p:  # 96 rows: above the automatic swap bound
        run_full(p, A, B, dtype, out=Cbuf[:, :3000])
        assert p.last_config()["swap_ab"] == 1
    assert torch.all(Cbuf[:, 3000:] == 3.0)


@pytest.mark.parametrize("variant,tile_n,swap", [(1, 256, 1), (1, 128, 1), (2, 256, 1),
                                                 (2, 128, 1), (1, 64, 2), (2, 128, 2)])
def test_cluster_launch_control_exact(variant, tile_n, swap):
    # many more tiles than co-resident clusters: most tiles are taken over
    # from cancelled cluster launches
    M, N, K = (4096, 2048, 192) if swap == 1 else (40, 16384, 192)
    A = make_matrix(M, K, "int2", seed=2200 + variant, device="cuda")
    B = make_matrix(N, K, "int2", seed=2300 + tile_n, device="cuda")
    with binding.Plan(0, variant=variant, tile_n=tile_n, swap_ab=swap,
                      schedule=binding.SCHEDULE_CLC) as p:
        for _ in range(2):
            run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["schedule"] == binding.SCHEDULE_CLC and c["grid"] == c["num_tiles"] * variant


def test_cluster_launch_control_normal_inputs():
    A = make_matrix(2000, 1000, "normal", seed=2400, device="cuda")
    B = make_matrix(3000, 1000, "normal", seed=2401, device="cuda")
    with binding.Plan(0, schedule=binding.SCHEDULE_CLC) as p:
        run_full(p, A, B, "bf16")


@pytest.mark.parametrize("opts", [dict(variant=2), dict(variant=1), dict(multicast=2),
                                  dict(swap_ab=2), dict(variant=2, split_k=2),
                                  dict(schedule=binding.SCHEDULE_STREAM_K)])
@pytest.mark.parametrize("N", [1300, 1297])
def test_columns_past_n_untouched(opts, N):
    # N not a multiple of 8: the last 16-byte chunk of each row of C straddles
    # the end of the row; the columns after N belong to the caller
    M, K = 200, 320
    A = make_matrix(M, K, "int2", seed=2900, device="cuda")
    B = make_matrix(N, K, "int2", seed=2901, device="cuda")
    C = torch.full((M, 1320), 7.0, dtype=torch.bfloat16, device="cuda")
    with binding.Plan(0, **opts) as p:
        run_full(p, A, B, "bf16", exact=True, out=C[:, :N])
    assert torch.all(C[:, N:] == 7.0)


# ------------------------------------- two K blocks per TMA copy (3-D operand views)
@pytest.mark.parametrize("K", [64, 128, 192, 200, 1000, 1088])
@pytest.mark.parametrize("opts", [dict(variant=2), dict(variant=1), dict(variant=1, tile_n=128),
                                  dict(variant=2, tile_n=128), dict(multicast=2),
                                  dict(schedule=binding.SCHEDULE_STREAM_K, max_ctas=24),
                                  dict(variant=2, split_k=3, schedule=binding.SCHEDULE_TILES)])
def test_paired_kblock_copies_exact(opts, K):
    # one chunk (no pairs), pairs only, pairs + a single, + a ragged tail;
    # stream-K and split-K units start at odd K blocks and odd ring stages
    A = make_matrix(520, K, "int2", seed=3000 + K, device="cuda")
    B = make_matrix(696, K, "int2", seed=3100 + K, device="cuda")
    outs = []
    for copy_kblocks in (1, 2):
        with binding.Plan(0, copy_kblocks=copy_kblocks, **opts) as p:
            _, C = run_full(p, A, B, "bf16", exact=True)
            outs.append(C.clone())
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("prefetch,opts", [(4, dict()), (3, dict(copy_kblocks=2)), (8, dict(swap_ab=2)),
                                           (6, dict(multicast=2)), (5, dict(schedule=binding.SCHEDULE_STREAM_K))])
def test_l2_prefetch_exact(prefetch, opts):
    # the prefetch stream of the operand with more rows (2-D or 3-D boxes)
    # changes no result
    A = make_matrix(264, 1000, "int2", seed=3300, device="cuda")
    B = make_matrix(2000, 1000, "int2", seed=3301, device="cuda")
    with binding.Plan(0, prefetch=prefetch, **opts) as p:
        run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["prefetch_kblocks"] == prefetch and c["prefetch_b"] == (0 if c["swap_ab"] else 1)


@pytest.mark.parametrize("swap", [2])
def test_paired_kblock_copies_swapped(swap):
    A = make_matrix(40, 1000, "int2", seed=3200, device="cuda")
    B = make_matrix(3000, 1000, "int2", seed=3201, device="cuda")
    with binding.Plan(0, swap_ab=swap, copy_kblocks=2) as p:
        run_full(p, A, B, "bf16", exact=True)
        assert p.last_config()["swap_ab"] == 1 and p.last_config()["copy_kblocks"] == 2


# ------------------------------------------------------------------ tuning
def test_tune_keeps_a_valid_config_per_shape():
    A = make_matrix(520, 1000, "int2", seed=3700, device="cuda")
    B = make_matrix(696, 1000, "int2", seed=3701, device="cuda")
    C = torch.full((520, 696), 5.0, dtype=torch.bfloat16, device="cuda")
    with binding.Plan(0) as p:
        best = p.tune(A, B, out=C, iters=3)
        assert p.tuned_count() == 1 and best["grid"] > 0
        ref = oracle.gemm(bits_of(A), bits_of(B), "bf16")
        compare(bits_of(C), ref, "bf16", 1000, exact=True)  # C holds the product
        # later runs of this shape use the tuned configuration
        run_full(p, A, B, "bf16", exact=True)
        got = p.last_config()
        assert {k: got[k] for k in best} == best
        # another shape is not affected; re-tuning replaces the entry
        A2 = make_matrix(256, 512, "int2", seed=3702, device="cuda")
        run_full(p, A2, B[:, :512].contiguous(), "bf16", exact=True)
        p.tune(A, B, out=C, iters=2)
        assert p.tuned_count() == 1


def test_tune_rejects_bad_arguments():
    A = make_matrix(64, 64, "int2", seed=3703, device="cuda")
    with binding.Plan(0) as p:
        with pytest.raises(binding.BwgemmError):
            p.tune(A, A, iters=0)
        C = torch.empty((64, 60), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(binding.BwgemmError):
            p.tune(A, A[:60].contiguous(), out=C[:, :60], iters=1)  # ldc 60: misaligned


# ------------------------------------------- 224-column tiles of the pair form
@pytest.mark.parametrize("M,N,K", [(256, 2048, 1024), (200, 1000, 1000), (500, 3000, 640),
                                   (40, 1800, 1088)])
@pytest.mark.parametrize("opts", [
    dict(schedule=binding.SCHEDULE_TILES),                                  # whole tiles
    dict(schedule=binding.SCHEDULE_TILES, copy_kblocks=2),
    dict(split_k=2, cluster_split=1, schedule=binding.SCHEDULE_TILES),      # slices through L2
    dict(split_k=2, cluster_split=2, schedule=binding.SCHEDULE_TILES),      # slices in one cluster
    dict(split_k=3, schedule=binding.SCHEDULE_TILES),
    dict(schedule=binding.SCHEDULE_STREAM_K, max_ctas=24),
    dict(schedule=binding.SCHEDULE_CLC),
])
@pytest.mark.parametrize("tile_n", [224, 320, 384])
def test_wide_tiles_exact(M, N, K, opts, tile_n):
    # 224: 7 store chunks of 32 columns per tile (an odd count: the two K
    # slices of a cluster own 4 and 3 of them), the second accumulator at TMEM
    # column 256.  320: two MMAs per K step (N = 256 and N = 64) into one
    # accumulator, its chunks mapped back to the tile's columns.  Ragged M, N
    # and K; integer inputs, run twice.  384: N = 256 and N = 128, no
    # clustered split form.
    if tile_n == 384 and opts.get("cluster_split") == 2:
        pytest.skip("no clustered split-K form of 384-column units")
    A = make_matrix(M, K, "int2", seed=3700 + M, device="cuda")
    B = make_matrix(N, K, "int2", seed=3710 + N, device="cuda")
    with binding.Plan(0, variant=2, tile_n=tile_n, swap_ab=1, **opts) as p:
        for _ in range(2):
            run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["tile_n"] == tile_n and c["variant"] == 2
        if opts.get("cluster_split") == 2:
            assert c["cluster_split"] == 1


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_tile320_auto_qkv_family(dtype):
    # the main kernel's choice for one row block over N = 10240 (32 tiles of
    # 320, two K slices each in one cluster; the planner's default there is the
    # whole-K pair kernel, turned off here) on N(0,1) activations and
    # N(0, 0.02^2) weights
    A = make_matrix(256, 1024, "normal", dtype, seed=3730, device="cuda")
    B = make_matrix(10240, 1024, "weight", dtype, seed=3731, device="cuda")
    with binding.Plan(0, wholek=1) as p:
        run_full(p, A, B, dtype)
        c = p.last_config()
        assert c["tile_n"] == 320 and c["num_tiles"] == 32 and c["split_k"] == 2
    with binding.Plan(0) as p:  # the default: 72 blocks of 144 weight rows, whole K
        run_full(p, A, B, dtype)
        c = p.last_config()
        assert c["wholek"] == 1 and c["tile_n"] == 144 and c["num_tiles"] == 72


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_tile384_auto_mlp_up_family(dtype):
    # the planner's choice for one row block over N = 28672 (75 whole tiles
    # of 384, one wave) on N(0,1) activations and N(0, 0.02^2) weights
    A = make_matrix(256, 512, "normal", dtype, seed=3740, device="cuda")
    B = make_matrix(28672, 512, "weight", dtype, seed=3741, device="cuda")
    with binding.Plan(0) as p:
        run_full(p, A, B, dtype)
        c = p.last_config()
        assert c["tile_n"] == 384 and c["num_tiles"] == 75 and c["split_k"] == 1


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_tile224_auto_two_row_blocks(dtype):
    # the planner's choice for two row blocks over N = 8192 (2 x 37 whole
    # tiles of 224 on 74 of 76 pairs) on N(0,1) activations and N(0, 0.02^2)
    # weights
    A = make_matrix(512, 512, "normal", dtype, seed=3720, device="cuda")
    B = make_matrix(8192, 512, "weight", dtype, seed=3721, device="cuda")
    with binding.Plan(0) as p:
        run_full(p, A, B, dtype)
        c = p.last_config()
        assert c["tile_n"] == 224 and c["num_tiles"] == 74 and c["split_k"] == 1


# ------------------------------ split-K slices exchanging in distributed shared memory
@pytest.mark.parametrize("M,N,K", [(256, 2048, 1024), (200, 2048, 1000), (130, 1024, 520),
                                   (16, 4096, 512), (40, 2048, 1088), (1, 2048, 640)])
def test_cluster_split_exact(M, N, K):
    # two K slices of each tile in one cluster against the same split through
    # L2: identical bits (a sum of two terms); padding rows past M take part
    A = make_matrix(M, K, "int2", seed=3400 + M, device="cuda")
    B = make_matrix(N, K, "int2", seed=3500 + N, device="cuda")
    outs = []
    for mode in (1, 2):
        with binding.Plan(0, split_k=2, cluster_split=mode, schedule=binding.SCHEDULE_TILES) as p:
            for _ in range(2):
                _, C = run_full(p, A, B, "bf16", exact=True)
            c = p.last_config()
            assert c["cluster_split"] == (1 if mode == 2 else 0) and c["split_k"] == 2
            outs.append(C.clone())
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_cluster_split_normal_inputs(dtype):
    A = make_matrix(256, 4096, "normal", dtype, seed=3600, device="cuda")
    B = make_matrix(3072, 4096, "weight", dtype, seed=3601, device="cuda")
    with binding.Plan(0, cluster_split=2, split_k=2, schedule=binding.SCHEDULE_TILES) as p:
        run_full(p, A, B, dtype)
        assert p.last_config()["cluster_split"] == 1


# ------------------------------------------------- A multicast across two pairs
@pytest.mark.parametrize("M,N,K", [(512, 1024, 192), (300, 768, 200), (1000, 1300, 520),
                                   (256, 256, 64)])
@pytest.mark.parametrize("tile_n", [256, 128])
def test_multicast_integers_exact(M, N, K, tile_n):
    # ragged M / N / K; an odd count of column blocks leaves the second pair
    # of the last group on padding columns (its boxes are never stored)
    ldc = (N + 7) // 8 * 8
    A = make_matrix(M, K, "int2", seed=2500 + M, device="cuda")
    B = make_matrix(N, K, "int2", seed=2600 + N, device="cuda")
    C = torch.full((M, ldc), 7.0, dtype=torch.bfloat16, device="cuda")
    with binding.Plan(0, multicast=2, tile_n=tile_n, schedule=binding.SCHEDULE_TILES) as p:
        for _ in range(2):
            run_full(p, A, B, "bf16", exact=True, out=C[:, :N])
        c = p.last_config()
        assert c["multicast"] == 2 and c["grid"] % 4 == 0
    assert torch.all(C[:, N:] == 7.0)


@pytest.mark.parametrize("schedule,split_k", [(binding.SCHEDULE_STREAM_K, 0),
                                              (binding.SCHEDULE_TILES, 3),
                                              (binding.SCHEDULE_CLC, 0)])
def test_multicast_schedules_exact(schedule, split_k):
    A = make_matrix(1536, 1024, "int2", seed=2700, device="cuda")
    B = make_matrix(2560, 1024, "int2", seed=2701, device="cuda")
    with binding.Plan(0, multicast=2, schedule=schedule, split_k=split_k, max_ctas=40) as p:
        for _ in range(2):
            run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["multicast"] == 2 and c["schedule"] == schedule
        if split_k:
            assert c["split_k"] == split_k
        if schedule == binding.SCHEDULE_STREAM_K:
            assert c["sk_tiles"] > 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_multicast_normal_inputs(dtype):
    A = make_matrix(2000, 1000, "normal", dtype, seed=2800, device="cuda")
    B = make_matrix(3000, 1000, "weight", dtype, seed=2801, device="cuda")
    with binding.Plan(0, multicast=2) as p:
        run_full(p, A, B, dtype)


def test_split_k_normal_inputs():
    A = make_matrix(200, 4096, "normal", seed=910, device="cuda")
    B = make_matrix(384, 4096, "weight", seed=911, device="cuda")
    with binding.Plan(0, split_k=4) as p:
        run_full(p, A, B, "bf16")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("M,N,K,max_ctas", [
    (512, 512, 512, 0),       # fewer tiles than workers: every tile split across workers
    (1024, 1024, 1280, 6),    # 16 tiles on 3 pairs / 6 CTAs: whole waves + stream-K tail
    (768, 1280, 4096, 8),     # pieces spanning several tiles per worker
    (5, 768, 2000, 0),        # mostly padding rows: predicated partial traffic
    (130, 264, 1600, 0),      # ragged M, N and K
])
def test_stream_k_exact(variant, M, N, K, max_ctas):
    A = make_matrix(M, K, "int2", seed=1000 + M, device="cuda")
    B = make_matrix(N, K, "int2", seed=1100 + N, device="cuda")
    with binding.Plan(0, variant=variant, schedule=binding.SCHEDULE_STREAM_K,
                      max_ctas=max_ctas) as p:
        _, C1 = run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["schedule"] == binding.SCHEDULE_STREAM_K and c["sk_tiles"] > 0
        C2 = p.gemm(A, B)
        assert p.status() == 0
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))  # deterministic


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_stream_k_normal_inputs(dtype):
    A = make_matrix(1000, 3000, "normal", dtype, seed=1200, device="cuda")
    B = make_matrix(696, 3000, "weight", dtype, seed=1201, device="cuda")
    with binding.Plan(0, schedule=binding.SCHEDULE_STREAM_K, max_ctas=10) as p:
        run_full(p, A, B, dtype)
        assert p.last_config()["dp_tiles"] > 0


def test_schedules_agree_on_integers():
    A = make_matrix(640, 1536, "int2", seed=1300, device="cuda")
    B = make_matrix(896, 1536, "int2", seed=1301, device="cuda")
    outs = []
    for sched in (binding.SCHEDULE_TILES, binding.SCHEDULE_STREAM_K, binding.SCHEDULE_AUTO):
        with binding.Plan(0, schedule=sched) as p:
            outs.append(p.gemm(A, B))
            assert p.status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_without_programmatic_dependent_launch():
    A = make_matrix(512, 512, "int2", seed=1400, device="cuda")
    B = make_matrix(512, 512, "int2", seed=1401, device="cuda")
    with binding.Plan(0, pdl_off=1) as p:
        run_full(p, A, B, "bf16", exact=True)


def test_back_to_back_launches_see_previous_results(plan):
    # with programmatic dependent launch the next GEMM's prologue overlaps the
    # previous one; the chain C1 = A B^T, C2 = C1 B^T must still read finished data
    A = make_matrix(384, 256, "int2", seed=1500, device="cuda")
    B = make_matrix(256, 256, "int2", seed=1501, device="cuda")
    C1 = plan.gemm(A, B)            # 384 x 256, exact small integers
    C2 = plan.gemm(C1, B)           # reads C1 right after it is written
    assert plan.status() == 0
    ref1 = oracle.gemm(bits_of(A), bits_of(B), "bf16")
    compare(bits_of(C1), ref1, "bf16", 256, exact=True)
    ref2 = oracle.gemm(ref1, bits_of(B), "bf16")
    compare(bits_of(C2), ref2, "bf16", 256)


def test_persistent_grid_smaller_than_units():
    # more work units than CTAs: every CTA walks several units, both TMEM
    # accumulators and the ring wrap many times
    A = make_matrix(1024, 512, "int2", seed=920, device="cuda")
    B = make_matrix(1024, 512, "int2", seed=921, device="cuda")
    for variant in (1, 2):
        with binding.Plan(0, variant=variant, max_ctas=6) as p:
            run_full(p, A, B, "bf16", exact=True)
            assert p.last_config()["grid"] == 6


def test_degenerate_shapes(plan):
    A = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(32, 64, dtype=torch.bfloat16, device="cuda")
    assert plan.gemm(A, B).shape == (0, 32)
    n_before = plan.launch_count()
    A = torch.ones(48, 0, dtype=torch.bfloat16, device="cuda")
    B = torch.ones(40, 0, dtype=torch.bfloat16, device="cuda")
    C = torch.full((48, 40), 3.0, dtype=torch.bfloat16, device="cuda")
    plan.gemm(A, B, out=C)  # K = 0: the empty sum
    assert plan.status() == 0
    assert torch.all(C == 0)
    assert plan.launch_count() == n_before  # no GEMM kernel for empty work


def test_rejects_misaligned_on_device(plan):
    A = torch.zeros(64, 72, dtype=torch.bfloat16, device="cuda")[:, 1:]  # base not 16 B aligned
    B = torch.zeros(64, 71, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.BwgemmError) as e:
        plan.gemm(A, B)
    assert e.value.status == 2


def test_rejects_operands_not_on_the_plan_device(plan):
    # pinned host memory is device-accessible, but no tensor map may cover
    # anything but this GPU's own memory: bwgemm_run refuses before encoding
    A = make_matrix(256, 512, "int2", seed=940, device="cuda")
    C = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    hA = torch.zeros(256, 512, dtype=torch.bfloat16).pin_memory()
    hC = torch.zeros(256, 256, dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    n_before = plan.launch_count()
    for a, b, c in ((hA, A, C), (A, hA, C), (A, A, hC)):
        rc = plan.run_raw(a.data_ptr(), b.data_ptr(), c.data_ptr(), 256, 256, 512, 512, 512, 256,
                          binding.BF16, stream)
        assert rc == 1  # BWGEMM_ERR_INVALID_ARG
    assert plan.launch_count() == n_before
    with pytest.raises(ValueError):
        plan.gemm(A, hA)  # the binding names the tensor first
    # device memory of this GPU is accepted, and the product is right
    C = plan.gemm(A, A, out=C)
    assert plan.status() == 0
    compare(bits_of(C), oracle.gemm(bits_of(A), bits_of(A), "bf16"), "bf16", 512, exact=True)


def test_host_buffers_round_trip(plan):
    A = make_matrix(300, 264, "int2", seed=930)
    B = make_matrix(200, 264, "int2", seed=931)
    C = plan.gemm_host(A.pin_memory(), B.pin_memory())
    ref = oracle.gemm(bits_of(A), bits_of(B), "bf16")
    compare(bits_of(C), ref, "bf16", 264, exact=True)


@pytest.mark.parametrize("M,N,K,lda_pad,ldc_pad", [(2000, 2048, 2048, 0, 0), (1536, 2048, 2048, 8, 16),
                                                   (1100, 2048, 2048, 24, 0), (8192, 7800, 512, 0, 8),
                                                   (1024, 1024, 2048, 0, 0)])
def test_host_buffers_pipelined(M, N, K, lda_pad, ldc_pad):
    # calls moving >= 16 MiB run as a pipeline over blocks of C (row blocks of
    # A and, once a block of C holds 64 tiles of 256 x 256, two column blocks
    # of B: A and B in, GEMM, C out on three streams); ragged last row and
    # column blocks, host strides wider than the rows, run twice on one plan
    Abuf = make_matrix(M, K + lda_pad, "int2", seed=940 + M).pin_memory()
    A = Abuf[:, :K]
    B = make_matrix(N, K, "int2", seed=941).pin_memory()
    Cbuf = torch.full((M, N + ldc_pad), 5.0, dtype=torch.bfloat16).pin_memory()
    C = Cbuf[:, :N]
    ref = oracle.gemm(bits_of(A.contiguous()), bits_of(B), "bf16")
    with binding.Plan(0) as p:
        for _ in range(2):
            p.gemm_host(A, B, out=C)
            compare(bits_of(C.contiguous()), ref, "bf16", K, exact=True)
    if ldc_pad:
        assert torch.all(Cbuf[:, N:] == 5.0)


# ------------------------------------------------------- the pages' full shapes
FULL = ["square4096", "square4096_fp16", "prefill_attn_out", "prefill_mlp_up",
        "decode_attn_out", "decode_qkv", "decode_mlp_up", "decode_mlp_down",
        "gemma_512x8192x5376", "tail_m1", "tail_m16", "tail_m64", "tail_m200"]


FULL_FP16 = [n for n in FULL if not n.endswith("_fp16")]


@pytest.mark.parametrize("name,dtype", [(n, None) for n in FULL] + [(n, "fp16") for n in FULL_FP16])
def test_full_shape_sampled(plan, name, dtype):
    # every configuration of the pages' shapes, in bf16 and in fp16
    s = SHAPES[name] if dtype is None else SHAPES[name].with_dtype(dtype)
    A, B = make_inputs(s, device="cuda")
    C = plan.gemm(A, B)
    assert plan.status() == 0
    rows = sample_indices(s.M, 64, seed=1)
    cols = sample_indices(s.N, 64, seed=2)
    a_bits, b_bits = bits_of(A), bits_of(B)
    c_rows = bits_of(C[torch.from_numpy(rows).cuda()])
    c_cols = bits_of(C[:, torch.from_numpy(cols).cuda()])
    ref_rows = oracle.gemm(a_bits, b_bits, s.dtype, rows=rows)
    ref_cols = oracle.gemm(a_bits, b_bits, s.dtype, cols=cols)
    compare(c_rows, ref_rows, s.dtype, s.K)
    compare(c_cols, ref_cols, s.dtype, s.K)


def test_full_square_integers_bit_exact(plan):
    # 4096^3 with integer entries: every partial sum is an exact integer in fp32
    s = SHAPES["square512_int"]
    A = make_matrix(4096, 4096, "int2", seed=940, device="cuda")
    B = make_matrix(4096, 4096, "int2", seed=941, device="cuda")
    C = plan.gemm(A, B)
    assert plan.status() == 0
    rows = sample_indices(4096, 64, seed=3)
    ref = oracle.gemm(bits_of(A), bits_of(B), "bf16", rows=rows)
    compare(bits_of(C[torch.from_numpy(rows).cuda()]), ref, "bf16", 4096, exact=True)
    del s


def test_timeline_trace_is_ordered():
    from dense_gemm_blackwell_03_gb300 import timeline
    A = make_matrix(1024, 2048, "int2", seed=1600, device="cuda")
    B = make_matrix(1536, 2048, "int2", seed=1601, device="cuda")
    with binding.Plan(0, trace=1, max_ctas=16) as p:
        run_full(p, A, B, "bf16", exact=True)
        tr = p.read_trace().astype(np.int64)
        c = p.last_config()
    assert tr.shape == (c["grid"], 64)
    for row in tr:
        e, r, f, l, d, x = (row[i] for i in range(6))
        assert 0 < e <= r <= f <= l <= x and r <= d <= x
    s = timeline.summarize(tr)
    assert s["ctas"] == c["grid"] and s["span_us"] > 0
    assert s["units_per_cta"]["max"] >= 2
    for ulist in timeline.units(tr):
        for ms, me, es, ee in ulist:
            if ms and me:
                assert ms <= me
            if es and ee:
                assert es <= ee


@pytest.mark.parametrize("variant,schedule", [(1, 1), (2, 1), (2, 2)])
def test_bounded_wait_reports_timeout_and_context_survives(variant, schedule):
    # the producer of CTA 0 never fills K block 1 of its first unit: the MMA's
    # wait on that stage runs out after timeout_ns, every role leaves its loop,
    # TMEM is freed and the call reports BWGEMM_ERR_TIMEOUT -- no trap, no hang
    A = make_matrix(512, 1024, "int2", seed=1700, device="cuda")
    B = make_matrix(512, 1024, "int2", seed=1701, device="cuda")
    with binding.Plan(0, variant=variant, schedule=schedule, stall_kblock=1,
                      timeout_ns=200_000_000) as p:
        p.gemm(A, B)
        assert p.status() == 6  # BWGEMM_ERR_TIMEOUT
        assert p.last_device_status() != 0
    # the context is still usable and a normal plan gives exact results
    with binding.Plan(0, variant=variant, schedule=schedule) as p:
        run_full(p, A, B, "bf16", exact=True)


def test_cuda_graph_capture_and_replay():
    # bwgemm_run enqueues one kernel and allocates nothing, so a stream can
    # capture it; replays see the operands' current contents
    A = make_matrix(384, 1024, "int2", seed=1800, device="cuda")
    B = make_matrix(640, 1024, "int2", seed=1801, device="cuda")
    C = torch.empty(384, 640, dtype=torch.bfloat16, device="cuda")
    with binding.Plan(0) as p:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            p.gemm(A, B, out=C, stream=s)  # warm-up launch outside the capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                p.gemm(A, B, out=C, stream=s)
        torch.cuda.synchronize()
        for seed in (1802, 1803):
            A.copy_(make_matrix(384, 1024, "int2", seed=seed, device="cuda"))
            C.fill_(0)
            g.replay()
            torch.cuda.synchronize()
            assert p.status() == 0
            compare(bits_of(C), oracle.gemm(bits_of(A), bits_of(B), "bf16"), "bf16", 1024, exact=True)


def test_probe_tensor_rate():
    """The per-SM tensor rate behind the nominal dense peak: a whole number of
    FLOP per SM clock in a plausible range, on every SM of the device, and a
    nominal peak at the top SM clock that is not below what cuBLAS reaches on
    this part (the measured burst figure, where the driver recorded one)."""
    import json
    import os
    import subprocess
    rate, sms = binding.probe_tensor_rate(0)
    assert sms == torch.cuda.get_device_properties(0).multi_processor_count
    assert 2048.0 <= rate <= 16384.0
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        out = subprocess.run(["nvidia-smi", "--id=0", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=30).stdout.strip()
        max_mhz = float(out.splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        pytest.skip("nvidia-smi clocks unavailable")
    if os.path.exists(path):
        measured = json.load(open(path)).get("bf16_tflops")
        if measured:
            assert sms * rate * max_mhz * 1e6 / 1e12 >= 0.95 * float(measured)


@pytest.mark.parametrize("layout", [0, 1, 2, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("source,ctas", [(0, 0), (1, 0), (1, 64)])
def test_load_path_microbench(layout, source, ctas):
    # the load path alone (no MMA) in each shared-memory layout, from L2 and
    # from HBM: every wait ends, and the landed bytes per second are plausible
    binding.load_library(build_if_missing=True)
    stages, kblocks = (3, 128) if layout >= 6 else (6, 256)
    gbs, ms = binding.bench_load_path(layout, source=source, ctas=ctas, stages=stages, kblocks=kblocks)
    assert ms > 0 and 100.0 < gbs < 200000.0


def test_epilogue_share_of_a_traced_launch():
    from dense_gemm_blackwell_03_gb300 import ablations
    (row,) = ablations.run_epilogue_share(["square512"], warmup=2)
    e = row["epilogue"]
    assert e["ctas"] > 0 and 0.0 < e["busy_share"] <= 1.0
    assert e["exposed_us"] is not None and 0.0 <= e["exposed_share"] <= 1.0


# ---------------------------------------------- whole-K kernel for a few rows
@pytest.mark.parametrize("M", [1, 5, 16, 17, 32, 33, 64])
@pytest.mark.parametrize("N,K", [(1088, 1024), (1104, 1000), (2048, 64), (1024, 200), (8192, 1600), (1024, 256),
                                 (1040, 328)])
def test_skinny_exact(M, N, K):
    # 64 weight rows per CTA (MMA M = 64), A's rows as the MMA's N, whole K:
    # K of one block, whole stages of four blocks only (1024, 256), whole
    # stages then single blocks (1000, 1600, 328: 5 whole chunks and a ragged
    # one), fewer than four chunks (200), a ragged last CTA (N not a multiple
    # of 64)
    A = make_matrix(M, K, "int2", seed=4000 + M, device="cuda")
    B = make_matrix(N, K, "int2", seed=4100 + N + K, device="cuda")
    with binding.Plan(0) as p:
        run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["skinny"] == 1 and c["split_k"] == 1 and c["tile_m"] == (128 if M > 32 else 64)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M", [1, 16, 64])
def test_skinny_normal_inputs(dtype, M):
    A = make_matrix(M, 4096, "normal", dtype, seed=4200 + M, device="cuda")
    B = make_matrix(8192, 4096, "weight", dtype, seed=4201, device="cuda")
    with binding.Plan(0) as p:
        run_full(p, A, B, dtype)
        assert p.last_config()["skinny"] == 1


@pytest.mark.parametrize("M", [20, 50])
@pytest.mark.parametrize("N", [1100, 1297, 1096])
def test_skinny_strided_operands_and_columns_untouched(M, N):
    # the row end of C inside the last output block (16 columns for one CTA,
    # 32 for a pair), off a 16-byte boundary (1100, 1297) or on one (1096);
    # the columns after N belong to the caller
    K = 520
    A = make_matrix(M, K, "int2", seed=4300, device="cuda", ld=K + 24)
    B = make_matrix(N, K, "int2", seed=4301, device="cuda", ld=K + 8)
    Cbuf = torch.full((M, 1320), 7.0, dtype=torch.bfloat16, device="cuda")
    with binding.Plan(0) as p:
        run_full(p, A, B, "bf16", exact=True, out=Cbuf[:, :N])
        assert p.last_config()["skinny"] == 1
    assert torch.all(Cbuf[:, N:] == 7.0), "wrote outside the output view"


def test_skinny_back_to_back_and_graph():
    # programmatic dependent launch chains and a captured graph: each launch
    # sees the previous one's output through C
    A = make_matrix(16, 2048, "int2", seed=4400, device="cuda")
    B = make_matrix(4096, 2048, "int2", seed=4401, device="cuda")
    want = oracle.gemm(bits_of(A), bits_of(B), "bf16")
    with binding.Plan(0) as p:
        outs = [p.gemm(A, B) for _ in range(4)]
        assert p.status() == 0 and p.last_config()["skinny"] == 1
        for C in outs:
            compare(bits_of(C), want, "bf16", 2048, exact=True)
        C = torch.empty(16, 4096, dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            p.gemm(A, B, out=C)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        C.zero_()
        with torch.cuda.graph(g):
            p.gemm(A, B, out=C)
        g.replay()
        torch.cuda.synchronize()
        assert p.status() == 0
        compare(bits_of(C), want, "bf16", 2048, exact=True)


@pytest.mark.parametrize("M", [16, 64])
def test_skinny_bounded_wait_reports_timeout(M):
    # one CTA (16 rows) and a CTA pair (64 rows): the even CTA's producer
    # never fills a stage, every wait of both CTAs ends
    A = make_matrix(M, 4096, "int2", seed=4500, device="cuda")
    B = make_matrix(2048, 4096, "int2", seed=4501, device="cuda")
    with binding.Plan(0, stall_kblock=3, timeout_ns=20_000_000) as p:
        p.gemm(A, B)
        assert p.last_config()["skinny"] == 1
        assert p.status() == 6  # BWGEMM_ERR_TIMEOUT, no trap
        assert p.last_device_status() != 0
    with binding.Plan(0) as p:  # the context is still usable
        run_full(p, A, B, "bf16", exact=True)


# ------------------------------------- whole-K pair kernel for 129-256 rows
@pytest.mark.parametrize("M", [129, 200, 256])
@pytest.mark.parametrize("N,K", [(8192, 1024), (1104, 1000), (2048, 64), (1040, 200), (10240, 328)])
def test_wholek_exact(M, N, K):
    # all rows of A on the MMA's M side (256 over a CTA pair), a block of
    # weight rows per pair sized to fill the pairs once, whole K: K of one
    # block, stages of two K blocks then a single one (1000: 15 whole chunks
    # and a ragged one; 328: 5 and a ragged one), fewer chunks than a stage
    # (200), ragged N (1104, 1040), a wide N (10240: blocks of 144)
    A = make_matrix(M, K, "int2", seed=5000 + M, device="cuda")
    B = make_matrix(N, K, "int2", seed=5100 + N + K, device="cuda")
    with binding.Plan(0, wholek=2) as p:
        run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["wholek"] == 1 and c["split_k"] == 1 and c["tile_m"] == 256 and c["variant"] == 2


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M", [200, 256])
def test_wholek_normal_inputs(dtype, M):
    A = make_matrix(M, 4096, "normal", dtype, seed=5200 + M, device="cuda")
    B = make_matrix(8192, 4096, "weight", dtype, seed=5201, device="cuda")
    with binding.Plan(0, wholek=2) as p:
        run_full(p, A, B, dtype)
        assert p.last_config()["wholek"] == 1


@pytest.mark.parametrize("N", [1100, 1297, 1096])
def test_wholek_strided_operands_and_columns_untouched(N):
    # the row end of C inside the last block of weight rows, off a 16-byte
    # boundary (1100, 1297) or on one (1096); the columns after N belong to
    # the caller
    M, K = 150, 520
    A = make_matrix(M, K, "int2", seed=5300, device="cuda", ld=K + 24)
    B = make_matrix(N, K, "int2", seed=5301, device="cuda", ld=K + 8)
    Cbuf = torch.full((M, 1320), 7.0, dtype=torch.bfloat16, device="cuda")
    with binding.Plan(0, wholek=2) as p:
        run_full(p, A, B, "bf16", exact=True, out=Cbuf[:, :N])
        assert p.last_config()["wholek"] == 1
    assert torch.all(Cbuf[:, N:] == 7.0), "wrote outside the output view"


def test_wholek_back_to_back_and_graph():
    A = make_matrix(256, 2048, "int2", seed=5400, device="cuda")
    B = make_matrix(4096, 2048, "int2", seed=5401, device="cuda")
    want = oracle.gemm(bits_of(A), bits_of(B), "bf16")
    with binding.Plan(0, wholek=2) as p:
        outs = [p.gemm(A, B) for _ in range(4)]
        assert p.status() == 0 and p.last_config()["wholek"] == 1
        for C in outs:
            compare(bits_of(C), want, "bf16", 2048, exact=True)
        C = torch.empty(256, 4096, dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            p.gemm(A, B, out=C)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        C.zero_()
        with torch.cuda.graph(g):
            p.gemm(A, B, out=C)
        g.replay()
        torch.cuda.synchronize()
        assert p.status() == 0
        compare(bits_of(C), want, "bf16", 2048, exact=True)


def test_wholek_bounded_wait_reports_timeout():
    # the even CTA's producer never fills a stage: every wait of both CTAs ends
    A = make_matrix(256, 4096, "int2", seed=5500, device="cuda")
    B = make_matrix(2048, 4096, "int2", seed=5501, device="cuda")
    with binding.Plan(0, wholek=2, stall_kblock=3, timeout_ns=20_000_000) as p:
        p.gemm(A, B)
        assert p.last_config()["wholek"] == 1
        assert p.status() == 6  # BWGEMM_ERR_TIMEOUT, no trap
        assert p.last_device_status() != 0
    with binding.Plan(0, wholek=2) as p:  # the context is still usable
        run_full(p, A, B, "bf16", exact=True)


@pytest.mark.parametrize("M,opts", [(16, {}), (64, {}), (200, {"wholek": 2})])
def test_whole_k_kernels_without_programmatic_dependent_launch(M, opts):
    # plain stream order between launches (no griddepcontrol overlap)
    A = make_matrix(M, 1000, "int2", seed=5600 + M, device="cuda")
    B = make_matrix(2048, 1000, "int2", seed=5601, device="cuda")
    with binding.Plan(0, pdl_off=1, **opts) as p:
        for _ in range(3):
            run_full(p, A, B, "bf16", exact=True)
        c = p.last_config()
        assert c["skinny"] == 1 if M <= 64 else c["wholek"] == 1


@pytest.mark.parametrize("M", [16, 200])
def test_tune_on_whole_k_shapes(M):
    # the tuner's candidates on a decode-batch shape: whatever it keeps is exact
    A = make_matrix(M, 1024, "int2", seed=5700 + M, device="cuda")
    B = make_matrix(2048, 1024, "int2", seed=5701, device="cuda")
    C = torch.zeros((M, 2048), dtype=torch.bfloat16, device="cuda")
    with binding.Plan(0) as p:
        p.tune(A, B, out=C, iters=3)
        assert p.tuned_count() == 1
        run_full(p, A, B, "bf16", exact=True)
