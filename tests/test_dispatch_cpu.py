"""Host logic of the whole kernel choice, through the C ABI, on the CPU.

sptg_plan makes the choice sptg_gemm_ex makes -- the square kernel or one of
the four skinny kernels, with its width, grid and cluster size -- without
touching a device. These tests pin the dispatch table that the skinny
kernels' measurements set (by output columns per SM, c = N / SMs rounded up
to a multiple of 8, and by rows of A), its edges, forced kernels, and over
many random shapes the invariants the kernels rely on.
"""
import random

import pytest

import software_pipelined_tiled_gb300 as sptg

SM = 152  # GB300


def plan(M, N, K, dtype="bf16_bf16", sm=SM, **cfg):
    c = None
    if cfg:
        c = sptg.Config()
        for k, v in cfg.items():
            setattr(c, k, sptg.KERNELS[v] if k == "kernel" else v)
    return sptg.plan(M, N, K, dtype, sm, c)


def cols(N, sm=SM):
    return max(8, (-(-N // sm) + 7) // 8 * 8)


@pytest.mark.parametrize("M,N,K,kernel,width,grid,cluster,mma_n", [
    # the measured skinny workload: 56 columns per CTA, 74 pairs
    (64, 8192, 8192, "skinny_pair", 56, 148, 2, 64),
    # up to 64 rows: pairs for 32 <= c <= 64, strips for 64 < c <= 256,
    # the cluster split below (even with SMs idle), stream-K past 256
    (64, 4096, 8192, "skinny_pair", 32, 128, 2, 64),
    (64, 9216, 8192, "skinny_pair", 64, 144, 2, 64),
    (64, 10240, 8192, "skinny_rows", 72, 143, 1, 64),
    (64, 16384, 4096, "skinny_rows", 112, 147, 1, 64),
    (64, 38912, 2048, "skinny_rows", 256, 152, 1, 64),
    (64, 1024, 8192, "skinny_cluster", 128, 32, 4, 64),
    (40, 3072, 4096, "skinny_cluster", 128, 96, 4, 64),
    (64, 40960, 1024, "skinny", 128, 152, 1, 64),
    (1, 8192, 8192, "skinny_pair", 56, 148, 2, 64),
    # 65-128 rows: pairs with MMA N = 128 up to c = 128
    (128, 8192, 8192, "skinny_pair", 56, 148, 2, 128),
    (65, 1024, 2048, "skinny_pair", 8, 128, 2, 128),
    (100, 16384, 1024, "skinny_pair", 112, 148, 2, 128),
    # 129-256 rows: pairs with MMA N = 256 up to c = 64
    (256, 8192, 2048, "skinny_pair", 56, 148, 2, 256),
    (129, 4096, 4096, "skinny_pair", 32, 128, 2, 256),
])
def test_skinny_choices(M, N, K, kernel, width, grid, cluster, mma_n):
    p = plan(M, N, K)
    assert (p["kernel"], p["width"], p["grid"], p["cluster"], p["mma_n"]) == \
        (kernel, width, grid, cluster, mma_n), p


def test_long_k_narrow_outputs_take_stream_k():
    # c < 32 and K past 16384: the cluster split must fill the GPU, which 8
    # column tiles cannot, so stream-K takes it
    assert plan(64, 1024, 32768)["kernel"] == "skinny"
    assert plan(64, 1024, 16384)["kernel"] == "skinny_cluster"


@pytest.mark.parametrize("M,N,K,dtype", [
    (4096, 4096, 4096, "f16_f16"), (256, 256, 256, "f16_f32"), (8192, 8192, 16384, "bf16_f32"),
    (64, 8192, 8192, "s8_s32"), (257, 8192, 8192, "bf16_bf16"), (256, 16384, 1024, "bf16_bf16"),
    (128, 24576, 1024, "bf16_bf16"), (64, 1000, 8192, "bf16_bf16")])
def test_square_kernel_elsewhere(M, N, K, dtype):
    # int8, more than 256 rows, N below 1024, wider than the skinny kernels
    # take: the square kernel, with the square planner's tile and schedule
    p = plan(M, N, K, dtype)
    sq = sptg.plan_square(M, N, K, dtype, SM)
    assert p["kernel"] == "square" and p["width"] == sq["bn"] and p["mma_n"] == 0
    assert p["cluster"] == (2 if sq["pair"] else 1)
    assert p["grid"] == sq["workers"] * p["cluster"]
    assert p["stream_k_tiles"] == sq["stream_k_tiles"]


def test_benchmark_shapes():
    assert plan(4096, 4096, 4096, "f16_f16")["width"] == 224
    assert plan(4096, 4096, 4096, "s8_s32")["width"] == 224
    assert plan(8192, 8192, 16384, "bf16_f32")["width"] == 512
    assert plan(64, 8192, 8192)["kernel"] == "skinny_pair"
    assert plan(256, 256, 256, "f16_f32")["cluster"] == 1


def test_fewer_sms_move_the_edges():
    # the choice follows the GPU's SM count, not a fixed N
    assert plan(64, 8192, 8192, sm=148)["width"] == cols(8192, 148)
    assert plan(64, 8192, 8192, sm=76)["kernel"] == "skinny_rows"  # 112 columns per SM


def test_forced_kernels():
    p = plan(64, 8192, 8192, kernel="skinny_rows", bn=64)
    assert (p["kernel"], p["width"], p["grid"]) == ("skinny_rows", 64, 128)
    p = plan(64, 8192, 8192, kernel="skinny_pair", bn=64)
    assert (p["kernel"], p["width"], p["grid"]) == ("skinny_pair", 64, 128)
    p = plan(64, 8192, 8192, kernel="skinny_cluster", splits=2)
    assert (p["kernel"], p["grid"], p["cluster"]) == ("skinny_cluster", 128, 2)
    p = plan(64, 8192, 8192, kernel="skinny", splits=24)
    assert (p["kernel"], p["grid"]) == ("skinny", 24)
    assert plan(64, 8192, 8192, kernel="square")["kernel"] == "square"
    for bad in (dict(kernel="skinny_rows", bn=12), dict(kernel="skinny_pair", bn=136),
                dict(kernel="skinny_cluster", splits=3)):
        with pytest.raises(sptg.SptgError):
            plan(64, 8192, 8192, **bad)
    with pytest.raises(sptg.SptgError):
        plan(65, 8192, 8192, kernel="skinny_rows")  # strips take up to 64 rows
    with pytest.raises(sptg.SptgError):
        plan(257, 8192, 8192, kernel="skinny_pair")
    with pytest.raises(sptg.SptgError):
        plan(64, 8192, 8192, "s8_s32", kernel="skinny_pair")


def test_invalid_arguments():
    for args in ((0, 8, 8), (8, 0, 8), (8, 8, 0)):
        with pytest.raises(sptg.SptgError):
            sptg.plan(*args, "bf16_bf16", SM)
    with pytest.raises(sptg.SptgError):
        sptg.plan(8, 8, 8, "bf16_bf16", 1)
    c = sptg.Config()
    c.kernel = 6
    with pytest.raises(sptg.SptgError):
        sptg.plan(8, 8, 8, "bf16_bf16", SM, c)


@pytest.mark.parametrize("seed", range(4))
def test_invariants_over_random_shapes(seed):
    rng = random.Random(seed)
    for _ in range(500):
        M = rng.choice([rng.randint(1, 64), rng.randint(65, 128), rng.randint(129, 300),
                        rng.randint(1, 4096)])
        N = 8 * rng.randint(1, 8000)
        K = 8 * rng.randint(1, 5000)
        sm = rng.choice([SM, 148, 132, 76])
        p = plan(M, N, K, sm=sm)
        k = p["kernel"]
        if k == "skinny_pair":
            assert M <= 256 and p["width"] % 8 == 0 and 8 <= p["width"] <= 128
            assert p["cluster"] == 2 and p["grid"] == 2 * -(-N // (2 * p["width"]))
            assert p["grid"] <= sm
            assert p["mma_n"] == (64 if M <= 64 else 128 if M <= 128 else 256)
        elif k == "skinny_rows":
            assert M <= 64 and p["width"] % 8 == 0 and 32 <= p["width"] <= 256
            assert p["grid"] == -(-N // p["width"]) and 3 * sm <= 4 * p["grid"] <= 4 * sm
        elif k == "skinny_cluster":
            assert M <= 128 and p["cluster"] in (1, 2, 4) and p["grid"] <= sm
            assert p["grid"] == -(-N // 128) * p["cluster"]
        elif k == "skinny":
            assert M <= 64 and p["grid"] <= sm
        else:
            assert k == "square"
        if M > 256 or N < 1024:
            assert k == "square"
