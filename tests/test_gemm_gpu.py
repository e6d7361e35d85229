"""GPU parity of the pipelined GEMM against the CPU oracle, through the C ABI.

Covers the five measured workloads (full comparison where the oracle finishes
in seconds, sampled positions for the 8192 x 8192 x 16384 product), the
pipeline-structure cases the method's pitfalls name (a dropped, doubled or
misplaced K-tile; ring wrap and phase flips; the last tile), ragged edges and
degenerate shapes, and the bounded-wait error path.
"""
import numpy as np
import pytest
import torch

import oracle
import software_pipelined_tiled_gb300 as sptg
from gpu_helpers import (assert_float_parity, assert_int_parity, run, sample_positions)
from workloads import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

F16, BF16, F32, I8, I32 = torch.float16, torch.bfloat16, torch.float32, torch.int8, torch.int32


# ----------------------------------------------------------------- workloads
# Float workloads meet the unmodified bound |C - C_ref| <= 1e-3 sum_k |A_ik B_kj|
# itself (plain=True): their K is large enough that the output rounding of a
# 16-bit C stays well inside it. Each prints its max |err| / (1e-3 sum|AB|).
def test_workload_f16_256_f32out():
    w = WORKLOADS["f16_256x256x256_f32out"]
    A, B = workload_inputs(w)
    C = run(A, B, F32)
    assert "kernel=square" in sptg.last_config()
    print(w.name, "max |err| / (1e-3 sum|ab|) =", assert_float_parity(C, A, B, plain=True))


def test_workload_f16_4096_f16out():
    w = WORKLOADS["f16_4096x4096x4096_f16out"]
    A, B = workload_inputs(w)
    C = run(A, B, F16)
    print(w.name, "max |err| / (1e-3 sum|ab|) =", assert_float_parity(C, A, B, plain=True))


def test_workload_s8_4096_bit_exact():
    w = WORKLOADS["s8_4096x4096x4096_s32out"]
    A, B = workload_inputs(w)
    C = run(A, B, I32)
    assert_int_parity(C, A, B)


def test_workload_bf16_skinny():
    w = WORKLOADS["bf16_skinny_64x8192x8192_bf16out"]
    A, B = workload_inputs(w)
    C = run(A, B, BF16)
    assert "kernel=skinny" in sptg.last_config()
    print(w.name, "max |err| / (1e-3 sum|ab|) =", assert_float_parity(C, A, B, plain=True))


def test_workload_bf16_8192x8192x16384_sampled():
    w = WORKLOADS["bf16_8192x8192x16384_f32out"]
    A, B = workload_inputs(w)
    C = run(A, B, F32)
    # 32 x 16 tiles of 256 x 512 over 76 pairs, data-parallel: sample one
    # whole tile densely too (both 256-column halves of each CTA's rows)
    assert "bn=512" in sptg.last_config() and _sk_tiles() == 0, sptg.last_config()
    rows, cols = sample_positions(w.M, w.N, 4000, seed=5)
    extra = np.arange(2560, 2816, dtype=np.int64)
    rows = np.concatenate([rows, np.repeat(extra, 16)])
    cols = np.concatenate([cols, np.tile(np.arange(4096, 4608, 32, dtype=np.int64), 256) + np.repeat(extra, 16) % 32])
    assert_float_parity(C, A, B, rows, cols, plain=True)
    # a whole row and a whole column as well
    r = np.full(w.N, 4097, dtype=np.int64)
    assert_float_parity(C, A, B, r, np.arange(w.N, dtype=np.int64), plain=True)
    c = np.full(w.M, 8191, dtype=np.int64)
    assert_float_parity(C, A, B, np.arange(w.M, dtype=np.int64), c, plain=True)


@pytest.mark.slow
def test_workload_bf16_8192x8192x16384_every_element():
    # all 67 M outputs against the oracle (about a minute of CPU time on the
    # host's cores)
    w = WORKLOADS["bf16_8192x8192x16384_f32out"]
    A, B = workload_inputs(w)
    C = run(A, B, F32)
    print(w.name, "max |err| / (1e-3 sum|ab|) =", assert_float_parity(C, A, B, plain=True))


# ---------------------------------------------------------- pipeline structure
def _marker_inputs(M, N, T, BK=64, dtype=F16):
    # A = 1, B[k][j] = floor(k / BK) + 1: C = BK * T (T + 1) / 2 exactly
    K = BK * T
    A = torch.ones(M, K, dtype=dtype)
    Bcm = (torch.arange(K) // BK + 1).to(dtype).repeat(N, 1).contiguous()
    return A, Bcm, BK * T * (T + 1) // 2


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 9, 17])
@pytest.mark.parametrize("stages", [1, 2, 3, 4])
@pytest.mark.parametrize("bn", [256, 224])
def test_k_tile_marker_square(T, stages, bn):
    # K/BK around the ring depth: fewer, equal, one more, wraps twice; three
    # CTAs over several tiles each, so accumulators and phases wrap as well
    A, B, expect = _marker_inputs(256, 512, T)
    C = run(A, B, F16, stages=stages, splits=3, bn=bn, cta_pair=1)
    assert "pair=0" in sptg.last_config()
    assert (C.to(torch.float64) == expect).all()


FLOAT_WIDTHS = [256, 240, 224, 208, 192, 176, 160, 144, 128, 112]


@pytest.mark.parametrize("bn", FLOAT_WIDTHS)
@pytest.mark.parametrize("pair", ["f16_f32", "f16_f16", "bf16_bf16", "bf16_f32"])
def test_every_tile_width(bn, pair):
    it, ot = pair.split("_")
    dt = {"f16": F16, "bf16": BF16, "f32": F32}
    A, B = make_inputs(300, 680, 328, it, "uniform", bn)
    C = run(A, B, dt[ot], kernel="square", bn=bn, cta_pair=1)
    assert f"bn={bn}" in sptg.last_config() and "pair=0" in sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("T", [1, 2, 5, 6, 7, 13])
@pytest.mark.parametrize("bn", [224, 128])
def test_k_tile_marker_cta_pair(T, bn):
    # 2-SM tiles: both CTAs' copies must land before the leader's MMA, and
    # both halves of the result must come back; 3 pairs over several tiles
    A, B, expect = _marker_inputs(512, 896, T)
    C = run(A, B, F16, cta_pair=2, bn=bn, splits=3)
    assert "pair=1" in sptg.last_config()
    assert (C.to(torch.float64) == expect).all()


@pytest.mark.parametrize("bn", FLOAT_WIDTHS)
@pytest.mark.parametrize("pair", ["f16_f32", "f16_f16", "bf16_bf16", "bf16_f32"])
def test_every_tile_width_cta_pair(bn, pair):
    it, ot = pair.split("_")
    dt = {"f16": F16, "bf16": BF16, "f32": F32}
    # M = 300: the second pair-tile's peer CTA sees only out-of-range rows
    A, B = make_inputs(300, 680, 328, it, "uniform", bn + 1)
    C = run(A, B, dt[ot], kernel="square", bn=bn, cta_pair=2)
    assert f"bn={bn}" in sptg.last_config() and "pair=1" in sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("bn", [112, 176, 240])
@pytest.mark.parametrize("cta_pair", [1, 2])
@pytest.mark.parametrize("it,ot,N", [("f16", F16, 1000), ("bf16", BF16, 696), ("bf16", F32, 692),
                                     ("f16", F32, 1056)])
def test_half_block_tiles_over_several_rounds(bn, cta_pair, it, ot, N):
    # widths ending in a 16-column block (stored from registers) on three
    # workers, so each holds several tiles and both accumulators take turns;
    # N = 696 / 692 end inside the last tile's 16-column block (one group of
    # 8 bfloat16 / 4 fp32 outputs in C, the rest past N), 1056 is a multiple
    # of 176 (every tile whole)
    A, B = make_inputs(700, N, 200, it, "uniform", bn + cta_pair)
    C = run(A, B, ot, kernel="square", bn=bn, cta_pair=cta_pair, splits=3, stream_k=1)
    cfg = sptg.last_config()
    assert f"bn={bn}" in cfg and f"pair={cta_pair - 1}" in cfg, cfg
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("bn", [112, 176, 240])
@pytest.mark.parametrize("cta_pair", [1, 2])
def test_half_block_tiles_cut_along_k(bn, cta_pair):
    # every tile cut along K: the last 16 columns of each partial go to the
    # scratch slot's last groups and come back through the reduction
    A, B = make_inputs(520, 776, 1096, "bf16", "uniform", 42 + bn)
    C = run(A, B, F32, kernel="square", bn=bn, cta_pair=cta_pair, stream_k=2, splits=5)
    assert _sk_tiles() > 0 and f"bn={bn}" in sptg.last_config()
    assert_float_parity(C, A, B)
    A, B = make_inputs(300, 528, 2000, "f16", "uniform", 43 + bn)
    C = run(A, B, F16, kernel="square", bn=bn, cta_pair=cta_pair, stream_k=2, splits=7)
    assert _sk_tiles() > 0
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("bn,it,ot", [(112, "f16", F16), (176, "f16", F16), (144, "bf16", BF16),
                                      (128, "bf16", F32), (112, "bf16", F32)])
def test_two_chunk_stages(bn, it, ot):
    # CTA pairs over K-loops of 32 K-chunks or more take two 64-wide K-chunks
    # per ring stage where that ring still holds four stages; K = 2056 leaves
    # the last stage's second chunk wholly past K (zero-filled)
    A, B = make_inputs(300, 680, 2056, it, "uniform", bn + 3)
    C = run(A, B, ot, kernel="square", bn=bn, cta_pair=2, splits=7, stream_k=1)
    cfg = sptg.last_config()
    assert "kch=2" in cfg and f"bn={bn}" in cfg and "pair=1" in cfg, cfg
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("bn,cta_pair,ot", [(176, 2, F32), (192, 2, F16), (176, 1, F16),
                                            (112, 1, F16)])
def test_one_chunk_stages_where_two_leave_a_shallow_ring(bn, cta_pair, ot):
    # fp32 C at 176 columns and 192-wide pairs would keep three two-chunk
    # stages, single CTAs two or three: one chunk per stage there
    A, B = make_inputs(300, 680, 2056, "f16", "uniform", bn + 5)
    C = run(A, B, ot, kernel="square", bn=bn, cta_pair=cta_pair)
    assert "kch=1" in sptg.last_config(), sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("T", [32, 33, 47])
def test_k_tile_marker_two_chunk_stages(T):
    # both chunks of every stage land in the sum exactly once (T odd: the
    # last stage holds one chunk inside K); three pairs over several tiles
    A, B, expect = _marker_inputs(512, 896, T)
    C = run(A, B, F32, kernel="square", bn=112, cta_pair=2, splits=3, stream_k=1)
    assert "kch=2" in sptg.last_config(), sptg.last_config()
    assert (C.to(torch.float64) == expect).all()


def test_two_chunk_stages_cut_along_k():
    # stream-K over stages of two K-chunks: the cut falls between stages
    A, B = make_inputs(520, 776, 4104, "bf16", "uniform", 62)
    C = run(A, B, F32, kernel="square", bn=112, cta_pair=2, stream_k=2, splits=5)
    assert _sk_tiles() > 0 and "kch=2" in sptg.last_config(), sptg.last_config()
    assert_float_parity(C, A, B)
    # a forced ring depth keeps one chunk per stage (the deepest one-chunk
    # ring of a 112-wide pair tile with fp32 C: 8 stages)
    C = run(A, B, F32, kernel="square", bn=112, cta_pair=2, stages=8)
    assert "kch=1" in sptg.last_config() and "stages=8" in sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("bn", [112, 176])
def test_half_block_columns_are_placed(bn):
    # each column of B distinct, A the identity block: C[i, j] = B[j, i]
    # exactly, so a 16-column block written to the wrong columns or rows shows
    M, N, K = 256, 3 * bn, 256
    A = torch.eye(M, K, dtype=F16)
    Bcm = ((torch.arange(N).unsqueeze(1) * 7 + torch.arange(K).unsqueeze(0)) % 1024).to(F16)
    for cta_pair in (1, 2):
        C = run(A, Bcm, F32, kernel="square", bn=bn, cta_pair=cta_pair, splits=1, stream_k=1)
        assert f"bn={bn}" in sptg.last_config()
        assert torch.equal(C, Bcm.t().to(F32)[:M])


def test_mid_rows_default_tiles():
    # 768 x 8192 x 8192 takes 256 x 176 pair tiles by default: sampled
    # outputs, a whole row, and the 16-column block that ends tile column 45
    # (the last tile column holds only 96 columns)
    M, N, K = 768, 8192, 8192
    A, B = make_inputs(M, N, K, "bf16", "normal", 46)
    C = run(A, B, BF16)
    cfg = sptg.last_config()
    assert "bn=176" in cfg and "pair=1" in cfg, cfg
    rows, cols = sample_positions(M, N, 3000, seed=46)
    tail = np.arange(45 * 176 + 160, 46 * 176, dtype=np.int64)
    rows = np.concatenate([rows, np.repeat(np.arange(0, M, 37, dtype=np.int64), 16)])
    cols = np.concatenate([cols, np.tile(tail, len(range(0, M, 37)))])
    assert_float_parity(C, A, B, rows, cols)
    r = np.full(N, 513, dtype=np.int64)
    assert_float_parity(C, A, B, r, np.arange(N, dtype=np.int64))


def test_cta_pair_operand_halves_are_not_swapped():
    # rows of A and columns of B differ everywhere: a swapped half or a
    # misplaced peer tile changes the result
    M, N, K = 256, 224, 64
    A = (torch.arange(M).unsqueeze(1) + 1).to(F32).expand(M, K).contiguous() / 256
    Bcm = (torch.arange(N).unsqueeze(1) + 1).to(F32).expand(N, K).contiguous() / 256
    A, Bcm = A.to(F16), Bcm.to(F16)
    C = run(A, Bcm, F32, cta_pair=2, bn=224)
    # every product and partial sum is a multiple of 2^-16 below 2^6: exact in
    # fp32, so the result must equal the oracle's sum exactly
    ref, _ = oracle.gemm_float(A, Bcm, oracle.IN_F16)
    assert np.array_equal(C.to(torch.float64).numpy(), ref)


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5, 6])
def test_cta_pair_stage_count_does_not_change_the_arithmetic(stages):
    A, B = make_inputs(512, 448, 640, "f16", "uniform", 13)
    ref = run(A, B, F16, bn=224, cta_pair=2)
    got = run(A, B, F16, stages=stages, bn=224, cta_pair=2)
    assert f"stages={stages}" in sptg.last_config() and "pair=1" in sptg.last_config()
    assert torch.equal(ref, got)
    # and against the oracle: a fault shared by every ring depth shows here
    assert_float_parity(got, A, B)


@pytest.mark.parametrize("T", [1, 2, 7, 8, 9, 17])
def test_k_tile_marker_skinny(T):
    A, B, expect = _marker_inputs(64, 1024, T, dtype=BF16)
    C = run(A, B, F32, kernel="skinny", splits=24)
    assert (C.to(torch.float64) == expect).all()


def test_only_last_k_tile_nonzero():
    # a dropped final tile ("Pipeline GPU Kernel", pitfalls) shows up as zeros
    M, N, K = 128, 256, 64 * 7
    A = torch.zeros(M, K, dtype=F16)
    B = torch.zeros(N, K, dtype=F16)
    A[:, -64:] = 1
    B[:, -64:] = 0.5
    C = run(A, B, F32)
    assert (C == 32.0).all()


def test_identity_and_ones():
    A, _ = make_inputs(256, 1, 256, "f16", "uniform", 3)
    eye = torch.eye(256, dtype=F16)
    C = run(A, eye, F32)
    assert torch.equal(C, A.to(F32))
    ones = torch.ones(128, 4096, dtype=BF16)
    C = run(ones, torch.ones(256, 4096, dtype=BF16), F32)
    assert (C == 4096).all()


def test_permutation_selects_columns():
    A, _ = make_inputs(256, 1, 512, "bf16", "normal", 4)
    perm = torch.randperm(512, generator=torch.Generator().manual_seed(1))[:384]
    Bcm = torch.zeros(384, 512, dtype=BF16)
    Bcm[torch.arange(384), perm] = 1
    C = run(A, Bcm, BF16)
    assert torch.equal(C, A[:, perm])


@pytest.mark.parametrize("stages", [1, 2, 3])
def test_stage_count_does_not_change_the_arithmetic(stages):
    # pipelining reorders loads only ("Pipeline GPU Kernel", Step 5): any
    # ring depth gives the same bits as the default one
    A, B = make_inputs(384, 512, 1024, "f16", "uniform", 12)
    ref = run(A, B, F16, bn=224, cta_pair=1)
    got = run(A, B, F16, stages=stages, bn=224, cta_pair=1)
    assert f"stages={stages}" in sptg.last_config()
    assert torch.equal(ref, got)
    assert_float_parity(got, A, B)


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5])
def test_long_k_ablation_rings_match(stages):
    # the shallower rings of the 256-wide bfloat16 pair tile give the bits of
    # the default ring
    A, B = make_inputs(512, 512, 2048, "bf16", "normal", 14)
    ref = run(A, B, F32, bn=256, cta_pair=2, stream_k=1)
    got = run(A, B, F32, bn=256, cta_pair=2, stream_k=1, stages=stages)
    assert f"stages={stages}" in sptg.last_config()
    assert torch.equal(ref, got)
    assert_float_parity(got, A, B)


@pytest.mark.parametrize("stages", [1, 2, 3])
def test_skinny_cluster_ablation_rings_match(stages):
    A, B = make_inputs(64, 2048, 4096, "bf16", "normal", 15)
    ref = run(A, B, BF16, kernel="skinny_cluster", splits=2)
    got = run(A, B, BF16, kernel="skinny_cluster", splits=2, stages=stages)
    assert f"stages={stages}" in sptg.last_config()
    assert torch.equal(ref, got)
    assert_float_parity(got, A, B)


# --------------------------------------------------------- ragged and edges
@pytest.mark.parametrize("M,N,K,dt,out", [
    (200, 136, 200, F16, F32),
    (1, 8, 8, F16, F16),
    (129, 264, 72, BF16, BF16),
    (300, 520, 1032, BF16, F32),
    (77, 4, 4104, F16, F32),
])
def test_ragged_shapes(M, N, K, dt, out):
    A, B = make_inputs(M, N, K, "f16" if dt == F16 else "bf16", "uniform", M + N + K)
    C = run(A, B, out, kernel="square")
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("M,N,K", [(256, 256, 2048), (129, 260, 1040), (64, 64, 16)])
def test_int8_exact_small(M, N, K):
    A, B = make_inputs(M, N, K, "s8", "int8", 7 + K)
    C = run(A, B, I32)
    assert_int_parity(C, A, B)


@pytest.mark.parametrize("M,N,K", [(512, 384, 2080), (300, 136, 1024)])
def test_int8_exact_cta_pair(M, N, K):
    A, B = make_inputs(M, N, K, "s8", "int8", 11 + K)
    C = run(A, B, I32, cta_pair=2)
    assert "pair=1" in sptg.last_config()
    assert_int_parity(C, A, B)


@pytest.mark.parametrize("cta_pair", [1, 2])
@pytest.mark.parametrize("bn", [256, 224, 192, 160, 128])
def test_int8_exact_every_width(bn, cta_pair):
    A, B = make_inputs(520, 488, 3136, "s8", "int8", 50 + bn)
    C = run(A, B, I32, bn=bn, cta_pair=cta_pair)
    assert f"bn={bn}" in sptg.last_config()
    assert_int_parity(C, A, B)


@pytest.mark.parametrize("K", [131056, 131072, 135168])
def test_int8_sum_range(K):
    # |a b| <= 2^14, so any K below 2^17 fits int32; at and beyond it the
    # all -128 product (16384 K) wraps modulo 2^32, as an int32 accumulator does
    A = torch.full((128, K), -128, dtype=I8)
    B = torch.full((128, K), -128, dtype=I8)
    C = run(A, B, I32)
    want = 16384 * K
    want = (want + 2**31) % 2**32 - 2**31
    assert (C.to(torch.int64) == want).all(), (int(C[0, 0]), want)


@pytest.mark.parametrize("K", [1024, 1040, 4096])
def test_int8_extremes_exact(K):
    # every chunk of 1024 products reaches 2^24 exactly
    A = torch.full((130, K), -128, dtype=I8)
    B = torch.full((136, K), -128, dtype=I8)
    C = run(A, B, I32)
    assert (C.to(torch.int64) == 16384 * K).all()
    alt = torch.tensor([-128 if k % 2 == 0 else 127 for k in range(K)], dtype=I8)
    C = run(alt.repeat(128, 1), (-alt.to(torch.int16)).clamp(-128, 127).to(I8).repeat(128, 1), I32)
    assert (C.to(torch.int64) == (K // 2) * (-128 * 127) + (K // 2) * (127 * -127)).all()


def test_zero_k_gives_zero_and_empty_is_noop():
    A = torch.zeros(64, 0, dtype=F16).cuda()
    B = torch.zeros(128, 0, dtype=F16).cuda()
    C = torch.full((64, 128), 7.0, dtype=F32).cuda()
    sptg.gemm(A, B, C=C)
    torch.cuda.synchronize()
    assert (C == 0).all()
    E = torch.empty(0, 128, dtype=F32).cuda()
    sptg.gemm(torch.zeros(0, 16, dtype=F16).cuda(), torch.zeros(128, 16, dtype=F16).cuda(), C=E)


# ----------------------------------------------------------------- skinny
@pytest.mark.parametrize("M,N,K,splits", [
    (64, 8192, 1024, 0), (1, 1024, 2048, 0), (17, 1000, 1000, 7), (64, 512, 4096, 200),
    (33, 2048, 520, 5), (64, 256, 64, 3)])
def test_skinny_split_and_ragged(M, N, K, splits):
    A, B = make_inputs(M, N, K, "bf16", "normal", M * 7 + K)
    C = run(A, B, BF16, kernel="skinny", splits=splits)
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("M,N,K,cs", [
    (64, 8192, 4096, 2), (64, 4096, 2048, 2), (17, 1000, 1000, 2), (1, 2048, 1040, 2),
    (40, 768, 520, 1), (64, 256, 64, 2), (33, 1024, 64, 1),
    (64, 4096, 8192, 4), (48, 1000, 1088, 4), (64, 512, 512, 4), (5, 2048, 4160, 4)])
def test_skinny_cluster_split(M, N, K, cs):
    A, B = make_inputs(M, N, K, "bf16", "normal", M * 3 + K)
    C = run(A, B, BF16, kernel="skinny_cluster", splits=cs)
    assert "kernel=skinny-cluster" in sptg.last_config() and f"cluster={cs}" in sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("T", [1, 2, 3, 8, 17])
@pytest.mark.parametrize("cs", [1, 2, 4])
def test_k_tile_marker_skinny_cluster(T, cs):
    # every rank's K-range lands in the sum exactly once
    A, B, expect = _marker_inputs(64, 1024, T * cs, dtype=BF16)
    C = run(A, B, F32, kernel="skinny_cluster", splits=cs)
    assert (C.to(torch.float64) == expect).all()


# One CTA per strip of output columns over the whole of K (M <= 64): strip
# widths from 8 to 128, ragged last strips (N not a multiple of the width),
# K not a multiple of the 128-wide stage (half-empty last stage, 2-D copies
# when K is not a multiple of 64), rows past M, all four float dtype pairs.
@pytest.mark.parametrize("M,N,K,nt,it,ot", [
    (64, 8192, 4096, 0, "bf16", BF16), (64, 8192, 1024, 56, "bf16", F32),
    (1, 2048, 1040, 16, "f16", F16), (17, 1000, 1000, 48, "f16", F32),
    (33, 4096, 520, 128, "bf16", BF16), (64, 256, 64, 8, "bf16", BF16),
    (48, 9216, 2056, 0, "f16", F16), (5, 1000, 4160, 120, "bf16", F32),
    (64, 1024, 8200, 32, "f16", F32),
    # strips past 160 columns (one K-chunk per stage) up to 256
    (64, 32768, 1024, 0, "bf16", BF16), (17, 5000, 1040, 256, "f16", F32),
    (40, 3000, 2056, 168, "bf16", F32), (64, 2048, 520, 200, "f16", F16)])
def test_skinny_rows(M, N, K, nt, it, ot):
    A, B = make_inputs(M, N, K, it, "normal", M * 5 + K)
    C = run(A, B, ot, kernel="skinny_rows", bn=nt)
    cfg = sptg.last_config()
    assert "kernel=skinny-rows" in cfg, cfg
    if nt:
        assert f"mma_n={nt} " in cfg, cfg
    assert_float_parity(C, A, B)


def test_skinny_rows_is_the_default_for_wide_outputs():
    # 64 x 16384 x 4096: more than 64 columns per SM, strips of at most one
    # per SM, the whole of K each
    A, B = make_inputs(64, 16384, 4096, "bf16", "normal", 44)
    C = run(A, B, BF16)
    cfg = sptg.last_config()
    assert "kernel=skinny-rows" in cfg, cfg
    grid = int(cfg.split("grid=")[1].split()[0])
    nt = int(cfg.split("mma_n=")[1].split()[0])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert nt % 8 == 0 and grid == -(-16384 // nt) and 3 * sms <= 4 * grid <= 4 * sms
    print(cfg, "max |err| / (1e-3 sum|ab|) =", assert_float_parity(C, A, B, plain=True))
    # deterministic: no split, no reduction order to vary
    assert torch.equal(C, run(A, B, BF16))


@pytest.mark.parametrize("T", [1, 2, 3, 8, 17])
@pytest.mark.parametrize("stages", [0, 1, 2, 3])
@pytest.mark.parametrize("nt", [64, 192])
def test_k_tile_marker_skinny_rows(T, stages, nt):
    # every K-chunk lands in the sum exactly once, whatever the ring depth;
    # an odd T leaves the second chunk of the last stage empty (two chunks per
    # stage up to 160 columns, one past that)
    A, B, expect = _marker_inputs(64, 1024, T, dtype=BF16)
    C = run(A, B, F32, kernel="skinny_rows", bn=nt, stages=stages)
    if stages:
        assert f"stages={stages}" in sptg.last_config()
    assert (C.to(torch.float64) == expect).all()


@pytest.mark.parametrize("T,nt", [(129, 64), (129, 192), (130, 112)])
def test_k_tile_marker_skinny_rows_staggered(T, nt):
    # K >= 8192 over 64 stages or more: the strips start their K-loops at
    # staggered chunks and wrap around; every K-chunk must still land in each
    # sum exactly once (binary16 markers: exact up to 2048)
    A, B, expect = _marker_inputs(64, 2000, T, dtype=F16)
    C = run(A, B, F32, kernel="skinny_rows", bn=nt)
    assert "k_rotate=1" in sptg.last_config(), sptg.last_config()
    assert (C.to(torch.float64) == expect).all()


@pytest.mark.parametrize("M,N,K,it,ot", [(64, 16384, 8200, "bf16", BF16),
                                         (40, 30000, 8192, "f16", F32)])
def test_skinny_rows_staggered_parity(M, N, K, it, ot):
    A, B = make_inputs(M, N, K, it, "normal", M + N)
    C = run(A, B, ot)
    cfg = sptg.last_config()
    assert "kernel=skinny-rows" in cfg and "k_rotate=1" in cfg, cfg
    rows, cols = sample_positions(M, N, 6000, seed=M)
    assert_float_parity(C, A, B, rows, cols)
    r = np.full(N, M - 1, dtype=np.int64)
    assert_float_parity(C, A, B, r, np.arange(N, dtype=np.int64))
    assert torch.equal(C, run(A, B, ot))  # the same order every call


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_skinny_rows_ablation_rings_match(stages):
    A, B = make_inputs(64, 2048, 4096, "bf16", "normal", 16)
    ref = run(A, B, BF16, kernel="skinny_rows", bn=56)
    got = run(A, B, BF16, kernel="skinny_rows", bn=56, stages=stages)
    assert f"stages={stages}" in sptg.last_config()
    assert torch.equal(ref, got)
    assert_float_parity(got, A, B)


def test_skinny_rows_limits():
    A, B = make_inputs(65, 2048, 1024, "bf16", "normal", 87)
    with pytest.raises(sptg.SptgError):
        run(A, B, BF16, kernel="skinny_rows")  # more than 64 rows
    A, B = make_inputs(64, 2048, 1024, "bf16", "normal", 88)
    for bad in (12, 264):
        with pytest.raises(sptg.SptgError):
            run(A, B, BF16, kernel="skinny_rows", bn=bad)
    with pytest.raises(sptg.SptgError):
        run(A, B, BF16, kernel="skinny_rows", bn=128, stages=5)  # 5 x 48 KB > the budget
    A, B = make_inputs(64, 2048, 1024, "s8", "int8", 89)
    with pytest.raises(sptg.SptgError):
        run(A, B, I32, kernel="skinny_rows")


# CTA pairs with the 2-SM MMA over the whole of K (M <= 64): columns per CTA
# from 8 to 64, ragged last pairs (a CTA whose columns all lie past N), rows of
# A past 32 (the second CTA's half of the MMA's N side) and past M, K not a
# multiple of the stage, all four float dtype pairs.
@pytest.mark.parametrize("M,N,K,nc,it,ot", [
    (64, 8192, 4096, 0, "bf16", BF16), (64, 8192, 1024, 56, "bf16", F32),
    (1, 2048, 1040, 16, "f16", F16), (17, 1000, 1000, 48, "f16", F32),
    (33, 4096, 520, 64, "bf16", BF16), (64, 256, 64, 8, "bf16", BF16),
    (48, 9216, 2056, 0, "f16", F16), (5, 1000, 4160, 40, "bf16", F32),
    (64, 1024, 8200, 32, "f16", F32), (40, 200, 640, 64, "bf16", F32),
    (8, 136, 256, 64, "f16", F16),  # the second CTA of the last pair lies wholly past N
    # 65-128 rows: the MMA's N side covers 128 rows of A, 64 copied per CTA
    (128, 8192, 2048, 0, "bf16", BF16), (65, 1000, 1040, 48, "f16", F32),
    (100, 4096, 520, 64, "bf16", BF16), (128, 200, 640, 8, "f16", F16),
    (96, 2056, 4160, 40, "bf16", F32),
    # past 64 columns per CTA: two 64-row blocks, two MMAs per K-step
    (64, 16384, 1024, 0, "bf16", BF16), (100, 12288, 520, 88, "f16", F32),
    (5, 2000, 1040, 128, "bf16", F32), (128, 1000, 2056, 72, "bf16", BF16),
    (33, 3000, 4104, 120, "f16", F16),
    # 129-256 rows: the MMA's N side covers 256 rows of A, 128 copied per CTA
    (256, 2048, 1024, 0, "bf16", BF16), (200, 1000, 1040, 72, "f16", F32),
    (129, 4096, 520, 128, "bf16", F32), (256, 8192, 2048, 0, "f16", F16)])
def test_skinny_pair(M, N, K, nc, it, ot):
    A, B = make_inputs(M, N, K, it, "normal", M * 11 + K)
    C = run(A, B, ot, kernel="skinny_pair", bn=nc)
    cfg = sptg.last_config()
    assert "kernel=skinny-pair" in cfg, cfg
    if nc:
        assert f"cols_per_cta={nc} " in cfg, cfg
    assert_float_parity(C, A, B)


def test_skinny_pair_is_the_default_for_the_memory_bound_workload():
    # 64 x 8192 x 8192: 56 columns per SM, so CTA pairs over the whole of K
    A, B = make_inputs(64, 8192, 8192, "bf16", "normal", 45)
    C = run(A, B, BF16)
    cfg = sptg.last_config()
    assert "kernel=skinny-pair" in cfg, cfg
    nc = int(cfg.split("cols_per_cta=")[1].split()[0])
    grid = int(cfg.split("grid=")[1].split()[0])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert nc % 8 == 0 and grid == 2 * -(-8192 // (2 * nc)) and 3 * sms <= 4 * grid <= 4 * sms
    print(cfg, "max |err| / (1e-3 sum|ab|) =", assert_float_parity(C, A, B, plain=True))
    assert torch.equal(C, run(A, B, BF16))


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 17])
@pytest.mark.parametrize("stages", [0, 1, 2, 3])
@pytest.mark.parametrize("M", [64, 128, 256])
def test_k_tile_marker_skinny_pair(T, stages, M):
    # every K-chunk lands in the sum exactly once; T not a multiple of the
    # stage's chunks leaves the last stage partly empty
    A, B, expect = _marker_inputs(M, 1024, T, dtype=BF16)
    if M == 256 and stages == 1:
        # one 47 KB stage cannot hold the 256 x 56 fp32 output block: refused
        with pytest.raises(sptg.SptgError):
            run(A, B, F32, kernel="skinny_pair", bn=56, stages=stages)
        return
    C = run(A, B, F32, kernel="skinny_pair", bn=56, stages=stages)
    if stages:
        assert f"stages={stages}" in sptg.last_config()
    assert (C.to(torch.float64) == expect).all()


@pytest.mark.parametrize("M,N,T,nc", [(64, 1024, 260, 56), (128, 2048, 260, 32),
                                      (256, 1000, 129, 40), (64, 4000, 257, 120)])
def test_k_tile_marker_skinny_pair_staggered(M, N, T, nc):
    # 64 stages or more: the pairs start their K-loops at staggered chunks and
    # wrap around; every K-chunk must still land in each sum exactly once
    # (T K-tiles of 64, the last stage partly empty, its chunk somewhere in
    # the middle of most pairs' loops); binary16 holds the markers up to 2048
    # exactly (bfloat16 only up to 256)
    A, B, expect = _marker_inputs(M, N, T, dtype=F16)
    C = run(A, B, F32, kernel="skinny_pair", bn=nc)
    cfg = sptg.last_config()
    assert "k_rotate=1" in cfg, cfg
    assert (C.to(torch.float64) == expect).all()


@pytest.mark.parametrize("M,N,K,it,ot", [(64, 4096, 16392, "bf16", BF16),
                                         (128, 8192, 8200, "f16", F32),
                                         (96, 6000, 16384, "bf16", F32)])
def test_skinny_pair_staggered_parity(M, N, K, it, ot):
    A, B = make_inputs(M, N, K, it, "normal", M + K)
    C = run(A, B, ot, kernel="skinny_pair")
    assert "k_rotate=1" in sptg.last_config(), sptg.last_config()
    assert_float_parity(C, A, B)
    assert torch.equal(C, run(A, B, ot, kernel="skinny_pair"))  # the same order every call


@pytest.mark.parametrize("M", [64, 128, 256])
def test_skinny_pair_places_every_row_and_column(M):
    # A[m, k] = m + 1 and Bcm[n, k] = n % 61 + 1: C[m, n] = K (m + 1)(n % 61 + 1),
    # exact, so a row or column of the accumulator read from the wrong place
    # cannot go unseen
    N, K = 2000, 128
    A = (torch.arange(M, dtype=torch.float32) + 1).repeat(K, 1).t().contiguous().to(BF16)
    Bcm = (torch.arange(N) % 61 + 1).to(torch.float32).repeat(K, 1).t().contiguous().to(BF16)
    expect = K * torch.outer(torch.arange(M, dtype=torch.float64) + 1,
                             (torch.arange(N) % 61 + 1).to(torch.float64))
    for nc in (8, 40, 56, 64, 72, 128):
        C = run(A, Bcm, F32, kernel="skinny_pair", bn=nc)
        assert f"mma_n={M} " in sptg.last_config()
        assert torch.equal(C.to(torch.float64), expect), nc


@pytest.mark.parametrize("stages", [1, 2, 3, 5])
def test_skinny_pair_ablation_rings_match(stages):
    A, B = make_inputs(64, 2048, 4096, "bf16", "normal", 17)
    ref = run(A, B, BF16, kernel="skinny_pair", bn=40)
    got = run(A, B, BF16, kernel="skinny_pair", bn=40, stages=stages)
    assert f"stages={stages}" in sptg.last_config()
    assert torch.equal(ref, got)
    assert_float_parity(got, A, B)


def test_skinny_pair_limits():
    A, B = make_inputs(257, 2048, 1024, "bf16", "normal", 90)
    with pytest.raises(sptg.SptgError):
        run(A, B, BF16, kernel="skinny_pair")  # more than 256 rows
    A, B = make_inputs(64, 2048, 1024, "bf16", "normal", 91)
    for bad in (12, 136):
        with pytest.raises(sptg.SptgError):
            run(A, B, BF16, kernel="skinny_pair", bn=bad)
    with pytest.raises(sptg.SptgError):
        run(A, B, BF16, kernel="skinny_pair", bn=64, stages=5)  # 5 x 48 KB > the budget


@pytest.mark.parametrize("M,N,K,it,ot", [
    (128, 8192, 4096, "bf16", BF16), (96, 8192, 2048, "f16", F16), (65, 9216, 1040, "bf16", F32),
    (128, 8192, 2048, "f16", F32), (100, 16384, 1024, "bf16", BF16)])
def test_skinny_cluster_up_to_128_rows(M, N, K, it, ot):
    # 64 < M <= 128: the cluster split with MMA N = 128 (the default only past
    # 64 columns per SM; the CTA pairs take narrower outputs)
    A, B = make_inputs(M, N, K, it, "normal", M + N + K)
    C = run(A, B, ot, kernel="skinny_cluster")
    cfg = sptg.last_config()
    assert "kernel=skinny-cluster" in cfg and "mma_n=128" in cfg, cfg
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("M,N,K,kernel", [
    (64, 1024, 8192, "kernel=skinny-cluster"), (40, 3072, 4096, "kernel=skinny-cluster"),
    (64, 1024, 32768, "kernel=skinny "), (64, 6144, 2048, "kernel=skinny-pair"),
    (64, 12288, 2048, "kernel=skinny-rows"), (64, 32768, 1024, "kernel=skinny-rows"),
    (64, 40960, 1024, "kernel=skinny ")])
def test_default_kernel_up_to_64_rows(M, N, K, kernel):
    # narrow outputs: the cluster split even with SMs idle (stream-K for long
    # K); 32-64 columns per SM: CTA pairs; 65-256: strips; wider: stream-K
    A, B = make_inputs(M, N, K, "bf16", "normal", M + N + 1)
    C = run(A, B, BF16)
    assert sptg.last_config().startswith(kernel), sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("M,N,K,ot", [(128, 8192, 8192, BF16), (96, 4096, 4096, F32),
                                      (65, 1024, 2048, BF16), (100, 16384, 1024, BF16),
                                      (128, 1536, 4096, F32), (128, 24576, 1024, BF16),
                                      (256, 8192, 2048, BF16), (160, 4096, 1024, F32),
                                      (256, 16384, 1024, BF16)])
def test_default_kernel_up_to_256_rows(M, N, K, ot):
    # CTA pairs with MMA N = 128 up to 128 columns per SM (past that the
    # 128-column tiles outnumber the SMs, so the square kernel takes it);
    # 129-256 rows: pairs with MMA N = 256 up to 64 columns per SM
    A, B = make_inputs(M, N, K, "bf16", "normal", M + N)
    C = run(A, B, ot)
    cfg = sptg.last_config()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    c = -(-N // sms)
    if c > (128 if M <= 128 else 64):
        assert cfg.startswith("kernel=square"), cfg
    else:
        assert "kernel=skinny-pair" in cfg and f"mma_n={128 if M <= 128 else 256}" in cfg, cfg
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("T", [1, 3, 8])
@pytest.mark.parametrize("cs", [1, 2])
def test_k_tile_marker_skinny_cluster_128_rows(T, cs):
    A, B, expect = _marker_inputs(128, 1024, T * cs, dtype=BF16)
    C = run(A, B, BF16, kernel="skinny_cluster", splits=cs)
    assert "mma_n=128" in sptg.last_config()
    assert (C.to(torch.float64) == expect).all()


def test_skinny_cluster_128_rows_limits():
    A, B = make_inputs(96, 2048, 1024, "bf16", "normal", 85)
    with pytest.raises(sptg.SptgError):
        run(A, B, BF16, kernel="skinny_cluster", splits=4)  # no room for 4 ranks
    # too few column tiles for the cluster split: CTA pairs over the whole of K
    A, B = make_inputs(100, 1024, 2048, "bf16", "normal", 86)
    C = run(A, B, BF16)
    assert "kernel=skinny-pair" in sptg.last_config()
    assert_float_parity(C, A, B)


def test_skinny_cluster_matches_stream_k_and_is_deterministic():
    A, B = make_inputs(64, 8192, 8192, "bf16", "normal", 19)
    c1 = run(A, B, F32, kernel="skinny_cluster", splits=2)
    c2 = run(A, B, F32, kernel="skinny_cluster", splits=2)
    assert torch.equal(c1, c2)
    assert_float_parity(c1, A, B)
    for pair in (("f16", F16), ("f16", F32)):
        A2, B2 = make_inputs(48, 4096, 2048, pair[0], "uniform", 20)
        assert_float_parity(run(A2, B2, pair[1], kernel="skinny_cluster", splits=2), A2, B2)


def test_skinny_is_deterministic():
    A, B = make_inputs(64, 4096, 4096, "bf16", "normal", 9)
    c1 = run(A, B, F32, kernel="skinny")
    c2 = run(A, B, F32, kernel="skinny")
    assert torch.equal(c1, c2)


def test_skinny_f16_out_and_f32_out():
    A, B = make_inputs(40, 2048, 2048, "f16", "uniform", 10)
    assert_float_parity(run(A, B, F16, kernel="skinny"), A, B)
    assert_float_parity(run(A, B, F32, kernel="skinny"), A, B)


# ------------------------------------------------------------ stream-K tiles
def _sk_tiles():
    return int(sptg.last_config().split("stream_k_tiles=")[1].split()[0])


@pytest.mark.parametrize("cta_pair", [1, 2])
@pytest.mark.parametrize("it,out", [("f16", F32), ("f16", F16), ("bf16", BF16), ("bf16", F32)])
def test_stream_k_every_tile(cta_pair, it, out):
    # every tile cut along K over five workers (ragged M, N and K): the
    # partial sums go to scratch and the last contributor of each tile adds
    # them up in contributor order
    A, B = make_inputs(520, 776, 1096, it, "uniform", 40)
    C = run(A, B, out, kernel="square", bn=224, cta_pair=cta_pair, stream_k=2, splits=5)
    assert _sk_tiles() > 0 and f"pair={cta_pair - 1}" in sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("cta_pair", [1, 2])
def test_stream_k_many_contributors(cta_pair):
    # one tile, all workers: each holds 8 K-tiles of it, so the reduction
    # adds dozens of partials
    A, B = make_inputs(256, 256, 8192, "bf16", "normal", 41)
    C = run(A, B, F32, kernel="square", bn=256, cta_pair=cta_pair, stream_k=2)
    assert _sk_tiles() == (1 if cta_pair == 2 else 2)
    assert "stream_k_workers=" in sptg.last_config()
    assert int(sptg.last_config().split("stream_k_workers=")[1].split()[0]) >= 8
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("T,splits", [(17, 7), (40, 3), (9, 16)])
def test_k_tile_marker_stream_k(T, splits):
    # the K-tile marker through split tiles: a dropped, doubled or misplaced
    # K-tile at a cut changes the exact result
    A, B, expect = _marker_inputs(256, 512, T)
    for cta_pair in (1, 2):
        C = run(A, B, F32, kernel="square", bn=256, cta_pair=cta_pair, stream_k=2, splits=splits)
        assert _sk_tiles() > 0
        assert (C.to(torch.float64) == expect).all()


@pytest.mark.parametrize("bn", [128, 160, 224, 256])
@pytest.mark.parametrize("cta_pair", [1, 2])
def test_stream_k_int8_exact(cta_pair, bn):
    # cuts fall inside the 1024-product chunks, and a contributor's piece spans
    # several chunks; the int32 partials add exactly
    A, B = make_inputs(512, 384, 4160, "s8", "int8", 42)
    C = run(A, B, I32, cta_pair=cta_pair, stream_k=2, splits=6, bn=bn)
    assert _sk_tiles() > 0
    assert_int_parity(C, A, B)
    A = torch.full((130, 4096), -128, dtype=I8)
    B = torch.full((136, 4096), -128, dtype=I8)
    C = run(A, B, I32, cta_pair=cta_pair, stream_k=2, splits=7)
    assert (C.to(torch.int64) == 16384 * 4096).all()


def test_stream_k_is_deterministic_and_matches_data_parallel():
    A, B = make_inputs(1024, 1536, 2048, "f16", "normal", 43)
    c1 = run(A, B, F32, kernel="square", stream_k=2, splits=9)
    c2 = run(A, B, F32, kernel="square", stream_k=2, splits=9)
    assert torch.equal(c1, c2)
    c3 = run(A, B, F32, kernel="square", stream_k=1)
    assert _sk_tiles() == 0
    assert_float_parity(c1, A, B)
    assert_float_parity(c3, A, B)


def test_headline_schedule_fills_whole_rounds():
    # 4096 x 4096 in 256 x 224 pair tiles: 16 x 19 = 304 tiles, four whole
    # rounds of the pairs; the last tile column holds 64 of its 224 columns
    A, B = make_inputs(4096, 4096, 4096, "f16", "uniform", 44)
    C = run(A, B, F16)
    cfg = sptg.last_config()
    assert "pair=1" in cfg and "bn=224" in cfg and _sk_tiles() == 0, cfg
    rows, cols = sample_positions(4096, 4096, 20000, seed=44)
    extra = np.arange(0, 4096, dtype=np.int64)
    rows = np.concatenate([rows, extra])
    cols = np.concatenate([cols, 18 * 224 + extra % 64])
    assert_float_parity(C, A, B, rows, cols)


# ------------------------------------------------ 256 x 512 CTA-pair tiles
@pytest.mark.parametrize("M,N,K,it,ot,stream_k", [
    (768, 1096, 520, "f16", F16, 1),     # ragged N: the last tile holds 72 of 512 columns
    (512, 1536, 1024, "bf16", F32, 0),
    (300, 2048, 2080, "bf16", BF16, 2),  # every tile cut along K: 512-wide partials
    (256, 512, 64, "f16", F32, 1),       # one tile, one K-tile
])
def test_wide_pair_tiles_parity(M, N, K, it, ot, stream_k):
    # two 256-column MMAs per K-step into one 512-column accumulator; each
    # CTA copies its 128 rows of each half of the tile's B
    A, B = make_inputs(M, N, K, it, "uniform", 71)
    kw = {"splits": 5} if stream_k == 2 else {}
    C = run(A, B, ot, kernel="square", cta_pair=2, bn=512, stream_k=stream_k, **kw)
    cfg = sptg.last_config()
    assert "bn=512" in cfg and "pair=1" in cfg, cfg
    assert_float_parity(C, A, B)


def test_wide_tiles_need_a_float_pair():
    A, B = make_inputs(256, 512, 64, "f16", "uniform", 72)
    with pytest.raises(sptg.SptgError):
        run(A, B, F32, kernel="square", cta_pair=1, bn=512)
    A, B = make_inputs(256, 512, 64, "s8", "int8", 72)
    with pytest.raises(sptg.SptgError):
        run(A, B, I32, kernel="square", cta_pair=2, bn=512)


# ------------------------------------------------------------ leading dimensions
def _in_wider(X, pitch, fill):
    """X placed in the leading columns of a rows x pitch device buffer."""
    buf = torch.full((X.shape[0], pitch), fill, dtype=X.dtype)
    buf[:, :X.shape[1]] = X
    return buf.cuda()


@pytest.mark.parametrize("kernel,M,N,K,it,ot,extra", [
    ("square", 300, 264, 520, "f16", F32, {}),
    ("square", 520, 776, 1096, "bf16", BF16, {"cta_pair": 2, "stream_k": 2, "splits": 5}),
    ("square", 384, 512, 1024, "f16", F16, {"cta_pair": 1, "stream_k": 2, "splits": 7}),
    ("skinny", 48, 2048, 1024, "bf16", BF16, {}),
    ("skinny_cluster", 64, 4096, 2048, "f16", F16, {"splits": 2}),
    ("skinny_pair", 64, 4096, 2048, "bf16", F32, {"bn": 56}),
    ("skinny_pair", 33, 1000, 1096, "f16", F16, {"bn": 24}),
    ("skinny_rows", 64, 4096, 2048, "f16", F16, {"bn": 72}),
    ("skinny_rows", 17, 2056, 1096, "bf16", F32, {"bn": 128}),
])
def test_leading_dimensions(kernel, M, N, K, it, ot, extra):
    # A, Bcm and C as column slices of wider buffers: the tiles are read and
    # written through the row pitch, and C's columns past N stay untouched
    A, B = make_inputs(M, N, K, it, "uniform", 60 + M)
    dA = _in_wider(A, K + 64, 7)[:, :K]
    dB = _in_wider(B, K + 32, -3)[:, :K]
    Cbuf = torch.full((M, N + 24), 5, dtype=ot, device="cuda")
    C = Cbuf[:, :N]
    sptg.gemm(dA, dB, C=C, kernel=kernel, **extra)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    assert kernel.replace("_", "-") in sptg.last_config()
    assert (Cbuf[:, N:].cpu().to(torch.float64) == 5).all()
    assert_float_parity(C.cpu().contiguous(), A, B)


@pytest.mark.parametrize("stream_k", [1, 2])
def test_leading_dimensions_int8(stream_k):
    A, B = make_inputs(264, 136, 1040, "s8", "int8", 61)
    dA = _in_wider(A, 1040 + 48, 1)[:, :1040]
    dB = _in_wider(B, 1040 + 16, -1)[:, :1040]
    Cbuf = torch.full((264, 136 + 4), 9, dtype=I32, device="cuda")
    sptg.gemm(dA, dB, C=Cbuf[:, :136], stream_k=stream_k, splits=7 if stream_k == 2 else 0)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    assert (Cbuf[:, 136:].cpu() == 9).all()
    assert_int_parity(Cbuf[:, :136].cpu().contiguous(), A, B)


@pytest.mark.parametrize("it,ot,M,N,K,kw", [
    ("f16", F32, 300, 264, 520, {"kernel": "square", "cta_pair": 1}),
    ("bf16", BF16, 300, 456, 1096, {"kernel": "square", "cta_pair": 2}),
    ("bf16", F32, 300, 1040, 520, {"kernel": "square", "cta_pair": 2, "bn": 512}),
    ("f16", F16, 520, 776, 1096, {"kernel": "square", "cta_pair": 2, "stream_k": 2, "splits": 5}),
    ("s8", I32, 264, 136, 1040, {}),
    ("s8", I32, 264, 456, 2080, {"cta_pair": 2, "stream_k": 2, "splits": 6}),
    ("bf16", BF16, 48, 2048, 1024, {"kernel": "skinny"}),
    ("bf16", F32, 40, 2056, 2048, {"kernel": "skinny_cluster", "splits": 2}),
    ("bf16", BF16, 40, 2056, 2048, {"kernel": "skinny_pair", "bn": 64}),
    ("f16", F32, 5, 1000, 1040, {"kernel": "skinny_rows", "bn": 40}),
])
def test_rows_outside_c_stay_untouched(it, ot, M, N, K, kw):
    # C is rows 8 .. 8 + M of a taller buffer filled with a sentinel: a store
    # past row M (a tile's rows beyond the matrix) or before row 0 would land
    # in those guard rows
    A, B = make_inputs(M, N, K, it, "int8" if it == "s8" else "uniform", 62 + M)
    sentinel = 77
    Cbuf = torch.full((M + 48, N), sentinel, dtype=ot, device="cuda")
    C = Cbuf[8:8 + M]
    sptg.gemm(A.cuda(), B.cuda(), C=C, **kw)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    guard = torch.cat([Cbuf[:8], Cbuf[8 + M:]]).cpu().to(torch.float64)
    assert (guard == sentinel).all()
    if it == "s8":
        assert_int_parity(C.cpu(), A, B)
    else:
        assert_float_parity(C.cpu(), A, B)


def test_leading_dimensions_zero_k():
    Cbuf = torch.full((40, 72), 3.0, dtype=F32, device="cuda")
    A = torch.zeros(40, 0, dtype=F16, device="cuda")
    B = torch.zeros(64, 0, dtype=F16, device="cuda")
    sptg.gemm(A, B, C=Cbuf[:, :64])
    torch.cuda.synchronize()
    assert (Cbuf[:, :64].cpu() == 0).all() and (Cbuf[:, 64:].cpu() == 3).all()


# ------------------------------------------------------------ host buffers
@pytest.mark.parametrize("M,N,K,it,ot,kernel", [
    (264, 520, 1040, "f16", F16, "square"), (264, 520, 1040, "bf16", F32, "square"),
    (264, 520, 1040, "s8", I32, "square"),
    # the skinny kernels behind the host-buffer entry point as well
    (64, 8192, 2048, "bf16", BF16, "skinny-pair"), (64, 16384, 1024, "f16", F16, "skinny-rows"),
    (40, 3072, 2048, "bf16", F32, "skinny-cluster"), (128, 4096, 1024, "bf16", BF16, "skinny-pair")])
def test_host_buffers(M, N, K, it, ot, kernel):
    # sptg_gemm_host: operands and result in pinned host memory, the copies
    # enqueued by the library around the product
    A, B = make_inputs(M, N, K, it, "int8" if it == "s8" else "uniform", 70)
    hA, hB = A.pin_memory(), B.pin_memory()
    C = sptg.gemm_host(hA, hB, out_dtype=ot)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    assert sptg.last_config().startswith(f"kernel={kernel} "), sptg.last_config()
    if it == "s8":
        assert_int_parity(C.clone(), A, B)
    else:
        assert_float_parity(C.clone(), A, B)


def test_host_buffers_pageable_and_two_streams():
    A, B = make_inputs(300, 256, 512, "f16", "uniform", 71)
    hA, hB = A.pin_memory(), B.pin_memory()
    C1 = torch.empty(300, 256, dtype=F32)               # pageable
    C2 = torch.empty(300, 256, dtype=F32).pin_memory()  # pinned
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    sptg.gemm_host(A, B, C=C1, stream=s1)
    sptg.gemm_host(hA, hB, C=C2, stream=s2)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    assert_float_parity(C1, A, B)
    assert torch.equal(C1, C2)


# ------------------------------------------------------------ CUDA graphs
def _replay_three_times(call, C, A, B):
    # one call captured in a graph and replayed: the split-K counters must be
    # back at 0 after each replay, since every replay carries the generation
    # the call was captured with
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(s)  # sizes the stream's library buffers before the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    torch.cuda.synchronize()
    for _ in range(3):
        C.fill_(-1)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sptg.device_error() == 0
        assert_float_parity(C.cpu(), A, B)


@pytest.mark.parametrize("cta_pair", [1, 2])
def test_graph_replays_of_a_stream_k_call(cta_pair):
    A, B = make_inputs(520, 776, 1096, "bf16", "uniform", 81)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(520, 776, dtype=F32, device="cuda")
    _replay_three_times(lambda s: sptg.gemm(dA, dB, C=C, stream=s, cta_pair=cta_pair,
                                            stream_k=2, splits=5), C, A, B)


@pytest.mark.parametrize("stream_k", [0, 2])
def test_graph_replays_of_an_int8_call_with_new_inputs(stream_k):
    # The captured call widens the int8 operands into the stream's scratch and
    # multiplies them; every replay gets new inputs, which the replay must
    # widen again (and, when tiles are cut along K, count and reduce anew).
    M, N, K = 520, 456, 2080
    dA = torch.empty(M, K, dtype=I8, device="cuda")
    dB = torch.empty(N, K, dtype=I8, device="cuda")
    C = torch.empty(M, N, dtype=I32, device="cuda")
    s = torch.cuda.Stream()
    kw = {"stream_k": 2, "splits": 7} if stream_k else {}

    def call():
        sptg.gemm(dA, dB, C=C, stream=s, **kw)

    A, B = make_inputs(M, N, K, "s8", "int8", 90)
    dA.copy_(A)
    dB.copy_(B)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        call()  # sizes the stream's scratch before the capture
    s.synchronize()
    assert_int_parity(C.cpu(), A, B)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    torch.cuda.synchronize()
    for r in range(3):
        A, B = make_inputs(M, N, K, "s8", "int8", 91 + r)
        dA.copy_(A)
        dB.copy_(B)
        C.fill_(0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sptg.device_error() == 0
        assert_int_parity(C.cpu(), A, B)


def test_graph_replays_of_a_skinny_split_call():
    A, B = make_inputs(48, 2048, 1024, "bf16", "normal", 82)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(48, 2048, dtype=BF16, device="cuda")
    _replay_three_times(lambda s: sptg.gemm(dA, dB, C=C, stream=s, kernel="skinny"), C, A, B)
    assert "units=" in sptg.last_config()


@pytest.mark.parametrize("M,N,K,kernel", [(64, 8192, 2048, "skinny-pair"),
                                           (128, 4096, 1024, "skinny-pair"),
                                           (64, 16384, 1024, "skinny-rows"),
                                           (40, 3072, 2048, "skinny-cluster")])
def test_graph_replays_of_the_skinny_kernels_with_new_inputs(M, N, K, kernel):
    # captured once, replayed with new operands copied into the same buffers
    dA = torch.empty(M, K, dtype=BF16, device="cuda")
    dB = torch.empty(N, K, dtype=BF16, device="cuda")
    C = torch.empty(M, N, dtype=BF16, device="cuda")
    s = torch.cuda.Stream()
    A, B = make_inputs(M, N, K, "bf16", "normal", 84)
    dA.copy_(A)
    dB.copy_(B)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        sptg.gemm(dA, dB, C=C, stream=s)
    s.synchronize()
    assert sptg.last_config().startswith(f"kernel={kernel} "), sptg.last_config()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sptg.gemm(dA, dB, C=C, stream=s)
    torch.cuda.synchronize()
    for r in range(3):
        A, B = make_inputs(M, N, K, "bf16", "normal", 85 + r)
        dA.copy_(A)
        dB.copy_(B)
        C.fill_(0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sptg.device_error() == 0
        assert_float_parity(C.cpu(), A, B)


def test_graph_replays_of_the_allocation_free_call():
    A, B = make_inputs(64, 4096, 2048, "bf16", "normal", 83)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(64, 4096, dtype=BF16, device="cuda")

    def call(s):
        rc = sptg.gemm_skinny_noalloc_raw(64, 4096, 2048, "bf16_bf16", dA.data_ptr(),
                                          dB.data_ptr(), C.data_ptr(), s.cuda_stream)
        assert rc == 0
    _replay_three_times(call, C, A, B)


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_graph_capture_before_the_buffers_exist_is_refused():
    A, B = make_inputs(512, 768, 1024, "f16", "uniform", 84)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(512, 768, dtype=F32, device="cuda")
    s = torch.cuda.Stream()  # never used before: no scratch for it yet
    g = torch.cuda.CUDAGraph()
    with pytest.raises(sptg.SptgError, match="before graph capture"):
        with torch.cuda.graph(g, stream=s):
            sptg.gemm(dA, dB, C=C, stream=s, stream_k=2, splits=7)
    torch.cuda.synchronize()
    # the library and the context are fine afterwards
    assert_float_parity(run(A, B, F32, stream_k=2, splits=7), A, B)


# ------------------------------------------------------- host-only plan
@pytest.mark.parametrize("M,N,K", [
    (64, 8192, 4096), (64, 16384, 1024), (64, 1024, 8192), (64, 1024, 32768), (40, 3072, 4096),
    (64, 40960, 1024), (128, 8192, 2048), (256, 4096, 1024), (256, 16384, 1024),
    (1024, 1024, 1024), (4096, 4096, 1024)])
def test_plan_matches_the_launch(M, N, K):
    # sptg_plan, computed on the host alone, names the kernel and grid the
    # call then launches
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = sptg.plan(M, N, K, "bf16_bf16", sms)
    A, B = make_inputs(M, N, K, "bf16", "normal", 5)
    run(A, B, BF16)
    cfg = sptg.last_config()
    prefix = {"square": "kernel=square ", "skinny": "kernel=skinny ",
              "skinny_cluster": "kernel=skinny-cluster ", "skinny_rows": "kernel=skinny-rows ",
              "skinny_pair": "kernel=skinny-pair "}[p["kernel"]]
    assert cfg.startswith(prefix), (p, cfg)
    assert int(cfg.split("grid=")[1].split()[0]) == p["grid"], (p, cfg)


# ------------------------------------------------------------ stream / errors
def test_async_on_a_side_stream():
    A, B = make_inputs(512, 512, 512, "f16", "uniform", 21)
    dA, dB = A.cuda(), B.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = sptg.gemm(dA, dB, out_dtype=F32, stream=s)
    s.synchronize()
    assert_float_parity(C.cpu(), A, B)


@pytest.mark.parametrize("kernel,pair,stream_k", [(1, 1, 0), (1, 2, 0), (1, 1, 2), (1, 2, 2),
                                                   (2, 0, 0), (3, 0, 0), (4, 0, 0), (5, 0, 0)])
def test_bounded_wait_reports_timeout_and_context_survives(kernel, pair, stream_k):
    # The producer withholds one K-tile; the consumer's wait runs out after
    # 100 ms, the kernel tears down, and the host reads SPTG_ERR_TIMEOUT.
    # With every tile cut along K, the other contributors of the stalled
    # CTA's tiles count their arrival and go on: none of them waits for it.
    M = 512 if kernel == 1 else 64
    A, B = make_inputs(M, 1024, 1024, "bf16", "normal", 30)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, 1024, dtype=BF16, device="cuda")
    cfg = sptg.Config(kernel, 0, 0, 2 if kernel == 3 else 4, 100, 1, pair)
    cfg.stream_k = stream_k
    rc = sptg.gemm_raw(M, 1024, 1024, "bf16_bf16", dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                       torch.cuda.current_stream().cuda_stream, cfg)
    assert rc == 0
    assert sptg.device_error() == -5
    assert sptg.device_error() == 0  # the word was cleared
    # the context still works
    C = run(A, B, BF16, kernel={1: "square", 2: "skinny", 3: "skinny_cluster",
                                4: "skinny_rows", 5: "skinny_pair"}[kernel])
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("cta_pair,stream_k", [(1, 0), (2, 0), (1, 2), (2, 2)])
def test_bounded_wait_int8_reports_timeout_and_context_survives(cta_pair, stream_k):
    # the exact-integer kernel's eight epilogue warps and two reduction warps
    # leave together when the producer withholds a K-tile
    M, N, K = 512, 448, 2080
    A, B = make_inputs(M, N, K, "s8", "int8", 33)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=I32, device="cuda")
    cfg = sptg.Config(1, 224, 0, 4, 100, 1, cta_pair)
    cfg.stream_k = stream_k
    rc = sptg.gemm_raw(M, N, K, "s8_s32", dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                       torch.cuda.current_stream().cuda_stream, cfg)
    assert rc == 0
    assert sptg.device_error() == -5
    assert sptg.device_error() == 0
    C = run(A, B, I32, cta_pair=cta_pair, stream_k=stream_k, splits=4 if stream_k else 0)
    assert_int_parity(C, A, B)


@pytest.mark.parametrize("kernel,cta_pair", [("square", 1), ("square", 2), ("skinny", 0),
                                             ("skinny_cluster", 0), ("skinny_rows", 0),
                                             ("skinny_pair", 0)])
def test_timeline_trace_is_ordered(kernel, cta_pair):
    # the optional in-kernel timeline: per CTA the events come in pipeline
    # order, and CTA 0's K-tiles are consumed after they were issued
    M = 64 if kernel.startswith("skinny") else 512
    A, B = make_inputs(M, 2048, 2048, "bf16", "normal", 31)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, 2048, dtype=BF16, device="cuda")
    buf = torch.zeros(8 * 1024 + 128, dtype=torch.int64, device="cuda")
    cfg = sptg.Config(sptg.KERNELS[kernel], 0, 0, 2 if kernel == "skinny_cluster" else 0, 0, 0,
                      cta_pair)
    cfg.trace = buf.data_ptr()
    sptg.gemm(dA, dB, C=C, config=cfg)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    grid = int(sptg.last_config().split("grid=")[1].split()[0])
    t = buf.cpu().numpy()
    ev = t[:8 * 1024].reshape(1024, 8)[:grid]
    assert (ev[:, 0] > 0).all() and (ev[:, 6] > 0).all()
    for row in ev:
        assert row[0] <= row[1] <= row[3], row       # set-up, first copy, last copy
        assert row[6] >= row[5] >= row[0], row       # epilogue done before exit
    leaders = ev[:, 2] > 0
    assert (ev[leaders, 1] <= ev[leaders, 2]).all()  # data after its copy
    assert (ev[leaders, 2] <= ev[leaders, 4]).all()
    issue, full = t[8192:8256], t[8256:8320]
    n = int((full > 0).sum())
    assert n > 0 and (full[:n] >= issue[:n]).all()
    assert_float_parity(C.cpu(), A, B)
