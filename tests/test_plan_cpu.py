"""Host logic of the square kernel's planning, through the C ABI, on the CPU.

sptg_plan_square runs the tile-shape model and the stream-K split of
sptg_gemm_ex without touching a device. These tests check the choices the
method depends on (whole rounds of 256 x 224 pair tiles at 4096^3, a
partial last round cut along K for a long K-loop, small products left
data-parallel, the int8 tile widths, no cluster-sharing mode) and, over
many random
shapes and configurations, the invariants the kernels rely on: a cut tile
never has more contributors than the scratch holds slots for, every
stream-K worker gets at least 8 K-tiles, and forced settings are honoured.
"""
import random

import pytest

import software_pipelined_tiled_gb300 as sptg

SM = 152  # GB300


def plan(M, N, K, dtype="f16_f16", sm=SM, **cfg):
    c = None
    if cfg:
        c = sptg.Config()
        for k, v in cfg.items():
            setattr(c, k, v)
    return sptg.plan_square(M, N, K, dtype, sm, c)


def test_headline_fills_whole_rounds():
    p = plan(4096, 4096, 4096)
    # 256 x 224 pair tiles: 16 x 19 = 304 tiles = exactly 4 rounds of 76 pairs
    assert (p["bn"], p["pair"], p["tiles"], p["workers"]) == (224, 1, 304, 76)
    assert p["tiles"] % p["workers"] == 0
    assert p["stream_k_tiles"] == 0


def test_long_k_takes_wide_pair_tiles():
    # 256 x 512 pair tiles (one accumulator, a quarter fewer copied bytes per
    # FLOP): 32 x 16 = 512 tiles = 6.7 rounds of 76 pairs, never cut along K
    p = plan(8192, 8192, 16384, "bf16_f32")
    assert (p["bn"], p["pair"], p["tiles"], p["workers"]) == (512, 1, 512, 76)
    assert p["stream_k_tiles"] == 0
    # short K-loops keep the double-buffered accumulators
    assert plan(8192, 8192, 4096)["bn"] == 256
    assert plan(16384, 16384, 4096, "bf16_bf16")["bn"] == 256


def test_widths_in_steps_of_16_fill_rounds():
    # 768 x 8192: 256 x 176 pair tiles, 3 x 47 = 141 tiles in two rounds of 76
    # pairs (256-wide tiles: 96 tiles, 1.26 rounds)
    p = plan(768, 8192, 8192, "bf16_bf16")
    assert (p["bn"], p["pair"], p["tiles"], p["stream_k_tiles"]) == (176, 1, 141, 0)
    # 256^3: six single-CTA tiles of 128 x 112 (four of 128 x 128 before)
    p = plan(256, 256, 256, "f16_f32")
    assert (p["bn"], p["pair"], p["tiles"]) == (112, 0, 6)
    # 512 x 4096 x 4096: 4 x 37 = 148 single-CTA tiles of 128 x 112, one round
    p = plan(512, 4096, 4096)
    assert (p["bn"], p["pair"], p["tiles"], p["workers"]) == (112, 0, 148, 148)


def test_long_k_at_256_columns_cuts_the_partial_last_round():
    p = plan(8192, 8192, 16384, "bf16_f32", bn=256)
    # 256 x 256 pair tiles: 32 x 32 = 1024 tiles = 13 rounds of 76 pairs + 36
    assert (p["bn"], p["pair"], p["tiles"], p["workers"]) == (256, 1, 1024, 76)
    assert p["stream_k_tiles"] == 1024 % 76 == 36
    assert p["stream_k_workers"] == 76


@pytest.mark.parametrize("size", [256, 512, 1024, 2048])
def test_small_products_stay_data_parallel(size):
    assert plan(size, size, size)["stream_k_tiles"] == 0


def test_int8_takes_the_float_tiles():
    # exact int8 keeps its int32 sums in the epilogue's registers: tensor
    # memory holds the two accumulators of a float tile, so int8 takes the
    # same widths (the 512-wide tile, with a single accumulator, excepted)
    for size in (1024, 4096, 8192):
        p = plan(size, size, size, "s8_s32")
        assert p["bn"] in (128, 160, 192, 224, 256)
    # whole rounds of 256 x 224 pair tiles at the int8 workload size
    p = plan(4096, 4096, 4096, "s8_s32")
    assert (p["bn"], p["pair"], p["stream_k_tiles"]) == (224, 1, 0)
    assert plan(4096, 4096, 4096, "s8_s32", cta_pair=1)["pair"] == 0


def test_stream_k_settings():
    assert plan(4096, 4096, 4096, stream_k=1)["stream_k_tiles"] == 0
    p = plan(4096, 4096, 4096, stream_k=2)
    assert p["stream_k_tiles"] == p["tiles"]


FLOAT_WIDTHS = tuple(range(112, 257, 16))


def test_forced_fields_are_honoured():
    for bn in FLOAT_WIDTHS:
        for pair in (1, 2):
            p = plan(3000, 5000, 700, bn=bn, cta_pair=pair)
            assert p["bn"] == bn and p["pair"] == pair - 1
    # int8 tiles in steps of 32 columns only
    for bn in (128, 160, 192, 224, 256):
        assert plan(3000, 5000, 704, "s8_s32", bn=bn)["bn"] == bn
    for bn in (112, 144, 176, 208, 240, 96):
        with pytest.raises(sptg.SptgError):
            plan(3000, 5000, 704, "s8_s32", bn=bn)
    assert plan(3000, 5000, 700, bn=512, cta_pair=2)["bn"] == 512
    for args, cfg in [((3000, 5000, 700), {"bn": 512, "cta_pair": 1}),
                      ((3000, 5000, 704, "s8_s32"), {"bn": 512})]:
        with pytest.raises(sptg.SptgError):
            plan(*args, **cfg)
    assert plan(4096, 4096, 4096, splits=10)["workers"] <= 10


def test_arguments_are_checked():
    for args in [(0, 64, 64, "f16_f16", SM), (64, 64, 64, "f16_f16", 1),
                 (64, 64, -1, "f16_f16", SM)]:
        with pytest.raises(sptg.SptgError):
            sptg.plan_square(*args)
    c = sptg.Config()
    c.stream_k = 3
    with pytest.raises(sptg.SptgError):
        sptg.plan_square(64, 64, 64, "f16_f16", SM, c)


def _owner(u, G, U):
    # the worker whose unit range [w * U / G, (w + 1) * U / G) holds unit u
    for w in range(G):
        if w * U // G <= u < (w + 1) * U // G:
            return w
    raise AssertionError("unit without a worker")


def test_plan_invariants_over_random_shapes():
    rng = random.Random(7)
    dtypes = ["f16_f16", "f16_f32", "bf16_bf16", "bf16_f32", "s8_s32"]
    for _ in range(300):
        M, N = rng.randint(1, 20000), rng.randint(1, 20000)
        K = rng.randint(1, 9000)
        dt = rng.choice(dtypes)
        sm = rng.choice([8, 20, 100, 132, 148, 152])
        cfg = {}
        if rng.random() < 0.3:
            cfg["stream_k"] = rng.choice([0, 1, 2])
        if rng.random() < 0.3:
            cfg["splits"] = rng.randint(1, 40)
        if cfg.get("stream_k") == 2 and M * N > 4e7:
            cfg["stream_k"] = 0  # every tile cut needs a counter per tile: keep it small
        p = plan(M, N, K, dt, sm, **cfg)
        rows = 256 if p["pair"] else 128
        assert p["bn"] in FLOAT_WIDTHS + (512,)
        if p["bn"] == 512:
            assert p["pair"] == 1 and dt != "s8_s32" and p["stream_k_tiles"] == 0
        if dt == "s8_s32":
            assert p["bn"] != 512 and p["bn"] % 32 == 0
        assert p["tiles"] == -(-M // rows) * -(-N // p["bn"])
        kt = -(-K // 64)
        t, g, mc = p["stream_k_tiles"], p["stream_k_workers"], p["max_contrib"]
        assert 0 <= t <= p["tiles"] and g <= max(p["workers"], 1)
        if cfg.get("stream_k") == 1:
            assert t == 0
        if t == 0:
            continue
        U = t * kt
        if g >= 2:
            assert U // g >= 8, "every stream-K worker gets at least 8 K-tiles"
        # contributors per cut tile never exceed the partial slots
        if U <= 20000:
            for sk in range(t):
                first, last = _owner(sk * kt, g, U), _owner((sk + 1) * kt - 1, g, U)
                assert last - first + 1 <= mc


def test_no_multicast_mode():
    # every CTA copies its own operand tiles: there is no cluster-sharing mode
    for cfg in ({"cta_pair": 3}, {"cta_pair": -1}):
        with pytest.raises(sptg.SptgError):
            plan(4096, 4096, 4096, **cfg)


def test_two_chunk_stages_count_in_the_stream_k_split():
    # Float CTA pairs over K-loops of 32 K-chunks or more whose two-chunk ring
    # keeps four stages take two 64-wide K-chunks per stage, and the stream-K
    # split counts in stages: one cut tile over every pair, at least 8 stages
    # (16 K-chunks) each. 176-wide pairs with 16-bit C qualify; with fp32 C
    # (three two-chunk stages) and single CTAs they keep one chunk per stage.
    K = 64 * 600  # 600 K-chunks, 300 two-chunk stages
    for dtype, pair, chunks in [("f16_f16", 2, 2), ("bf16_bf16", 2, 2), ("f16_f32", 2, 1),
                                ("bf16_f32", 2, 1), ("f16_f16", 1, 1)]:
        p = plan(256 if pair == 2 else 128, 176, K, dtype, bn=176, cta_pair=pair, stream_k=2)
        assert p["stream_k_tiles"] == p["tiles"] == 1
        stages = -(-K // (64 * chunks))
        workers = SM // 2 if pair == 2 else SM
        assert p["stream_k_workers"] == min(workers, stages // 8), (dtype, pair)
    # a short K-loop (fewer than 32 K-chunks) keeps one chunk per stage
    p = plan(256, 176, 64 * 31, "f16_f16", bn=176, cta_pair=2, stream_k=2)
    assert p["stream_k_workers"] == min(SM // 2, 31 // 8)
    # int8 never takes two chunks (its exact sums are cut every 1024 products)
    p = plan(256, 192, 64 * 600, "s8_s32", bn=192, cta_pair=2, stream_k=2)
    assert p["stream_k_workers"] == min(SM // 2, 600 // 8)
