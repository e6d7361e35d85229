"""Seeded random sweep over shapes, dtype pairs and forced configurations.

Every case is small enough for the full oracle, so each element of C is
checked: int8 bit-exact, float within the element-wise bound. The shapes are
ragged (no tile multiple) within the library's 16-byte row-pitch rule, and the
configurations cover the automatic choice, one-CTA and CTA-pair tiles of
every width, stream-K never / chosen / every tile, and the three skinny kernels with their
cluster sizes, strip widths and ring depths.
"""
import random

import pytest
import torch

import software_pipelined_tiled_gb300 as sptg
from gpu_helpers import assert_float_parity, assert_int_parity, run
from workloads import make_inputs

pytestmark = pytest.mark.gpu

OUT = {"f16_f16": torch.float16, "f16_f32": torch.float32, "bf16_bf16": torch.bfloat16,
       "bf16_f32": torch.float32, "s8_s32": torch.int32}


def _case(i):
    rng = random.Random(1000 + i)
    dt = rng.choice(list(OUT))
    it = dt.split("_")[0]
    kind = rng.choice(["auto", "single", "pair", "pair", "pair", "skinny", "skinny_cluster"])
    if dt == "s8_s32" and kind in ("skinny", "skinny_cluster"):
        kind = "pair"
    kmul = 16 if it == "s8" else 8          # 16-byte rows of A and B
    nmul = 4 if OUT[dt].itemsize == 4 else 8  # 16-byte rows of C
    if kind.startswith("skinny"):
        M = rng.randint(1, 64 if kind == "skinny" else 128)
        N = nmul * rng.randint(1024 // nmul, 2600 // nmul)
    else:
        M = rng.randint(1, 700)
        N = nmul * rng.randint(1, 700 // nmul)
    K = kmul * rng.randint(1, 700 // kmul)
    kw = {}
    if kind in ("single", "pair"):
        kw["kernel"] = "square"
        kw["cta_pair"] = {"single": 1, "pair": 2}[kind]
        widths = (256, 224, 192, 160, 128) + ((512,) if kind == "pair" and it != "s8" else ())
        if it != "s8":
            widths += (240, 208, 176, 144, 112)
        kw["bn"] = rng.choice(widths)
        if kw["bn"] != 512:
            kw["stream_k"] = rng.choice([0, 1, 2])
            if kw["stream_k"] == 2:
                kw["splits"] = rng.randint(2, 40)
    elif kind == "skinny":
        kw["kernel"] = "skinny"
        kw["splits"] = rng.randint(1, 64)
    elif kind == "skinny_cluster":
        kw["kernel"] = "skinny_cluster"
        kw["splits"] = rng.choice([1, 2] if M > 64 else [1, 2, 4])
    return dt, it, M, N, K, kind, kw


@pytest.mark.parametrize("i", range(120))
def test_random_configuration(i):
    dt, it, M, N, K, kind, kw = _case(i)
    A, B = make_inputs(M, N, K, it, "int8" if it == "s8" else "uniform", 2000 + i)
    C = run(A, B, OUT[dt], **kw)
    cfg = sptg.last_config()
    if kind in ("single", "pair"):
        assert f"pair={int(kind == 'pair')}" in cfg, cfg
    if it == "s8":
        assert_int_parity(C, A, B)
    else:
        assert_float_parity(C, A, B)


@pytest.mark.parametrize("i", range(40))
def test_random_skinny_rows(i):
    # the column-strip skinny kernel: any strip width (multiple of 8 up to
    # 256), any ring depth that fits, ragged N and K, rows 1 ... 64
    rng = random.Random(5000 + i)
    dt = rng.choice(["f16_f16", "f16_f32", "bf16_bf16", "bf16_f32"])
    it = dt.split("_")[0]
    nmul = 4 if OUT[dt].itemsize == 4 else 8
    M = rng.randint(1, 64)
    N = nmul * rng.randint(8 // nmul, 2600 // nmul)
    K = 8 * rng.randint(1, 1400 // 8)
    nt = 8 * rng.randint(1, 32)
    stages = rng.randint(0, 4)
    A, B = make_inputs(M, N, K, it, "uniform", 6000 + i)
    C = run(A, B, OUT[dt], kernel="skinny_rows", bn=nt, stages=stages)
    assert "kernel=skinny-rows" in sptg.last_config()
    assert_float_parity(C, A, B)


@pytest.mark.parametrize("i", range(60))
def test_random_skinny_pair(i):
    # the CTA-pair skinny kernel: any column count per CTA (multiple of 8 up
    # to 128), any ring depth from 2 that fits (one stage cannot hold every
    # output block), ragged N and K, rows 1 ... 256
    rng = random.Random(7000 + i)
    dt = rng.choice(["f16_f16", "f16_f32", "bf16_bf16", "bf16_f32"])
    it = dt.split("_")[0]
    nmul = 4 if OUT[dt].itemsize == 4 else 8
    M = rng.randint(1, 256)
    N = nmul * rng.randint(8 // nmul, 2600 // nmul)
    K = 8 * rng.randint(1, 1400 // 8)
    nc = 8 * rng.randint(1, 16)
    stages = rng.choice([0, 2, 3, 4] if M <= 128 else [0, 2, 3])
    A, B = make_inputs(M, N, K, it, "uniform", 8000 + i)
    C = run(A, B, OUT[dt], kernel="skinny_pair", bn=nc, stages=stages)
    assert "kernel=skinny-pair" in sptg.last_config()
    assert_float_parity(C, A, B)
