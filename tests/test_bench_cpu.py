"""Host logic of bench.py on the CPU: the parity verdict a bench line carries
and its roofline arithmetic.

The verdict must say "ok" for a result within the element-wise bound and
must catch a single element outside it; the roofline must divide the
algorithmic work by the measured time and by the right peak.
"""
import pytest
import torch

import bench
import oracle
from workloads import DTYPE_PAIRS, Workload, make_inputs


def _exact_float(A, B):
    ref, _ = oracle.gemm_float(A, B, oracle.IN_F16)
    return torch.from_numpy(ref).to(torch.float32)


def test_parity_verdict_float_passes_and_catches_one_element():
    w = Workload("f16_48x40x64_f32out", 48, 40, 64, "f16_f32", "uniform", 1.0, 7)
    A, B = make_inputs(w.M, w.N, w.K, "f16", "uniform", w.seed)
    C = _exact_float(A, B)
    res = oracle.gemm_float(A, B, oracle.IN_F16)
    v = bench.parity_verdict(w, C, A, B, w.M, res)
    assert v["ok"] and v["checked"] == "every element" and v["elements"] == w.M * w.N
    assert v["max_err_over_1e-3_sum_abs"] < 1e-3  # fp32 rounding only
    # one element off by twice its bound fails, and only that one
    _, S = res
    bad = C.clone()
    bad[5, 7] += float(2.5e-3 * S[5, 7])
    v = bench.parity_verdict(w, bad, A, B, w.M, res)
    assert not v["ok"] and v["outside"] == 1 and v["max_err_over_bound"] > 2.0


def test_parity_verdict_sampled_rows_and_random_positions():
    w = Workload("f16_64x32x32_f32out", 64, 32, 32, "f16_f32", "uniform", 1.0, 8)
    A, B = make_inputs(w.M, w.N, w.K, "f16", "uniform", w.seed)
    C = _exact_float(A, B)
    res = oracle.gemm_float(A[:10], B, oracle.IN_F16)
    v = bench.parity_verdict(w, C, A, B, 10, res, n_random=50)
    assert v["ok"] and v["elements"] == 10 * w.N + 50
    assert "rows 0..9" in v["checked"] and "50 random" in v["checked"]
    # an error inside the sampled rows is always found
    bad = C.clone()
    bad[3, 3] += 1.0
    assert not bench.parity_verdict(w, bad, A, B, 10, res, n_random=50)["ok"]


def test_parity_verdict_int8_is_exact():
    w = Workload("s8_20x24x48_s32out", 20, 24, 48, "s8_s32", "int8", 1.0, 9)
    A, B = make_inputs(w.M, w.N, w.K, "s8", "int8", w.seed)
    ref = oracle.gemm_s8(A, B)
    C = torch.from_numpy(ref).to(torch.int32)
    v = bench.parity_verdict(w, C, A, B, w.M, ref)
    assert v["ok"] and v["mismatches"] == 0 and v["rule"] == "bit-exact"
    C[0, 0] += 1
    v = bench.parity_verdict(w, C, A, B, w.M, ref)
    assert not v["ok"] and v["mismatches"] == 1


def test_roofline_arithmetic():
    peaks, _ = bench.measured_peaks()
    # a square product is tensor-bound: achieved = 2 M N K / time
    w = Workload("f16_4096x4096x4096_f16out", 4096, 4096, 4096, "f16_f16", "uniform", 1.0, 2)
    r = bench.roofline(w, 0.08, 1.6, {"reasons": []}, "square", bench.algorithmic_bytes(w))
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(2 * 4096 ** 3 / 80e-6 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / peaks["bf16_tflops"])
    assert r["frac_dense_spec"] == pytest.approx(r["achieved"] / 2250.0)
    assert r["frac_dense_spec_nvl72"] == pytest.approx(r["achieved"] / 2500.0)
    assert r["algorithmic_bytes"] == 3 * 4096 * 4096 * 2
    # a timed region over a second takes the sustained peak
    r = bench.roofline(w, 0.08, 2000.0, {"reasons": []}, "square", bench.algorithmic_bytes(w))
    assert r["peak"] == peaks["bf16_tflops_sustained"]
    assert r["frac_burst"] == pytest.approx(r["achieved"] / peaks["bf16_tflops"])
    # so does a power cap that pulled the SM clock down ...
    capped = {"reasons": ["sw_power_cap"], "sm_mhz": 1500.0, "sm_max_mhz": 2070.0}
    r = bench.roofline(w, 0.08, 20.0, capped, "square", bench.algorithmic_bytes(w))
    assert r["peak"] == peaks["bf16_tflops_sustained"]
    # ... but not a cap flagged while the clock stayed at its maximum
    flagged = {"reasons": ["sw_power_cap"], "sm_mhz": 2070.0, "sm_max_mhz": 2070.0}
    r = bench.roofline(w, 0.08, 20.0, flagged, "square", bench.algorithmic_bytes(w))
    assert r["peak"] == peaks["bf16_tflops"]
    # the skinny product is bound by HBM: achieved = (A + B + C bytes) / time
    w = Workload("bf16_skinny_64x8192x8192_bf16out", 64, 8192, 8192, "bf16_bf16", "normal", 1.0, 4)
    b = bench.algorithmic_bytes(w)
    assert b == 136314880
    r = bench.roofline(w, 0.025, 0.5, {"reasons": []}, "skinny-cluster", b)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(b / 25e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / peaks["hbm_gbs"])


def test_job_throughput_counts_every_rank():
    # units of all ranks over the slowest rank's time
    assert bench.job_throughput(10.0, 4, 2.0) == pytest.approx(20.0)


def test_versus_torch_calls():
    # the PyTorch call timed beside each dtype pair computes the same product
    assert bench.torch_product("f16_f16")[1] == "torch.matmul"
    assert bench.torch_product("bf16_bf16")[1] == "torch.matmul"
    assert bench.torch_product("bf16_f32")[1] == "torch.mm(out_dtype=float32)"
    assert bench.torch_product("s8_s32")[1] == "torch._int_mm"
    A = torch.randn(8, 16, dtype=torch.float32)
    Bcm = torch.randn(4, 16, dtype=torch.float32)
    C = torch.empty(8, 4)
    bench.torch_product("f32_f32")[0](A, Bcm, C)
    assert torch.allclose(C, A @ Bcm.t())
    for spec in bench.VERSUS_SHAPES.split(";"):
        m, n, k, pair = spec.split(",")
        assert int(m) > 0 and int(n) > 0 and int(k) > 0 and pair in DTYPE_PAIRS


def test_clock_summary_counts_samples_under_load():
    # idle samples before and after the timed region read the maximum clock;
    # only those drawing at least half the run's highest power count
    s = bench.ClockSampler(0)
    idle = "0, 2070, 2070, 180.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    busy = "0, {c}, 2070, {p}, 0x4, Not Active, Not Active, Not Active, Active"
    s.lines = [idle, idle, idle, busy.format(c=1500, p=1390.0), busy.format(c=1480, p=1395.0),
               busy.format(c=1520, p=1380.0), idle]
    r = s.summary()
    assert r["sm_mhz"] == 1500 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"] and r["samples"] == 7 and r["samples_under_load"] == 3
    # the roofline then takes the sustained peak: the cap pulled the clock down
    peaks, _ = bench.measured_peaks()
    w = Workload("f16_4096x4096x4096_f16out", 4096, 4096, 4096, "f16_f16", "uniform", 1.0, 2)
    assert bench.roofline(w, 0.08, 100.0, r, "square",
                          bench.algorithmic_bytes(w))["peak"] == peaks["bf16_tflops_sustained"]
    # no power figure: the clock filter of before
    s.lines = ["0, 2070, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1900, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 300, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active"]
    r = s.summary()
    assert r["sm_mhz"] == 2070 and r["samples_under_load"] == 2
