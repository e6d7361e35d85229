"""Pins the CPU oracle to facts that do not come from the oracle itself.

The oracle computes the plain product C = A * B (the definition the method
leaves unchanged: "Pipeline GPU Kernel", Step 5 item 4; "Hiding Memory
Latency in CUDA", section 15).  It is checked here against:

* exact rational arithmetic on tiny random shapes (brute force with
  ``fractions.Fraction``; input values decoded by numpy/torch, not by the
  oracle's own decoder), with the fp64 summation error bound K * 2^-53 * S;
* closed forms that must come out exact: identity, all-ones, one-hot column
  selection, the k-tile marker and the int8 extremes;
* a library routine: ``torch.matmul`` in float64;
* mutants of the oracle source (a dropped last term, a transposed operand, a
  sign error, a wrong exponent bias), each of which one of the pins rejects.
"""
import os
import random
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from workloads import make_inputs

EPS64 = 2.0 ** -53


# --------------------------------------------------------------------------
# helpers independent of the oracle
# --------------------------------------------------------------------------
def _exact_values(t: torch.Tensor):
    """Exact python Fractions of a f16/bf16/int8 tensor, via torch's own casts."""
    if t.dtype == torch.int8:
        return [[int(v) for v in row] for row in t.tolist()]
    as64 = t.to(torch.float64).tolist()  # f16/bf16 -> f64 is exact
    return [[Fraction(v) for v in row] for row in as64]


def _brute(A: torch.Tensor, Bcm: torch.Tensor):
    a, b = _exact_values(A), _exact_values(Bcm)
    M, K = A.shape
    N = Bcm.shape[0]
    C = [[sum((a[i][k] * b[j][k] for k in range(K)), Fraction(0) if A.dtype != torch.int8 else 0)
          for j in range(N)] for i in range(M)]
    S = [[sum((abs(a[i][k] * b[j][k]) for k in range(K)), Fraction(0) if A.dtype != torch.int8 else 0)
          for j in range(N)] for i in range(M)]
    return C, S


def _in_type(dt):
    return oracle.IN_BF16 if dt == torch.bfloat16 else oracle.IN_F16


# --------------------------------------------------------------------------
# decoders: all 65536 patterns against numpy (binary16) and torch (bfloat16)
# --------------------------------------------------------------------------
def test_decode_f16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode(int(b), oracle.IN_F16) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_bf16_all_patterns_match_torch():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode(int(b) & 0xFFFF, oracle.IN_BF16) for b in bits.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_f16_hand_values():
    # values fixed by the binary16 format itself
    cases = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24,
             0x0400: 2.0 ** -14, 0x3555: 0.333251953125, 0x8000: -0.0}
    for b, v in cases.items():
        assert oracle.decode(b, oracle.IN_F16) == v


# --------------------------------------------------------------------------
# brute force on tiny shapes
# --------------------------------------------------------------------------
def _tiny_cases(n, seed):
    rnd = random.Random(seed)
    return [(rnd.randint(1, 17), rnd.randint(1, 17), rnd.randint(1, 17), rnd.randint(0, 10 ** 6))
            for _ in range(n)]


@pytest.mark.parametrize("in_type,dist", [("f16", "uniform"), ("bf16", "normal"), ("f16", "normal")])
def test_float_oracle_against_exact_rationals(in_type, dist):
    for (M, N, K, seed) in _tiny_cases(70, hash((in_type, dist)) & 0xFFFF):
        A, Bcm = make_inputs(M, N, K, in_type, dist, seed, scale=3.0)
        C, S = oracle.gemm_float(A, Bcm, _in_type(A.dtype))
        Ce, Se = _brute(A, Bcm)
        for i in range(M):
            for j in range(N):
                exact, sabs = Ce[i][j], Se[i][j]
                bound = K * EPS64 * float(sabs)
                assert abs(Fraction(C[i, j]) - exact) <= Fraction(bound), (M, N, K, seed, i, j)
                assert abs(Fraction(S[i, j]) - sabs) <= Fraction(bound), (M, N, K, seed, i, j)


def test_int8_oracle_against_python_integers():
    for (M, N, K, seed) in _tiny_cases(80, 7):
        A, Bcm = make_inputs(M, N, K, "s8", "int8", seed)
        C = oracle.gemm_s8(A, Bcm)
        Ce, _ = _brute(A, Bcm)
        assert C.tolist() == Ce, (M, N, K, seed)


def test_operand_roles_on_a_rectangular_case():
    # A 2x3, B 3x2 written out by hand; B column-major means Bcm rows are B's columns.
    A = torch.tensor([[1, 2, 3], [4, 5, 6]], dtype=torch.float16)
    B = torch.tensor([[7, 8], [9, 10], [11, 12]], dtype=torch.float16)
    C, S = oracle.gemm_float(A, B.t().contiguous(), oracle.IN_F16)
    assert C.tolist() == [[58.0, 64.0], [139.0, 154.0]]
    assert S.tolist() == C.tolist()  # all products positive
    Ci = oracle.gemm_s8(A.to(torch.int8), B.t().contiguous().to(torch.int8))
    assert Ci.tolist() == [[58, 64], [139, 154]]


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_identity_gives_A():
    A, _ = make_inputs(37, 1, 24, "f16", "uniform", 11)
    eye = torch.eye(24, dtype=torch.float16)  # symmetric: its column-major form is itself
    C, _ = oracle.gemm_float(A, eye, oracle.IN_F16)
    assert np.array_equal(C, A.to(torch.float64).numpy())


def test_all_ones_gives_K():
    for K in (1, 63, 64, 4096):
        A = torch.ones(3, K, dtype=torch.bfloat16)
        Bcm = torch.ones(5, K, dtype=torch.bfloat16)
        C, S = oracle.gemm_float(A, Bcm, oracle.IN_BF16)
        assert (C == K).all() and (S == K).all()


def test_one_hot_selects_columns():
    A, _ = make_inputs(9, 1, 31, "bf16", "normal", 5)
    perm = [(7 * j + 3) % 31 for j in range(13)]
    Bcm = torch.zeros(13, 31, dtype=torch.bfloat16)
    for j, p in enumerate(perm):
        Bcm[j, p] = 1.0
    C, _ = oracle.gemm_float(A, Bcm, oracle.IN_BF16)
    assert np.array_equal(C, A.to(torch.float64).numpy()[:, perm])


@pytest.mark.parametrize("BK,T", [(64, 1), (64, 4), (64, 5), (128, 9), (32, 17)])
def test_k_tile_marker(BK, T):
    # A = 1 and B[k][j] = floor(k / BK) + 1: C = BK * T (T + 1) / 2 exactly.
    # A dropped, doubled or reordered k-tile changes the integer.
    K = BK * T
    A = torch.ones(4, K, dtype=torch.float16)
    col = (torch.arange(K) // BK + 1).to(torch.float16)
    Bcm = col.repeat(6, 1)
    C, _ = oracle.gemm_float(A, Bcm, oracle.IN_F16)
    assert (C == BK * T * (T + 1) // 2).all()


def test_int8_extremes():
    K = 4096
    A = torch.full((3, K), -128, dtype=torch.int8)
    B = torch.full((2, K), -128, dtype=torch.int8)
    assert (oracle.gemm_s8(A, B) == 16384 * K).all()
    alt = torch.tensor([-128 if k % 2 == 0 else 127 for k in range(K)], dtype=torch.int8)
    C = oracle.gemm_s8(alt.repeat(2, 1), alt.repeat(3, 1))
    assert (C == (K // 2) * 16384 + (K // 2) * 127 * 127).all()
    C2 = oracle.gemm_s8(alt.repeat(2, 1), (-alt.to(torch.int16)).clamp(-128, 127).to(torch.int8).repeat(3, 1))
    # (-128)*(127) + 127*(-127) per pair
    assert (C2 == (K // 2) * (-128 * 127) + (K // 2) * (127 * -127)).all()


def test_empty_inner_dimension_gives_zeros():
    A = torch.zeros(3, 0, dtype=torch.float16)
    B = torch.zeros(4, 0, dtype=torch.float16)
    C, S = oracle.gemm_float(A, B, oracle.IN_F16)
    assert C.shape == (3, 4) and (C == 0).all() and (S == 0).all()
    Ci = oracle.gemm_s8(torch.zeros(2, 0, dtype=torch.int8), torch.zeros(5, 0, dtype=torch.int8))
    assert Ci.shape == (2, 5) and (Ci == 0).all()


# --------------------------------------------------------------------------
# library special case: float64 matmul
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,in_type", [(256, "f16"), (1024, "bf16")])
def test_against_torch_float64_matmul(n, in_type):
    A, Bcm = make_inputs(n, n, n, in_type, "uniform", 99)
    C, S = oracle.gemm_float(A, Bcm, _in_type(A.dtype))
    ref = A.to(torch.float64) @ Bcm.to(torch.float64).t()
    err = np.abs(C - ref.numpy())
    assert (err <= 4 * n * EPS64 * S).all()


def test_sampled_positions_match_full_product():
    A, Bcm = make_inputs(40, 33, 70, "bf16", "normal", 3)
    C, S = oracle.gemm_float(A, Bcm, oracle.IN_BF16)
    rows = np.array([0, 39, 17, 5, 39])
    cols = np.array([0, 32, 9, 31, 0])
    c, s = oracle.gemm_float_at(A, Bcm, oracle.IN_BF16, rows, cols)
    assert np.array_equal(c, C[rows, cols]) and np.array_equal(s, S[rows, cols])
    Ai, Bi = make_inputs(40, 33, 70, "s8", "int8", 3)
    Ci = oracle.gemm_s8(Ai, Bi)
    assert np.array_equal(oracle.gemm_s8_at(Ai, Bi, rows, cols), Ci[rows, cols])


# --------------------------------------------------------------------------
# mutants: every plausible slip in the oracle is caught by a pin above
# --------------------------------------------------------------------------
_MUTANTS = {
    "drops_last_term": ("for (int64_t k = 0; k < K; ++k) {\n                double p = ai[k] * bj[k];",
                        "for (int64_t k = 0; k < K - 1; ++k) {\n                double p = ai[k] * bj[k];"),
    "transposed_B": ("double p = ai[k] * bj[k];\n                sum += p;", "double p = ai[k] * b[k * N + j];\n                sum += p;"),
    "sign_error": ("sum += p;\n                sabs", "sum += (k == 0 ? -p : p);\n                sabs"),
    "wrong_f16_bias": ("expo - 25", "expo - 24"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle_gemm.c")).read()
    old, new = _MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    stream_src = os.path.join(os.path.dirname(oracle.__file__), "oracle_stream.c")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(so), str(path),
                    stream_src, "-lm"], check=True)
    return so


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_pins_reject_mutants(tmp_path, name, monkeypatch):
    so = _build_mutant(tmp_path, name)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: str(so))
    failed = False
    for pin in (lambda: test_float_oracle_against_exact_rationals("f16", "uniform"),
                test_operand_roles_on_a_rectangular_case,
                test_decode_f16_hand_values,
                lambda: test_k_tile_marker(64, 4)):
        try:
            pin()
        except AssertionError:
            failed = True
            break
    monkeypatch.setattr(oracle, "_lib", None)
    assert failed, f"mutant {name} passed every pin"
