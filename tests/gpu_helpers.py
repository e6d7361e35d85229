"""Shared helpers of the GPU parity tests: run the library, ask the oracle, compare.

The float bar is the per-element bound |C - C_ref| <= 1e-3 * sum_k |A_ik B_kj|
on the fp32-accumulated sum (C_ref the oracle's fp64 sum), plus, for a 16-bit
output type, the rounding of that sum to the output type: at most u |x| with
u = 2^-11 (binary16) or 2^-8 (bfloat16) for round-to-nearest.  The int8 bar
is equality with the oracle's int64 sum.
"""
import numpy as np
import torch

import oracle
import software_pipelined_tiled_gb300 as sptg

TOL = 1e-3  # relative to sum_k |A_ik B_kj|
# unit roundoff of the output type (round to nearest even)
OUT_ROUNDING = {torch.float32: 0.0, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}

IN_TYPE = {torch.float16: oracle.IN_F16, torch.bfloat16: oracle.IN_BF16}


def run(A, Bcm, out_dtype, **kw):
    """Runs the library on CPU tensors A, Bcm; returns C on the CPU."""
    dA, dB = A.cuda(), Bcm.cuda()
    C = sptg.gemm(dA, dB, out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    return C.cpu()


def assert_float_parity(C, A, Bcm, rows=None, cols=None, plain=False):
    """Element-wise bound against the oracle (full, or at sampled positions).

    Returns max |err| / (1e-3 * S), the error against the unmodified bound of
    the fp32 sum. With plain=True that bound itself must hold as well (it can
    where the output rounding u |C| is small against 1e-3 * S, i.e. at large K
    or with a 4-byte output)."""
    it = IN_TYPE[A.dtype]
    got = C.to(torch.float64).numpy()
    if rows is None:
        ref, S = oracle.gemm_float(A, Bcm, it)
    else:
        ref, S = oracle.gemm_float_at(A, Bcm, it, rows, cols)
        got = got[rows, cols]
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref)
    u = OUT_ROUNDING[C.dtype]
    bound = TOL * S + u * (np.abs(ref) + TOL * S)
    tiny = np.finfo(np.float64).tiny
    ratio = err / np.maximum(bound, tiny)
    worst = float(ratio.max()) if ratio.size else 0.0
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} elements outside the bound; "
                           f"max |err|/bound = {worst:.3e}")
    plain_ratio = err / np.maximum(TOL * S, tiny)
    worst_plain = float(plain_ratio.max()) if plain_ratio.size else 0.0
    if plain:
        assert (err <= TOL * S).all(), f"max |err| / (1e-3 sum|ab|) = {worst_plain:.3e} > 1"
    return worst_plain


def assert_int_parity(C, A, Bcm, rows=None, cols=None):
    got = C.to(torch.int64).numpy()
    if rows is None:
        ref = oracle.gemm_s8(A, Bcm)
    else:
        ref = oracle.gemm_s8_at(A, Bcm, rows, cols)
        got = got[rows, cols]
    mism = got != ref
    assert not mism.any(), f"{int(mism.sum())} int8 results differ from the oracle"


def sample_positions(M, N, n, seed=0):
    """n positions: the four corners, tile edges, and uniform random ones."""
    g = np.random.default_rng(seed)
    fixed_r = [0, 0, M - 1, M - 1, min(127, M - 1), min(128, M - 1)]
    fixed_c = [0, N - 1, 0, N - 1, min(255, N - 1), min(256, N - 1)]
    r = np.concatenate([fixed_r, g.integers(0, M, n)])
    c = np.concatenate([fixed_c, g.integers(0, N, n)])
    return r.astype(np.int64), c.astype(np.int64)
