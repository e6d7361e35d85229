"""The largest shapes: matrices of more than 2^31 elements.

Every address a kernel forms -- tensor-copy coordinates, row pitches times
rows, scratch offsets, the int8 widening's element counts -- must be 64-bit
where the product needs it. C or B here hold 2.5e9 to 4.3e9 elements. The
operands too large to draw on the host are drawn on the GPU from a seeded
generator; the oracle then checks sampled positions (corners, tile edges,
random ones), fed with just the rows of A and B those positions need.
"""
import numpy as np
import pytest
import torch

import oracle
import software_pipelined_tiled_gb300 as sptg
from gpu_helpers import IN_TYPE, OUT_ROUNDING, TOL, sample_positions
from workloads import make_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

F16, BF16, F32, I8, I32 = torch.float16, torch.bfloat16, torch.float32, torch.int8, torch.int32


def _check_sampled(C, dA, dB, r, c):
    """C (on the GPU) at (r, c) against the oracle on the needed rows only."""
    got = C[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].cpu()
    rr, ri = np.unique(r, return_inverse=True)
    cc, ci = np.unique(c, return_inverse=True)
    A_rows = dA[torch.from_numpy(rr).cuda()].cpu()
    B_rows = dB[torch.from_numpy(cc).cuda()].cpu()
    if dA.dtype == I8:
        ref = oracle.gemm_s8_at(A_rows, B_rows, ri, ci)
        assert (got.to(torch.int64).numpy() == ref).all()
        return
    ref, S = oracle.gemm_float_at(A_rows, B_rows, IN_TYPE[dA.dtype], ri, ci)
    err = np.abs(got.to(torch.float64).numpy() - ref)
    bound = TOL * S + OUT_ROUNDING[C.dtype] * (np.abs(ref) + TOL * S)
    assert np.isfinite(got.to(torch.float64).numpy()).all()
    assert (err <= bound).all(), f"max |err|/bound = {float((err / np.maximum(bound, 1e-300)).max()):.3e}"


def _gpu_operand(rows, K, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    if dtype == I8:
        return torch.randint(-128, 128, (rows, K), generator=g, device="cuda", dtype=I8)
    return (torch.rand((rows, K), generator=g, device="cuda") * 2 - 1).to(dtype)


@pytest.mark.parametrize("it,ot", [("f16", F16), ("s8", I32)])
def test_output_of_more_than_2_to_31_elements(it, ot):
    # square kernel: C is 65536 x 40960 = 2.7e9 elements
    M, N, K = 65536, 40960, 64
    A, B = make_inputs(M, N, K, it, "int8" if it == "s8" else "uniform", 93)
    dA, dB = A.cuda(), B.cuda()
    C = sptg.gemm(dA, dB, out_dtype=ot)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0 and "kernel=square" in sptg.last_config()
    r, c = sample_positions(M, N, 600, seed=3)
    _check_sampled(C, dA, dB, r, c)
    del C


@pytest.mark.parametrize("M,N,K,kernel", [
    (64, 9728, 262144, "kernel=skinny-pair"),     # 64 columns per CTA
    (40, 38912, 65536, "kernel=skinny-rows"),     # 256-column strips
    (64, 1048576, 4096, "kernel=skinny "),        # wider than the strips: stream-K
])
def test_skinny_operand_of_more_than_2_to_31_elements(M, N, K, kernel):
    # B is N x K = 2.5e9 to 4.3e9 elements, drawn on the GPU
    A, _ = make_inputs(M, 8, K, "bf16", "uniform", 94)
    dA = A.cuda()
    dB = _gpu_operand(N, K, BF16, 95)
    C = sptg.gemm(dA, dB, out_dtype=BF16)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0 and sptg.last_config().startswith(kernel), sptg.last_config()
    r, c = sample_positions(M, N, 200, seed=4)
    _check_sampled(C, dA, dB, r, c)
    del dB, C
