"""The allocation-free skinny entry point, called through the C ABI.

Some callers cannot let a library allocate device memory: a serving process
that reserved the GPU's memory for its own pool up front, or latency-critical
code that cannot take the synchronisation an allocation may imply.  For them
sptg_gemm_skinny_noalloc runs the skinny kernel with its split-K scratch in a
fixed array compiled into the library.  Its output must agree with
sptg_gemm's, on every call: the array is shared by all calls and keeps the
last call's partial sums, so a second call in a row must not be disturbed by
what the first one left there.
"""
import numpy as np
import pytest
import torch

import oracle
import software_pipelined_tiled_gb300 as sptg
from gpu_helpers import OUT_ROUNDING, TOL
from workloads import make_inputs

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


def _bound(A, B, out_dtype):
    ref, S = oracle.gemm_float(A, B, oracle.IN_BF16)
    u = OUT_ROUNDING[out_dtype]
    return ref, TOL * S + u * (np.abs(ref) + TOL * S)


@pytest.mark.parametrize("M,N,K", [(64, 8192, 8192), (17, 1000, 1000), (64, 2048, 3072)])
def test_noalloc_matches_the_allocating_entry_on_two_calls(M, N, K):
    A, B = make_inputs(M, N, K, "bf16", "normal", 40 + M + K)
    dA, dB = A.cuda(), B.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    ref_gpu = torch.empty(M, N, dtype=BF16, device="cuda")
    skinny = sptg.Config(2, 0, 0, 0, 0, 0)  # the same kernel through sptg_gemm_ex
    assert sptg.gemm_raw(M, N, K, "bf16_bf16", dA.data_ptr(), dB.data_ptr(), ref_gpu.data_ptr(),
                         stream, skinny) == 0
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    existing = ref_gpu.cpu().to(torch.float64).numpy()
    ref, bound = _bound(A, B, BF16)
    # The calls below go to a new stream, for which the allocating entry
    # points hold no cached scratch: had this entry point asked for scratch
    # after all, it would have to allocate some, and the device's free memory
    # would drop. The outputs are allocated before the free memory is read.
    side = torch.cuda.Stream()
    outs = [torch.full((M, N), float("nan"), dtype=BF16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for call, out in enumerate(outs):
        rc = sptg.gemm_skinny_noalloc_raw(M, N, K, "bf16_bf16", dA.data_ptr(), dB.data_ptr(),
                                          out.data_ptr(), side.cuda_stream)
        assert rc == 0, sptg.last_error()
        side.synchronize()
        assert sptg.device_error(side) == 0
        got = out.cpu().to(torch.float64).numpy()
        assert np.isfinite(got).all(), f"call {call}: output not fully written"
        assert (np.abs(got - existing) <= bound).all(), f"call {call}: differs from sptg_gemm"
        assert (np.abs(got - ref) <= bound).all(), f"call {call}: outside the oracle bound"
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, f"device memory changed by {free_before - free_after} bytes"


def test_noalloc_rejects_what_it_cannot_hold():
    stream = torch.cuda.current_stream().cuda_stream
    # a split that needs ~128 MiB of partial tiles: far beyond the fixed array
    # (3 K-steps of 128 per column tile, 6144 units over the CTAs: the CTA
    # boundaries fall inside column tiles)
    M, N, K = 64, 262144, 384
    A = torch.zeros(M, K, dtype=BF16, device="cuda")
    B = torch.zeros(N, K, dtype=BF16, device="cuda")
    C = torch.empty(M, N, dtype=BF16, device="cuda")
    rc = sptg.gemm_skinny_noalloc_raw(M, N, K, "bf16_bf16", A.data_ptr(), B.data_ptr(),
                                      C.data_ptr(), stream)
    assert rc == -7 and "fixed scratch" in sptg.last_error()
    # int8 and more than 64 rows are outside this entry point
    A8 = torch.zeros(16, 64, dtype=torch.int8, device="cuda")
    B8 = torch.zeros(256, 64, dtype=torch.int8, device="cuda")
    C32 = torch.empty(16, 256, dtype=torch.int32, device="cuda")
    assert sptg.gemm_skinny_noalloc_raw(16, 256, 64, "s8_s32", A8.data_ptr(), B8.data_ptr(),
                                        C32.data_ptr(), stream) == -7
    A2 = torch.zeros(65, 64, dtype=BF16, device="cuda")
    C2 = torch.empty(65, 256, dtype=BF16, device="cuda")
    B2 = torch.zeros(256, 64, dtype=BF16, device="cuda")
    assert sptg.gemm_skinny_noalloc_raw(65, 256, 64, "bf16_bf16", A2.data_ptr(), B2.data_ptr(),
                                        C2.data_ptr(), stream) == -7
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
