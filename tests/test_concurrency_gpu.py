"""Calls from several host threads at once, each thread on its own stream.

The library keeps its tensor-map caches per host thread, its scratch and
host-call buffers per (device, stream), and its plan caches under one lock,
so concurrent calls must neither mix their buffers nor change their results:
every kernel here is deterministic, so each result must equal, bit for bit,
the same call made alone (which is itself checked against the oracle).
"""
import threading

import pytest
import torch

import software_pipelined_tiled_gb300 as sptg
from gpu_helpers import assert_float_parity, assert_int_parity, run
from workloads import make_inputs

pytestmark = pytest.mark.gpu

F16, BF16, F32, I32 = torch.float16, torch.bfloat16, torch.float32, torch.int32

# square pairs, square with every tile cut along K (scratch and counters),
# int8 (widened operands in scratch), the skinny CTA pairs, column strips,
# cluster split and stream-K (scratch and counters)
CASES = [
    (512, 768, 1040, "f16", F32, {}),
    (256, 1024, 4096, "bf16", F32, {"stream_k": 2, "splits": 9}),
    (300, 448, 2080, "s8", I32, {}),
    (64, 8192, 2048, "bf16", BF16, {}),
    (64, 16384, 1024, "f16", F16, {}),
    (40, 3072, 2048, "bf16", F32, {}),
    (48, 2048, 1024, "bf16", BF16, {"kernel": "skinny"}),
]


def test_concurrent_threads_and_streams():
    inputs = []
    for i, (M, N, K, it, ot, kw) in enumerate(CASES):
        A, B = make_inputs(M, N, K, it, "int8" if it == "s8" else "uniform", 700 + i)
        alone = run(A, B, ot, **kw)
        if it == "s8":
            assert_int_parity(alone, A, B)
        else:
            assert_float_parity(alone, A, B)
        inputs.append((A.cuda(), B.cuda(), ot, kw, alone))

    results, errors = {}, []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for rep in range(6):
                    for j in range(len(inputs)):
                        k = (j + t + rep) % len(inputs)  # threads interleave different kernels
                        dA, dB, ot, kw, _ = inputs[k]
                        outs.append((k, sptg.gemm(dA, dB, out_dtype=ot, stream=s, **kw)))
            s.synchronize()
            results[t] = outs
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    assert sorted(results) == [0, 1, 2, 3]
    for t, outs in results.items():
        assert len(outs) == 6 * len(inputs)
        for k, C in outs:
            assert torch.equal(C.cpu(), inputs[k][4]), (t, CASES[k])
