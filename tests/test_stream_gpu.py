"""GPU parity of the streaming ring (out = alpha * in) against its oracle.

Bit-exact: one binary32 multiplication per element on both sides. Covers the
pages' worked example (N = 2^20, in[i] = (i % 113) * 0.25, alpha = 2,
max_error = 0), ragged lengths around the 16-byte vector and the 32 KB tile,
several tiles per CTA (ring wrap), in-place use and the bounded-wait path.
"""
import numpy as np
import pytest
import torch

import oracle
import software_pipelined_tiled_gb300 as sptg

pytestmark = pytest.mark.gpu


def _run(x_cpu, alpha, **kw):
    x = x_cpu.cuda()
    out = sptg.stream_scale(x, alpha, **kw)
    torch.cuda.synchronize()
    assert sptg.device_error() == 0
    return out.cpu().numpy()


def test_pages_worked_example():
    n = 1 << 20
    x = torch.from_numpy(((np.arange(n) % 113) * 0.25).astype(np.float32))
    got = _run(x, 2.0)
    assert float(np.max(np.abs(got.astype(np.float64) - 2.0 * x.numpy().astype(np.float64)))) == 0.0
    assert np.array_equal(got.view(np.uint32), oracle.scale_f32(x, 2.0).view(np.uint32))


@pytest.mark.parametrize("n", [1, 3, 4, 5, 8191, 8192, 8193, 8195, 1000003, (1 << 26) + 7])
@pytest.mark.parametrize("alpha", [2.0, -1.5, 1.0 / 3.0])
def test_bit_exact_against_oracle(n, alpha):
    g = torch.Generator().manual_seed(n % 1000)
    x = torch.randn(n, generator=g) * 100
    got = _run(x, alpha)
    assert np.array_equal(got.view(np.uint32), oracle.scale_f32(x, alpha).view(np.uint32))


def test_in_place_and_empty():
    x = torch.randn(100000, generator=torch.Generator().manual_seed(2))
    ref = oracle.scale_f32(x, 0.5)
    d = x.cuda()
    sptg.stream_scale(d, 0.5, out=d)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    e = torch.empty(0, device="cuda")
    sptg.stream_scale(e, 2.0)


def test_bounded_wait_in_the_ring():
    x = torch.randn(1 << 22, device="cuda")
    cfg = sptg.Config(0, 0, 0, 0, 100, 1)
    sptg.stream_scale(x, 2.0, config=cfg)
    assert sptg.device_error() == -5
    assert sptg.device_error() == 0
    out = sptg.stream_scale(x, 2.0)
    torch.cuda.synchronize()
    assert torch.equal(out, x * 2)
