"""Host-side checks of the C ABI that need no GPU.

The library must build, load without a driver, and export every function
that include/sptgemm.h declares; argument checks that come before any device
work must return their documented codes.  No compute call is made here.
"""
import ctypes
import os
import re

import pytest

import software_pipelined_tiled_gb300 as sptg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sptgemm.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sptg_[a-z_0-9]+)\s*\(", text)))


def _header_enum(name):
    text = open(HEADER).read()
    m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
    assert m, name
    return int(m.group(1))


@pytest.fixture(scope="module")
def lib():
    sptg.build()
    return sptg.load()


def test_library_exports_every_declared_function(lib):
    declared = _declared_functions()
    assert declared, "no declarations found in the header"
    assert set(declared) == set(sptg.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
        getattr(lib, name)  # resolves through dlsym


def test_dtype_and_status_values_match_header():
    for key, val in {"SPTG_F16_F32": "f16_f32", "SPTG_F16_F16": "f16_f16", "SPTG_S8_S32": "s8_s32",
                     "SPTG_BF16_BF16": "bf16_bf16", "SPTG_BF16_F32": "bf16_f32"}.items():
        assert _header_enum(key) == sptg.DTYPES[val]
    for code, name in sptg.STATUS.items():
        assert _header_enum(name) == code


def test_version_and_status_strings(lib):
    assert lib.sptg_version() == 101
    for code in sptg.STATUS:
        assert sptg.status_string(code) and sptg.status_string(code) != "unknown status"
    assert sptg.status_string(12345) == "unknown status"


def test_argument_errors_before_device_work(lib):
    ok16 = 1 << 20  # a 16-byte aligned fake address; never dereferenced on these paths
    bad = ok16 + 8
    assert lib.sptg_gemm(4, 4, 16, 99, ok16, ok16, ok16, None) == -1          # unknown dtype
    assert lib.sptg_gemm(-1, 4, 16, 1, ok16, ok16, ok16, None) == -1          # negative M
    assert lib.sptg_gemm(4, 4, 1 << 31, 1, ok16, ok16, ok16, None) == -1      # K too large
    assert lib.sptg_gemm(4, 8, 16, 1, None, ok16, ok16, None) == -1           # null A
    assert lib.sptg_gemm(4, 8, 16, 1, ok16, ok16, None, None) == -1           # null C
    assert lib.sptg_gemm(4, 8, 16, 1, bad, ok16, ok16, None) == -2            # A misaligned
    assert lib.sptg_gemm(4, 8, 12, 1, ok16, ok16, ok16, None) == -2           # K*2 % 16 != 0
    assert lib.sptg_gemm(4, 4, 16, 1, ok16, ok16, ok16, None) == -2           # N*2 % 16 != 0
    assert lib.sptg_gemm(4, 2, 16, 0, ok16, ok16, ok16, None) == -2           # N*4 % 16 != 0
    assert lib.sptg_gemm(4, 4, 8, 2, ok16, ok16, ok16, None) == -2            # int8 K % 16 != 0
    # leading dimensions (elements): too small, or a pitch off the 16-byte rule
    g = lib.sptg_gemm_strided
    assert g(4, 8, 16, 1, ok16, 8, ok16, 16, ok16, 8, None, None) == -1        # lda < K
    assert g(4, 8, 16, 1, ok16, 16, ok16, 8, ok16, 8, None, None) == -1        # ldb < K
    assert g(4, 8, 16, 1, ok16, 16, ok16, 16, ok16, 4, None, None) == -1       # ldc < N
    assert g(4, 8, 16, 1, ok16, 20, ok16, 16, ok16, 8, None, None) == -2       # lda*2 % 16
    assert g(4, 8, 16, 1, ok16, 16, ok16, 16, ok16, 12, None, None) == -2      # ldc*2 % 16
    assert g(4, 8, 16, 1, ok16, 1 << 31, ok16, 16, ok16, 8, None, None) == -1  # lda >= 2^31
    # empty outputs are a no-op that touches nothing
    assert lib.sptg_gemm(0, 8, 16, 1, None, None, ok16, None) == 0
    assert lib.sptg_gemm(8, 0, 16, 1, None, None, ok16, None) == 0
    assert "empty" in sptg.last_config()


def test_invalid_config_fields(lib):
    ok16 = 1 << 20
    for cfg in (sptg.Config(6, 0, 0, 0, 0, 0), sptg.Config(0, -1, 0, 0, 0, 0),
                sptg.Config(0, 0, -2, 0, 0, 0), sptg.Config(0, 0, 0, 0, -5, 0),
                sptg.Config(0, 0, 0, 0, 0, 7), sptg.Config(0, 0, 0, 0, 0, 0, 4)):
        assert lib.sptg_gemm_ex(4, 8, 16, 1, ok16, ok16, ok16, None, ctypes.byref(cfg)) == -1
    cfg = sptg.Config()
    cfg.stream_k = 3
    assert lib.sptg_gemm_ex(4, 8, 16, 1, ok16, ok16, ok16, None, ctypes.byref(cfg)) == -1


def test_no_device_is_reported_not_hidden(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ok16 = 1 << 20
    rc = lib.sptg_gemm(128, 128, 64, 1, ok16, ok16, ok16, None)
    assert rc in (-3, -4)  # unsupported / runtime error; never a silent success
    assert sptg.last_error()


def test_python_binding_rejects_bad_tensors():
    import torch
    A = torch.zeros(4, 16, dtype=torch.float16)
    with pytest.raises(ValueError):
        sptg.gemm(A, torch.zeros(8, 8, dtype=torch.float16))
    with pytest.raises(ValueError):
        sptg.gemm(A, torch.zeros(8, 16, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        sptg.gemm(A, torch.zeros(8, 16, dtype=torch.float16))  # CPU tensors
    with pytest.raises(ValueError):
        sptg._dtype_key(torch.float16, torch.int32)
    with pytest.raises(ValueError):
        sptg._row_pitch(torch.zeros(16, 8).t(), "A")  # columns not contiguous
    wide = torch.zeros(4, 24)
    assert sptg._row_pitch(wide[:, :16], "A") == 24
