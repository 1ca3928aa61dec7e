"""The measured FP8 tensor-core ceiling (an MMA-only kernel on every SM): it runs, reports a
plausible rate for a 152-SM GB300-class part, and the GEMM kernels stay below it."""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


def test_mma_ceiling_is_plausible(lib):
    tflops, ms = lib.dg_measure_fp8_mma_tflops(1024)
    assert ms > 0.0
    # dense FP8 on this class of part is a few PFLOP/s; anything outside this band means the
    # kernel is not doing (or not timing) the work
    assert 1000.0 < tflops < 12000.0, tflops


def test_mma_ceiling_rejects_bad_arguments(lib):
    raw = lib.load_library()
    import ctypes
    x = ctypes.c_double(0.0)
    assert raw.dg_measure_fp8_mma_tflops(0, ctypes.byref(x), None) == 1
    assert raw.dg_measure_fp8_mma_tflops(16, None, None) == 1
