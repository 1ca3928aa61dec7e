"""Programmatic dependent launch on and off (dg_set_pdl, README "Utilities": set_pdl /
get_pdl): every GEMM form must give bit-identical results either way, since each kernel
waits for its predecessor before touching global memory; and with PDL on, inputs written
by the kernel right before the GEMM in the same stream must be the ones it reads."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import bf16_bits, run_contiguous, run_dense, run_k_grouped, run_masked, run_wgrad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    yield L
    L.dg_set_pdl(True)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy().copy()


CASES = {
    "dense_tile": lambda L: run_dense(L, W.make_dense(512, 1024, 1024, seed=41, with_c=True)),
    "dense_stream_k": lambda L: run_dense(L, W.make_dense(200, 384, 4096, seed=42, with_c=True)),
    "dense_split_k_pairs": lambda L: run_dense(L, W.make_dense(128, 7168, 4096, seed=43, with_c=True)),
    "dense_cta_pairs": lambda L: run_dense(L, W.make_dense(2048, 4096, 1024, seed=44, with_c=False)),
    "contiguous": lambda L: run_contiguous(L, W.make_contiguous(G=4, tokens=3000, N=1024, K=512, seed=45)),
    "masked": lambda L: run_masked(L, W.make_masked(G=6, max_m=256, N=512, K=512, seed=46,
                                                    masked_m=[0, 1, 255, 256, 100, 129])),
    "wgrad": lambda L: run_wgrad(L, W.make_wgrad(1024, 2048, 1024, seed=47)),
    "k_grouped": lambda L: run_k_grouped(L, W.make_k_grouped(G=3, M=512, N=768, tokens=1500, seed=48)),
    "fp4_dense": lambda L: run_dense(L, W.make_dense_fp4(1024, 2048, 1024, seed=49)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_pdl_on_and_off_bit_identical(lib, name):
    out = {}
    for pdl in (False, True):
        lib.dg_set_pdl(pdl)
        assert lib.dg_get_pdl() == pdl
        out[pdl] = _bits(CASES[name](lib))
        assert lib.dg_get_device_status() == 0
    lib.dg_set_pdl(True)
    assert np.array_equal(out[False], out[True]), name
