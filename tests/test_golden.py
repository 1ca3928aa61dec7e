"""Hand-worked examples (tests/golden/*.txt) against the oracle and, on a GPU, the library.

Each fixture is derived by hand from the format definitions and the operation as the pages
state it, with its arithmetic written out in the file, so it checks the oracle against
something other than itself. Every expected value is exact in FP64. Each value's rounding to
the output type (BF16, or FP32 for the weight-gradient forms) either sits far from a
rounding boundary or is worked out in the file. The library must therefore reproduce the
output values bit for bit, in any order of FP32 accumulation.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from golden_util import all_fixtures, check_oracle, load, stored

GEMM_FIXTURES = [n for n in all_fixtures() if not n.startswith("pack_sf")]
PACK_FIXTURES = [n for n in all_fixtures() if n.startswith("pack_sf")]
FORMS = {"dense_e4m3", "dense_e2m1", "masked_e4m3", "masked_e2m1", "contiguous_e4m3", "contiguous_e2m1",
         "wgrad_fp32", "k_grouped_fp32"}


def test_fixtures_cover_every_form():
    assert {load(n).form for n in GEMM_FIXTURES} == FORMS and PACK_FIXTURES
    layouts = {(load(n).form, load(n).layout) for n in GEMM_FIXTURES}
    assert {("dense_e4m3", x) for x in ("nt", "nn", "tn", "tt")} <= layouts
    assert {("contiguous_e4m3", "nn"), ("k_grouped_fp32", "tn")} <= layouts
    for name in GEMM_FIXTURES:
        assert (load(name).out != 0).any(), name


@pytest.mark.parametrize("name", GEMM_FIXTURES)
def test_oracle_reproduces_hand_worked_example(name):
    g = load(name)
    exact = np.vectorize(float, otypes=[np.float64])(g.exact)
    assert (np.vectorize(Fraction, otypes=[object])(exact) == g.exact).all(), "a worked value is not an FP64"
    check_oracle(O, g)
    # the output values in the fixture are round-to-nearest-even of the exact ones
    out_dtype = torch.float32 if g.form in ("wgrad_fp32", "k_grouped_fp32") else torch.bfloat16
    rounded = torch.from_numpy(exact).to(out_dtype).to(torch.float64).numpy()
    rows = np.ones(exact.shape[:-1], bool) if g.valid is None else g.valid
    assert np.array_equal(rounded[rows], g.out[rows]), f"{name}: hand rounding to {out_dtype}"


def _ue8m0_round_up(x: float) -> int:
    """Smallest code e with 2^(e-127) >= x, clamped to [0, 254] (exact rational arithmetic)."""
    v = Fraction(x)
    assert v > 0
    t = v.numerator.bit_length() - v.denominator.bit_length()
    while Fraction(2) ** t < v:
        t += 1
    while Fraction(2) ** (t - 1) >= v:
        t -= 1
    return min(max(t + 127, 0), 254)


@pytest.mark.parametrize("name", PACK_FIXTURES)
def test_pack_fixture_follows_the_definition(name):
    g = load(name)
    mn, kg = g.sf.shape
    codes = np.array([[_ue8m0_round_up(float(x)) for x in row] for row in g.sf], np.uint8)
    assert np.array_equal(W.pack_sf(codes).view(np.uint32), g.words)
    assert np.array_equal(O.unpack_sf(g.words.view(np.int32), mn, kg), codes)


# --------------------------------------------------------------------------------------
# the library, through its C ABI
# --------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


def _run_library(lib, g):
    from gpu_util import dev, run_contiguous, run_dense, run_k_grouped, run_masked, run_wgrad, sentinel_like
    p = g.problem
    if g.form == "contiguous_e4m3" and g.layout == "nn":
        _, b = stored(g)
        d = sentinel_like((p.M_total, p.N))
        lib.dg_m_grouped_fp8_gemm_nn_contiguous(dev(p.a), dev(p.sfa), dev(b), dev(p.sfb), d, dev(p.m_indices))
        torch.cuda.synchronize()
        return d
    if g.form == "k_grouped_fp32" and g.layout == "tn":
        a, b = stored(g)
        c = dev(p.c) if p.c is not None else None
        d = torch.full((p.G, p.M, p.N), float("nan"), dtype=torch.float32, device="cuda")
        lib.dg_k_grouped_fp8_gemm_tn_contiguous(dev(a), dev(p.sfa), dev(b), dev(p.sfb), c, d,
                                                dev(np.asarray(p.ks, np.int32)))
        torch.cuda.synchronize()
        return d
    if g.form == "dense_e4m3" and g.layout != "nt":
        a, b = stored(g)
        c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
        d = sentinel_like((p.M, p.N))
        getattr(lib, f"dg_fp8_gemm_{g.layout}")(dev(a), dev(p.sfa), dev(b), dev(p.sfb), c, d)
        torch.cuda.synchronize()
        return d
    run = {"dense_e4m3": run_dense, "dense_e2m1": run_dense, "masked_e4m3": run_masked, "masked_e2m1": run_masked,
           "contiguous_e4m3": run_contiguous, "contiguous_e2m1": run_contiguous, "wgrad_fp32": run_wgrad,
           "k_grouped_fp32": run_k_grouped}
    return run[g.form](lib, p)


@pytest.mark.gpu
@pytest.mark.parametrize("name", GEMM_FIXTURES)
def test_library_reproduces_hand_worked_example(lib, name):
    from gpu_util import SENTINEL, bf16_bits, bf16_f64
    g = load(name)
    lib.dg_get_device_status()
    d = _run_library(lib, g)
    assert lib.dg_get_device_status() == 0
    rows = np.ones(g.out.shape[:-1], bool) if g.valid is None else g.valid
    got = d.cpu().numpy().astype(np.float64) if d.dtype == torch.float32 else bf16_f64(d)
    bad = np.argwhere(got[rows] != g.out[rows])
    assert bad.size == 0, f"{name}: {len(bad)} entries differ, first {bad[:4].tolist()}"
    if d.dtype == torch.bfloat16:
        assert (bf16_bits(d)[~rows] == SENTINEL).all(), f"{name}: rows outside the computed set were written"


@pytest.mark.gpu
@pytest.mark.parametrize("name", PACK_FIXTURES)
def test_library_packs_hand_worked_scales(lib, name):
    from gpu_util import dev
    g = load(name)
    lib.dg_get_device_status()
    out = lib.dg_pack_sf_ue8m0(dev(g.sf)).cpu().numpy()
    assert lib.dg_get_device_status() == 0
    assert np.array_equal(out.view(np.uint32), g.words)
    # the same scales given MN-major ([kgroups, mn]) pack to the same words
    out_t = lib.dg_pack_sf_ue8m0(dev(np.ascontiguousarray(g.sf.T)), mn_major=True).cpu().numpy()
    assert lib.dg_get_device_status() == 0
    assert np.array_equal(out_t.view(np.uint32), g.words)
