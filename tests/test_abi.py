"""Host-side checks of the C ABI that need no GPU: the library builds, loads, exports
every entry point declared in include/dg.h, and rejects bad arguments before it
touches the device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from fp8_gemm_nt_gb300 import build
    build.build()
    import fp8_gemm_nt_gb300 as L
    return L.load_library()


def test_header_declares_the_three_gemms():
    names = declared_symbols()
    for n in ("dg_fp8_gemm_nt", "dg_m_grouped_fp8_gemm_nt_contiguous", "dg_m_grouped_fp8_gemm_nt_masked"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    import fp8_gemm_nt_gb300 as L
    bound = {name for name, _, _ in L.SIGNATURES}
    assert set(declared_symbols()) == bound
    for name in declared_symbols():
        assert callable(getattr(L, name)), name


def test_host_helpers(lib):
    assert lib.dg_get_mk_alignment_for_contiguous_layout() == 128
    assert lib.dg_get_tma_aligned_size(5, 4) == 8
    assert lib.dg_get_tma_aligned_size(16, 4) == 16
    assert lib.dg_get_tma_aligned_size(17, 1) == 32
    assert lib.dg_get_tma_aligned_size(3, 2) == 8
    assert lib.dg_get_tma_aligned_size(3, 3) == -1
    assert lib.dg_status_string(6) == b"DG_ERR_BAD_INDEX"


def test_invalid_arguments_rejected_before_launch(lib):
    P = ctypes.c_void_p
    x = P(0x10000)           # never dereferenced: validation fails first
    INVALID, MISALIGNED = 1, 3
    # null pointers
    assert lib.dg_fp8_gemm_nt(None, x, x, x, None, x, 128, 128, 128, None) == INVALID
    assert lib.dg_fp8_gemm_nt(x, x, x, x, None, None, 128, 128, 128, None) == INVALID
    # K not a multiple of 128, N not a multiple of 16, negative M
    assert lib.dg_fp8_gemm_nt(x, x, x, x, None, x, 128, 128, 100, None) == INVALID
    assert lib.dg_fp8_gemm_nt(x, x, x, x, None, x, 128, 120, 128, None) == INVALID
    assert lib.dg_fp8_gemm_nt(x, x, x, x, None, x, -1, 128, 128, None) == INVALID
    assert lib.dg_fp8_gemm_nt(x, x, x, x, None, x, 128, 128, 0, None) == INVALID
    # misaligned base pointer
    assert lib.dg_fp8_gemm_nt(P(0x10008), x, x, x, None, x, 128, 128, 128, None) == MISALIGNED
    # grouped forms: G <= 0
    assert lib.dg_m_grouped_fp8_gemm_nt_contiguous(x, x, x, x, x, x, 128, 128, 128, 0, None) == INVALID
    assert lib.dg_m_grouped_fp8_gemm_nt_masked(x, x, x, x, x, x, 0, 128, 128, 128, None) == INVALID
    assert lib.dg_m_grouped_fp8_gemm_nt_masked(x, x, x, x, x, x, 4, -1, 128, 128, None) == INVALID
    assert lib.dg_m_grouped_fp8_gemm_nt_contiguous(x, x, x, x, x, P(0x10002), 128, 128, 128, 2, None) == MISALIGNED
    assert lib.dg_pack_sf_ue8m0(None, x, 4, 4, 0, None) == INVALID
    assert lib.dg_pack_sf_ue8m0(x, x, 4, 4, 2, None) == INVALID          # orientation flag is 0 or 1


def test_mk_alignment_setter(lib):
    try:
        assert lib.dg_get_theoretical_mk_alignment_for_contiguous_layout() == 128
        assert lib.dg_set_mk_alignment_for_contiguous_layout(256) == 0
        assert lib.dg_get_mk_alignment_for_contiguous_layout() == 256
        for bad in (0, -128, 100, 192 + 1, 1 << 21):
            assert lib.dg_set_mk_alignment_for_contiguous_layout(bad) == 1
        assert lib.dg_get_mk_alignment_for_contiguous_layout() == 256
    finally:
        assert lib.dg_set_mk_alignment_for_contiguous_layout(128) == 0
    assert lib.dg_get_mk_alignment_for_contiguous_layout() == 128


def test_pdl_setter(lib):
    # host-only: the setting is process-wide and touches no device
    before = lib.dg_get_pdl()
    try:
        assert lib.dg_set_pdl(0) == 0 and lib.dg_get_pdl() == 0
        assert lib.dg_set_pdl(1) == 0 and lib.dg_get_pdl() == 1
        for bad in (-1, 2, 7):
            assert lib.dg_set_pdl(bad) == 1        # DG_ERR_INVALID_ARG, setting unchanged
            assert lib.dg_get_pdl() == 1
    finally:
        lib.dg_set_pdl(before)


def test_weight_gradient_forms_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    x = P(0x10000)
    INVALID, MISALIGNED = 1, 3
    assert lib.dg_wgrad_gemm_fp8_fp8_fp32_nt(x, x, x, x, None, None, 128, 128, 128, None) == INVALID
    assert lib.dg_wgrad_gemm_fp8_fp8_fp32_nt(x, x, x, x, None, x, 128, 120, 128, None) == INVALID
    assert lib.dg_wgrad_gemm_fp8_fp8_fp32_nt(x, x, x, x, P(0x10004), x, 128, 128, 128, None) == MISALIGNED
    # K-grouped: G <= 0, K_total not a multiple of 128, null ks, misaligned ks
    assert lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(x, x, x, x, None, x, x, 0, 128, 128, 128, 1, None) == INVALID
    assert lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(x, x, x, x, None, x, x, 2, 128, 128, 100, 1, None) == INVALID
    assert lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(x, x, x, x, None, x, None, 2, 128, 128, 128, 1, None) == INVALID
    assert lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(x, x, x, x, None, x, P(0x10002), 2, 128, 128, 128, 1,
                                                       None) == MISALIGNED


def test_fp8_fp4_forms_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    x = P(0x10000)
    INVALID, MISALIGNED = 1, 3
    assert lib.dg_fp8_fp4_gemm_nt(None, x, x, x, None, x, 128, 128, 128, None) == INVALID
    assert lib.dg_fp8_fp4_gemm_nt(x, x, x, x, None, x, 128, 128, 64, None) == INVALID      # K % 128
    assert lib.dg_fp8_fp4_gemm_nt(x, x, x, x, None, x, 128, 120, 128, None) == INVALID     # N % 16
    # the packed FP4 operand must be 32-byte aligned; 16 is not enough
    assert lib.dg_fp8_fp4_gemm_nt(x, x, P(0x10010), x, None, x, 128, 128, 128, None) == MISALIGNED
    assert lib.dg_fp8_fp4_gemm_nt(x, x, x, x, P(0x10008), x, 128, 128, 128, None) == MISALIGNED
    assert lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(x, x, x, x, x, x, 128, 128, 128, 0, None) == INVALID
    assert lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(x, x, x, x, x, None, 128, 128, 128, 2, None) == INVALID
    assert lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(x, x, P(0x10010), x, x, x, 128, 128, 128, 2,
                                                       None) == MISALIGNED
    assert lib.dg_m_grouped_fp8_fp4_gemm_nt_masked(x, x, x, x, x, x, 0, 128, 128, 128, None) == INVALID
    assert lib.dg_m_grouped_fp8_fp4_gemm_nt_masked(x, x, x, x, x, P(0x10002), 2, 128, 128, 128, None) == MISALIGNED
    # empty problems launch nothing and accept null pointers
    assert lib.dg_fp8_fp4_gemm_nt(None, None, None, None, None, None, 0, 128, 128, None) == 0
    assert lib.dg_m_grouped_fp8_fp4_gemm_nt_masked(None, None, None, None, None, None, 2, 0, 128, 128, None) == 0


def test_binding_rejects_tensors_outside_the_current_device(lib):
    # host tensors never reach the library: the binding raises before any call
    import torch
    import fp8_gemm_nt_gb300 as L
    M = N = K = 128
    a = torch.zeros((M, K), dtype=torch.uint8)
    sf = torch.zeros(L.sf_shape(M, K), dtype=torch.int32)
    sfb = torch.zeros(L.sf_shape(1, K), dtype=torch.int32)
    d = torch.zeros((M, N), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        L.dg_fp8_gemm_nt(a, sf, a, sfb, None, d)
    with pytest.raises(ValueError, match="CUDA"):
        L.dg_wgrad_gemm_fp8_fp8_fp32_nt(a, sf, a, sfb, None, d.float())
    with pytest.raises(ValueError, match="CUDA"):
        L.dg_fp8_fp4_gemm_nt(a, sf, a[:, :K // 2].contiguous(), torch.zeros((1, N), dtype=torch.int32), None, d)
    with pytest.raises(ValueError, match="CUDA"):
        L.dg_pack_sf_ue8m0(torch.ones((4, 4), dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        L.dg_fp8_gemm_nt_no_alloc(a, sf, a, sfb, None, d, torch.zeros(1, dtype=torch.int32))


def _param_kind(param: str) -> str:
    if "*" in param or "cudaStream_t" in param:
        return "pointer"
    if "unsigned long long" in param or re.match(r"^\s*size_t\s+\w+$", param):
        return "u64"
    assert re.match(r"^(const\s+)?(int|dg_status)\s+\w+$", param.strip()), param
    return "int"


def declared_prototypes():
    """name -> parameter kinds ("pointer", "int", "u64") of every dg_ function in include/*.h."""
    protos = {}
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        src = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
        for name, params in re.findall(r"\b(dg_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
            params = params.strip()
            protos[name] = [] if params in ("", "void") else [_param_kind(x) for x in params.split(",")]
    return protos


def _ctypes_kind(t) -> str:
    if t is ctypes.c_void_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "pointer"
    if t in (ctypes.c_ulonglong, ctypes.c_size_t):
        return "u64"
    assert t is ctypes.c_int, t
    return "int"


def test_binding_arguments_match_the_header():
    # ctypes passes whatever it is told: a parameter added to the header but not to the
    # binding (or the reverse), or an int where a pointer is expected, would corrupt the call
    from fp8_gemm_nt_gb300 import SIGNATURES
    protos = declared_prototypes()
    assert set(protos) == {name for name, _, _ in SIGNATURES}
    for name, _, args in SIGNATURES:
        assert [_ctypes_kind(t) for t in args] == protos[name], name
