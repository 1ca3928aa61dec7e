"""Python binding of libdg, the GB300 (sm_103a) fine-grained-scaled FP8 GEMM library.

Argument marshalling only: every function below passes device pointers, sizes and the
current CUDA stream to the C ABI declared in include/dg.h; all arithmetic runs in the
library's CUDA kernels. There is no fallback: if libdg.so is missing or the call
fails, an exception is raised.

The GEMM computes D = C + A @ B.T (DeepGEMM README, "Interfaces / Notices", as
reproduced on the page "Weight gradient kernels for dense and MoE models #95"), with
A and B in E4M3, UE8M0 scales packed four per int32 (A: per row per 128-K group,
B: per 128x128 block), FP32 accumulation and a BF16 result.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdg.so")

DG_OK = 0
STATUS_NAMES = {0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_UNSUPPORTED", 3: "DG_ERR_MISALIGNED",
                4: "DG_ERR_CUDA", 5: "DG_ERR_TIMEOUT", 6: "DG_ERR_BAD_INDEX"}

# (name, restype, argtypes) of every entry point in include/dg.h
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = [
    ("dg_fp8_gemm_nt", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("dg_wgrad_gemm_fp8_fp8_fp32_nt", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("dg_fp8_gemm_nn", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("dg_fp8_gemm_tn", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("dg_fp8_gemm_tt", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt", _I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    ("dg_k_grouped_fp8_gemm_tn_contiguous", _I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    ("dg_m_grouped_fp8_gemm_nn_contiguous", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("dg_m_grouped_fp8_gemm_nt_contiguous", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("dg_m_grouped_fp8_gemm_nt_masked", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("dg_fp8_fp4_gemm_nt", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    ("dg_m_grouped_fp8_fp4_gemm_nt_contiguous", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("dg_m_grouped_fp8_fp4_gemm_nt_masked", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    ("dg_pack_sf_ue8m0", _I, [_P, _P, _I, _I, _I, _P]),
    ("dg_get_mk_alignment_for_contiguous_layout", _I, []),
    ("dg_set_mk_alignment_for_contiguous_layout", _I, [_I]),
    ("dg_get_theoretical_mk_alignment_for_contiguous_layout", _I, []),
    ("dg_get_tma_aligned_size", _I, [_I, _I]),
    ("dg_set_num_sms", _I, [_I]),
    ("dg_reserve_workspace", _I, [_P, ctypes.c_size_t]),
    ("dg_release_workspace", _I, [_P]),
    ("dg_get_workspace_size", ctypes.c_size_t, [_P]),
    ("dg_set_pdl", _I, [_I]),
    ("dg_get_pdl", _I, []),
    ("dg_get_num_sms", _I, []),
    ("dg_get_device_status", _I, [_P]),
    ("dg_status_string", ctypes.c_char_p, [_I]),
    ("dg_last_cuda_error", _I, []),
    ("dg_set_debug", _I, [_I, ctypes.c_ulonglong]),
    ("dg_measure_fp8_mma_tflops", _I, [_I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    ("dg_fp8_gemm_nt_no_alloc", _I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
]


class DGError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdg.so (built by fp8_gemm_nt_gb300.build) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m fp8_gemm_nt_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(name: str, status: int) -> None:
    if status != DG_OK:
        raise DGError(name, status)


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _here(t: torch.Tensor, name: str) -> None:
    # the library works on the current device (and its stream): memory of another GPU would be
    # read through the wrong device's mappings
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.device.index == torch.cuda.current_device(),
          f"{name} is on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")


def _fp8(t: torch.Tensor, name: str) -> None:
    _here(t, name)
    _need(t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(t.dtype in (torch.float8_e4m3fn, torch.uint8), f"{name} must be float8_e4m3fn (or its uint8 bytes)")


def _i32(t: torch.Tensor, name: str) -> None:
    _here(t, name)
    _need(t.is_contiguous() and t.dtype == torch.int32, f"{name} must be a contiguous CUDA int32 tensor")


def _bf16(t: torch.Tensor, name: str) -> None:
    _here(t, name)
    _need(t.is_contiguous() and t.dtype == torch.bfloat16, f"{name} must be a contiguous CUDA bf16 tensor")


def _f32(t: torch.Tensor, name: str) -> None:
    _here(t, name)
    _need(t.is_contiguous() and t.dtype == torch.float32, f"{name} must be a contiguous CUDA float32 tensor")


def sf_shape(mn: int, k: int, groups: Optional[int] = None):
    """Shape of a packed scale tensor for an MN extent and K: [(G,) ceil(K/512), ceil4(mn)]."""
    shape = (-(-(k // 128) // 4), 4 * (-(-mn // 4)))
    return shape if groups is None else (groups,) + shape


def dg_fp8_gemm_nt(a, sfa, b, sfb, c, d, stream=None) -> torch.Tensor:
    """D = C + A @ B.T. a [M, K] e4m3, sfa [KP, ceil4(M)] int32, b [N, K] e4m3,
    sfb [KP, ceil4(ceil(N/128))] int32, c [M, N] bf16 or None, d [M, N] bf16 (written)."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d")
    M, K = a.shape
    N = b.shape[0]
    _need(b.shape[1] == K and tuple(d.shape) == (M, N), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_shape(-(-N // 128), K), "scale shape mismatch")
    if c is not None:
        _bf16(c, "c")
        _need(tuple(c.shape) == (M, N), "c shape mismatch")
    _check("dg_fp8_gemm_nt", lib.dg_fp8_gemm_nt(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                                                M, N, K, _stream(stream)))
    return d


def _dense_layout(name, a_kmajor, b_kmajor, a, sfa, b, sfb, c, d, stream):
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d")
    M, K = a.shape if a_kmajor else a.shape[::-1]
    N = b.shape[0] if b_kmajor else b.shape[1]
    Kb = b.shape[1] if b_kmajor else b.shape[0]
    _need(Kb == K and tuple(d.shape) == (M, N), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_shape(-(-N // 128), K), "scale shape mismatch")
    if c is not None:
        _bf16(c, "c")
        _need(tuple(c.shape) == (M, N), "c shape mismatch")
    _check(name, getattr(lib, name)(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d), M, N, K,
                                    _stream(stream)))
    return d


def dg_fp8_gemm_nn(a, sfa, b, sfb, c, d, stream=None) -> torch.Tensor:
    """D = C + A @ B with a [M, K] (K-major) and b [K, N] (N-major); scales as dg_fp8_gemm_nt."""
    return _dense_layout("dg_fp8_gemm_nn", True, False, a, sfa, b, sfb, c, d, stream)


def dg_fp8_gemm_tn(a, sfa, b, sfb, c, d, stream=None) -> torch.Tensor:
    """D = C + A.T @ B with a [K, M] (M-major, M a multiple of 16) and b [K, N]."""
    return _dense_layout("dg_fp8_gemm_tn", False, False, a, sfa, b, sfb, c, d, stream)


def dg_fp8_gemm_tt(a, sfa, b, sfb, c, d, stream=None) -> torch.Tensor:
    """D = C + A.T @ B.T with a [K, M] (M-major, M a multiple of 16) and b [N, K]."""
    return _dense_layout("dg_fp8_gemm_tt", False, True, a, sfa, b, sfb, c, d, stream)


def dg_wgrad_gemm_fp8_fp8_fp32_nt(a, sfa, b, sfb, c, d, stream=None) -> torch.Tensor:
    """Weight-gradient GEMM, D = C + A @ B.T with FP32 C and D (C may be D itself, which then
    accumulates in place). a, sfa, b, sfb as dg_fp8_gemm_nt; c [M, N] float32 or None;
    d [M, N] float32 (written)."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _f32(d, "d")
    M, K = a.shape
    N = b.shape[0]
    _need(b.shape[1] == K and tuple(d.shape) == (M, N), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_shape(-(-N // 128), K), "scale shape mismatch")
    if c is not None:
        _f32(c, "c")
        _need(tuple(c.shape) == (M, N), "c shape mismatch")
    _check("dg_wgrad_gemm_fp8_fp8_fp32_nt",
           lib.dg_wgrad_gemm_fp8_fp8_fp32_nt(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                                             M, N, K, _stream(stream)))
    return d


def dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(a, sfa, b, sfb, c, d, ks, stream=None) -> torch.Tensor:
    """K-grouped weight-gradient GEMM: D[g] = C[g] + A[:, slice_g] @ B[:, slice_g].T in FP32,
    expert g owning the K-slice of length ks[g]. a [M, K_total] e4m3, sfa [R, ceil4(M)] int32
    (packed per expert, R word rows), b [N, K_total], sfb [R, ceil4(ceil(N/128))],
    c [G, M, N] float32 or None (may be d), d [G, M, N] float32, ks [G] int32 (CUDA)."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _f32(d, "d"); _i32(ks, "ks")
    M, K = a.shape
    N = b.shape[0]
    G = ks.shape[0]
    _need(b.shape[1] == K and tuple(d.shape) == (G, M, N), "shape mismatch")
    R = sfa.shape[0]
    _need(sfa.dim() == 2 and sfa.shape[1] == 4 * (-(-M // 4)) and sfb.dim() == 2 and sfb.shape[0] == R
          and sfb.shape[1] == 4 * (-(-(-(-N // 128)) // 4)), "scale shape mismatch")
    if c is not None:
        _f32(c, "c")
        _need(tuple(c.shape) == (G, M, N), "c shape mismatch")
    _check("dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt",
           lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                                                       _ptr(ks), G, M, N, K, R, _stream(stream)))
    return d


def dg_k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, c, d, ks, stream=None) -> torch.Tensor:
    """K-grouped GEMM, TN layout: a [K_total, M] e4m3 (M a multiple of 16), b [K_total, N] e4m3,
    scales packed per expert as for dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt, c [G, M, N] float32
    or None (may be d), d [G, M, N] float32, ks [G] int32 (CUDA)."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _f32(d, "d"); _i32(ks, "ks")
    K, M = a.shape
    Kb, N = b.shape
    G = ks.shape[0]
    _need(Kb == K and tuple(d.shape) == (G, M, N), "shape mismatch")
    R = sfa.shape[0]
    _need(sfa.dim() == 2 and sfa.shape[1] == 4 * (-(-M // 4)) and sfb.dim() == 2 and sfb.shape[0] == R
          and sfb.shape[1] == 4 * (-(-(-(-N // 128)) // 4)), "scale shape mismatch")
    if c is not None:
        _f32(c, "c")
        _need(tuple(c.shape) == (G, M, N), "c shape mismatch")
    _check("dg_k_grouped_fp8_gemm_tn_contiguous",
           lib.dg_k_grouped_fp8_gemm_tn_contiguous(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                                                   _ptr(ks), G, M, N, K, R, _stream(stream)))
    return d


def dg_m_grouped_fp8_gemm_nn_contiguous(a, sfa, b, sfb, d, m_indices, stream=None) -> torch.Tensor:
    """Contiguous M-grouped GEMM with N-major weights: a [M_total, K], b [G, K, N] (N contiguous),
    other arguments as dg_m_grouped_fp8_gemm_nt_contiguous."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d"); _i32(m_indices, "m_indices")
    M, K = a.shape
    G, Kb, N = b.shape
    _need(Kb == K and tuple(d.shape) == (M, N) and tuple(m_indices.shape) == (M,), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_shape(-(-N // 128), K, G),
          "scale shape mismatch")
    _check("dg_m_grouped_fp8_gemm_nn_contiguous",
           lib.dg_m_grouped_fp8_gemm_nn_contiguous(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d),
                                                   _ptr(m_indices), M, N, K, G, _stream(stream)))
    return d


def dg_m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, d, m_indices, stream=None) -> torch.Tensor:
    """Contiguous M-grouped GEMM. a [M_total, K], sfa [KP, ceil4(M_total)], b [G, N, K],
    sfb [G, KP, ceil4(ceil(N/128))], d [M_total, N] bf16, m_indices [M_total] int32 (-1 = pad)."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d"); _i32(m_indices, "m_indices")
    M, K = a.shape
    G, N, Kb = b.shape
    _need(Kb == K and tuple(d.shape) == (M, N) and tuple(m_indices.shape) == (M,), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_shape(-(-N // 128), K, G),
          "scale shape mismatch")
    _check("dg_m_grouped_fp8_gemm_nt_contiguous",
           lib.dg_m_grouped_fp8_gemm_nt_contiguous(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d),
                                                   _ptr(m_indices), M, N, K, G, _stream(stream)))
    return d


def dg_m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, d, masked_m, stream=None) -> torch.Tensor:
    """Masked M-grouped GEMM. a [G, max_m, K], sfa [G, KP, ceil4(max_m)], b [G, N, K],
    sfb [G, KP, ceil4(ceil(N/128))], d [G, max_m, N] bf16, masked_m [G] int32 on the device."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d"); _i32(masked_m, "masked_m")
    G, max_m, K = a.shape
    Gb, N, Kb = b.shape
    _need(Gb == G and Kb == K and tuple(d.shape) == (G, max_m, N) and tuple(masked_m.shape) == (G,),
          "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(max_m, K, G) and tuple(sfb.shape) == sf_shape(-(-N // 128), K, G),
          "scale shape mismatch")
    _check("dg_m_grouped_fp8_gemm_nt_masked",
           lib.dg_m_grouped_fp8_gemm_nt_masked(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(masked_m),
                                               G, max_m, N, K, _stream(stream)))
    return d


# --------------------------------------------------------------------------------------
# FP8 x FP4: b holds packed E2M1 (two per byte, the even element in the low nibble), one
# UE8M0 scale per row per 32 K packed four per int32: sfb [(G,) K/128, ceil4(N)]
# --------------------------------------------------------------------------------------

_FP4_DTYPES = (torch.uint8,) + ((torch.float4_e2m1fn_x2,) if hasattr(torch, "float4_e2m1fn_x2") else ())


def _fp4(t: torch.Tensor, name: str) -> None:
    _here(t, name)
    _need(t.is_contiguous(), f"{name} must be a contiguous CUDA tensor")
    _need(t.dtype in _FP4_DTYPES, f"{name} must hold packed E2M1 bytes (uint8 or float4_e2m1fn_x2)")


def sf_fp4_shape(n: int, k: int, groups: Optional[int] = None):
    """Shape of the FP4 operand's packed scales: [(G,) K/128, ceil4(n)]."""
    shape = (k // 128, 4 * (-(-n // 4)))
    return shape if groups is None else (groups,) + shape


def dg_fp8_fp4_gemm_nt(a, sfa, b, sfb, c, d, stream=None) -> torch.Tensor:
    """D = C + A @ B.T with B in FP4. a [M, K] e4m3, sfa [KP, ceil4(M)] int32, b [N, K/2] packed
    E2M1 (32-byte aligned), sfb [K/128, ceil4(N)] int32, c [M, N] bf16 or None, d [M, N] bf16."""
    lib = load_library()
    _fp8(a, "a"); _fp4(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d")
    M, K = a.shape
    N = b.shape[0]
    _need(b.shape[1] * 2 == K and tuple(d.shape) == (M, N), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_fp4_shape(N, K), "scale shape mismatch")
    if c is not None:
        _bf16(c, "c")
        _need(tuple(c.shape) == (M, N), "c shape mismatch")
    _check("dg_fp8_fp4_gemm_nt", lib.dg_fp8_fp4_gemm_nt(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                                                        M, N, K, _stream(stream)))
    return d


def dg_m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, d, m_indices, stream=None) -> torch.Tensor:
    """Contiguous M-grouped FP8 x FP4 GEMM. a [M_total, K], sfa [KP, ceil4(M_total)], b [G, N, K/2]
    packed E2M1, sfb [G, K/128, ceil4(N)], d [M_total, N] bf16, m_indices [M_total] int32 (-1 = pad)."""
    lib = load_library()
    _fp8(a, "a"); _fp4(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d"); _i32(m_indices, "m_indices")
    M, K = a.shape
    G, N, Kh = b.shape
    _need(Kh * 2 == K and tuple(d.shape) == (M, N) and tuple(m_indices.shape) == (M,), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_fp4_shape(N, K, G), "scale shape mismatch")
    _check("dg_m_grouped_fp8_fp4_gemm_nt_contiguous",
           lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d),
                                                       _ptr(m_indices), M, N, K, G, _stream(stream)))
    return d


def dg_m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, d, masked_m, stream=None) -> torch.Tensor:
    """Masked M-grouped FP8 x FP4 GEMM. a [G, max_m, K], sfa [G, KP, ceil4(max_m)], b [G, N, K/2]
    packed E2M1, sfb [G, K/128, ceil4(N)], d [G, max_m, N] bf16, masked_m [G] int32 on the device."""
    lib = load_library()
    _fp8(a, "a"); _fp4(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d"); _i32(masked_m, "masked_m")
    G, max_m, K = a.shape
    Gb, N, Kh = b.shape
    _need(Gb == G and Kh * 2 == K and tuple(d.shape) == (G, max_m, N) and tuple(masked_m.shape) == (G,),
          "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(max_m, K, G) and tuple(sfb.shape) == sf_fp4_shape(N, K, G),
          "scale shape mismatch")
    _check("dg_m_grouped_fp8_fp4_gemm_nt_masked",
           lib.dg_m_grouped_fp8_fp4_gemm_nt_masked(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(masked_m),
                                                   G, max_m, N, K, _stream(stream)))
    return d


def dg_pack_sf_ue8m0(sf: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None,
                     mn_major: bool = False) -> torch.Tensor:
    """FP32 scales [mn, kgroups] (or [kgroups, mn] with mn_major) -> packed UE8M0 int32
    [ceil(kgroups/4), ceil4(mn)] (MN-major)."""
    lib = load_library()
    _here(sf, "sf")
    _need(sf.is_contiguous() and sf.dtype == torch.float32 and sf.dim() == 2,
          "sf must be a contiguous 2-D CUDA float32 tensor")
    mn, kg = (sf.shape[1], sf.shape[0]) if mn_major else (sf.shape[0], sf.shape[1])
    shape = (-(-kg // 4), 4 * (-(-mn // 4)))
    if out is None:
        out = torch.empty(shape, dtype=torch.int32, device=sf.device)
    _i32(out, "out")
    _need(tuple(out.shape) == shape, "out shape mismatch")
    _check("dg_pack_sf_ue8m0", lib.dg_pack_sf_ue8m0(_ptr(sf), _ptr(out), mn, kg, int(mn_major), _stream(stream)))
    return out


def dg_get_mk_alignment_for_contiguous_layout() -> int:
    return load_library().dg_get_mk_alignment_for_contiguous_layout()


def dg_set_mk_alignment_for_contiguous_layout(alignment: int) -> None:
    """Set the segment alignment callers are told to pad to (a positive multiple of 128)."""
    _check("dg_set_mk_alignment_for_contiguous_layout",
           load_library().dg_set_mk_alignment_for_contiguous_layout(int(alignment)))


def dg_get_theoretical_mk_alignment_for_contiguous_layout() -> int:
    return load_library().dg_get_theoretical_mk_alignment_for_contiguous_layout()


def dg_get_tma_aligned_size(mn: int, elem_bytes: int) -> int:
    return load_library().dg_get_tma_aligned_size(mn, elem_bytes)


def dg_set_num_sms(n: int) -> None:
    _check("dg_set_num_sms", load_library().dg_set_num_sms(n))


def dg_get_num_sms() -> int:
    return load_library().dg_get_num_sms()


def dg_reserve_workspace(nbytes: int, stream=None) -> None:
    """Reserve (at least nbytes of) the library's workspace for the stream (current by default)."""
    _check("dg_reserve_workspace", load_library().dg_reserve_workspace(_stream(stream), nbytes))


def dg_release_workspace(stream=None) -> None:
    _check("dg_release_workspace", load_library().dg_release_workspace(_stream(stream)))


def dg_get_workspace_size(stream=None) -> int:
    return int(load_library().dg_get_workspace_size(_stream(stream)))


def dg_set_pdl(enable: bool) -> None:
    """Programmatic dependent launch on (True) or off (False) for later launches."""
    _check("dg_set_pdl", load_library().dg_set_pdl(1 if enable else 0))


def dg_get_pdl() -> bool:
    return bool(load_library().dg_get_pdl())


def dg_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device-side error status code."""
    return load_library().dg_get_device_status(_stream(stream))


def dg_status_string(status: int) -> str:
    return load_library().dg_status_string(status).decode()


def dg_last_cuda_error() -> int:
    """The last CUDA error code the library saw on this host thread (0 if none)."""
    return load_library().dg_last_cuda_error()


def dg_set_debug(fault_mode: int, wait_timeout_ns: int = 0) -> None:
    """Failure-detection test hook: fault_mode 1 makes later launches time out on purpose
    (their producer issues nothing); wait_timeout_ns bounds every pipeline wait (0 = 2 s)."""
    _check("dg_set_debug", load_library().dg_set_debug(fault_mode, wait_timeout_ns))


def dg_measure_fp8_mma_tflops(iters_per_sm: int = 4096) -> tuple[float, float]:
    """Measured FP8 tensor-core ceiling of the current device: (TFLOP/s, kernel ms) of an
    MMA-only kernel (block-scaled 128 x 256 x 32 MMAs from shared memory on every SM)."""
    tf, ms = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _check("dg_measure_fp8_mma_tflops",
           load_library().dg_measure_fp8_mma_tflops(int(iters_per_sm), ctypes.byref(tf), ctypes.byref(ms)))
    return tf.value, ms.value


def dg_fp8_gemm_nt_no_alloc(a, sfa, b, sfb, c, d, status, stream=None) -> torch.Tensor:
    """D = C + A @ B.T without any device allocation by the library, for callers that
    cannot allocate at call time (graph capture, fixed-footprint servers, custom
    allocators). Same tensors as dg_fp8_gemm_nt plus `status`, a CUDA uint32/int32 tensor
    of one element that receives device-side error bits. The library's fixed 16 MiB
    scratch bounds the problem size (DG_ERR_INVALID_ARG beyond it); calls that overlap on
    the GPU race on that scratch."""
    lib = load_library()
    _fp8(a, "a"); _fp8(b, "b"); _i32(sfa, "sfa"); _i32(sfb, "sfb"); _bf16(d, "d")
    _here(status, "status")
    _need(status.numel() == 1 and status.element_size() == 4, "status must be one 4-byte CUDA word")
    M, K = a.shape
    N = b.shape[0]
    _need(b.shape[1] == K and tuple(d.shape) == (M, N), "shape mismatch")
    _need(tuple(sfa.shape) == sf_shape(M, K) and tuple(sfb.shape) == sf_shape(-(-N // 128), K), "scale shape mismatch")
    if c is not None:
        _bf16(c, "c")
        _need(tuple(c.shape) == (M, N), "c shape mismatch")
    _check("dg_fp8_gemm_nt_no_alloc",
           lib.dg_fp8_gemm_nt_no_alloc(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d), _ptr(status),
                                       M, N, K, _stream(stream)))
    return d
