"""Helpers shared by the GPU tests: move seeded workloads to the device, run the
library through its binding, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workloads as W

SENTINEL = W.sentinel_bits()


def dev(x: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def sentinel_like(shape) -> torch.Tensor:
    return torch.full(shape, SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_dense(lib, p: W.Dense, c_alias: bool = False) -> torch.Tensor:
    a, b = dev(p.a), dev(p.b)
    sfa, sfb = dev(p.sfa), dev(p.sfb)
    c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
    if c_alias and c is not None:
        d = c
    else:
        d = sentinel_like((p.M, p.N))
    fn = lib.dg_fp8_fp4_gemm_nt if p.b_format == "e2m1" else lib.dg_fp8_gemm_nt
    fn(a, sfa, b, sfb, c, d)
    torch.cuda.synchronize()
    return d


def run_wgrad(lib, p: W.Wgrad, in_place: bool = False) -> torch.Tensor:
    """FP32 D = C + A @ B.T; with in_place, D is the C buffer itself (accumulation)."""
    c = dev(p.c) if p.c is not None else None
    if in_place and c is not None:
        d = c
    else:
        d = torch.full((p.M, p.N), float("nan"), dtype=torch.float32).cuda()
    lib.dg_wgrad_gemm_fp8_fp8_fp32_nt(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c, d)
    torch.cuda.synchronize()
    return d


def run_k_grouped(lib, p: W.KGrouped, in_place: bool = False) -> torch.Tensor:
    """FP32 D[g] = C[g] + A_g @ B_g.T per expert; with in_place, D is the C buffer itself."""
    c = dev(p.c) if p.c is not None else None
    if in_place and c is not None:
        d = c
    else:
        d = torch.full((p.G, p.M, p.N), float("nan"), dtype=torch.float32).cuda()
    lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c, d,
                                                dev(np.asarray(p.ks, np.int32)))
    torch.cuda.synchronize()
    return d


def run_contiguous(lib, p: W.Contiguous) -> torch.Tensor:
    d = sentinel_like((p.M_total, p.N))
    fn = lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous if p.b_format == "e2m1" else lib.dg_m_grouped_fp8_gemm_nt_contiguous
    fn(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), d, dev(p.m_indices))
    torch.cuda.synchronize()
    return d


def run_masked(lib, p: W.Masked) -> torch.Tensor:
    d = sentinel_like((p.G, p.max_m, p.N))
    fn = lib.dg_m_grouped_fp8_fp4_gemm_nt_masked if p.b_format == "e2m1" else lib.dg_m_grouped_fp8_gemm_nt_masked
    fn(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), d, dev(p.masked_m))
    torch.cuda.synchronize()
    return d


def assert_parity(d_f64: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    rep = O.parity_report(d_f64, ref)
    assert rep["ok"], f"parity failed {what}: {rep}"
    return rep
