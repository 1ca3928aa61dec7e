"""Worked examples derived by hand (tests/golden/*.txt): their line format and parser.

A fixture names its source in '#' lines, shows the arithmetic that gives each expected
value, then lists one item per line:

  form    dense_e4m3 | dense_e2m1 | masked_e4m3 | masked_e2m1 | contiguous_e4m3 |
          contiguous_e2m1 | wgrad_fp32 | k_grouped_fp32 | pack_sf   (e2m1: B in FP4)
  shape   dense, wgrad: M N K;  masked: G max_m N K;  contiguous: G M_total N K;
          k_grouped: M N (with "ks");  pack_sf: mn kgroups
  layout  nt | nn | tn | tt (dense_e4m3), nt | nn (contiguous_e4m3), nt | tn (k_grouped_fp32);
          default nt. The rows below always give the logical A' [M, K] and B [N, K]; the
          layout says how the library receives them.
  ks      K of each expert (k_grouped)
  a  IDX RUNS     one row of A: IDX is "r" ("g,r" for masked); codes fill from k = 0, zeros after
  b  IDX RUNS     one row of B: IDX is "n" ("g,n" for the grouped forms); E2M1 codes are nibbles
  sfa IDX E...    UE8M0 codes of one row of A, one per 128-wide K-group, from the first
                  (codes and rows not listed: 127)
  sfb IDX E...    E4M3 B: one 128-row block of B ("j" or "g,j"), one code per K-group;
                  E2M1 B: one row of B ("n" or "g,n"), one code per 32-wide K-block
                  (not listed: 127)
  c  IDX N VALUE  one entry of C (IDX "r", or "g,r" for k_grouped); entries not listed are 0
  masked_m COUNTS / m_indices VALUE*COUNT ...
  d  IDX N EXACT OUT   one entry of D (IDX "r" or "g,r"): its exact value, and that value
                  rounded to the output type (BF16, or FP32 for wgrad and k_grouped); every
                  other computed entry is exactly 0 (k_grouped: exactly C)
  sf R VALUES     pack_sf: one row of scales, each taken as its nearest FP32 value
  word Q I HEX    pack_sf: packed word (q, i) of the result; words not listed are 0

Numbers are decimals or hex-floats such as 0x1p-30. A run of codes is "XX" (one code),
"XX*n" (n copies) or "XX,YY*n" (the pair n times); codes are hexadecimal. This module only
builds inputs and expected values from that text: it holds none of the GEMM's arithmetic.
"""
from __future__ import annotations

import dataclasses
import os
from fractions import Fraction
from typing import Dict, List, Optional, Tuple

import numpy as np

import workloads as W

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@dataclasses.dataclass
class Golden:
    name: str
    form: str
    problem: object                        # W.Dense / Masked / Contiguous / Wgrad / KGrouped; None for pack_sf
    layout: str = "nt"
    exact: Optional[np.ndarray] = None     # object array of Fraction, shape of D
    out: Optional[np.ndarray] = None       # float64 values of D in the output type
    valid: Optional[np.ndarray] = None     # rows the operation computes (M-grouped forms)
    sf: Optional[np.ndarray] = None        # pack_sf: FP32 [mn, kgroups]
    words: Optional[np.ndarray] = None     # pack_sf: uint32 [ceil(kgroups/4), ceil4(mn)]


def number(tok: str) -> Fraction:
    t = tok.lower().lstrip("+-")
    if t.startswith("0x"):
        return Fraction(float.fromhex(tok))
    return Fraction(tok)


def _codes(tokens: List[str], limit: int) -> np.ndarray:
    out: List[int] = []
    for t in tokens:
        pat, _, rep = t.partition("*")
        n = int(rep) if rep else 1
        out.extend([int(x, 16) for x in pat.split(",")] * n)
    assert len(out) <= limit, f"{len(out)} codes for a row of {limit}"
    return np.array(out + [0] * (limit - len(out)), np.uint8)


def _idx(tok: str) -> Tuple[int, ...]:
    return tuple(int(x) for x in tok.split(","))


def _pack_grouped(exps: np.ndarray) -> np.ndarray:
    return np.stack([W.pack_sf(e) for e in exps])


def _f32(v: Fraction) -> float:
    x = float(np.float32(float(v)))
    assert Fraction(x) == v, f"{v} is not an FP32 value"
    return x


def load(name: str) -> Golden:
    items: Dict[str, List[List[str]]] = {}
    with open(os.path.join(GOLDEN_DIR, name), encoding="utf-8") as f:
        for raw in f:
            s = raw.split("#", 1)[0].split()
            if s:
                items.setdefault(s[0], []).append(s[1:])
    form = items["form"][0][0]
    shape = [int(x) for x in items["shape"][0]]
    layout = items["layout"][0][0] if "layout" in items else "nt"
    assert layout == "nt" or form == "dense_e4m3" or (form, layout) in (("contiguous_e4m3", "nn"),
                                                                         ("k_grouped_fp32", "tn"))

    if form == "pack_sf":
        mn, kg = shape
        sf = np.full((mn, kg), np.nan, np.float32)
        for r, *vals in items["sf"]:
            sf[int(r)] = [np.float32(float(number(v))) for v in vals]   # nearest FP32
        assert not np.isnan(sf).any(), "every scale must be listed"
        words = np.zeros((-(-kg // 4), 4 * (-(-mn // 4))), np.uint32)
        for q, i, h in items.get("word", []):
            words[int(q), int(i)] = int(h, 16)
        return Golden(name, form, None, sf=sf, words=words)

    fp4 = form.endswith("_e2m1")
    ks = None
    if form in ("dense_e4m3", "dense_e2m1", "wgrad_fp32"):
        M, N, K = shape
        G, rows = 1, M
    elif form.startswith(("masked_", "contiguous_")):
        G, rows, N, K = shape
    elif form == "k_grouped_fp32":
        rows, N = shape
        ks = np.array([int(v) for v in items["ks"][0]], np.int32)
        G, K = len(ks), int(ks.sum())
    else:
        raise ValueError(form)
    KG, NB = K // 128, -(-N // 128)
    grouped_a = form.startswith("masked_")
    grouped_b = form.startswith(("masked_", "contiguous_"))
    a = np.zeros((G, rows, K) if grouped_a else (rows, K), np.uint8)
    b = np.zeros((G, N, K) if grouped_b else (N, K), np.uint8)
    ea = np.full((G, rows, KG) if grouped_a else (rows, KG), 127, np.uint8)
    eb_shape = (N, K // 32) if fp4 else (NB, KG)
    eb = np.full((G,) + eb_shape if grouped_b else eb_shape, 127, np.uint8)
    for key, arr, width in (("a", a, K), ("b", b, K)):
        for tok, *runs in items.get(key, []):
            arr[_idx(tok)] = _codes(runs, width)
    for key, arr in (("sfa", ea), ("sfb", eb)):
        for tok, *vals in items.get(key, []):
            row = arr[_idx(tok)]
            assert len(vals) <= len(row), f"{key} {tok}: {len(vals)} codes for {len(row)}"
            row[:len(vals)] = [int(v) for v in vals]
    if fp4:
        assert (b < 16).all(), "E2M1 codes are nibbles"

    f32_out = form in ("wgrad_fp32", "k_grouped_fp32")
    dshape = (G, rows, N) if grouped_a or form == "k_grouped_fp32" else (rows, N)
    cv = None
    if "c" in items:
        cv = np.zeros(dshape, np.float32)
        for tok, n, v in items["c"]:
            cv[_idx(tok) + (int(n),)] = _f32(number(v))
    valid = None
    b_dev, b_format = (W.pack_fp4(b), "e2m1") if fp4 else (b, "e4m3")
    if grouped_a:
        counts = np.array([int(v) for v in items["masked_m"][0]], np.int32)
        valid = np.zeros((G, rows), bool)
        for g in range(G):
            valid[g, :min(max(int(counts[g]), 0), rows)] = True
        p = W.Masked(a, _pack_grouped(ea), b_dev, _pack_grouped(eb), counts, G, rows, N, K, b_format=b_format)
    elif form.startswith("contiguous_"):
        idx: List[int] = []
        for t in items["m_indices"][0]:
            v, _, n = t.partition("*")
            idx.extend([int(v)] * (int(n) if n else 1))
        assert len(idx) == rows
        m_indices = np.array(idx, np.int32)
        valid = m_indices >= 0
        p = W.Contiguous(a, W.pack_sf(ea), b_dev, _pack_grouped(eb), m_indices, rows, N, K, G, b_format=b_format)
    elif form == "wgrad_fp32":
        p = W.Wgrad(a, W.pack_sf(ea), b, W.pack_sf(eb), cv, rows, N, K)
    elif form == "k_grouped_fp32":
        p = W.KGrouped(a, W.pack_sf_k_grouped(ea, ks), b, W.pack_sf_k_grouped(eb, ks), cv, ks, rows, N)
    else:
        c = None
        if cv is not None:
            c = W.to_bf16_bits(cv)
            assert np.array_equal((c.astype(np.uint32) << 16).view(np.float32), cv), "C must hold BF16 values"
        if fp4:
            p = W.Dense(a, W.pack_sf(ea), W.pack_fp4(b), W.pack_sf(eb), c, rows, N, K, b_format="e2m1")
        else:
            p = W.Dense(a, W.pack_sf(ea), b, W.pack_sf(eb), c, rows, N, K, layout=layout)

    exact = np.empty(dshape, object)
    exact.fill(Fraction(0))
    out = np.zeros(dshape, np.float64)
    if form == "k_grouped_fp32" and cv is not None:
        for at in zip(*np.nonzero(cv)):
            exact[at] = Fraction(float(cv[at]))
            out[at] = cv[at]
    for tok, n, ex, o in items.get("d", []):
        at = _idx(tok) + (int(n),)
        exact[at] = number(ex)
        out[at] = float(number(o))
    if f32_out:
        for at in zip(*np.nonzero(out)):
            _f32(Fraction(out[at]))
    return Golden(name, form, p, layout=layout, exact=exact, out=out, valid=valid)


def all_fixtures() -> List[str]:
    return sorted(f for f in os.listdir(GOLDEN_DIR) if f.endswith(".txt"))


def stored(g: Golden):
    """A and B as the library receives them in the fixture's layout. A transposed A is
    [K, M]; a transposed B is [K, N], or [G, K, N] for the grouped weights."""
    p = g.problem
    a = p.a if g.layout[0] == "n" else np.ascontiguousarray(p.a.T)
    if g.layout[1] == "t":
        b = p.b
    elif p.b.ndim == 3:
        b = np.ascontiguousarray(p.b.transpose(0, 2, 1))
    else:
        b = np.ascontiguousarray(p.b.T)
    return a, b


def oracle_result(O_, g: Golden):
    """Run the fixture through the oracle module O_: (D, rows it computes or None)."""
    p = g.problem
    if g.form == "dense_e4m3":
        a, b = stored(g)
        return getattr(O_, f"fp8_gemm_{g.layout}")(a, p.sfa, b, p.sfb, p.c, p.M, p.N, p.K), None
    if g.form == "dense_e2m1":
        return O_.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K), None
    if g.form == "wgrad_fp32":
        return O_.wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K), None
    if g.form == "k_grouped_fp32" and g.layout == "tn":
        a, b = stored(g)
        return O_.k_grouped_fp8_gemm_tn_contiguous(a, p.sfa, b, p.sfb, p.c, p.ks, p.M, p.N), None
    if g.form == "k_grouped_fp32":
        return O_.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.ks, p.M, p.N), None
    if g.form == "masked_e2m1":
        return O_.m_grouped_fp8_fp4_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    if g.form == "contiguous_e2m1":
        return O_.m_grouped_fp8_fp4_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K,
                                                       p.G)
    if g.form == "masked_e4m3":
        return O_.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    if g.form == "contiguous_e4m3" and g.layout == "nn":
        _, b = stored(g)
        return O_.m_grouped_fp8_gemm_nn_contiguous(p.a, p.sfa, b, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    if g.form == "contiguous_e4m3":
        return O_.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K,
                                                   p.G)
    raise ValueError(g.form)


def check_oracle(O_, g: Golden) -> None:
    """The oracle reproduces every exact value of the fixture, computes exactly the rows the
    fixture computes, and marks the others as not computed (NaN)."""
    ref, valid = oracle_result(O_, g)
    exact = np.vectorize(float, otypes=[np.float64])(g.exact)
    rows = np.ones(exact.shape[:-1], bool) if g.valid is None else g.valid
    if g.valid is not None:
        assert np.array_equal(valid, g.valid), f"{g.name}: computed rows differ"
        assert np.isnan(ref[~rows]).all(), f"{g.name}: a row outside the computed set has a value"
    bad = np.argwhere(ref[rows] != exact[rows])
    assert bad.size == 0, f"{g.name}: {len(bad)} entries differ from the worked values, first {bad[:4].tolist()}"
