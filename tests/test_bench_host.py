"""Host logic of the benchmark that needs no GPU: the algorithmic work behind the roofline
fraction, and the summary of the clocks sampled during the timed regions."""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _zeros_dense(M, N, K, with_c):
    KP, NB = -(-K // 512), -(-N // 128)
    return W.Dense(np.zeros((M, K), np.uint8), np.zeros((KP, W.ceil4(M)), np.int32), np.zeros((N, K), np.uint8),
                   np.zeros((KP, W.ceil4(NB)), np.int32), np.zeros((M, N), np.uint16) if with_c else None, M, N, K)


def test_algorithmic_work_of_the_headline():
    # A 128 x 16384, B 7168 x 16384, their packed scales, C read and D written once (BF16)
    flops, by = bench.algorithmic(_zeros_dense(128, 7168, 16384, with_c=True))
    assert flops == 2 * 128 * 7168 * 16384
    assert by == 128 * 16384 + 7168 * 16384 + 32 * 128 * 4 + 32 * 56 * 4 + 2 * 128 * 7168 * 2 == 123_231_232


def test_algorithmic_work_counts_valid_rows_and_used_experts_only():
    G, max_m, N, K = 3, 8, 256, 256
    KP = 1
    p = W.Masked(np.zeros((G, max_m, K), np.uint8), np.zeros((G, KP, 8), np.int32), np.zeros((G, N, K), np.uint8),
                 np.zeros((G, KP, 4), np.int32), np.array([0, 5, 9], np.int32), G, max_m, N, K)
    flops, by = bench.algorithmic(p)
    v = 5 + 8                                  # a count above max_m is clamped; expert 0 has none
    assert flops == 2 * v * N * K
    assert by == v * K + p.sfa.nbytes + 2 * (N * K + KP * 4 * 4) + v * N * 2
    m_idx = np.array([1] * 3 + [-1] * 125 + [2] * 128, np.int32)       # expert 0 unused, padding rows
    c = W.Contiguous(np.zeros((256, K), np.uint8), np.zeros((KP, 256), np.int32), np.zeros((G, N, K), np.uint8),
                     np.zeros((G, KP, 4), np.int32), m_idx, 256, N, K, G)
    flops, by = bench.algorithmic(c)
    assert flops == 2 * 131 * N * K
    assert by == 131 * K + c.sfa.nbytes + 2 * (N * K + KP * 4 * 4) + 131 * N * 2


def test_clock_summary():
    lines = [
        "0, 1980, 2070, 300.0, 0, 0x0, Not Active, Not Active, Not Active, Not Active",     # idle
        "0, 2070, 2070, 1350.5, 100, 0x4, Not Active, Not Active, Not Active, Active",     # power cap
        "0, 1995, 2070, 1390.0, 98, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 1200.0, 97, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0, 0x0, Not Active, Not Active, Not Active, Not Active",        # unparseable
    ]
    c = bench.summarize_clocks(lines)
    assert c["sm_mhz"] == 2040 and c["sm_max_mhz"] == 2070          # median of the samples under load
    assert c["reasons"] == ["sw_power_cap"]
    assert c["samples"] == 4 and c["samples_under_load"] == 3
    # a slowdown in any sample of the window is reported, even one taken at low utilisation
    idle_slow = ["0, 900, 2070, 100, 0, 0x8, Active, Not Active, Not Active, Not Active"] + lines[1:4]
    c = bench.summarize_clocks(idle_slow)
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"] and c["reasons_under_load"] == ["sw_power_cap"]
    assert c["sm_mhz"] == 2040
    assert bench.summarize_clocks(["header only"]) is None


def test_oracle_sample_rows_are_one_experts_valid_rows():
    G, K, N = 3, 128, 16
    m_idx = np.array([0] * 100 + [-1] * 28 + [1] * 40 + [-1] * 88 + [2] * 128, np.int32)
    c = W.Contiguous(np.zeros((384, K), np.uint8), np.zeros((1, 384), np.int32), np.zeros((G, N, K), np.uint8),
                     np.zeros((G, 1, 4), np.int32), m_idx, 384, N, K, G)
    for call in range(7):
        rows = bench.oracle_sample_rows(c, call, 32)
        assert len(rows) == 32 and len(set(rows.tolist())) == 32
        assert (m_idx[rows] == call % G).all()                 # valid rows of one expert, never padding


def test_headline_is_the_largest_configuration():
    # the contiguous G=8 workload: the most FLOPs of the five configurations
    assert bench.HEADLINE == "contiguous_g8_t32768_n4096_k7168"
    assert bench.HEADLINE_TRAFFIC["kernel"].startswith("pair 256x")
