"""The benchmark's headline facts that need the GPU: the configuration the dispatcher picks
for the headline workload is the one the recorded DRAM traffic was measured on."""
from __future__ import annotations

import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


def test_headline_traffic_names_the_dispatched_kernel(capfd, monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    import fp8_gemm_nt_gb300 as L
    import workloads as W
    L.load_library()
    prob = bench.DeviceProblem(L, W.make_workload(bench.HEADLINE), torch, max_bytes=0)
    monkeypatch.setenv("DG_PRINT_CONFIGS", "1")
    prob.launch(0)
    torch.cuda.synchronize()
    monkeypatch.delenv("DG_PRINT_CONFIGS")
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("[dg]")]
    assert len(lines) == 1, err
    assert bench.HEADLINE_TRAFFIC["kernel"] in lines[0], (bench.HEADLINE_TRAFFIC["kernel"], lines[0])
    assert L.dg_get_device_status() == 0
