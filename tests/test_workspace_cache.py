"""The per-stream workspace cache policy (csrc/workspace_cache.h), checked on the host.

tests/workspace_cache_check.cpp instantiates the policy with fake CUDA calls and walks
through the situations that must stay safe: streams that come and go (evictions ordered after
the evicted block's last use), reserved workspaces (no allocation, free or event on a call that
fits), a captured graph whose workspace must outlive any later eviction, growth or release,
and captures during which nothing may be freed. The fake API has no synchronisation call, so
the policy cannot synchronise. No GPU is needed.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_workspace_cache_policy(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "workspace_cache_check"
    build = subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror",
                            "-I", os.path.join(ROOT, "fp8_gemm_nt_gb300", "csrc"),
                            os.path.join(ROOT, "tests", "workspace_cache_check.cpp"), "-o", str(exe)],
                           capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert out.stdout.startswith("ok"), out.stdout
