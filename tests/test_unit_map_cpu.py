"""The decode unit map (per-row unit counts and offsets, owner warps) checked
on the host: a small C++ program built with nvcc against csrc/kvq_device.cuh
(host code only, no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_unit_map_partitions_units_and_slots(tmp_path):
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    if not (os.path.exists(nvcc) or shutil.which("nvcc")):
        pytest.skip("no nvcc")
    exe = tmp_path / "unit_map_check"
    subprocess.check_call([nvcc, "-std=c++17", "-O1",
                           "-I", os.path.join(ROOT, "bit_kv_cache_11_gb300", "csrc"),
                           "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "harness", "unit_map_check.cu"),
                           "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "failures 0" in out.stdout
