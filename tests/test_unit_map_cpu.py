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


def _oracle_slots(oracle_mod, side, bits, D):
    """Element index (token * D + channel) stored in each (word, bit) field of
    a block's K or V code region, recovered from the oracle's packing one bit
    plane of the index at a time."""
    import numpy as np
    G = 32
    n = G * D
    off = oracle_mod.block_offsets(D, G, bits, bits)
    lo = off[0] if side == "K" else off[2]
    nwords = G * D * bits // 32
    found = np.zeros((nwords, 32 // bits), np.int64)
    idx = np.arange(n).reshape(G, D)
    for k in range(int(np.ceil(np.log2(n)))):
        plane = ((idx >> k) & 1).astype(np.uint8)
        zeros = np.zeros((G, D), np.uint8)
        st = dict(G=G, bk=bits, bv=bits, ak=0, av=1,
                  kcodes=plane if side == "K" else zeros, kscale=np.zeros((1, D), np.uint16),
                  kzero=np.zeros((1, D), np.uint16), vcodes=plane if side == "V" else zeros,
                  vscale=np.zeros((G, D // G), np.uint16), vzero=np.zeros((G, D // G), np.uint16))
        blk = oracle_mod.pack_pair(st)[0]
        words = np.frombuffer(bytes(blk[lo:lo + G * D * bits // 8]), "<u4").astype(np.int64)
        for f in range(32 // bits):
            found[:, f] |= ((words >> (f * bits)) & 1) << k
    return found


def test_device_code_order_matches_the_oracle(tmp_path, oracle_mod):
    """The device function that places codes in fragment order (used by the
    dequantizer, and the layout the quantizer and decode kernels follow) puts
    every element of a block at the word and bit where the oracle packs it."""
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    if not (os.path.exists(nvcc) or shutil.which("nvcc")):
        pytest.skip("no nvcc")
    exe = tmp_path / "frag_dump"
    subprocess.check_call([nvcc, "-std=c++17", "-O1",
                           "-I", os.path.join(ROOT, "bit_kv_cache_11_gb300", "csrc"),
                           "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "harness", "frag_position_dump.cu"),
                           "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120).stdout.split("\n")
    slots = {}
    checked = 0
    for line in out:
        if not line:
            continue
        side, bits, D, j, d, w, b = line.split()
        bits, D, j, d, w, b = int(bits), int(D), int(j), int(d), int(w), int(b)
        key = (side, bits, D)
        if key not in slots:
            slots[key] = _oracle_slots(oracle_mod, side, bits, D)
        assert b % bits == 0
        assert slots[key][w, b // bits] == j * D + d, (side, bits, D, j, d, w, b)
        checked += 1
    assert checked == 2 * 32 * (64 + 128) * 3
