"""Host-side checks of the C ABI (no GPU needed): the library builds, loads
and exports exactly the calls include/kvq.h declares; config validation and
size queries run on the host."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib_path():
    from bit_kv_cache_11_gb300 import build
    return build.build()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]*?\b(kvq_\w+)\s*\(", text)))


def test_header_declares_the_five_calls_and_helpers():
    syms = declared_symbols()
    for name in ("kvq_create", "kvq_quantize_prefill", "kvq_append", "kvq_decode_attention",
                 "kvq_dequantize", "kvq_destroy"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    kvq_exported = sorted(s for s in exported if s.startswith("kvq_"))
    assert kvq_exported == declared_symbols()


def _kvq(lib_path):
    import importlib
    return importlib.import_module("bit_kv_cache_11_gb300.kvq")


def test_config_check_on_host(lib_path):
    k = _kvq(lib_path)
    good = k.make_config(8, 32, 32, 128, 8192)
    assert k.kvq_config_check(good) == k.KVQ_OK
    cases = [
        (dict(batch=0), k.KVQ_ERR_INVALID_ARG),
        (dict(n_q_heads=30), k.KVQ_ERR_INVALID_ARG),      # not a multiple of n_kv_heads... 30 % 32
        (dict(bits_k=3), k.KVQ_ERR_INVALID_ARG),
        (dict(bits_v=16), k.KVQ_ERR_INVALID_ARG),
        (dict(axis_k=2), k.KVQ_ERR_INVALID_ARG),
        (dict(head_dim=96), k.KVQ_ERR_UNSUPPORTED),
        (dict(group=16), k.KVQ_ERR_UNSUPPORTED),
        (dict(n_q_heads=32 * 16), k.KVQ_ERR_UNSUPPORTED),  # GQA ratio 16
        (dict(keys_pre_rope=True, rope_base=0.5), k.KVQ_ERR_INVALID_ARG),
        (dict(head_dim=64, group=128, axis_v=1), k.KVQ_ERR_INVALID_ARG),  # D % G != 0
        (dict(max_ctx=0), k.KVQ_ERR_INVALID_ARG),
        (dict(n_sink=-1), k.KVQ_ERR_INVALID_ARG),
        (dict(n_sink=1025), k.KVQ_ERR_INVALID_ARG),
        (dict(residual=-32), k.KVQ_ERR_INVALID_ARG),
        (dict(residual=4097), k.KVQ_ERR_INVALID_ARG),
        (dict(n_sink=1024, residual=4096), k.KVQ_OK),
        (dict(n_sink=4, residual=100, group=64), k.KVQ_OK),
        (dict(fp8=True), k.KVQ_ERR_INVALID_ARG),                  # FP8 needs 8-bit sides
        (dict(fp8=True, bits_k=8, bits_v=4), k.KVQ_ERR_INVALID_ARG),
        (dict(fp8=True, bits_k=8, bits_v=8), k.KVQ_OK),
        (dict(fp8=True, bits_k=8, bits_v=8, axis_k=1, group=128), k.KVQ_OK),
        (dict(n_outliers=32), k.KVQ_OK),
        (dict(n_outliers=30), k.KVQ_ERR_INVALID_ARG),              # a multiple of 4
        (dict(n_outliers=128), k.KVQ_ERR_INVALID_ARG),             # at most 64
        (dict(n_outliers=32, bits_k=8), k.KVQ_ERR_UNSUPPORTED),
        (dict(n_outliers=32, group=64), k.KVQ_ERR_UNSUPPORTED),
    ]
    base = dict(batch=8, n_q_heads=32, n_kv_heads=32, head_dim=128, max_ctx=8192)
    for over, status in cases:
        kw = dict(base)
        kw.update(over)
        assert k.kvq_config_check(k.make_config(**kw)) == status, over
    # D % G is only required when an axis groups along channels of one token
    assert k.kvq_config_check(k.make_config(1, 2, 2, 64, 256, group=128, axis_k=0, axis_v=0)) == k.KVQ_OK


def test_cache_bytes_on_host(lib_path):
    k = _kvq(lib_path)
    cfg = k.make_config(8, 32, 32, 128, 4096 + 32)
    n = k.kvq_cache_bytes(cfg)
    P, NB = 8 * 32, (4096 + 32) // 32
    block = 32 * 128 * 4 // 8 + 8 * 128          # 3072 bytes per 32-token block at 2/2 bits
    assert block == 3072
    tails = 4 * P * 32 * 128 * 2
    assert n >= P * NB * block + tails
    assert n < P * NB * block + tails + 64 << 20


def test_cache_bytes_count_the_windows(lib_path):
    """Sink windows are fp16 [P][n_sink][D] for K and V; each of the four tail
    buffers grows to [P][residual + G][D]."""
    k = _kvq(lib_path)
    P, D = 8 * 32, 128
    base = k.kvq_cache_bytes(k.make_config(8, 32, 32, D, 4096))
    win = k.kvq_cache_bytes(k.make_config(8, 32, 32, D, 4096, n_sink=4, residual=128))
    assert win - base == 2 * P * 4 * D * 2 + 4 * P * 128 * D * 2


def test_status_strings(lib_path):
    k = _kvq(lib_path)
    for s in range(7):
        assert k.kvq_status_string(s)
    assert k.kvq_status_string(99) == "unknown status"


def test_null_handles_are_rejected_on_host(lib_path):
    k = _kvq(lib_path)
    lib = k._lib
    assert lib.kvq_append(None, None, None, 1, None) == k.KVQ_ERR_INVALID_ARG
    assert lib.kvq_decode_attention(None, None, None, 1.0, None) == k.KVQ_ERR_INVALID_ARG
    assert lib.kvq_destroy(None) == k.KVQ_OK
    T = ctypes.c_int(0)
    assert lib.kvq_get_state(None, ctypes.byref(T), ctypes.byref(T)) == k.KVQ_ERR_INVALID_ARG


def test_ctypes_structs_match_the_header(lib_path, tmp_path):
    """The binding's kvq_config and kvq_buffers have the C layout of
    include/kvq.h: every field at the same offset, the same sizes (a C program
    built against the header prints them)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    k = _kvq(lib_path)
    structs = {"kvq_config": k.kvq_config, "kvq_buffers": k.kvq_buffers}
    lines = []
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "kvq.h"\nint main(void) {\n'
                   + "\n".join(lines) + "\nreturn 0;\n}\n")
    exe = tmp_path / "layout"
    include = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.check_call(["gcc", "-std=c99", "-I", include, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split("\n")
    got = {}
    for line in out:
        if line:
            struct, field, value = line.split()
            got[(struct, field)] = int(value)
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert got[(name, field)] == getattr(cls, field).offset, (name, field)


def test_noalloc_refuses_windows_on_host(lib_path):
    """kvq_decode_attention_noalloc takes no sink or residual buffers: a config
    with either window is refused before any device work (no GPU needed)."""
    k = _kvq(lib_path)
    for kw in (dict(n_sink=4), dict(residual=32), dict(keys_pre_rope=True)):
        cfg = k.make_config(2, 8, 8, 128, 256, **kw)
        status = k._lib.kvq_decode_attention_noalloc(ctypes.byref(cfg), None, None, None, 0, 0,
                                                    None, None, 0.1, None, None)
        assert status == k.KVQ_ERR_UNSUPPORTED, kw
    bad = k.make_config(2, 8, 8, 128, 256, fp8=True, bits_k=8, bits_v=4)
    assert k._lib.kvq_decode_attention_noalloc(ctypes.byref(bad), None, None, None, 0, 0, None,
                                               None, 0.1, None, None) == k.KVQ_ERR_INVALID_ARG
