"""Host-side accounting of bench.py (no GPU): the algorithmic bytes of the
Llama-2-7B-shaped layer worked by hand, and the append rule the variant legs
replay, pinned to the oracle's window definition."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def test_decode_bytes_of_the_bench_layer(bench):
    from bit_kv_cache_11_gb300 import synth
    w = synth.WORKLOADS[2]
    # B8, 32 kv heads, D128, 2/2 bits, G32, 4096 quantized + 17 tail tokens:
    codes = 256 * 4096 * 128 * 4 // 8          # 67,108,864
    meta = 2 * 256 * (4096 * 128 // 32) * 4    # 33,554,432 (half2 scale/zero, K and V)
    tail = 256 * 17 * 128 * 2 * 2              # 2,228,224 (fp16 K and V rows)
    qo = 8 * 32 * 128 * (2 + 4)                # 196,608 (fp16 q in, fp32 out)
    assert bench.decode_bytes(w, 4096, 17) == codes + meta + tail + qo == 103_088_128


def test_quantize_bytes_per_token(bench):
    from bit_kv_cache_11_gb300 import synth
    w4 = synth.WORKLOADS[4]
    # 8 kv heads x D128: fp16 K+V in (4096 B), 2+2-bit codes (512 B), scales/zeros (256 B)
    assert bench.quantize_bytes_per_token(w4) == 4096 + 512 + 256 == 4864


@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("n_sink,residual", [(0, 0), (3, 0), (0, 40), (4, 128)])
def test_append_rule_replay_matches_the_oracle(bench, oracle_mod, G, n_sink, residual):
    for T0 in (0, 1, 2, G - 1, G, 3 * G + 5, residual + G - 1):
        row = list(oracle_mod.window_lengths(T0, G, n_sink, residual))
        for i in range(1, 3 * G + residual + 4):
            row = bench.append_one(row, n_sink, residual, G)
            assert tuple(row) == oracle_mod.window_lengths(T0 + i, G, n_sink, residual), (T0, i)
