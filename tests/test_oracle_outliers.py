"""Pins of the oracle's dense-and-sparse outlier isolation (CPU).

KVQuant keeps "a small fraction of outliers" apart ("Why KV Cache Geometry
Matters More Than Bit Precision", section "KV Cache Size, GPU Memory
Efficiency, and the Shift to Geometry-Aware Quantization"; "Your KV cache
doesn't have a bit problem, it has a geometry problem", section "Rotary
Embeddings Complicate the Keys").  The pages give no selection rule or
format; the reading (kept identical by the oracle and the CUDA path): the n
elements of largest magnitude in a G-token block of one side (ties: lower
position j*D + d) are kept in fp16 with their positions, every group takes
min/max over its remaining elements, kept positions get code 0 and
dequantize to their kept value.

Pinned here by: hand-worked blocks (tests/golden/outlier_cases.txt), the
selection against a sort written with numpy, the half-step bound on the
dense elements and exactness of the kept ones, the reduction to the plain
quantizer (n = 0, and the dense group equal to the plain group of the
remaining elements), the packed layout and its round trip, and the
direction the pages give for isolating extreme values: on a cache with
sparse massive activations the attention errors fall.
"""
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden_rows():
    rows = []
    with open(os.path.join(HERE, "golden", "outlier_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


@pytest.mark.parametrize("row", _golden_rows())
def test_outlier_hand_cases(oracle_mod, row):
    head, rows, outs, sc, zs, codes = [x.strip() for x in row.split("|")]
    G, D, bits, axis, n = map(int, head.split())
    X = np.array([[float(v) for v in r.split()] for r in rows.split(";")], np.float16)
    Tq, c, s, z, o = oracle_mod.quantize_tensor_sparse(X, G, bits, axis, n)
    want_o = [] if outs == "-" else [int(v, 16) for v in outs.split()]
    assert o.reshape(-1).tolist() == want_o
    assert s.reshape(-1).tolist() == [int(v, 16) for v in sc.split()]
    assert z.reshape(-1).tolist() == [int(v, 16) for v in zs.split()]
    assert c.reshape(-1).tolist() == [int(v) for v in codes.split()]


def test_selection_is_top_magnitude_with_lower_position_first(oracle_mod):
    rng = np.random.default_rng(1)
    for trial in range(60):
        G, D = [(32, 128), (32, 64), (4, 8), (128, 128)][trial % 4]
        # few distinct magnitudes, so that ties are common
        vals = np.array([0.0, -0.0, 0.5, -0.5, 3.0, -3.0, 7.25, -7.25, 100.0], np.float16)
        tile = vals[rng.integers(0, vals.size, (G, D))]
        n = int(rng.integers(0, min(64, G * D) + 1))
        got = oracle_mod.select_outliers(tile, n)
        mag = np.abs(tile.astype(np.float64)).reshape(-1)
        order = np.lexsort((np.arange(G * D), -mag))   # magnitude desc, then position
        assert got.tolist() == sorted(order[:n].tolist())


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_dense_bound_and_exact_outliers(oracle_mod, axis, bits):
    rng = np.random.default_rng(10 * bits + axis)
    G, D, n = 32, 128, 32
    X = rng.standard_normal((3 * G, D)).astype(np.float32)
    hot = rng.random(X.shape) < 0.004
    X[hot] *= 400.0                                     # sparse massive activations
    X = X.astype(np.float16)
    st = oracle_mod.build_pair(X, X, G, bits, bits, axis, 1 - axis, n_outliers=n)
    kh, _ = oracle_mod.dequantize_pair(st)
    xf = X.astype(np.float64)
    kept = np.zeros(X.shape, bool)
    for i in range(3):
        for e in st["kout"][i]:
            p = int(e) >> 16
            kept[i * G + p // D, p % D] = True
            assert (int(e) & 0xffff) == int(X.view(np.uint16)[i * G + p // D, p % D])
    assert kept.sum() == 3 * n
    assert np.array_equal(kh[kept], xf[kept])           # kept elements are exact
    # dense elements: within half a step of their group (subnormal steps add
    # their own rounding, as for the plain quantizer)
    for i in range(3):
        for gi in range(D if axis == 0 else G * (D // G)):
            if axis == 0:
                rows, cols = slice(i * G, (i + 1) * G), slice(gi, gi + 1)
                s_bits, z_bits = st["kscale"][i, gi], st["kzero"][i, gi]
            else:
                j, g = divmod(gi, D // G)
                rows, cols = slice(i * G + j, i * G + j + 1), slice(g * G, (g + 1) * G)
                s_bits, z_bits = st["kscale"][i * G + j, g], st["kzero"][i * G + j, g]
            m = ~kept[rows, cols]
            x = xf[rows, cols][m]
            xh = kh[rows, cols][m].astype(np.float64)
            s = float(np.uint16(s_bits).view(np.float16))
            if x.size == 0:
                assert s == 0.0
                continue
            assert float(np.uint16(z_bits).view(np.float16)) == x.min()
            slack = 0.0 if s >= 2.0 ** -14 else ((1 << bits) - 1) * 2.0 ** -25
            assert np.all(np.abs(x - xh) <= s / 2 + slack + 2.0 ** -21 * np.abs(x - x.min()))


def test_dense_group_is_the_plain_group_of_the_remaining_elements(oracle_mod):
    rng = np.random.default_rng(2)
    for _ in range(200):
        bits = int(rng.choice([2, 4, 8]))
        x = (rng.standard_normal(32) * 10.0 ** rng.uniform(-2, 2)).astype(np.float16)
        skip = rng.random(32) < 0.2
        skip[0] = False
        s, z, c = oracle_mod.quantize_group_masked(x, bits, skip.astype(np.uint8))
        s2, z2, c2 = oracle_mod.quantize_group(x[~skip], bits)
        assert (s, z) == (s2, z2)
        assert np.array_equal(c[~skip], c2)
        assert not c[skip].any()
    # no element left: scale 0, zero +0, codes 0
    s, z, c = oracle_mod.quantize_group_masked(np.ones(8, np.float16), 2, np.ones(8, np.uint8))
    assert (s, z) == (0, 0) and not c.any()


@pytest.mark.parametrize("ak,av", [(0, 1), (1, 0)])
def test_no_outliers_is_the_plain_format(oracle_mod, ak, av):
    rng = np.random.default_rng(3)
    K = rng.standard_normal((70, 128), dtype=np.float32).astype(np.float16)
    V = rng.standard_normal((70, 128), dtype=np.float32).astype(np.float16)
    a = oracle_mod.pack_pair(oracle_mod.build_pair(K, V, 32, 2, 4, ak, av))
    b = oracle_mod.pack_pair(oracle_mod.build_pair(K, V, 32, 2, 4, ak, av, n_outliers=0))
    assert np.array_equal(a, b)
    assert oracle_mod.block_bytes(128, 32, 2, 4, 0) == oracle_mod.block_bytes(128, 32, 2, 4)


def test_block_layout_with_outlier_sections(oracle_mod):
    # [K codes | K meta 4D | K outliers 4n | V codes | V meta 4D | V outliers 4n]
    D, G, bk, bv, n = 128, 32, 2, 4, 16
    off = oracle_mod.block_offsets(D, G, bk, bv, n)
    assert off == [0, 1024, 1024 + 512, 1024 + 512 + 64, 1600 + 2048, 1600 + 2048 + 512]
    assert oracle_mod.block_bytes(D, G, bk, bv, n) == off[5] + 64
    rng = np.random.default_rng(4)
    K = rng.standard_normal((96, D), dtype=np.float32).astype(np.float16)
    V = rng.standard_normal((96, D), dtype=np.float32).astype(np.float16)
    st = oracle_mod.build_pair(K, V, G, bk, bv, n_outliers=n)
    blk = oracle_mod.pack_pair(st)
    # the K outlier section holds the entries as little-endian uint32
    words = blk[1][off[2]:off[3]].view("<u4")
    assert np.array_equal(words, st["kout"][1])
    back = oracle_mod.unpack_pair(blk, D, G, bk, bv, 0, 1, n)
    for key in ("kcodes", "kscale", "kzero", "vcodes", "vscale", "vzero", "kout", "vout"):
        assert np.array_equal(back[key], st[key])


def test_isolating_outliers_lowers_attention_error(oracle_mod):
    """Sparse massive activations (0.3 % of key and value elements x300, the
    kind "Keys: The Outliers Live in Fixed Channels" describes as rare and
    four orders of magnitude above the median) widen the steps of their
    groups; keeping the 32 largest elements of every block side apart lowers
    the attention-score and attention-output errors at 2 bits."""
    from bit_kv_cache_11_gb300 import synth
    w = synth.WORKLOADS[2].with_(batch=1, n_kv_heads=4, n_q_heads=4, T=512)
    case = synth.make_case(w, seed=17)
    err = {}
    for n in (0, 32):
        se, oe = [], []
        for h in range(w.n_kv_heads):
            K = case["K"][0, h].astype(np.float32)
            V = case["V"][0, h].astype(np.float32)
            hk = np.random.default_rng(100 + h).random(K.shape) < 0.003
            hv = np.random.default_rng(200 + h).random(V.shape) < 0.003
            K[hk] *= 300.0
            V[hv] *= 300.0
            K, V = K.astype(np.float16), V.astype(np.float16)
            q = case["q"][0, h:h + 1]
            st = oracle_mod.build_pair(K, V, w.group, 2, 2, 0, 1, n_outliers=n)
            o_q, s_q = oracle_mod.decode_pair(st, q, w.scale, want_scores=True)
            o_r, s_r = oracle_mod.reference_pair(K, V, q, w.scale, want_scores=True)
            se.append(oracle_mod.rel_fro(s_q, s_r))
            oe.append(oracle_mod.rel_fro(o_q, o_r))
        err[n] = (np.mean(se), np.mean(oe))
    assert err[32][0] < 0.5 * err[0][0]
    assert err[32][1] < err[0][1]
