"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own formulas: they use hand-worked
cases (tests/golden/), a brute-force search for the nearest quantization
level, the error bound the pages state, closed forms of softmax attention and
RoPE, library routines (numpy float16 casts and float64 linear algebra) and
invariants.

Sources: "Your KV cache doesn't have a bit problem, it has a geometry
problem" — "What Quantization Error Is Actually Made Of" (quantizer, the
half-step error bound), "Keys: The Outliers Live in Fixed Channels" (key
grouping and the direction of the score error), "Values: Where the Intuition
Breaks" (value grouping, attention as a weighted sum), "Rotary Embeddings
Complicate the Keys" (RoPE after dequantization), "The Systems Tax" (the fp16
residual).
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([p.strip() for p in line.split("|")])
    return rows


# ---- fp16 conversions -------------------------------------------------------

def test_h2f_all_patterns_match_numpy(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.h2f(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f2h_matches_numpy_on_ties_and_random_floats(oracle_mod):
    rng = np.random.default_rng(7)
    finite = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    finite = finite[np.isfinite(finite)].astype(np.float32)
    srt = np.unique(finite.astype(np.float64))
    mids = ((srt[1:] + srt[:-1]) / 2).astype(np.float32)  # exact ties of fp16 rounding
    rand = rng.integers(0, 2**32, size=1 << 21, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rand = rand[np.isfinite(rand)]
    for x in (finite, mids, rand, np.array([65519.99, 65520.0, 1e-8, -1e-8, 2.0**-25, 3 * 2.0**-26],
                                            np.float32)):
        got = oracle_mod.f2h(x)
        with np.errstate(over="ignore"):
            ref = x.astype(np.float16).view(np.uint16)
        assert np.array_equal(got, ref)


# ---- the quantizer ----------------------------------------------------------

@pytest.mark.parametrize("row", _read_golden("quantizer_cases.txt"))
def test_quantizer_hand_cases(oracle_mod, row):
    bits = int(row[0])
    vals = np.array([float(v) for v in row[1].split()], np.float16)
    exp_s, exp_z = (int(h, 16) for h in row[2].split())
    exp_codes = [int(c) for c in row[3].split()]
    s, z, codes = oracle_mod.quantize_group(vals, bits)
    assert (s, z) == (exp_s, exp_z)
    assert codes.tolist() == exp_codes


def _nearest_level_ok(x, s, z, c, bits):
    """c is a nearest level of x on the grid z + k*s, k in [0, 2^bits - 1]
    (exact fp64 distances; near-ties may go either way within fp32 rounding
    of (x - min) / s)."""
    ks = np.arange(1 << bits, dtype=np.float64)
    dist = np.abs(x - (z + ks * s))
    best = dist.min()
    return dist[c] <= best + 2.0 ** -21 * max(abs(x - z), s)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("n", [1, 2, 4, 32, 128])
def test_quantizer_brute_force_invariants(oracle_mod, bits, n):
    rng = np.random.default_rng(100 * bits + n)
    for trial in range(40):
        spread = 10.0 ** rng.uniform(-3, 3)
        x = (rng.standard_normal(n) * spread).astype(np.float16)
        if trial % 10 == 0:
            x[rng.integers(0, n)] = np.float16(spread * 50)  # an outlier
        s_bits, z_bits, codes = oracle_mod.quantize_group(x, bits)
        s = float(np.uint16(s_bits).view(np.float16))
        z = float(np.uint16(z_bits).view(np.float16))
        xf = x.astype(np.float64)
        assert codes.max() <= (1 << bits) - 1
        assert z == xf.min()                       # zero point = group minimum
        if xf.max() == xf.min():
            assert s == 0.0 and not codes.any()
            continue
        # the minimum reconstructs exactly: its code is 0
        assert codes[int(np.argmin(xf))] == 0
        if s == 0.0:
            assert not codes.any()
            continue
        normal = s >= 2.0 ** -14
        if normal:
            # the maximum takes the top level
            assert codes[int(np.argmax(xf))] == (1 << bits) - 1
        # half a step when the stored fp16 step is a normal number; a
        # subnormal stored step adds its own rounding, at most 2^-25 per level
        slack = 0.0 if normal else ((1 << bits) - 1) * 2.0 ** -25
        for xi, ci in zip(xf, codes):
            assert abs(xi - (z + ci * s)) <= s / 2 + slack + 2.0 ** -21 * abs(xi - z)
            assert _nearest_level_ok(xi, s, z, int(ci), bits)


@pytest.mark.parametrize("bits,lo,hi", [(2, -1.0, 2.5), (4, -3.0, 0.5), (8, 0.25, 7.0)])
def test_quantizer_every_fp16_between_fixed_extremes(oracle_mod, bits, lo, hi):
    """Sweeps every fp16 value x in [lo, hi] through the group {lo, x, hi}."""
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    xs = np.unique(allh[np.isfinite(allh) & (allh >= lo) & (allh <= hi)])
    for x in xs:
        g = np.array([lo, x, hi], np.float16)
        s_bits, z_bits, codes = oracle_mod.quantize_group(g, bits)
        s = float(np.uint16(s_bits).view(np.float16))
        z = float(np.uint16(z_bits).view(np.float16))
        assert z == lo and codes[0] == 0 and codes[2] == (1 << bits) - 1
        assert _nearest_level_ok(float(x), s, z, int(codes[1]), bits)


def test_quantize_tensor_groups_along_the_right_axis(oracle_mod):
    """Channel axis: one group per channel over G tokens; token axis: one
    group per G channels of a token.  A single large value must change only
    its own group's step."""
    rng = np.random.default_rng(3)
    T, D, G = 64, 64, 32
    X = rng.standard_normal((T, D)).astype(np.float16)
    Y = X.copy()
    Y[5, 7] = np.float16(200.0)
    for axis in (0, 1):
        _, _, s0, _ = oracle_mod.quantize_tensor(X, G, 2, axis)
        _, _, s1, _ = oracle_mod.quantize_tensor(Y, G, 2, axis)
        changed = np.argwhere(s0 != s1)
        if axis == 0:
            assert changed.tolist() == [[0, 7]]      # block 0, channel 7
        else:
            assert changed.tolist() == [[5, 0]]      # token 5, channels 0..31


def test_dequantize_is_a_single_rounding_of_code_times_scale_plus_zero(oracle_mod):
    rng = np.random.default_rng(11)
    X = (rng.standard_normal((64, 64)) * 3).astype(np.float16)
    for axis in (0, 1):
        _, codes, sc, zr = oracle_mod.quantize_tensor(X, 32, 4, axis)
        got = oracle_mod.dequantize_tensor(codes, sc, zr, 32, axis)
        s = sc.view(np.float16).astype(np.float64)
        z = zr.view(np.float16).astype(np.float64)
        if axis == 0:
            s = np.repeat(s, 32, axis=0)
            z = np.repeat(z, 32, axis=0)
        else:
            s = np.repeat(s, 32, axis=1)
            z = np.repeat(z, 32, axis=1)
        # codes*s + z is exact in fp64 (few significant bits), so one rounding
        # to fp32 is what a fused multiply-add gives
        ref = (codes.astype(np.float64) * s + z).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ---- packing ----------------------------------------------------------------

@pytest.mark.parametrize("row", _read_golden("packed_words.txt"))
def test_packed_words(oracle_mod, row):
    kind, bits = row[0].split()
    bits = int(bits)
    codes = [int(c) for c in row[1].split()]
    word = int(row[2], 16)
    per = 32 // bits
    D = 128 if kind == "K" else 128
    G = 32
    st = dict(G=G, bk=bits, bv=bits, ak=0, av=0,
              kcodes=np.zeros((G, D), np.uint8), kscale=np.zeros((1, D), np.uint16),
              kzero=np.zeros((1, D), np.uint16), vcodes=np.zeros((G, D), np.uint8),
              vscale=np.zeros((1, D), np.uint16), vzero=np.zeros((1, D), np.uint16))
    if kind == "K":   # codes of token 0, channels 0..per-1
        st["kcodes"][0, :per] = codes
        blk = oracle_mod.pack_pair(st)[0]
        got = int.from_bytes(bytes(blk[0:4]), "little")
    else:             # codes of channel 0, tokens 0..per-1
        st["vcodes"][:per, 0] = codes
        off = oracle_mod.block_offsets(D, G, bits, bits)[2]
        blk = oracle_mod.pack_pair(st)[0]
        got = int.from_bytes(bytes(blk[off:off + 4]), "little")
    assert got == word


def test_code_order_rule(oracle_mod):
    # fragment order only for keys per channel + values per token, G = 32,
    # D in {64, 128}, every bit width
    for D in (64, 128):
        assert oracle_mod.code_order(D, 32, 2, 0, 1) == 1
        assert oracle_mod.code_order(D, 32, 4, 0, 1) == 1
        assert oracle_mod.code_order(D, 32, 8, 0, 1) == 1
        assert oracle_mod.code_order(D, 128, 2, 0, 1) == 0
        assert oracle_mod.code_order(D, 64, 4, 0, 1) == 0
        for ak, av in ((0, 0), (1, 0), (1, 1)):
            assert oracle_mod.code_order(D, 32, 2, ak, av) == 0
    assert oracle_mod.code_order(32, 32, 2, 0, 1) == 0


@pytest.mark.parametrize("row", _read_golden("fragment_words.txt"))
def test_fragment_words(oracle_mod, row):
    kind, bits, D = row[0].split()
    bits, D = int(bits), int(D)
    tok, ch, code = (int(v) for v in row[1].split())
    word_index = int(row[2])
    word = int(row[3], 16)
    G = 32
    st = dict(G=G, bk=bits, bv=bits, ak=0, av=1,
              kcodes=np.zeros((G, D), np.uint8), kscale=np.zeros((1, D), np.uint16),
              kzero=np.zeros((1, D), np.uint16), vcodes=np.zeros((G, D), np.uint8),
              vscale=np.zeros((G, D // G), np.uint16), vzero=np.zeros((G, D // G), np.uint16))
    (st["kcodes"] if kind == "K" else st["vcodes"])[tok, ch] = code
    off = oracle_mod.block_offsets(D, G, bits, bits)
    blk = oracle_mod.pack_pair(st)[0]
    lo = off[0] if kind == "K" else off[2]
    region = bytes(blk[lo:lo + G * D * bits // 8])
    words = np.frombuffer(region, "<u4")
    assert int(words[word_index]) == word
    assert np.count_nonzero(words) == 1


def test_block_geometry_by_hand(oracle_mod):
    # G*D*(bk+bv)/8 + 8*D bytes; K codes, K meta, V codes, V meta in that order
    assert oracle_mod.block_bytes(128, 32, 2, 2) == 2048 + 1024 == 3072
    assert oracle_mod.block_offsets(128, 32, 2, 2) == [0, 1024, 1536, 2560]
    assert oracle_mod.block_offsets(64, 32, 2, 2) == [0, 512, 768, 1280]
    assert oracle_mod.block_bytes(128, 128, 8, 4) == 128 * 128 * 12 // 8 + 1024
    assert oracle_mod.block_offsets(128, 128, 8, 4) == [0, 16384, 16896, 16896 + 8192]


def test_block_bytes_by_hand(oracle_mod):
    """A whole 32-token block with hand-chosen codes and metadata."""
    D, G = 32, 32
    t = np.arange(G)[:, None]
    d = np.arange(D)[None, :]
    st = dict(G=G, bk=2, bv=2, ak=0, av=1,
              kcodes=np.broadcast_to(d % 4, (G, D)).astype(np.uint8),
              kscale=(0x3C00 + np.arange(D))[None, :].astype(np.uint16),
              kzero=(0x8000 + np.arange(D))[None, :].astype(np.uint16),
              vcodes=np.broadcast_to(3 - t % 4, (G, D)).astype(np.uint8),
              vscale=(0x4000 + np.arange(G))[:, None].astype(np.uint16),
              vzero=np.arange(G)[:, None].astype(np.uint16))
    blk = bytes(oracle_mod.pack_pair(st)[0])
    assert len(blk) == 768
    assert blk[0:256] == b"\xe4" * 256                      # K codes
    assert blk[256:264] == bytes([0x00, 0x3C, 0x00, 0x80, 0x01, 0x3C, 0x01, 0x80])
    assert blk[384:640] == b"\x1b" * 256                    # V codes
    assert blk[640:648] == bytes([0x00, 0x40, 0x00, 0x00, 0x01, 0x40, 0x01, 0x00])
    assert blk[764:768] == bytes([0x1F, 0x40, 0x1F, 0x00])


def test_fragment_block_by_hand(oracle_mod):
    """A whole 32-token block (D = 64) in fragment order, worked by hand from
    the definition.  Keys (2 bits), code d % 4: column 16 ks + 8 kh + 2 t + e
    has d % 4 = 2 (t % 2) + e, so the low half (e = 0) of every word of lane
    l holds eight codes 2 (l % 2) and the high half eight codes 2 (l % 2) + 1.
    Values (4 bits), code (token % 4) + 4 (channel % 2): token % 4 = 2 (t % 2)
    + e and channel % 2 = g % 2, the same in all four nibbles of a half."""
    D, G = 64, 32
    t = np.arange(G)[:, None]
    d = np.arange(D)[None, :]
    st = dict(G=G, bk=2, bv=4, ak=0, av=1,
              kcodes=np.broadcast_to(d % 4, (G, D)).astype(np.uint8),
              kscale=np.zeros((1, D), np.uint16), kzero=np.zeros((1, D), np.uint16),
              vcodes=np.broadcast_to(t % 4 + 4 * (d % 2), (G, D)).astype(np.uint8),
              vscale=np.zeros((G, D // G), np.uint16), vzero=np.zeros((G, D // G), np.uint16))
    off = oracle_mod.block_offsets(D, G, 2, 4)
    blk = bytes(oracle_mod.pack_pair(st)[0])
    kw = np.frombuffer(blk[off[0]:off[1]], "<u4").reshape(-1, 32, 4)  # [w/4][lane][w%4]
    vw = np.frombuffer(blk[off[2]:off[3]], "<u4").reshape(-1, 32, 4)
    for lane in range(32):
        g, tt = lane // 4, lane % 4
        assert np.all(kw[:, lane, :] == (0x55550000 if tt % 2 == 0 else 0xFFFFAAAA))
        v0 = 2 * (tt % 2) + 4 * (g % 2)
        assert np.all(vw[:, lane, :] == ((v0 + 1) * 0x1111) << 16 | v0 * 0x1111)


@pytest.mark.parametrize("bk,bv,ak,av,G,D", [(2, 2, 0, 1, 32, 128), (4, 8, 1, 0, 128, 128),
                                             (8, 4, 0, 1, 32, 64), (2, 4, 1, 1, 64, 128),
                                             (4, 2, 0, 1, 32, 64), (2, 2, 0, 1, 128, 128)])
def test_pack_unpack_round_trip(oracle_mod, bk, bv, ak, av, G, D):
    rng = np.random.default_rng(bk * 10 + bv)
    X = rng.standard_normal((2 * G + 5, D)).astype(np.float16)
    Y = rng.standard_normal((2 * G + 5, D)).astype(np.float16)
    st = oracle_mod.build_pair(X, Y, G, bk, bv, ak, av)
    back = oracle_mod.unpack_pair(oracle_mod.pack_pair(st), D, G, bk, bv, ak, av)
    for key in ("kcodes", "kscale", "kzero", "vcodes", "vscale", "vzero"):
        assert np.array_equal(back[key], st[key]), key


# ---- RoPE -------------------------------------------------------------------

def test_rope_closed_forms(oracle_mod):
    # D = 2: one pair turning at angle pos * base^0 = pos
    for pos in (0, 1, 7, 1000):
        got = oracle_mod.rope(np.array([1.0, 0.0]), pos, 10000.0)
        assert np.allclose(got, [math.cos(pos), math.sin(pos)], atol=1e-12)
    # D = 4, base 10000: pair 1 turns at pos * 10000^(-1/2) = pos / 100
    got = oracle_mod.rope(np.array([0.0, 2.0, 0.0, 0.0]), 100, 10000.0)
    assert np.allclose(got, [0.0, 2 * math.cos(1.0), 0.0, 2 * math.sin(1.0)], atol=1e-12)
    got = oracle_mod.rope(np.array([0.0, 0.0, 0.0, 3.0]), 100, 10000.0)
    assert np.allclose(got, [0.0, -3 * math.sin(1.0), 0.0, 3 * math.cos(1.0)], atol=1e-12)


def test_rope_is_a_relative_rotation(oracle_mod):
    rng = np.random.default_rng(5)
    D = 64
    q = rng.standard_normal(D)
    k = rng.standard_normal(D)
    assert np.allclose(oracle_mod.rope(k, 0, 10000.0), k)
    assert math.isclose(np.linalg.norm(oracle_mod.rope(k, 1234, 10000.0)), np.linalg.norm(k),
                        rel_tol=1e-12)
    dots = [oracle_mod.rope(q, m + 17, 10000.0) @ oracle_mod.rope(k, m, 10000.0)
            for m in (0, 5, 300, 4000)]
    assert np.allclose(dots, dots[0], rtol=1e-9, atol=1e-9)


# ---- attention --------------------------------------------------------------

def _as_pair(oracle_mod, K, V, G=32, bk=4, bv=4):
    return oracle_mod.build_pair(K, V, G, bk, bv, 0, 1)


def test_attention_zero_query_is_the_mean_of_values(oracle_mod):
    rng = np.random.default_rng(1)
    K = rng.standard_normal((77, 64)).astype(np.float16)
    V = rng.standard_normal((77, 64)).astype(np.float16)
    st = _as_pair(oracle_mod, K, V)
    kh, vh = oracle_mod.dequantize_pair(st)
    q = np.zeros((1, 64), np.float16)
    out = oracle_mod.decode_pair(st, q, 0.125)
    allv = np.concatenate([vh.astype(np.float64), st["vtail"].astype(np.float64)])
    assert np.allclose(out[0], allv.mean(0), rtol=1e-12, atol=1e-12)


def test_attention_two_tokens_logistic(oracle_mod):
    D = 8
    K = np.zeros((2, D), np.float16)
    K[0, 0], K[1, 0] = 3.0, -1.0
    V = np.zeros((2, D), np.float16)
    V[0, 1], V[1, 2] = 1.0, 1.0
    q = np.zeros((1, D), np.float16)
    q[0, 0] = 1.0
    scale = 0.5
    out = oracle_mod.reference_pair(K, V, q, scale)
    w0 = 1.0 / (1.0 + math.exp(-(scale * 3.0 - scale * -1.0)))
    assert np.allclose(out[0, 1:3], [w0, 1.0 - w0], rtol=1e-14)
    assert np.allclose(np.delete(out[0], [1, 2]), 0.0)


def test_attention_dominant_token(oracle_mod):
    rng = np.random.default_rng(2)
    D = 32
    K = (rng.standard_normal((50, D)) * 0.1).astype(np.float16)
    V = rng.standard_normal((50, D)).astype(np.float16)
    q = np.zeros((1, D), np.float16)
    q[0, 3] = 10.0
    K[17, 3] = 20.0                              # score 200*scale above the rest
    out = oracle_mod.reference_pair(K, V, q, 1.0)
    assert np.allclose(out[0], V[17].astype(np.float64), rtol=0, atol=1e-12)


def test_attention_matches_float64_linear_algebra(oracle_mod):
    rng = np.random.default_rng(9)
    R, T, D = 4, 45, 64
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((R, D)).astype(np.float16)
    out, scores = oracle_mod.reference_pair(K, V, q, 0.125, want_scores=True)
    s = 0.125 * q.astype(np.float64) @ K.astype(np.float64).T
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.allclose(scores, s, rtol=1e-13, atol=1e-13)
    assert np.allclose(out, p @ V.astype(np.float64), rtol=1e-12, atol=1e-13)


def test_attention_rope_matches_rotated_keys(oracle_mod):
    rng = np.random.default_rng(4)
    T, D = 40, 64
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((2, D)).astype(np.float16)
    out = oracle_mod.reference_pair(K, V, q, 0.125, rope_on=True, base=10000.0)
    Kr = np.stack([oracle_mod.rope(K[t].astype(np.float64), t, 10000.0) for t in range(T)])
    s = 0.125 * q.astype(np.float64) @ Kr.T
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.allclose(out, p @ V.astype(np.float64), rtol=1e-12, atol=1e-13)


def test_empty_sequence_gives_zero(oracle_mod):
    D = 64
    e = np.zeros((0, D), np.float16)
    out = oracle_mod.reference_pair(e, e, np.ones((2, D), np.float16), 0.125)
    assert not out.any()


def test_tail_equals_prefix_split(oracle_mod):
    """A cache of T tokens is the G-aligned quantized prefix plus the fp16
    tail; the tail tokens enter attention unquantized."""
    rng = np.random.default_rng(12)
    T, D, G = 3 * 32 + 17, 64, 32
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    st = oracle_mod.build_pair(K, V, G, 2, 2)
    assert st["Tq"] == 96 and st["Tt"] == 17
    assert np.array_equal(st["ktail"], K[96:]) and np.array_equal(st["vtail"], V[96:])
    head = oracle_mod.build_pair(K[:96], V[:96], G, 2, 2)
    for key in ("kcodes", "kscale", "kzero", "vcodes", "vscale", "vzero"):
        assert np.array_equal(head[key], st[key])


# ---- the geometry direction the pages report ------------------------------

def test_per_channel_keys_beat_per_token_keys_on_outlier_channels(oracle_mod):
    """Tiny case: 2-bit, G = 32, key channels {3, 17} scaled x50.  Grouping
    keys per channel gives lower key-reconstruction and attention-score error
    than grouping them per token (pages: 4.55 vs 13.67 and 9.60 vs 47.00 on
    Llama-2-13B; only the direction is expected to carry over)."""
    from bit_kv_cache_11_gb300 import synth
    w = synth.WORKLOADS[1]
    case = synth.make_case(w)
    err = {}
    for ak in (0, 1):
        ke, se = [], []
        for h in range(w.n_kv_heads):
            K, V = case["K"][0, h], case["V"][0, h]
            q = case["q"][0, h:h + 1]
            st = oracle_mod.build_pair(K, V, w.group, w.bits_k, w.bits_v, ak, 1)
            kh, _ = oracle_mod.dequantize_pair(st)
            _, s_q = oracle_mod.decode_pair(st, q, w.scale, want_scores=True)
            _, s_r = oracle_mod.reference_pair(K, V, q, w.scale, want_scores=True)
            ke.append(oracle_mod.rel_fro(kh, K))
            se.append(oracle_mod.rel_fro(s_q, s_r))
        err[ak] = (np.mean(ke), np.mean(se))
    assert err[0][0] < err[1][0]
    assert err[0][1] < err[1][1]


# ---- fp16 windows: attention sinks and the recent-token residual ------------

def _append_rule(T, G, n_sink, residual):
    """The windows grown one token at a time: a token fills the sink window
    first, then joins the tail; whenever the tail holds a full group beyond
    the residual window, its oldest G tokens are quantized."""
    Ts = Tq = Tt = 0
    for _ in range(T):
        if Ts < n_sink:
            Ts += 1
            continue
        Tt += 1
        while Tt >= residual + G:
            Tq += G
            Tt -= G
    return Ts, Tq, Tt


@pytest.mark.parametrize("G", [32, 64])
def test_window_lengths_follow_the_append_rule(oracle_mod, G):
    for n_sink in (0, 1, 4, 40):
        for residual in (0, 3, G, 2 * G + 5):
            for T in range(0, 4 * G + 2 * residual + n_sink + 3):
                got = oracle_mod.window_lengths(T, G, n_sink, residual)
                assert got == _append_rule(T, G, n_sink, residual), (T, n_sink, residual)
                Ts, Tq, Tt = got
                assert Tq % G == 0 and Tt < residual + G


@pytest.mark.parametrize("rope_on", [False, True])
def test_all_fp16_windows_reduce_to_plain_attention(oracle_mod, rope_on):
    """When the sink and residual windows cover every token nothing is
    quantized, and the decode is the textbook attention over the fp16 keys
    and values (same fp64 sums, bit for bit)."""
    rng = np.random.default_rng(21)
    T, D = 70, 64
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((2, D)).astype(np.float16)
    ref = oracle_mod.reference_pair(K, V, q, 0.125, rope_on, 10000.0)
    for n_sink, residual in ((T, 0), (0, T), (30, 40), (T + 5, 200)):
        st = oracle_mod.build_pair(K, V, 32, 2, 2, 0, 1, n_sink, residual)
        assert st["Tq"] == 0
        out = oracle_mod.decode_pair(st, q, 0.125, rope_on, 10000.0)
        assert np.array_equal(out, ref), (n_sink, residual)


@pytest.mark.parametrize("rope_on", [False, True])
def test_window_tokens_keep_exact_scores(oracle_mod, rope_on):
    """Sink tokens and the tail keep their fp16 keys: their scores equal the
    unquantized scores exactly (RoPE at their absolute positions), while the
    quantized tokens' scores move."""
    rng = np.random.default_rng(22)
    T, D, G = 150, 64, 32
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((1, D)).astype(np.float16)
    _, s_ref = oracle_mod.reference_pair(K, V, q, 0.125, rope_on, 10000.0, want_scores=True)
    st = oracle_mod.build_pair(K, V, G, 2, 2, 0, 1, n_sink=5, residual=40)
    Ts, Tq, Tt = st["Ts"], st["Tq"], st["Tt"]
    assert (Ts, Tq, Tt) == (5, 96, 49)
    _, s = oracle_mod.decode_pair(st, q, 0.125, rope_on, 10000.0, want_scores=True)
    assert np.array_equal(s[:, :Ts], s_ref[:, :Ts])
    assert np.array_equal(s[:, Ts + Tq:], s_ref[:, Ts + Tq:])
    assert not np.array_equal(s[:, Ts:Ts + Tq], s_ref[:, Ts:Ts + Tq])
    kh, _ = oracle_mod.dequantize_pair(oracle_mod.build_pair(K[Ts:Ts + Tq], V[Ts:Ts + Tq], G, 2, 2))
    assert np.array_equal(kh, oracle_mod.dequantize_pair(st)[0])


def _window_errors(oracle_mod, n_sink, residual):
    from bit_kv_cache_11_gb300 import synth
    w = synth.small(synth.WORKLOADS[2], batch=1, n_kv_heads=4, T=300)
    case = synth.make_case(w, seed=2024)
    se, oe = [], []
    for h in range(w.n_kv_heads):
        K, V, q = case["K"][0, h], case["V"][0, h], case["q"][0, h:h + 1]
        st = oracle_mod.build_pair(K, V, w.group, w.bits_k, w.bits_v, 0, 1, n_sink, residual)
        o, s = oracle_mod.decode_pair(st, q, w.scale, want_scores=True)
        o_r, s_r = oracle_mod.reference_pair(K, V, q, w.scale, want_scores=True)
        se.append(oracle_mod.rel_fro(s, s_r))
        oe.append(oracle_mod.rel_fro(o, o_r))
    return np.mean(se), np.mean(oe)


def _sink_spike_errors(oracle_mod, n_sink):
    """Attention sinks with massive activations: K, V ~ N(0, 1); tokens 0-3
    have keys 8 q / |q| (they draw attention) plus 40 on two fixed channels
    (the sink channels).  2-bit, G = 32, D = 128, T = 300, four heads."""
    rng = np.random.default_rng(77)
    T, D = 300, 128
    se, oe = [], []
    for _ in range(4):
        q = rng.standard_normal((1, D)).astype(np.float16)
        K = rng.standard_normal((T, D)).astype(np.float32)
        V = rng.standard_normal((T, D)).astype(np.float16)
        qf = q[0].astype(np.float32)
        K[:4] = 8.0 * qf / np.linalg.norm(qf)
        K[:4, [5, 77]] += 40.0
        K = K.astype(np.float16)
        st = oracle_mod.build_pair(K, V, 32, 2, 2, 0, 1, n_sink, 0)
        o, s = oracle_mod.decode_pair(st, q, D ** -0.5, want_scores=True)
        o_r, s_r = oracle_mod.reference_pair(K, V, q, D ** -0.5, want_scores=True)
        se.append(oracle_mod.rel_fro(s[:, 4:32], s_r[:, 4:32]))
        oe.append(oracle_mod.rel_fro(o, o_r))
    return np.mean(se), np.mean(oe)


def test_sink_window_lowers_error_on_sink_tokens(oracle_mod):
    """Outliers in the sink tokens' channels widen the key groups they share
    with ordinary tokens; keeping the sinks in fp16 (quantized groups start
    after them) lowers the score error of the ordinary tokens that would have
    shared the sinks' groups (positions 4-31) and the attention-output error
    — the pages' reason for high-precision sink windows (direction only)."""
    s0, o0 = _sink_spike_errors(oracle_mod, 0)
    s4, o4 = _sink_spike_errors(oracle_mod, 4)
    assert s4 < s0 and o4 < 0.5 * o0


def test_residual_window_lowers_error(oracle_mod):
    """A full-precision window of the most recent tokens lowers the
    attention error (the pages' residual-buffer result, direction only)."""
    s0, o0 = _window_errors(oracle_mod, 0, 0)
    s1, o1 = _window_errors(oracle_mod, 0, 128)
    assert s1 < s0 and o1 < o0


# ---- FP8 (E4M3) -----------------------------------------------------------

def test_e4m3_anchor_values(oracle_mod):
    """Codes whose values the format fixes: zero, the smallest subnormal and
    normal, one, two, the largest finite value, signs, NaN."""
    v = oracle_mod.e4m3_value
    assert v(0x00) == 0.0 and v(0x80) == 0.0 and np.signbit(v(0x80))
    assert v(0x01) == 2.0 ** -9 and v(0x07) == 7 * 2.0 ** -9
    assert v(0x08) == 2.0 ** -6 and v(0x38) == 1.0 and v(0x40) == 2.0
    assert v(0x3F) == 1.875 and v(0x77) == 240.0 and v(0x7E) == 448.0
    assert v(0xB8) == -1.0 and v(0xFE) == -448.0
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    pos = oracle_mod.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                      # increasing over the finite codes
    neg = oracle_mod.e4m3_value(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)


def test_e4m3_matches_torch_float8(oracle_mod):
    """An independent implementation: torch's float8_e4m3fn (decode every
    code; encode values inside the finite range, where both round to the
    nearest value with ties to even)."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = oracle_mod.e4m3_value(codes)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~fin)
    assert np.array_equal(got[fin], ref[fin])
    rng = np.random.default_rng(31)
    y = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 2.0 ** -7,
                        oracle_mod.e4m3_value(codes[fin]).astype(np.float64) * (1 + 2.0 ** -5)])
    y = np.clip(y, -448, 448).astype(np.float32)
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_mod.e4m3_encode(y), want)


def test_e4m3_encode_is_nearest_even(oracle_mod):
    """Brute force over the finite values, hand-made ties and saturation."""
    finite = np.arange(0x7F, dtype=np.uint8)
    vals = oracle_mod.e4m3_value(finite).astype(np.float64)
    rng = np.random.default_rng(32)
    y = np.concatenate([rng.uniform(0, 460, 5000), rng.uniform(0, 2.0 ** -5, 5000)]).astype(np.float32)
    got = oracle_mod.e4m3_encode(y)
    for yi, ci in zip(y.astype(np.float64), got):
        d = np.abs(vals - yi)
        best = np.flatnonzero(d == d.min())
        want = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
        if yi >= 448:
            want = 0x7E
        assert ci == want, (yi, ci, want)
    ties = {1.0625: 0x38, 1.1875: 0x3A, 2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02,
            432.0: 0x7E, 400.0: 0x7C, 464.0: 0x7E, 1.0e6: 0x7E}
    for yi, ci in ties.items():
        assert oracle_mod.e4m3_encode(np.float32(yi)) == ci, yi
        assert oracle_mod.e4m3_encode(np.float32(-yi)) == ci | 0x80, -yi


def test_fp8_group_rule(oracle_mod):
    """Scale = fp16(max|x| / 448), zero 0; the largest magnitude codes to
    +-448; every other element to its nearest E4M3 multiple of the scale; a
    group of zeros gives scale 0 and codes 0."""
    rng = np.random.default_rng(33)
    for _ in range(200):
        x = (rng.standard_normal(32) * rng.choice([1e-3, 1.0, 30.0, 3000.0])).astype(np.float16)
        s_h, z_h, codes = oracle_mod.quantize_group_fp8(x)
        xf = x.astype(np.float32)
        amax = np.abs(xf).max()
        assert s_h == oracle_mod.f2h(np.float32(amax / np.float32(448.0))).item() and z_h == 0
        s = oracle_mod.h2f(np.uint16(s_h)).item()
        i = int(np.argmax(np.abs(xf)))
        assert codes[i] & 0x7F == 0x7E
        assert np.array_equal(codes, oracle_mod.e4m3_encode((xf / np.float32(s)).astype(np.float32)))
        xh = oracle_mod.e4m3_value(codes).astype(np.float64) * s
        # relative error at most 2^-4 (three mantissa bits) above the subnormal range
        big = np.abs(xf) >= 2.0 ** -6 * s * 1.0001
        assert np.all(np.abs(xh - xf)[big] <= 2.0 ** -4 * np.abs(xf)[big] * (1 + 2.0 ** -10))
    s_h, z_h, codes = oracle_mod.quantize_group_fp8(np.zeros(32, np.float16))
    assert s_h == 0 and not codes.any()


def test_fp8_dequantize_is_value_times_scale(oracle_mod):
    rng = np.random.default_rng(34)
    X = (rng.standard_normal((64, 64)) * 5).astype(np.float16)
    for axis in (0, 1):
        _, codes, sc, zr = oracle_mod.quantize_tensor(X, 32, 8, axis, fp8=True)
        assert not zr.any()
        got = oracle_mod.dequantize_tensor(codes, sc, zr, 32, axis, fp8=True)
        s = oracle_mod.h2f(sc).astype(np.float64)
        s = np.repeat(s, 32, axis=0) if axis == 0 else np.repeat(s, 32, axis=1)
        want = oracle_mod.e4m3_value(codes).astype(np.float64) * s
        assert np.array_equal(got.astype(np.float64), want)
        # FP8 keeps more of the signal than 4-bit integer codes on the same groups
        _, c4, s4, z4 = oracle_mod.quantize_tensor(X, 32, 4, axis)
        e8 = oracle_mod.rel_fro(got, X.astype(np.float32))
        e4 = oracle_mod.rel_fro(oracle_mod.dequantize_tensor(c4, s4, z4, 32, axis), X.astype(np.float32))
        assert e8 < e4


def test_fp8_cache_error_is_small_next_to_low_bit_codes(oracle_mod):
    """On the Llama-2-7B-shaped recipe (outlier key channels, sink tokens) an
    FP8 cache keeps the attention output much closer to the fp16 result than
    4- and 2-bit integer codes on the same groups: the pages' case for trying
    FP8 first (direction only)."""
    from bit_kv_cache_11_gb300 import synth
    w = synth.small(synth.WORKLOADS[2], batch=1, n_kv_heads=4, T=300)
    case = synth.make_case(w, seed=2025)
    err = {}
    for name, bits, fp8 in (("fp8", 8, True), ("int4", 4, False), ("int2", 2, False)):
        oe = []
        for h in range(w.n_kv_heads):
            K, V, q = case["K"][0, h], case["V"][0, h], case["q"][0, h:h + 1]
            st = oracle_mod.build_pair(K, V, 32, bits, bits, 0, 1, fp8=fp8)
            out = oracle_mod.decode_pair(st, q, w.scale)
            ref = oracle_mod.reference_pair(K, V, q, w.scale)
            oe.append(oracle_mod.rel_fro(out, ref))
        err[name] = np.mean(oe)
    assert err["fp8"] < 0.6 * err["int4"]
    assert err["fp8"] < 0.1 * err["int2"]
