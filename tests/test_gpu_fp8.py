"""FP8 (E4M3) cache on the GPU, through the C ABI, against the CPU oracle.

The format (oracle, pinned in test_oracle_pins): the integer path's groups,
scale = fp16(max|x| / 448), zero 0, codes E4M3(x / scale) with ties to even
and saturation.  Bars: packed blocks (E4M3 codes, scales, zeros) and tails
bit-exact; dequantized values bit-exact; decode within 2e-3 max abs and 1e-3
relative L2 of the fp64 attention over the same dequantized values.
"""
import zlib

import numpy as np
import pytest

from bit_kv_cache_11_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = 2e-3
RTOL_L2 = 1e-3


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_kv_cache_11_gb300 import kvq as k
    return k


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def workload(D, R, ak, av, G, rope, T, batch=2, hkv=3):
    return synth.Workload("fp8", batch, hkv * R, hkv, D, T, 8, 8, G, ak, av, rope,
                          outlier_scales=(20.0, 100.0), n_outliers=2, config_id=9)


def make_cache(kvq, w, max_ctx, n_sink=0, residual=0):
    return kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_ctx=max_ctx, bits_k=8, bits_v=8,
                       group=w.group, axis_k=w.axis_k, axis_v=w.axis_v,
                       keys_pre_rope=w.keys_pre_rope, rope_base=w.rope_base,
                       n_sink=n_sink, residual=residual, fp8=True)


def pair_state(orc, w, K, V, p, n_sink=0, residual=0):
    b, h = divmod(p, w.n_kv_heads)
    return orc.build_pair(K[b, h], V[b, h], w.group, 8, 8, w.axis_k, w.axis_v, n_sink, residual,
                          fp8=True)


def check_state(orc, cache, w, K, V, pairs, n_sink=0, residual=0):
    T = K.shape[2]
    Ts, Tq, Tt = orc.window_lengths(T, w.group, n_sink, residual)
    assert cache.state == (Tq, Tt)
    blocks = cache.block_bytes_view()
    kt, vt = cache.tail_views()
    for p in pairs:
        st = pair_state(orc, w, K, V, p, n_sink, residual)
        assert np.array_equal(blocks[p, : Tq // w.group].cpu().numpy(), orc.pack_pair(st)), p
        assert np.array_equal(kt[p, :Tt].cpu().numpy().view(np.uint16), st["ktail"].view(np.uint16))
        assert np.array_equal(vt[p, :Tt].cpu().numpy().view(np.uint16), st["vtail"].view(np.uint16))


def check_decode(orc, cache, w, K, V, q, pairs, n_sink=0, residual=0, out=None):
    if out is None:
        out = cache.decode(dev(q), softmax_scale=w.scale)
    torch.cuda.synchronize()
    out = out.cpu().numpy().astype(np.float64)
    R = w.gqa
    got, want = [], []
    for p in pairs:
        b, h = divmod(p, w.n_kv_heads)
        st = pair_state(orc, w, K, V, p, n_sink, residual)
        want.append(orc.decode_pair(st, q[b, h * R:(h + 1) * R], w.scale, w.keys_pre_rope,
                                    w.rope_base))
        got.append(out[b, h * R:(h + 1) * R])
    got, want = np.stack(got), np.stack(want)
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert err <= ATOL, f"max abs {err:.3e}"
    assert rel <= RTOL_L2, f"rel L2 {rel:.3e}"


# name, D, R, ak, av, G, rope, T
CASES = [
    ("mma-d128-r1", 128, 1, 0, 1, 32, False, 5 * 32 + 9),
    ("mma-d64-r8", 64, 8, 0, 1, 32, False, 4 * 32 + 31),
    ("mma-d128-r4-rope", 128, 4, 0, 1, 32, True, 3 * 32 + 7),
    ("mma-d64-r1-rope", 64, 1, 0, 1, 32, True, 100),
    ("gen-g128-ch/tok", 128, 2, 0, 1, 128, False, 2 * 128 + 45),
    ("gen-g32-tok/tok", 128, 4, 1, 1, 32, False, 6 * 32 + 1),
    ("gen-g64-ch/ch-rope", 64, 2, 0, 0, 64, True, 3 * 64 + 20),
    ("gen-g32-tok/ch", 128, 1, 1, 0, 32, False, 4 * 32),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fp8_prefill_dequant_decode(kvq, orc, case):
    name, D, R, ak, av, G, rope, T = case
    w = workload(D, R, ak, av, G, rope, T)
    c = synth.make_case(w, seed=zlib.crc32(name.encode()) % 10000)
    pairs = list(range(w.n_pairs))
    with make_cache(kvq, w, T + 64) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        check_state(orc, cache, w, c["K"], c["V"], pairs)
        kh, vh = cache.dequantize()
        torch.cuda.synchronize()
        for p in pairs:
            b, h = divmod(p, w.n_kv_heads)
            okh, ovh = orc.dequantize_pair(pair_state(orc, w, c["K"], c["V"], p))
            assert np.array_equal(kh[b, h].cpu().numpy().view(np.uint32), okh.view(np.uint32))
            assert np.array_equal(vh[b, h].cpu().numpy().view(np.uint32), ovh.view(np.uint32))
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], pairs)
        cache.check()


@pytest.mark.parametrize("case,T0,ns", [
    (CASES[0], 3, [1, 28, 1, 1, 33, 64, 5]),
    (CASES[4], 100, [27, 1, 128, 129, 2]),
], ids=["mma", "gen-g128"])
def test_fp8_append_flush(kvq, orc, case, T0, ns):
    name, D, R, ak, av, G, rope, _ = case
    total = T0 + sum(ns)
    w = workload(D, R, ak, av, G, rope, total)
    c = synth.make_case(w, seed=61)
    K, V = c["K"], c["V"]
    pairs = list(range(w.n_pairs))
    with make_cache(kvq, w, total) as cache:
        cache.prefill(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
        T = T0
        for n in ns:
            cache.append(dev(K[:, :, T:T + n]), dev(V[:, :, T:T + n]))
            T += n
            torch.cuda.synchronize()
            check_state(orc, cache, w, K[:, :, :T], V[:, :, :T], pairs)
            check_decode(orc, cache, w, K[:, :, :T], V[:, :, :T], c["q"], pairs)
        cache.check()


def test_fp8_append_decode_with_windows(kvq, orc):
    """FP8 with 4 sink tokens and a 40-token residual window, one decode step
    at a time through kvq_append_decode."""
    w = workload(128, 2, 0, 1, 32, True, 300)
    n_sink, residual = 4, 40
    c = synth.make_case(w, seed=62)
    K, V = c["K"], c["V"]
    pairs = list(range(w.n_pairs))
    q = dev(c["q"])
    with make_cache(kvq, w, 300, n_sink, residual) as cache:
        cache.prefill(dev(K[:, :, :150]), dev(V[:, :, :150]))
        T = 150
        for n in [1, 1, 30, 1, 1, 40, 1, 20]:
            out = cache.append_decode(dev(K[:, :, T:T + n]), dev(V[:, :, T:T + n]), q,
                                      softmax_scale=w.scale)
            T += n
            torch.cuda.synchronize()
            check_state(orc, cache, w, K[:, :, :T], V[:, :, :T], pairs, n_sink, residual)
            check_decode(orc, cache, w, K[:, :, :T], V[:, :, :T], c["q"], pairs, n_sink, residual,
                         out=out)
        cache.check()


def test_fp8_full_size_sampled(kvq, orc):
    """Llama-2-7B-shaped layer (B8, H32, D128, T4113) as an FP8 cache,
    sampled pairs."""
    w = synth.WORKLOADS[2].with_(bits_k=8, bits_v=8)
    c = synth.make_case(w)
    rng = np.random.default_rng(8)
    pairs = sorted({0, w.n_pairs - 1, *rng.choice(w.n_pairs, 5, replace=False).tolist()})
    with make_cache(kvq, w, w.T + 64) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        check_state(orc, cache, w, c["K"], c["V"], pairs)
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], pairs)
        cache.check()
