"""fp16 windows (attention sinks and the recent-token residual) on the GPU,
through the C ABI, against the CPU oracle.

The oracle's definition (``oracle.window_lengths`` / ``oracle.build_pair``):
the first n_sink tokens stay fp16; of the rest, a group of G is quantized only
when at least ``residual`` newer tokens remain in the fp16 tail.  Bars as in
test_gpu_parity: packed blocks, sink rows and tail rows bit-exact; decode
within 2e-3 max abs and 1e-3 relative L2 of the fp64 attention.
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


def workload(D, R, bk, bv, ak, av, G, rope, T, batch=2, hkv=3):
    return synth.Workload("windows", batch, hkv * R, hkv, D, T, bk, bv, G, ak, av, rope,
                          outlier_scales=(20.0, 100.0), n_outliers=2, config_id=9)


def make_cache(kvq, w, max_ctx, n_sink, residual):
    return kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_ctx=max_ctx, bits_k=w.bits_k, bits_v=w.bits_v,
                       group=w.group, axis_k=w.axis_k, axis_v=w.axis_v,
                       keys_pre_rope=w.keys_pre_rope, rope_base=w.rope_base,
                       n_sink=n_sink, residual=residual)


def pair_state(orc, w, K, V, p, n_sink, residual):
    b, h = divmod(p, w.n_kv_heads)
    return orc.build_pair(K[b, h], V[b, h], w.group, w.bits_k, w.bits_v, w.axis_k, w.axis_v,
                          n_sink, residual)


def check_state(orc, cache, w, K, V, n_sink, residual, pairs):
    """K, V: fp16 [B][Hkv][T][D], every token the cache received so far."""
    T = K.shape[2]
    Ts, Tq, Tt = orc.window_lengths(T, w.group, n_sink, residual)
    b = cache.buffers()
    assert (b.T_sink, b.T_q, b.T_tail) == (Ts, Tq, Tt)
    assert b.tail_rows == residual + w.group
    assert cache.state == (Tq, Tt)
    blocks = cache.block_bytes_view()
    kt, vt = cache.tail_views()
    sv = cache.sink_views()
    assert (sv is None) == (n_sink == 0)
    for p in pairs:
        st = pair_state(orc, w, K, V, p, n_sink, residual)
        assert np.array_equal(blocks[p, : Tq // w.group].cpu().numpy(), orc.pack_pair(st)), p
        assert np.array_equal(kt[p, :Tt].cpu().numpy().view(np.uint16), st["ktail"].view(np.uint16))
        assert np.array_equal(vt[p, :Tt].cpu().numpy().view(np.uint16), st["vtail"].view(np.uint16))
        if sv is not None:
            assert np.array_equal(sv[0][p, :Ts].cpu().numpy().view(np.uint16),
                                  st["ksink"].view(np.uint16))
            assert np.array_equal(sv[1][p, :Ts].cpu().numpy().view(np.uint16),
                                  st["vsink"].view(np.uint16))


def expected(orc, w, K, V, q, n_sink, residual, pairs):
    R = w.gqa
    out = []
    for p in pairs:
        b, h = divmod(p, w.n_kv_heads)
        st = pair_state(orc, w, K, V, p, n_sink, residual)
        out.append(orc.decode_pair(st, q[b, h * R:(h + 1) * R], w.scale, w.keys_pre_rope,
                                   w.rope_base))
    return np.stack(out)


def compare(got_bhd, w, want, pairs):
    R = w.gqa
    got = np.stack([got_bhd[p // w.n_kv_heads, (p % w.n_kv_heads) * R:(p % w.n_kv_heads + 1) * R]
                    for p in pairs]).astype(np.float64)
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert err <= ATOL, f"max abs {err:.3e}"
    assert rel <= RTOL_L2, f"rel L2 {rel:.3e}"


def check_decode(orc, cache, w, K, V, q, n_sink, residual, pairs):
    out = cache.decode(dev(q), softmax_scale=w.scale)
    torch.cuda.synchronize()
    compare(out.cpu().numpy(), w, expected(orc, w, K, V, q, n_sink, residual, pairs), pairs)


# name, D, R, bk, bv, ak, av, G, rope, T, n_sink, residual
CASES = [
    ("mma-2/2-s4-r64", 128, 1, 2, 2, 0, 1, 32, False, 5 * 32 + 9, 4, 64),
    ("mma-2/2-r4-s4-r32-rope", 128, 4, 2, 2, 0, 1, 32, True, 4 * 32 + 3, 4, 32),
    ("mma-4/4-d64-s1-r100", 64, 2, 4, 4, 0, 1, 32, False, 300, 1, 100),
    ("mma-T-below-sinks", 128, 1, 2, 2, 0, 1, 32, False, 3, 4, 0),
    ("mma-T-below-residual-rope", 128, 1, 2, 2, 0, 1, 32, True, 50, 4, 128),
    ("mma-8/2-s7", 128, 1, 8, 2, 0, 1, 32, False, 200, 7, 0),
    ("mma-2/4-r8-s40-rope", 128, 8, 2, 4, 0, 1, 32, True, 200, 40, 0),
    ("mma-2/2-r0-s0-r96", 128, 2, 2, 2, 0, 1, 32, False, 7 * 32 + 1, 0, 96),
    ("gen-g128-rope-s4-r128", 128, 1, 2, 2, 0, 1, 128, True, 3 * 128 + 50, 4, 128),
    ("gen-tok/tok-g32-s3-r40", 128, 4, 2, 2, 1, 1, 32, False, 250, 3, 40),
    ("gen-ch/ch-g64-d64-s16-r64-rope", 64, 2, 4, 2, 0, 0, 64, True, 400, 16, 64),
    ("gen-tok/ch-g64-8/2-s5", 128, 1, 8, 2, 1, 0, 64, False, 2 * 64 + 63, 5, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_windows(kvq, orc, case):
    name, D, R, bk, bv, ak, av, G, rope, T, n_sink, residual = case
    w = workload(D, R, bk, bv, ak, av, G, rope, T)
    c = synth.make_case(w, seed=zlib.crc32(name.encode()) % 10000)
    pairs = list(range(w.n_pairs))
    with make_cache(kvq, w, T + 64, n_sink, residual) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        check_state(orc, cache, w, c["K"], c["V"], n_sink, residual, pairs)
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], n_sink, residual, pairs)
        cache.check()


@pytest.mark.parametrize("case,T0,ns", [
    (CASES[0], 2, [1, 1, 1, 30, 33, 1, 64, 5, 100]),
    (CASES[1], 0, [3, 2, 40, 1, 1, 31, 70]),
    (CASES[2], 1, [150, 1, 31, 1, 60, 2]),
    (CASES[8], 3, [2, 200, 127, 1, 128, 129]),
    (CASES[9], 0, [1, 1, 1, 1, 39, 1, 31, 40]),
], ids=["mma-s4-r64", "mma-rope-r4", "mma-d64-r100", "gen-g128-rope", "gen-tok-tok"])
def test_append_windows(kvq, orc, case, T0, ns):
    """Appends fill the sink window first, then the tail; the residual window
    delays every flush; the state after each call equals the oracle's
    whole-sequence state."""
    name, D, R, bk, bv, ak, av, G, rope, _, n_sink, residual = case
    total = T0 + sum(ns)
    w = workload(D, R, bk, bv, ak, av, G, rope, total)
    c = synth.make_case(w, seed=88)
    K, V = c["K"], c["V"]
    pairs = list(range(w.n_pairs))
    with make_cache(kvq, w, total, n_sink, residual) as cache:
        cache.prefill(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
        T = T0
        for n in ns:
            cache.append(dev(K[:, :, T:T + n]), dev(V[:, :, T:T + n]))
            T += n
            torch.cuda.synchronize()
            check_state(orc, cache, w, K[:, :, :T], V[:, :, :T], n_sink, residual, pairs)
            check_decode(orc, cache, w, K[:, :, :T], V[:, :, :T], c["q"], n_sink, residual, pairs)
        cache.check()


@pytest.mark.parametrize("case,T0,ns", [
    (CASES[0], 1, [1, 1, 1, 1, 5, 20, 1, 40, 1, 1, 60, 1]),
    (CASES[1], 6, [1, 1, 29, 1, 2, 1]),
    (CASES[7], 0, [1, 130, 1, 1, 30, 1, 33]),
], ids=["mma-s4-r64", "mma-rope-r4", "mma-r96"])
def test_append_decode_windows(kvq, orc, case, T0, ns):
    """kvq_append_decode with windows: one launch when the tokens go to the
    tail and no group leaves the residual window; bit-identical to append +
    decode on a second cache; matches the oracle."""
    name, D, R, bk, bv, ak, av, G, rope, _, n_sink, residual = case
    total = T0 + sum(ns)
    w = workload(D, R, bk, bv, ak, av, G, rope, total)
    c = synth.make_case(w, seed=93)
    K, V = c["K"], c["V"]
    pairs = list(range(w.n_pairs))
    q = dev(c["q"])
    with make_cache(kvq, w, total, n_sink, residual) as fused, \
            make_cache(kvq, w, total, n_sink, residual) as split:
        fused.prefill(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
        split.prefill(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
        T = T0
        for n in ns:
            k, v = dev(K[:, :, T:T + n]), dev(V[:, :, T:T + n])
            Ts, _, Tt = orc.window_lengths(T, G, n_sink, residual)
            launches = kvq.kvq_launch_count()
            a = fused.append_decode(k, v, q, softmax_scale=w.scale)
            torch.cuda.synchronize()
            if Ts == n_sink and Tt + n < residual + G:
                assert kvq.kvq_launch_count() - launches == 1
            split.append(k, v)
            b = split.decode(q, softmax_scale=w.scale)
            T += n
            torch.cuda.synchronize()
            assert torch.equal(a, b)
            assert fused.state == split.state
            check_state(orc, fused, w, K[:, :, :T], V[:, :, :T], n_sink, residual, pairs)
            compare(a.cpu().numpy(), w,
                    expected(orc, w, K[:, :, :T], V[:, :, :T], c["q"], n_sink, residual, pairs), pairs)
        fused.check()
        split.check()


def test_full_size_windows_sampled(kvq, orc):
    """Llama-2-7B-shaped layer (B8, H32, D128, T4113, 2-bit) with four sink
    tokens and a 128-token residual window: sampled pairs."""
    w = synth.WORKLOADS[2]
    n_sink, residual = 4, 128
    c = synth.make_case(w)
    rng = np.random.default_rng(3)
    pairs = sorted({0, w.n_pairs - 1, *rng.choice(w.n_pairs, 5, replace=False).tolist()})
    with make_cache(kvq, w, w.T + 64, n_sink, residual) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        assert cache.buffers().T_sink == 4 and cache.state == (3968, 141)
        check_state(orc, cache, w, c["K"], c["V"], n_sink, residual, pairs)
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], n_sink, residual, pairs)
        cache.check()


def test_capacity_counts_the_sinks(kvq):
    w = workload(128, 1, 2, 2, 0, 1, 32, False, 40)
    c = synth.make_case(w, seed=4)
    K, V = dev(c["K"]), dev(c["V"])
    with make_cache(kvq, w, 48, 4, 32) as cache:
        cache.prefill(K, V)
        torch.cuda.synchronize()
        assert cache.buffers().T_sink == 4 and cache.state == (0, 36)
        with pytest.raises(kvq.KvqError) as ei:
            kvq.kvq_append(cache.handle, K, V, 9)          # 4 + 36 + 9 > 48
        assert ei.value.status == kvq.KVQ_ERR_CAPACITY
        kvq.kvq_append(cache.handle, K, V, 8)              # exactly full: 4 + 0 + 44
        torch.cuda.synchronize()
        assert cache.state == (0, 44)
        cache.check()
