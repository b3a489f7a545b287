"""CUDA path vs the CPU oracle, through the C ABI.

Bars (from the method's definition, see the oracle):
  * packed blocks (codes, fp16 scales and zeros, layout) and the fp16 tail are
    bit-exact;
  * dequantized values are bit-exact (both sides use one fused multiply-add);
  * decode attention is within 2e-3 max abs and 1e-3 relative L2 of the
    oracle's fp64 attention over the same dequantized values.
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


def make_cache(kvq, w, max_ctx):
    return kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_ctx=max_ctx, bits_k=w.bits_k, bits_v=w.bits_v,
                       group=w.group, axis_k=w.axis_k, axis_v=w.axis_v,
                       keys_pre_rope=w.keys_pre_rope, rope_base=w.rope_base)


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def check_state(orc, cache, w, K, V, pairs):
    """K, V: fp16 [B][Hkv][T][D], every token the cache received so far."""
    T = K.shape[2]
    tq, tt = cache.state
    assert tq == (T // w.group) * w.group and tt == T - tq
    blocks = cache.block_bytes_view()
    kt, vt = cache.tail_views()
    for p in pairs:
        b, h = divmod(p, w.n_kv_heads)
        st = orc.build_pair(K[b, h], V[b, h], w.group, w.bits_k, w.bits_v, w.axis_k, w.axis_v)
        want = orc.pack_pair(st)
        got = blocks[p, : tq // w.group].cpu().numpy()
        assert np.array_equal(got, want), f"pair {p}: packed blocks differ"
        assert np.array_equal(kt[p, :tt].cpu().numpy().view(np.uint16), st["ktail"].view(np.uint16))
        assert np.array_equal(vt[p, :tt].cpu().numpy().view(np.uint16), st["vtail"].view(np.uint16))


def check_dequant(orc, cache, w, K, V, pairs):
    kh, vh = cache.dequantize()
    torch.cuda.synchronize()
    for p in pairs:
        b, h = divmod(p, w.n_kv_heads)
        st = orc.build_pair(K[b, h], V[b, h], w.group, w.bits_k, w.bits_v, w.axis_k, w.axis_v)
        okh, ovh = orc.dequantize_pair(st)
        assert np.array_equal(kh[b, h].cpu().numpy().view(np.uint32), okh.view(np.uint32))
        assert np.array_equal(vh[b, h].cpu().numpy().view(np.uint32), ovh.view(np.uint32))


def check_decode(orc, cache, w, K, V, q, pairs):
    out = cache.decode(dev(q), softmax_scale=w.scale)
    torch.cuda.synchronize()
    out = out.cpu().numpy().astype(np.float64)
    R = w.gqa
    got, want = [], []
    for p in pairs:
        b, h = divmod(p, w.n_kv_heads)
        st = orc.build_pair(K[b, h], V[b, h], w.group, w.bits_k, w.bits_v, w.axis_k, w.axis_v)
        ref = orc.decode_pair(st, q[b, h * R:(h + 1) * R], w.scale, w.keys_pre_rope, w.rope_base)
        got.append(out[b, h * R:(h + 1) * R])
        want.append(ref)
    got, want = np.stack(got), np.stack(want)
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert err <= ATOL, f"max abs {err:.3e}"
    assert rel <= RTOL_L2, f"rel L2 {rel:.3e}"
    return err, rel


# name, D, R, bk, bv, ak, av, G, rope, T
SMALL = [
    ("d128-r1-2/2-ch/tok-g32", 128, 1, 2, 2, 0, 1, 32, False, 4 * 32 + 17),
    ("d64-r1-2/2-ch/tok-g32", 64, 1, 2, 2, 0, 1, 32, False, 256),
    ("d128-r4-2/2-ch/tok-g32", 128, 4, 2, 2, 0, 1, 32, False, 7 * 32 + 3),
    ("d128-r1-4/4-rope", 128, 1, 4, 4, 0, 1, 32, True, 3 * 32 + 5),
    ("d128-r1-2/2-rope-g128", 128, 1, 2, 2, 0, 1, 128, True, 2 * 128 + 77),
    ("d128-r2-8/8", 128, 2, 8, 8, 0, 1, 32, False, 100),
    ("d128-r8-8/4-g128", 128, 8, 8, 4, 0, 1, 128, False, 2 * 128 + 45),
    ("d128-r4-4/4-tok/ch-g32", 128, 4, 4, 4, 1, 0, 32, False, 5 * 32 + 9),
    ("d128-r4-2/2-ch/ch-g128", 128, 4, 2, 2, 0, 0, 128, False, 3 * 128 + 1),
    ("d128-r4-2/2-tok/tok-g128", 128, 4, 2, 2, 1, 1, 128, False, 3 * 128 + 100),
    ("d64-r4-2/8-tok/tok-g32-rope", 64, 4, 2, 8, 1, 1, 32, True, 70),
    ("d64-r2-4/2-ch/ch-g64", 64, 2, 4, 2, 0, 0, 64, False, 64 * 3 + 1),
    ("d128-r1-8/2-tok/ch-g64-rope", 128, 1, 8, 2, 1, 0, 64, True, 64 * 2 + 63),
    ("tail-only", 128, 1, 2, 2, 0, 1, 32, False, 17),
    ("no-tail", 128, 4, 4, 4, 0, 1, 32, False, 96),
    ("single-token-rope", 64, 1, 8, 8, 0, 1, 32, True, 1),
    # tensor-core kernel (keys per channel, values per token, G = 32): every
    # bit-width pair, every GQA ratio, both head dims, keys before RoPE
    ("mma-2/4-d128-r2", 128, 2, 2, 4, 0, 1, 32, False, 3 * 32 + 11),
    ("mma-4/2-d64-r8", 64, 8, 4, 2, 0, 1, 32, False, 5 * 32 + 30),
    ("mma-2/8-d128-r4-rope", 128, 4, 2, 8, 0, 1, 32, True, 2 * 32 + 7),
    ("mma-8/2-d64-r1", 64, 1, 8, 2, 0, 1, 32, False, 6 * 32 + 1),
    ("mma-4/8-d128-r8", 128, 8, 4, 8, 0, 1, 32, False, 3 * 32 + 20),
    ("mma-8/4-d128-r1-rope", 128, 1, 8, 4, 0, 1, 32, True, 4 * 32 + 13),
    ("mma-2/2-d128-r8", 128, 8, 2, 2, 0, 1, 32, False, 4 * 32 + 31),
    ("mma-4/4-d64-r2-rope", 64, 2, 4, 4, 0, 1, 32, True, 3 * 32 + 2),
    ("mma-2/2-d128-r8-rope", 128, 8, 2, 2, 0, 1, 32, True, 2 * 32 + 9),
    ("mma-4/4-d64-r4", 64, 4, 4, 4, 0, 1, 32, False, 4 * 32),
]


def small_workload(D, R, bk, bv, ak, av, G, rope, T, batch=2, hkv=3):
    return synth.Workload("small", batch, hkv * R, hkv, D, T, bk, bv, G, ak, av, rope,
                          outlier_scales=(20.0, 100.0), n_outliers=2, config_id=9)


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_prefill_dequant_decode_small(kvq, orc, case):
    name, D, R, bk, bv, ak, av, G, rope, T = case
    w = small_workload(D, R, bk, bv, ak, av, G, rope, T)
    c = synth.make_case(w, seed=zlib.crc32(name.encode()) % 10000)
    pairs = list(range(w.n_pairs))
    with make_cache(kvq, w, max_ctx=T + 300) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        check_state(orc, cache, w, c["K"], c["V"], pairs)
        check_dequant(orc, cache, w, c["K"], c["V"], pairs)
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], pairs)
        cache.check()


@pytest.mark.parametrize("case,T0,ns", [
    (SMALL[0], 0, [1, 1, 30, 1, 33, 64, 2, 95]),
    (SMALL[2], 17, [15, 1, 31, 32, 33, 1]),
    (SMALL[4], 31, [97, 1, 127, 128, 129, 3]),
    (SMALL[10], 5, [26, 1, 1, 40, 70]),
], ids=["g32-r1", "g32-r4", "g128-rope", "d64-tok"])
def test_append_flush_sequences(kvq, orc, case, T0, ns):
    name, D, R, bk, bv, ak, av, G, rope, _ = case
    total = T0 + sum(ns)
    w = small_workload(D, R, bk, bv, ak, av, G, rope, total)
    c = synth.make_case(w, seed=77)
    K, V = c["K"], c["V"]
    pairs = list(range(w.n_pairs))
    with make_cache(kvq, w, max_ctx=total) as cache:
        cache.prefill(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
        T = T0
        for n in ns:
            cache.append(dev(K[:, :, T:T + n]), dev(V[:, :, T:T + n]))
            T += n
            torch.cuda.synchronize()
            check_state(orc, cache, w, K[:, :, :T], V[:, :, :T], pairs)
            check_decode(orc, cache, w, K[:, :, :T], V[:, :, :T], c["q"], pairs)
        cache.check()


@pytest.mark.parametrize("case,T0,ns", [
    (SMALL[0], 3, [1, 1, 5, 20, 2, 1, 1, 33, 1, 60]),
    (SMALL[2], 30, [1, 1, 1, 29, 1, 2]),
    (SMALL[1], 0, [1, 31, 1, 1]),
    (SMALL[3], 10, [1, 20, 1, 9, 1]),
], ids=["g32-r1", "g32-r4", "d64-from-empty", "rope-4bit"])
def test_append_decode_steps(kvq, orc, case, T0, ns):
    """kvq_append_decode (one launch when no group completes) equals
    kvq_append + kvq_decode_attention on a second cache bit for bit, keeps the
    same state, and matches the oracle."""
    name, D, R, bk, bv, ak, av, G, rope, _ = case
    total = T0 + sum(ns)
    w = small_workload(D, R, bk, bv, ak, av, G, rope, total)
    c = synth.make_case(w, seed=91)
    K, V = c["K"], c["V"]
    pairs = list(range(w.n_pairs))
    q = dev(c["q"])
    with make_cache(kvq, w, max_ctx=total) as fused, make_cache(kvq, w, max_ctx=total) as split:
        fused.prefill(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
        split.prefill(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
        T = T0
        for n in ns:
            k, v = dev(K[:, :, T:T + n]), dev(V[:, :, T:T + n])
            launches = kvq.kvq_launch_count()
            a = fused.append_decode(k, v, q, softmax_scale=w.scale)
            torch.cuda.synchronize()
            if (T - (T // G) * G) + n < G:
                assert kvq.kvq_launch_count() - launches == 1   # one fused launch
            split.append(k, v)
            b = split.decode(q, softmax_scale=w.scale)
            T += n
            torch.cuda.synchronize()
            assert torch.equal(a, b)
            assert fused.state == split.state
            check_state(orc, fused, w, K[:, :, :T], V[:, :, :T], pairs)
            got = a.cpu().numpy().astype(np.float64)
            for p in pairs:
                bb, h = divmod(p, w.n_kv_heads)
                st = orc.build_pair(K[bb, h, :T], V[bb, h, :T], G, bk, bv, ak, av)
                ref = orc.decode_pair(st, c["q"][bb, h * R:(h + 1) * R], w.scale, rope, w.rope_base)
                assert np.abs(got[bb, h * R:(h + 1) * R] - ref).max() <= ATOL
        fused.check()
        split.check()


def test_empty_cache_decodes_to_zero(kvq):
    w = small_workload(128, 4, 2, 2, 0, 1, 32, False, 0)
    with make_cache(kvq, w, max_ctx=64) as cache:
        q = torch.randn(w.batch, w.n_q_heads, w.head_dim, device="cuda").half()
        out = torch.full((w.batch, w.n_q_heads, w.head_dim), 7.0, device="cuda")
        cache.decode(q, out)
        torch.cuda.synchronize()
        assert not out.any()


def test_errors_leave_state_unchanged(kvq, orc):
    w = small_workload(128, 1, 2, 2, 0, 1, 32, False, 40)
    c = synth.make_case(w, seed=5)
    K, V = dev(c["K"]), dev(c["V"])
    with make_cache(kvq, w, max_ctx=48) as cache:
        cache.prefill(K, V)
        torch.cuda.synchronize()
        before = cache.block_bytes_view().clone(), [t.clone() for t in cache.tail_views()], cache.state
        raw = torch.empty(K.numel() * 2 + 16, dtype=torch.uint8, device="cuda")
        mis = raw[2:].data_ptr()                                   # not 16-byte aligned
        cases = [
            (lambda: kvq.kvq_append(cache.handle, mis, V, 1), kvq.KVQ_ERR_INVALID_ARG),
            (lambda: kvq.kvq_append(cache.handle, K, V, 9), kvq.KVQ_ERR_CAPACITY),   # 40 + 9 > 48
            (lambda: kvq.kvq_append(cache.handle, K, V, -1), kvq.KVQ_ERR_INVALID_ARG),
            (lambda: kvq.kvq_quantize_prefill(cache.handle, K, V, 49), kvq.KVQ_ERR_CAPACITY),
            (lambda: kvq.kvq_decode_attention(cache.handle, mis, K, 0.1), kvq.KVQ_ERR_INVALID_ARG),
            (lambda: kvq.kvq_decode_attention(cache.handle, K, K, float("nan")), kvq.KVQ_ERR_INVALID_ARG),
            (lambda: kvq.kvq_dequantize(cache.handle, None, K), kvq.KVQ_ERR_INVALID_ARG),
        ]
        for fn, status in cases:
            with pytest.raises(kvq.KvqError) as ei:
                fn()
            assert ei.value.status == status
        torch.cuda.synchronize()
        assert cache.state == before[2]
        assert torch.equal(cache.block_bytes_view(), before[0])
        for a, b in zip(cache.tail_views(), before[1]):
            assert torch.equal(a, b)
        check_state(orc, cache, w, c["K"], c["V"], range(w.n_pairs))
        cache.check()


def test_launch_counter_counts_kernels(kvq):
    w = small_workload(128, 1, 2, 2, 0, 1, 32, False, 64)
    c = synth.make_case(w, seed=6)
    with make_cache(kvq, w, max_ctx=128) as cache:
        n0 = kvq.kvq_launch_count()
        cache.prefill(dev(c["K"]), dev(c["V"]))
        cache.decode(dev(c["q"]))
        torch.cuda.synchronize()
        # quantize, then one decode kernel: this geometry runs the tensor-core
        # kernel, which merges the split partials in place
        assert kvq.kvq_launch_count() - n0 == 2


# ---- the full-size workloads, sampled pairs ----------------------------------

def _sample_pairs(w, k, seed):
    rng = np.random.default_rng(seed)
    picks = {0, w.n_pairs - 1}
    picks.update(rng.choice(w.n_pairs, size=min(k, w.n_pairs), replace=False).tolist())
    return sorted(picks)


@pytest.mark.parametrize("cfg,bits", [(1, 2), (2, 2), (3, 2), (3, 4)],
                         ids=["tiny-b1-h2-d64-t256", "llama7b-b8", "llama13b-2bit", "llama13b-4bit"])
def test_full_size_decode_sampled(kvq, orc, cfg, bits):
    """The workloads at their stated sizes (the tiny case exactly as stated:
    batch 1, 2 heads, head_dim 64, 256 tokens, x50 outliers on channels
    {3, 17}; every pair checked), in the launch configuration the bench
    uses."""
    w = synth.WORKLOADS[cfg].with_(bits_k=bits, bits_v=bits)
    c = synth.make_case(w)
    pairs = _sample_pairs(w, 6, cfg)
    with make_cache(kvq, w, max_ctx=w.T + 64) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        check_state(orc, cache, w, c["K"], c["V"], pairs)
        if cfg == 1:
            assert pairs == [0, 1]
            check_dequant(orc, cache, w, c["K"], c["V"], pairs)
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], pairs)
        cache.check()


def test_long_context_prefill_then_decode_steps(kvq, orc):
    w = synth.WORKLOADS[4]
    steps = w.decode_steps
    c = synth.make_case(w)
    st = synth.make_decode_steps(w, steps, outliers=c["outliers"])
    K = np.concatenate([c["K"]] + [s["k"] for s in st], axis=2)
    V = np.concatenate([c["V"]] + [s["v"] for s in st], axis=2)
    pairs = [0, 5]
    check_at = {0, 30, 31, 32, steps - 1}
    with make_cache(kvq, w, max_ctx=w.T + steps) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        T = w.T
        for i, s in enumerate(st):
            cache.append(dev(s["k"]), dev(s["v"]))
            T += 1
            q = s["q"]
            out = cache.decode(dev(q), softmax_scale=w.scale)
            if i in check_at:
                torch.cuda.synchronize()
                check_state(orc, cache, w, K[:, :, :T], V[:, :, :T], pairs)
                check_decode(orc, cache, w, K[:, :, :T], V[:, :, :T], q, pairs)
        del out
        cache.check()


@pytest.mark.parametrize("sw", synth.sweep_workloads(), ids=lambda s: s.name.split("d128-t2048-")[-1])
def test_sweep_reduced_batch(kvq, orc, sw):
    w = sw.with_(batch=2)
    c = synth.make_case(w)
    pairs = list(range(w.n_pairs))
    with make_cache(kvq, w, max_ctx=w.T) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        check_state(orc, cache, w, c["K"], c["V"], pairs)
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], pairs)
        cache.check()


def test_sweep_full_size_main_geometry_sampled(kvq, orc):
    w = synth.WORKLOADS[5]
    c = synth.make_case(w)
    pairs = _sample_pairs(w, 8, 5)
    with make_cache(kvq, w, max_ctx=w.T) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        torch.cuda.synchronize()
        check_state(orc, cache, w, c["K"], c["V"], pairs)
        check_decode(orc, cache, w, c["K"], c["V"], c["q"], pairs)
        cache.check()
