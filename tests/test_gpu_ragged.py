"""Ragged batches (batch rows of different lengths) on the GPU, through the C
ABI, against the CPU oracle: every row is checked as its own sequence
(oracle.build_pair on that row's tokens).  Bars as in test_gpu_parity."""
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


def workload(D, R, bk, bv, ak, av, G, rope, T, batch, hkv=2):
    return synth.Workload("ragged", batch, hkv * R, hkv, D, T, bk, bv, G, ak, av, rope,
                          outlier_scales=(20.0, 100.0), n_outliers=2, config_id=9)


def make_cache(kvq, w, max_ctx, n_sink=0, residual=0, fp8=False):
    return kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_ctx=max_ctx, bits_k=w.bits_k, bits_v=w.bits_v,
                       group=w.group, axis_k=w.axis_k, axis_v=w.axis_v,
                       keys_pre_rope=w.keys_pre_rope, rope_base=w.rope_base,
                       n_sink=n_sink, residual=residual, fp8=fp8)


class Rows:
    """Per-row token arrays and the matching oracle states."""

    def __init__(self, orc, w, n_sink, residual, fp8):
        self.orc, self.w = orc, w
        self.kw = dict(n_sink=n_sink, residual=residual, fp8=fp8)

    def state(self, K, V, b, h, L):
        w = self.w
        return self.orc.build_pair(K[b, h, :L], V[b, h, :L], w.group, w.bits_k, w.bits_v,
                                   w.axis_k, w.axis_v, **self.kw)


def check_rows(orc, cache, w, K, V, lengths, q, n_sink=0, residual=0, fp8=False, out=None):
    """K, V: fp16 [B][Hkv][T_max][D]; row b holds lengths[b] tokens."""
    rows = Rows(orc, w, n_sink, residual, fp8)
    blocks = cache.block_bytes_view()
    sv = cache.sink_views()
    if out is None:
        out = cache.decode(dev(q), softmax_scale=w.scale)
    torch.cuda.synchronize()
    out = out.cpu().numpy().astype(np.float64)
    R, hkv = w.gqa, w.n_kv_heads
    got, want = [], []
    for b, L in enumerate(lengths):
        Ts, Tq, Tt = orc.window_lengths(L, w.group, n_sink, residual)
        assert cache.row_state(b)[:3] == (Ts, Tq, Tt), (b, L)
        kt, vt = cache.row_tail_views(b)
        for h in range(hkv):
            p = b * hkv + h
            st = rows.state(K, V, b, h, L)
            assert np.array_equal(blocks[p, : Tq // w.group].cpu().numpy(), orc.pack_pair(st)), (b, h)
            assert np.array_equal(kt[h, :Tt].cpu().numpy().view(np.uint16), st["ktail"].view(np.uint16))
            assert np.array_equal(vt[h, :Tt].cpu().numpy().view(np.uint16), st["vtail"].view(np.uint16))
            if sv is not None:
                assert np.array_equal(sv[0][p, :Ts].cpu().numpy().view(np.uint16), st["ksink"].view(np.uint16))
            want.append(orc.decode_pair(st, q[b, h * R:(h + 1) * R], w.scale, w.keys_pre_rope,
                                        w.rope_base))
            got.append(out[b, h * R:(h + 1) * R])
    got, want = np.stack(got), np.stack(want)
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert err <= ATOL, f"max abs {err:.3e}"
    assert rel <= RTOL_L2, f"rel L2 {rel:.3e}"


# name, D, R, bk, bv, ak, av, G, rope, lengths, n_sink, residual, fp8
CASES = [
    ("mma-2/2", 128, 1, 2, 2, 0, 1, 32, False, [1, 31, 32, 100, 257], 0, 0, False),
    ("mma-4/4-r4-rope", 128, 4, 4, 4, 0, 1, 32, True, [65, 3, 200], 0, 0, False),
    ("mma-2/2-d64-r2-windows", 64, 2, 2, 2, 0, 1, 32, False, [2, 40, 150, 300], 4, 32, False),
    ("mma-fp8-rope-windows", 128, 2, 8, 8, 0, 1, 32, True, [10, 170, 90], 3, 40, True),
    ("gen-g128-rope", 128, 1, 2, 2, 0, 1, 128, True, [129, 500, 7, 256], 0, 0, False),
    ("gen-tok/tok-windows", 128, 4, 4, 2, 1, 1, 32, False, [33, 1, 64, 95], 2, 32, False),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ragged_prefill_decode(kvq, orc, case):
    name, D, R, bk, bv, ak, av, G, rope, lengths, n_sink, residual, fp8 = case
    Tm = max(lengths)
    w = workload(D, R, bk, bv, ak, av, G, rope, Tm, batch=len(lengths))
    c = synth.make_case(w, seed=zlib.crc32(name.encode()) % 10000)
    with make_cache(kvq, w, Tm + 64, n_sink, residual, fp8) as cache:
        cache.prefill_ragged(dev(c["K"]), dev(c["V"]), lengths)
        torch.cuda.synchronize()
        assert cache.buffers().ragged == 1
        check_rows(orc, cache, w, c["K"], c["V"], lengths, c["q"], n_sink, residual, fp8)
        cache.check()


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4]], ids=["mma", "mma-windows", "gen-g128"])
def test_ragged_appends(kvq, orc, case):
    """Uniform appends and per-row appends (some rows idle) on a ragged
    cache: every row's state and decode after every call."""
    name, D, R, bk, bv, ak, av, G, rope, lengths, n_sink, residual, fp8 = case
    steps = [("all", 1), ("all", 1), ("rows", [3, 0, 31, 1, 2][:len(lengths)]), ("all", 30),
             ("rows", [0, 64, 1, 0, 40][:len(lengths)]), ("all", 1), ("all", 33)]
    extra = sum(n if kind == "all" else max(n) for kind, n in steps)
    Tm = max(lengths) + extra
    w = workload(D, R, bk, bv, ak, av, G, rope, Tm, batch=len(lengths))
    c = synth.make_case(w, seed=55)
    K, V = c["K"], c["V"]
    cur = list(lengths)
    # row b's tokens are K[b, :, :cur[b]]: appends take the next tokens of each row
    with make_cache(kvq, w, Tm, n_sink, residual, fp8) as cache:
        Tmax = max(cur)
        kin = np.zeros((w.batch, w.n_kv_heads, Tmax, D), np.float16)
        vin = np.zeros_like(kin)
        for b, L in enumerate(cur):
            kin[b, :, :L], vin[b, :, :L] = K[b, :, :L], V[b, :, :L]
        cache.prefill_ragged(dev(kin), dev(vin), cur)
        for kind, n in steps:
            ns = [n] * w.batch if kind == "all" else list(n)
            m = max(ns)
            kn = np.zeros((w.batch, w.n_kv_heads, m, D), np.float16)
            vn = np.zeros_like(kn)
            for b in range(w.batch):
                kn[b, :, :ns[b]] = K[b, :, cur[b]:cur[b] + ns[b]]
                vn[b, :, :ns[b]] = V[b, :, cur[b]:cur[b] + ns[b]]
            if kind == "all":
                cache.append(dev(kn), dev(vn))
            else:
                cache.append_ragged(dev(kn), dev(vn), ns)
            cur = [x + y for x, y in zip(cur, ns)]
            torch.cuda.synchronize()
            check_rows(orc, cache, w, K, V, cur, c["q"], n_sink, residual, fp8)
        cache.check()


def test_ragged_append_decode_fused(kvq, orc):
    """One decode step per call on a ragged cache: a single launch while no
    row flushes, bit-identical to append + decode on a second cache."""
    name, D, R, bk, bv, ak, av, G, rope, lengths, n_sink, residual, fp8 = CASES[0]
    n_steps = 40
    Tm = max(lengths) + n_steps
    w = workload(D, R, bk, bv, ak, av, G, rope, Tm, batch=len(lengths))
    c = synth.make_case(w, seed=56)
    K, V = c["K"], c["V"]
    q = dev(c["q"])
    cur = list(lengths)

    def prefill(cache):
        kin = np.zeros((w.batch, w.n_kv_heads, max(cur), D), np.float16)
        vin = np.zeros_like(kin)
        for b, L in enumerate(cur):
            kin[b, :, :L], vin[b, :, :L] = K[b, :, :L], V[b, :, :L]
        cache.prefill_ragged(dev(kin), dev(vin), cur)

    with make_cache(kvq, w, Tm) as fused, make_cache(kvq, w, Tm) as split:
        prefill(fused)
        prefill(split)
        for i in range(n_steps):
            kn = np.stack([K[b, :, cur[b]:cur[b] + 1] for b in range(w.batch)])
            vn = np.stack([V[b, :, cur[b]:cur[b] + 1] for b in range(w.batch)])
            will_fuse = all(orc.window_lengths(L, G)[2] + 1 < G for L in cur)
            n0 = kvq.kvq_launch_count()
            a = fused.append_decode(dev(kn), dev(vn), q, softmax_scale=w.scale)
            torch.cuda.synchronize()
            if will_fuse:
                assert kvq.kvq_launch_count() - n0 == 1
            split.append(dev(kn), dev(vn))
            b_ = split.decode(q, softmax_scale=w.scale)
            torch.cuda.synchronize()
            assert torch.equal(a, b_)
            cur = [L + 1 for L in cur]
            if i % 8 == 7 or i == n_steps - 1:
                check_rows(orc, fused, w, K, V, cur, c["q"], out=a)
        fused.check()
        split.check()


def test_ragged_one_long_row_among_short(kvq, orc):
    """A 20000-token row beside short rows: the long row's pair spreads over
    thousands of warps, so the two-level merge runs with wide chunks."""
    lengths = [20000, 40, 3, 100, 64, 1, 33, 2]
    w = workload(128, 1, 2, 2, 0, 1, 32, False, max(lengths), batch=len(lengths), hkv=1)
    c = synth.make_case(w, seed=57)
    with make_cache(kvq, w, max(lengths) + 32) as cache:
        cache.prefill_ragged(dev(c["K"]), dev(c["V"]), lengths)
        n0 = kvq.kvq_launch_count()
        check_rows(orc, cache, w, c["K"], c["V"], lengths, c["q"])
        assert kvq.kvq_launch_count() - n0 == 2  # decode + two-level merge
        cache.check()


def test_ragged_rules(kvq):
    w = workload(128, 1, 2, 2, 0, 1, 32, False, 64, batch=3)
    c = synth.make_case(w, seed=58)
    K, V = dev(c["K"]), dev(c["V"])
    with make_cache(kvq, w, 80) as cache:
        for lengths, status in (([0, 5, 6], kvq.KVQ_ERR_INVALID_ARG),
                                ([65, 5, 6], kvq.KVQ_ERR_INVALID_ARG)):  # > T_stride
            with pytest.raises(kvq.KvqError) as ei:
                cache.prefill_ragged(K, V, lengths)
            assert ei.value.status == status
        cache.prefill_ragged(K, V, [10, 10, 10])          # equal lengths: a uniform cache
        assert cache.buffers().ragged == 0 and cache.state == (0, 10)
        cache.prefill_ragged(K, V, [10, 64, 1])
        for fn in (lambda: cache.state, lambda: cache.dequantize()):
            with pytest.raises(kvq.KvqError) as ei:
                fn()
            assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
        with pytest.raises(kvq.KvqError) as ei:
            cache.append(K[:, :, :17], V[:, :, :17])        # row 1: 64 + 17 > 80
        assert ei.value.status == kvq.KVQ_ERR_CAPACITY
        assert cache.row_state(1)[:3] == (0, 64, 0)
        cache.check()
    wb = workload(64, 1, 2, 2, 0, 1, 32, False, 8, batch=65, hkv=1)
    cb = synth.make_case(wb, seed=59)
    with make_cache(kvq, wb, 16) as cache:
        with pytest.raises(kvq.KvqError) as ei:
            cache.prefill_ragged(dev(cb["K"]), dev(cb["V"]), [8] * 64 + [7])
        assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
