"""Dense-and-sparse outlier isolation on the GPU, through the C ABI, against
the CPU oracle.

The format (oracle, pinned in test_oracle_outliers): in every G-token block
and side, the n_outliers elements of largest magnitude (ties: lower
position) are kept in fp16 with their positions in a section after the
side's metadata; every group takes min/max over its other elements; kept
positions hold code 0 and dequantize to their kept value.  Bars: packed
blocks (codes, metadata, outlier sections) and fp16 tails bit-exact;
dequantized values bit-exact; decode within 2e-3 max abs and 1e-3 relative
L2 of the oracle's fp64 attention over the same dequantized values.

Inputs: the seeded workload recipe plus sparse massive activations (a few
per mille of the key and value elements scaled up), the kind of extreme
values the isolation is for ("Keys: The Outliers Live in Fixed Channels").
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


def massive(case, seed, frac=0.003, scale=8.0):
    """The case with a fraction of key and value elements scaled by `scale`
    (and a few equal magnitudes, so that selection ties occur)."""
    rng = np.random.default_rng(seed)
    K = case["K"].astype(np.float32)
    V = case["V"].astype(np.float32)
    K[rng.random(K.shape) < frac] *= scale
    V[rng.random(V.shape) < frac] *= scale
    tie = rng.random(K.shape) < frac / 4
    K[tie] = np.float32(-21.0)
    return dict(case, K=K.astype(np.float16), V=V.astype(np.float16))


def make_cache(kvq, w, max_ctx, n_out):
    return kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_ctx=max_ctx, bits_k=w.bits_k, bits_v=w.bits_v,
                       group=w.group, n_outliers=n_out)


def check_pairs(orc, cache, w, K, V, q, n_out, pairs, dequant=True):
    T = K.shape[2]
    tq, tt = cache.state
    assert tq == (T // 32) * 32 and tt == T - tq
    b = cache.buffers()
    assert b.n_outliers == n_out
    assert b.block_bytes == orc.block_bytes(w.head_dim, 32, w.bits_k, w.bits_v, n_out)
    blocks = cache.block_bytes_view()
    kt, vt = cache.tail_views()
    if dequant and tq > 0:
        kh, vh = cache.dequantize()
    out = cache.decode(dev(q), softmax_scale=w.scale)
    torch.cuda.synchronize()
    out = out.cpu().numpy().astype(np.float64)
    R = w.gqa
    got, want = [], []
    for p in pairs:
        bb, h = divmod(p, w.n_kv_heads)
        st = orc.build_pair(K[bb, h], V[bb, h], 32, w.bits_k, w.bits_v, 0, 1, n_outliers=n_out)
        assert np.array_equal(blocks[p, :tq // 32].cpu().numpy(), orc.pack_pair(st)), f"pair {p}"
        assert np.array_equal(kt[p, :tt].cpu().numpy().view(np.uint16), st["ktail"].view(np.uint16))
        assert np.array_equal(vt[p, :tt].cpu().numpy().view(np.uint16), st["vtail"].view(np.uint16))
        if dequant and tq > 0:
            okh, ovh = orc.dequantize_pair(st)
            assert np.array_equal(kh[bb, h].cpu().numpy().view(np.uint32), okh.view(np.uint32))
            assert np.array_equal(vh[bb, h].cpu().numpy().view(np.uint32), ovh.view(np.uint32))
        want.append(orc.decode_pair(st, q[bb, h * R:(h + 1) * R], w.scale))
        got.append(out[bb, h * R:(h + 1) * R])
    got, want = np.stack(got), np.stack(want)
    err = np.abs(got - want).max()
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert err <= ATOL, f"max abs {err:.3e}"
    assert rel <= RTOL_L2, f"rel L2 {rel:.3e}"


# name, D, R, bk, bv, n, T
CASES = [
    ("d128-r1-2/2-n32", 128, 1, 2, 2, 32, 5 * 32 + 7),
    ("d128-r4-2/4-n4", 128, 4, 2, 4, 4, 4 * 32 + 31),
    ("d64-r2-4/2-n64", 64, 2, 4, 2, 64, 3 * 32),
    ("d128-r8-4/4-n16", 128, 8, 4, 4, 16, 2 * 32 + 1),
    ("d64-r1-2/2-n8-one-block", 64, 1, 2, 2, 8, 32),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_blocks_dequant_decode(kvq, orc, case):
    name, D, R, bk, bv, n, T = case
    w = synth.Workload("outl", 2, 3 * R, 3, D, T, bk, bv, 32, 0, 1, False,
                       outlier_scales=(20.0, 100.0), n_outliers=2, config_id=9)
    c = massive(synth.make_case(w, seed=zlib.crc32(name.encode()) % 10000), 7)
    with make_cache(kvq, w, T + 64, n) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        check_pairs(orc, cache, w, c["K"], c["V"], c["q"], n, range(w.n_pairs))
        cache.check()


def test_append_flush_and_fused_steps(kvq, orc):
    """Appends across flushes, then kvq_append_decode steps (one launch while
    no group completes), each state against the oracle; the fused steps equal
    append + decode on a second cache bit for bit."""
    w = synth.Workload("outl", 2, 4, 2, 128, 200, 2, 2, 32, 0, 1, False, config_id=9)
    c = massive(synth.make_case(w, seed=3), 8)
    K, V, n = c["K"], c["V"], 16
    with make_cache(kvq, w, 256, n) as a, make_cache(kvq, w, 256, n) as b:
        a.prefill(dev(K[:, :, :20]), dev(V[:, :, :20]))
        b.prefill(dev(K[:, :, :20]), dev(V[:, :, :20]))
        T = 20
        for step in [1, 11, 33, 1, 40]:
            a.append(dev(K[:, :, T:T + step]), dev(V[:, :, T:T + step]))
            b.append(dev(K[:, :, T:T + step]), dev(V[:, :, T:T + step]))
            T += step
            check_pairs(orc, a, w, K[:, :, :T], V[:, :, :T], c["q"], n, range(w.n_pairs),
                        dequant=False)
        q = dev(c["q"])
        while T < 200:
            k1, v1 = dev(K[:, :, T:T + 1]), dev(V[:, :, T:T + 1])
            o1 = a.append_decode(k1, v1, q, softmax_scale=w.scale)
            b.append(k1, v1)
            o2 = b.decode(q, softmax_scale=w.scale)
            T += 1
            torch.cuda.synchronize()
            assert torch.equal(o1, o2)
        check_pairs(orc, a, w, K[:, :, :T], V[:, :, :T], c["q"], n, range(w.n_pairs))
        a.check()
        b.check()


def test_full_size_layer_sampled(kvq, orc):
    """The Llama-2-7B-shaped layer with 32 outliers kept per block side, in
    the bench's launch configuration (sampled pairs)."""
    w = synth.WORKLOADS[2]
    c = massive(synth.make_case(w), 9)
    rng = np.random.default_rng(2)
    pairs = sorted({0, w.n_pairs - 1} | set(rng.choice(w.n_pairs, 6, replace=False).tolist()))
    with make_cache(kvq, w, w.T + 64, 32) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        check_pairs(orc, cache, w, c["K"], c["V"], c["q"], 32, pairs, dequant=False)
        cache.check()


def test_outlier_configs_checked(kvq):
    base = dict(batch=2, n_q_heads=4, n_kv_heads=4, head_dim=128, max_ctx=256)
    cases = [
        (dict(n_outliers=16), kvq.KVQ_OK),
        (dict(n_outliers=64, bits_k=4, bits_v=2), kvq.KVQ_OK),
        (dict(n_outliers=6), kvq.KVQ_ERR_INVALID_ARG),              # not a multiple of 4
        (dict(n_outliers=68), kvq.KVQ_ERR_INVALID_ARG),
        (dict(n_outliers=-4), kvq.KVQ_ERR_INVALID_ARG),
        (dict(n_outliers=16, bits_k=8, bits_v=8), kvq.KVQ_ERR_UNSUPPORTED),
        (dict(n_outliers=16, group=128), kvq.KVQ_ERR_UNSUPPORTED),
        (dict(n_outliers=16, axis_k=1, axis_v=0), kvq.KVQ_ERR_UNSUPPORTED),
        (dict(n_outliers=16, keys_pre_rope=True, rope_base=10000.0), kvq.KVQ_ERR_UNSUPPORTED),
    ]
    for over, status in cases:
        kw = dict(base)
        kw.update(over)
        assert kvq.kvq_config_check(kvq.make_config(**kw)) == status, over
    cfg = kvq.make_config(**dict(base, n_outliers=16))
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as ei:
        kvq.kvq_decode_attention_noalloc(cfg, dummy, dummy, dummy, 32, 1, dummy, dummy, 0.1)
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
