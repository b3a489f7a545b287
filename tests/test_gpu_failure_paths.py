"""Failure paths of the C ABI, with every fault made on the host.

Nothing here faults, traps or hangs the GPU:
  * allocation failure: kvq_debug_fail_allocations makes the library's k-th
    device allocation fail; kvq_create must return KVQ_ERR_OOM, leave no
    handle and free what it had allocated, and the next create must work;
  * the device error word: kvq_debug_set_device_error writes it from the
    host as a kernel whose bounded wait ran out would;
    kvq_check_device_error must report KVQ_ERR_DEVICE_CHECK once, then OK;
  * a bounded wait that runs out: kvq_debug_set_wait_limit(cache, 0) makes
    every main-loop wait of the decode kernels give up at once (the warp
    records the error, drains its own bulk copies with the normal limit and
    leaves); the status comes back through kvq_check_device_error, and the
    next decode with the normal limit is correct again.
"""
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


def _cfg(kvq, **kw):
    base = dict(batch=2, n_q_heads=4, n_kv_heads=4, head_dim=128, max_ctx=512)
    base.update(kw)
    return kvq.make_config(**base)


def test_allocation_failure_returns_oom_and_frees(kvq):
    cfg = _cfg(kvq, keys_pre_rope=True, rope_base=10000.0, n_sink=4)
    # count the allocations of one create: fail the k-th for every k until a
    # create succeeds with the injection still armed
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    k = 0
    while True:
        kvq.kvq_debug_fail_allocations(k, 1)
        try:
            h = kvq.kvq_create(cfg)
        except kvq.KvqError as e:
            assert e.status == kvq.KVQ_ERR_OOM
            k += 1
            assert k < 64
            continue
        kvq.kvq_debug_fail_allocations(0, 0)
        kvq.kvq_destroy(h)
        break
    assert k >= 10   # blocks, 4 tails, 2 sink windows, RoPE table, workspace ...
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    # every failed create freed what it had allocated (allow allocator slack)
    assert free0 - free1 < 64 << 20
    # a create after the failures works normally
    h = kvq.kvq_create(cfg)
    kvq.kvq_destroy(h)


def test_debug_hooks_reject_bad_arguments(kvq):
    for args in [(-1, 1), (0, -1)]:
        with pytest.raises(kvq.KvqError) as ei:
            kvq.kvq_debug_fail_allocations(*args)
        assert ei.value.status == kvq.KVQ_ERR_INVALID_ARG
    with pytest.raises(kvq.KvqError) as ei:
        kvq.kvq_debug_set_device_error(None, 1)
    assert ei.value.status == kvq.KVQ_ERR_INVALID_ARG
    with pytest.raises(kvq.KvqError) as ei:
        kvq.kvq_debug_set_wait_limit(None, 0)
    assert ei.value.status == kvq.KVQ_ERR_INVALID_ARG


def _decode_ok(orc, w, K, V, q, out):
    got = out.cpu().numpy().astype(np.float64)
    R = w.gqa
    g_all, w_all = [], []
    for p in range(w.n_pairs):
        b, h = divmod(p, w.n_kv_heads)
        st = orc.build_pair(K[b, h], V[b, h], w.group, w.bits_k, w.bits_v, w.axis_k, w.axis_v)
        w_all.append(orc.decode_pair(st, q[b, h * R:(h + 1) * R], w.scale))
        g_all.append(got[b, h * R:(h + 1) * R])
    g_all, w_all = np.stack(g_all), np.stack(w_all)
    err = np.abs(g_all - w_all).max()
    rel = np.linalg.norm(g_all - w_all) / np.linalg.norm(w_all)
    return err <= ATOL and rel <= RTOL_L2, (err, rel)


def test_device_error_word_is_reported_and_cleared(kvq, orc):
    w = synth.WORKLOADS[2].with_(batch=2, n_kv_heads=4, n_q_heads=4, T=3 * 32 + 5)
    c = synth.make_case(w, seed=3)
    with kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                     head_dim=w.head_dim, max_ctx=256) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        cache.check()                                   # clean
        kvq.kvq_debug_set_device_error(cache.handle, 1)
        assert kvq.kvq_check_device_error(cache.handle) == kvq.KVQ_ERR_DEVICE_CHECK
        assert kvq.kvq_check_device_error(cache.handle) == kvq.KVQ_OK   # cleared
        out = cache.decode(dev(c["q"]), softmax_scale=w.scale)
        torch.cuda.synchronize()
        ok, detail = _decode_ok(orc, w, c["K"], c["V"], c["q"], out)
        assert ok, detail
        cache.check()


# name, G, axis_k, axis_v, T: the tensor-core kernel with its in-place merge,
# the CUDA-core kernel with the two-level merge kernel, and a long context
# whose pairs go to the two-level merge in the tensor-core geometry
WAIT_CASES = [
    ("tensor-core", 32, 0, 1, 7 * 32 + 9, 2),
    ("cuda-core", 128, 1, 0, 3 * 128 + 5, 2),
    ("tensor-core-long", 32, 0, 1, 20000, 1),
]


@pytest.mark.parametrize("case", WAIT_CASES, ids=[c[0] for c in WAIT_CASES])
def test_wait_that_runs_out_is_reported_then_decode_recovers(kvq, orc, case):
    name, G, ak, av, T, batch = case
    w = synth.WORKLOADS[2].with_(batch=batch, n_kv_heads=2, n_q_heads=2, T=T, group=G,
                                 axis_k=ak, axis_v=av)
    c = synth.make_case(w, seed=4)
    with kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                     head_dim=w.head_dim, max_ctx=T + 64, group=G, axis_k=ak,
                     axis_v=av) as cache:
        cache.prefill(dev(c["K"]), dev(c["V"]))
        q = dev(c["q"])
        cache.check()
        kvq.kvq_debug_set_wait_limit(cache.handle, 0)   # every wait gives up at once
        out = torch.full((w.batch, w.n_q_heads, w.head_dim), 7.0, device="cuda")
        cache.decode(q, out, w.scale)
        assert kvq.kvq_check_device_error(cache.handle) == kvq.KVQ_ERR_DEVICE_CHECK
        kvq.kvq_debug_set_wait_limit(cache.handle, -1)  # the normal limit again
        for _ in range(2):
            out = cache.decode(q, softmax_scale=w.scale)
            torch.cuda.synchronize()
            ok, detail = _decode_ok(orc, w, c["K"], c["V"], c["q"], out)
            assert ok, detail
            assert kvq.kvq_check_device_error(cache.handle) == kvq.KVQ_OK
