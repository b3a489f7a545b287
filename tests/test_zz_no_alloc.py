"""The decode entry point that allocates no device memory.

Callers that cannot call cudaMalloc while they decode (a runtime that keeps
all device memory in its own arena, a plugin host that only hands out its
own buffers, a loop where an allocation's device synchronization is not
acceptable) decode a packed cache they own with
kvq_decode_attention_noalloc, whose workspace is a static device array.
This test checks, through the C ABI, that two calls in a row give the same
output as kvq_decode_attention on the same cache and as the CPU oracle's
fp64 attention, within the decode tolerance of the parity tests (both decode
kernels, the FP8 format, with and without an fp16 tail), and that a shape too
large for the static workspace is refused.  It sits in its own file, named to be collected last,
and passes alone in a fresh process as well as after the other tests.
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


def _close(a, b):
    a = a.double()
    b = b.double()
    err = (a - b).abs().max().item()
    rel = ((a - b).norm() / b.norm()).item()
    return err <= ATOL and rel <= RTOL_L2, (err, rel)


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


# name, gqa, bits, G, axis_k, axis_v, fp8, T: the tensor-core kernel (keys per
# channel, values per token, G = 32), its FP8 variant, and the CUDA-core
# kernel with the separate merge kernel (G = 128, both axis assignments);
# T a multiple of G leaves the fp16 tail empty at the first call.
CASES = [
    ("mha-2bit", 1, 2, 32, 0, 1, False, 5 * 32 + 9),
    ("gqa4-4bit", 4, 4, 32, 0, 1, False, 5 * 32 + 9),
    ("mha-2bit-empty-tail", 1, 2, 32, 0, 1, False, 6 * 32),
    ("fp8", 2, 8, 32, 0, 1, True, 4 * 32 + 5),
    ("g128-ktok-vch", 2, 2, 128, 1, 0, False, 3 * 128 + 77),
    ("g128-kch-vtok-empty-tail", 4, 4, 128, 0, 1, False, 2 * 128),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_cache_decode_and_oracle_twice(kvq, orc, case):
    name, gqa, bits, G, ak, av, fp8, T = case
    w = synth.WORKLOADS[2].with_(batch=2, n_kv_heads=4, n_q_heads=4 * gqa, T=T, bits_k=bits,
                                 bits_v=bits, group=G, axis_k=ak, axis_v=av)
    c = synth.make_case(w, seed=11)
    steps = synth.make_decode_steps(w, 2, seed=12, outliers=c["outliers"])
    K, V = c["K"], c["V"]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    with kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                     head_dim=w.head_dim, max_ctx=w.T + 64, bits_k=w.bits_k, bits_v=w.bits_v,
                     group=w.group, axis_k=ak, axis_v=av, fp8=fp8) as cache:
        cache.prefill(dev(K), dev(V))
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        for i, s in enumerate(steps):       # two calls in a row
            if i > 0:                       # the second one after a new token
                cache.append(dev(s["k"]), dev(s["v"]))
                K = np.concatenate([K, s["k"]], axis=2)
                V = np.concatenate([V, s["v"]], axis=2)
            q = dev(s["q"])
            want = cache.decode(q, softmax_scale=w.scale)
            b = cache.buffers()
            got = torch.full_like(want, float("nan"))
            kvq.kvq_decode_attention_noalloc(cache.cfg, b.blocks, b.k_tail, b.v_tail, b.T_q,
                                             b.T_tail, q, got, w.scale, err)
            torch.cuda.synchronize()
            ok, detail = _close(got, want)
            assert ok, detail
            assert err.item() == 0
            # against the oracle's fp64 attention over the same dequantized cache
            out = got.cpu().numpy().astype(np.float64)
            R = w.gqa
            g_all, w_all = [], []
            for p in range(w.n_pairs):
                bb, h = divmod(p, w.n_kv_heads)
                st = orc.build_pair(K[bb, h], V[bb, h], G, bits, bits, ak, av, fp8=fp8)
                w_all.append(orc.decode_pair(st, s["q"][bb, h * R:(h + 1) * R], w.scale))
                g_all.append(out[bb, h * R:(h + 1) * R])
            ok, detail = _close(torch.from_numpy(np.stack(g_all)), torch.from_numpy(np.stack(w_all)))
            assert ok, detail
        cache.check()


def test_noalloc_rejects_shapes_beyond_its_workspace(kvq):
    # 32768 pairs x 8 query heads x 128 channels of partials exceed 8 MiB.
    cfg = kvq.make_config(batch=512, n_q_heads=512, n_kv_heads=64, head_dim=128, max_ctx=64)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as ei:
        kvq.kvq_decode_attention_noalloc(cfg, dummy, dummy, dummy, 32, 1, dummy, dummy, 0.1)
    assert ei.value.status == kvq.KVQ_ERR_CAPACITY
