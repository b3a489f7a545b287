"""Host-side logic of the multi-rank bench path, run as two gloo ranks on
CPU: every rank is an independent replica (its own seeded batch, no data-path
collective); the job's value is the sum of the ranks' bytes over the slowest
rank's time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    assert bench.dist_env() == (ws, rank, rank)
    t = bench.reduce_max(10.0 * (rank + 1), ws, device="cpu")
    b = bench.reduce_sum(1000.0 + rank, ws, device="cpu")
    seeds = [bench.rank_seed(2, rank, layer) for layer in range(8)]
    from bit_kv_cache_11_gb300 import synth
    w = synth.WORKLOADS[1]
    k0 = synth.make_case(w, seed=seeds[0])["K"]
    obj = [None] * ws
    dist.all_gather_object(obj, (seeds, float(k0.astype("float64").sum())))
    dist.barrier()
    dist.destroy_process_group()
    out[rank] = (t, b, obj)


def test_two_rank_replicas_gloo():
    ws = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(ws, _free_port(), out), nprocs=ws, join=True)
    for rank in range(ws):
        t, b, obj = out[rank]
        assert t == 20.0                      # slowest rank's time
        assert b == 2001.0                    # all ranks' bytes
        (s0, k0), (s1, k1) = obj
        assert not set(s0) & set(s1)          # independent replicas
        assert k0 != k1
