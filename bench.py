"""Decode-step benchmark of the low-bit KV cache on one GB300 (or N, one
process per GPU, each rank an independent replica).

Headline workload: a Llama-2-7B-shaped attention layer at decode time —
batch 8, 32 heads (MHA), head_dim 128, context 4096 + 17-token fp16 tail,
2-bit keys (per channel) and values (per token), group 32 — synthetic seeded
inputs.  A step runs the hot path once over a stack of L such layers (default
8, each with its own cache, 825 MB in total, so every layer is read cold from
HBM): for each layer, append the step's new token and run split-K decode
attention — one kvq_append_decode call, a single launch unless the token
completes a group of 32 (then the flush kernel runs before the decode).

value = algorithmic decode bytes of all layers and ranks / step time (GB/s):
packed codes + fp16 metadata + fp16 tail + q in + out, per decode call.

The same JSON line carries the decode kernel's roofline (back-to-back launches
timed by region, median / min / max per launch), the end-to-end rate through
the C ABI from pinned host memory, the CPU oracle's rate on one core and on
all cores, and the other workloads: the quantize prefill, the fp16 windows,
the FP8 cache, a ragged batch, the Llama-2-13B-shaped layer with keys stored
before RoPE (2 and 4 bits), the long-context request (prefill, then 64
append + decode steps with their flushes) and the geometry / bit-width sweep
(GB/s and quantization error per combination).

`python bench.py --profile-case --config N` runs one workload's prefill and a
few decode (or append, or prefill) calls alone: the small program that
profiler captures wrap.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_11_gb300 import synth  # noqa: E402

METRIC = "quantized decode-attention HBM GB/s"


# ---------------------------------------------------------------- byte counts

def decode_bytes(w, T_q, T_t):
    """Algorithmic bytes of one decode call (T_t counts every fp16 row: tail
    and sink window)."""
    P = w.batch * w.n_kv_heads
    codes = P * T_q * w.head_dim * (w.bits_k + w.bits_v) // 8
    meta = 2 * P * (T_q * w.head_dim // w.group) * 4
    tail = P * T_t * w.head_dim * 2 * 2
    qo = w.batch * w.n_q_heads * w.head_dim * (2 + 4)
    return codes + meta + tail + qo


def quantize_bytes_per_token(w):
    Hkv, D = w.n_kv_heads, w.head_dim
    return 2 * Hkv * D * 2 + Hkv * D * (w.bits_k + w.bits_v) // 8 + 2 * Hkv * D // w.group * 4


def append_one(row, n_sink, residual, group):
    """Row lengths [T_sink, T_q, T_tail] after one appended token: it fills
    the sink window first, then the tail; a group of `group` tokens is
    quantized once it leaves `residual` newer tail tokens (the cache's append
    rule, used to account the bytes of steps timed without host queries)."""
    ts, tq, tt = row
    if ts < n_sink:
        return [ts + 1, tq, tt]
    tt += 1
    if tt >= residual + group:
        tq += group
        tt -= group
    return [ts, tq, tt]


# ---------------------------------------------------------------- environment

def csrc_hash() -> str:
    """Hash of the CUDA sources and the C ABI header (identifies the kernels)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "bit_kv_cache_11_gb300", "csrc", "*.cu*")))
    for f in files + [os.path.join(ROOT, "include", "kvq.h")]:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernels changed since that capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        return rec["dram_bytes_per_launch"] if rec["csrc_sha"] == csrc_hash() else None
    except Exception:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                mhz.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _reduce(x: float, ws: int, op: str, device: str) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def reduce_max(x: float, ws: int, device: str = "cuda") -> float:
    """Slowest rank's value (timings)."""
    return _reduce(x, ws, "max", device)


def reduce_sum(x: float, ws: int, device: str = "cuda") -> float:
    """Whole-job total (bytes processed by all ranks)."""
    return _reduce(x, ws, "sum", device)


def rank_seed(config_id: int, rank: int, layer: int) -> int:
    """Each rank is an independent replica with its own batch: distinct seeds
    per (rank, layer)."""
    return 1000 * config_id + 100 * rank + layer


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def spread(xs):
    """Median, min and max of a list of per-launch times (ms)."""
    return {"median_ms": statistics.median(xs), "min_ms": min(xs), "max_ms": max(xs),
            "samples": len(xs)}


def tiled_case(w, reps: int, seed: int | None = None) -> dict:
    """The workload's synthetic case drawn for batch / reps rows and repeated
    reps times along the batch (same recipe and shape; fewer random draws)."""
    sub = w.with_(batch=max(1, w.batch // reps))
    c = synth.make_case(sub, seed=seed)
    k = w.batch // sub.batch
    return dict(K=np.tile(c["K"], (k, 1, 1, 1)), V=np.tile(c["V"], (k, 1, 1, 1)),
                q=np.tile(c["q"], (k, 1, 1)), outliers=c["outliers"])


def make_cache(kvq, w, max_ctx, **kw):
    return kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                       head_dim=w.head_dim, max_ctx=max_ctx, bits_k=w.bits_k, bits_v=w.bits_v,
                       group=w.group, axis_k=w.axis_k, axis_v=w.axis_v,
                       keys_pre_rope=w.keys_pre_rope, rope_base=w.rope_base, **kw)


def region_times(torch, stream, body, n_regions, n_warm=3):
    """Runs body() n_warm + n_regions times back to back; returns the CUDA-event
    time (ms) of each of the last n_regions runs."""
    for _ in range(n_warm):
        body()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_regions)]
    for a, b in ev:
        a.record(stream)
        body()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def flushed_launch_times(torch, stream, fn, n, flush):
    """Per-launch CUDA-event times of fn() with L2 flushed (a buffer larger
    than L2 rewritten) before each launch, outside the event pair."""
    out = []
    for i in range(n):
        flush.fill_(i & 0xff)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b))
    return out


# ---------------------------------------------------------------- CPU oracle arm

def oracle_decode_sample(w, case, pairs, T, threads=1):
    """Oracle decode (dequantize + fp64 attention) of the given pairs on
    `threads` host threads (the oracle's C calls release the interpreter
    lock); returns (seconds, algorithmic bytes of those pairs)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    states = []
    for p in pairs:
        b, h = divmod(p, w.n_kv_heads)
        states.append((b, h, oracle.build_pair(case["K"][b, h, :T], case["V"][b, h, :T], w.group,
                                               w.bits_k, w.bits_v, w.axis_k, w.axis_v)))
    R = w.gqa

    def one(item):
        b, h, st = item
        oracle.decode_pair(st, case["q"][b, h * R:(h + 1) * R], w.scale, w.keys_pre_rope,
                           w.rope_base)

    t0 = time.perf_counter()
    if threads <= 1:
        for item in states:
            one(item)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, states))
    dt = time.perf_counter() - t0
    T_q = (T // w.group) * w.group
    one_pair = w.with_(batch=1, n_kv_heads=1, n_q_heads=R)
    return dt, len(pairs) * decode_bytes(one_pair, T_q, T - T_q)


def oracle_quantize_sample(w4, tokens):
    import oracle
    rng = np.random.default_rng(4242)
    K = rng.standard_normal((tokens, w4.head_dim), dtype=np.float32).astype(np.float16)
    V = rng.standard_normal((tokens, w4.head_dim), dtype=np.float32).astype(np.float16)
    t0 = time.perf_counter()
    oracle.pack_pair(oracle.build_pair(K, V, w4.group, w4.bits_k, w4.bits_v, w4.axis_k, w4.axis_v))
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baselines(w, case):
    """The oracle as it stands, timed on one layer of the headline workload
    (all 256 pairs: dequantize + fp64 attention), on one core and on every
    core this process may use."""
    pairs = list(range(w.n_pairs))
    out = []
    for threads in (1, host_cores()):
        dt, b = oracle_decode_sample(w, case, pairs, w.T, threads=threads)
        out.append({"value": b / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                    "sample": f"one layer: all {len(pairs)} (batch, kv-head) pairs, dequantize + "
                              f"fp64 attention, {threads} thread(s)", "seconds": dt})
    return out


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    case = synth.make_case(w)
    pairs = list(range(16))
    for _ in range(args.warmup):
        oracle_decode_sample(w, case, pairs[:1], w.T)
    times, nbytes = [], 0
    for _ in range(args.steps):
        dt, b = oracle_decode_sample(w, case, pairs, w.T)
        times.append(dt)
        nbytes = b
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": f"{len(pairs)} of {w.n_pairs} (batch, kv-head) pairs per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(pairs)} pairs of {w.n_pairs} per step, dequantize + fp64 attention"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU legs

def decode_roofline(torch, kvq, w, caches, qs, outs, stream, n_regions=64):
    """The decode kernel alone: regions of one decode per layer cache, back to
    back (each read is cold in L2: the other layers' caches evict it)."""
    def body():
        for c, q, o in zip(caches, qs, outs):
            c.decode(q, o, w.scale)
    reg = region_times(torch, stream, body, n_regions)
    per = [r / len(caches) for r in reg]
    tq, tt = caches[0].state
    nb = decode_bytes(w, tq, tt)
    sp = spread(per)
    return nb, sp


def variant_leg(torch, kvq, w, dev, stream, n_layers, steps, n_sink=0, residual=0, fp8=False,
                lengths=None, n_outliers=0):
    """The decode step on a variant of the cache: fp16 windows (the first
    n_sink tokens and `residual` recent tokens kept in fp16), the FP8 (E4M3)
    format (w with 8-bit sides), a ragged batch (row b holds lengths[b]
    tokens), or dense-and-sparse blocks (n_outliers kept per block side).
    Algorithmic bytes count sink rows like tail rows, per row, and the
    outlier sections (8 n bytes per block).  The decode kernel is timed as
    regions of one kvq_decode_attention per layer."""
    caches, qs = [], []
    for layer in range(n_layers):
        seed = rank_seed(w.config_id, 0, layer) + 7
        case = synth.make_case(w, seed=seed)
        c = make_cache(kvq, w, w.T + 32, n_sink=n_sink, residual=residual, fp8=fp8,
                       n_outliers=n_outliers)
        if lengths is None:
            c.prefill(torch.from_numpy(case["K"]).to(dev), torch.from_numpy(case["V"]).to(dev))
        else:
            c.prefill_ragged(torch.from_numpy(case["K"]).to(dev), torch.from_numpy(case["V"]).to(dev),
                             lengths)
        caches.append(c)
        qs.append(torch.from_numpy(case["q"]).to(dev))
    outs = [torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev)
            for _ in range(n_layers)]

    def body():
        for c, q, o in zip(caches, qs, outs):
            c.decode(q, o, w.scale)
    per = [r / n_layers for r in region_times(torch, stream, body, steps)]
    nb = 0
    for b in range(w.batch):
        ts, tq, tt, _ = caches[0].row_state(b)
        nb += decode_bytes(w.with_(batch=1), tq, tt + ts)
        nb += w.n_kv_heads * (tq // w.group) * 8 * n_outliers
    for c in caches:
        c.check()
        c.close()
    peak, src = load_peaks()
    sp = spread(per)
    gbs = nb / (sp["median_ms"] * 1e-3) / 1e9
    if fp8:
        name = w.name.replace("-2bit", "-fp8")
    elif lengths is not None:
        name = w.name.replace("-t4113", f"-ragged-t{min(lengths)}..{max(lengths)}")
    elif n_outliers:
        name = f"{w.name}-outliers{n_outliers}"
    else:
        name = f"{w.name}-sink{n_sink}-res{residual}"
    return {"workload": name, "n_sink": n_sink, "residual": residual, "fp8": fp8,
            "lengths": lengths, "n_outliers": n_outliers, "GB/s": gbs, "frac": gbs / peak, "peak_source": f"hbm_gbs of {src}",
            "bytes_per_launch": nb, **sp}


def rope_leg(torch, kvq, dev, stream, bits_list=(2, 4), n_caches=2, n_launches=10):
    """Llama-2-13B-shaped layer (B16, H40, D128, T8192), keys stored before
    RoPE and rotated after dequantization inside the decode: per bit width,
    decode launches alternating over n_caches caches (each 504-839 MB, cold in
    L2), one event pair per launch."""
    w3 = synth.WORKLOADS[3]
    case = tiled_case(w3, 8)
    K = torch.from_numpy(case["K"]).to(dev)
    V = torch.from_numpy(case["V"]).to(dev)
    q = torch.from_numpy(case["q"]).to(dev)
    peak, src = load_peaks()
    out = []
    for bits in bits_list:
        w = w3.with_(bits_k=bits, bits_v=bits)
        caches = [make_cache(kvq, w, w.T) for _ in range(n_caches)]
        for c in caches:
            c.prefill(K, V)
        o = torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev)
        k = [0]

        def body():
            caches[k[0] % n_caches].decode(q, o, w.scale)
            k[0] += 1
        per = region_times(torch, stream, body, n_launches, n_warm=2)
        nb = decode_bytes(w, w.T, 0)
        sp = spread(per)
        gbs = nb / (sp["median_ms"] * 1e-3) / 1e9
        for c in caches:
            c.check()
            c.close()
        out.append({"workload": w.name.replace("prerope", f"prerope-{bits}bit"), "bits": bits,
                    "GB/s": gbs, "frac": gbs / peak, "peak_source": f"hbm_gbs of {src}",
                    "bytes_per_launch": nb, **sp})
    del K, V
    return out


def long_context_leg(torch, kvq, dev, stream, case4=None):
    """One long request (B1, 32 query / 8 KV heads, D128): a 131072-token
    prefill, then 64 decode steps of kvq_append_decode (the steps that
    complete a group run the flush kernel too).  Reports the steps' GB/s
    including the flushes, and the decode kernel alone."""
    w4 = synth.WORKLOADS[4]
    if case4 is None:
        case4 = synth.make_case(w4)
    steps = synth.make_decode_steps(w4, w4.decode_steps, outliers=case4["outliers"])
    sd = [{k: torch.from_numpy(v).to(dev) for k, v in s.items()} for s in steps]
    K = torch.from_numpy(case4["K"]).to(dev)
    V = torch.from_numpy(case4["V"]).to(dev)
    peak, src = load_peaks()
    with make_cache(kvq, w4, w4.T + w4.decode_steps) as c:
        c.prefill(K, V)
        o = torch.empty(w4.batch, w4.n_q_heads, w4.head_dim, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        lens = []
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for s in sd:
            c.append_decode(s["k"], s["v"], s["q"], o, w4.scale)
            lens.append(c.state)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        nb = sum(decode_bytes(w4, tq, tt) for tq, tt in lens)
        flushes = sum(1 for (tq0, _), (tq1, _) in zip([(w4.T, 0)] + lens[:-1], lens) if tq1 != tq0)
        q = sd[-1]["q"]
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        per = flushed_launch_times(torch, stream, lambda: c.decode(q, o, w4.scale), 3 + 16,
                                   flush)[3:]
        del flush
        tq, tt = c.state
        nb1 = decode_bytes(w4, tq, tt)
        sp = spread(per)
        c.check()
    gbs_steps = nb / (ms * 1e-3) / 1e9
    gbs_dec = nb1 / (sp["median_ms"] * 1e-3) / 1e9
    del K, V
    return {"workload": w4.name, "steps": w4.decode_steps, "flushes": flushes,
            "ms_per_step": ms / w4.decode_steps, "GB/s_steps": gbs_steps,
            "frac_steps": gbs_steps / peak,
            "decode": {"GB/s": gbs_dec, "frac": gbs_dec / peak, "bytes_per_launch": nb1,
                       "l2": "flushed (512 MB written) before each launch", **sp},
            "peak_source": f"hbm_gbs of {src}"}


def sweep_leg(torch, kvq, dev, stream, n_caches=4, n_regions=8, n_err_pairs=16):
    """Geometry and bit-width sweep (B64, 32 query / 8 KV heads, D128, T2048):
    per combination, the decode GB/s (regions of one launch on each of
    n_caches caches, cold in L2) and the quantization errors against fp64
    attention over the unquantized fp16 cache, on sampled pairs: key
    reconstruction, attention-score (pre-softmax) and attention-output
    relative Frobenius errors, computed in torch float64 from the library's
    dequantized keys (kvq_dequantize) and its decode output."""
    base = synth.WORKLOADS[5]
    case = tiled_case(base, 8)
    K = torch.from_numpy(case["K"]).to(dev)
    V = torch.from_numpy(case["V"]).to(dev)
    q = torch.from_numpy(case["q"]).to(dev)
    rng = np.random.default_rng(5)
    pairs = sorted(rng.choice(base.n_pairs, n_err_pairs, replace=False).tolist())
    R = base.gqa
    # fp64 reference on the sampled pairs
    ref = []
    for p in pairs:
        b, h = divmod(p, base.n_kv_heads)
        qq = q[b, h * R:(h + 1) * R].double()
        kk, vv = K[b, h].double(), V[b, h].double()
        s = (qq @ kk.T) * base.scale
        ref.append((s, torch.softmax(s, dim=-1) @ vv, kk))
    peak, src = load_peaks()
    out = []
    for w in synth.sweep_workloads():
        caches = [make_cache(kvq, w, w.T) for _ in range(n_caches)]
        for c in caches:
            c.prefill(K, V)
        o = torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev)

        def body():
            for c in caches:
                c.decode(q, o, w.scale)
        per = [r / n_caches for r in region_times(torch, stream, body, n_regions)]
        sp = spread(per)
        nb = decode_bytes(w, w.T, 0)
        gbs = nb / (sp["median_ms"] * 1e-3) / 1e9
        kh, _ = caches[0].dequantize()
        o = caches[0].decode(q, softmax_scale=w.scale)
        torch.cuda.synchronize()
        num = {"k": 0.0, "s": 0.0, "o": 0.0}
        den = {"k": 0.0, "s": 0.0, "o": 0.0}
        for p, (s_ref, o_ref, k_ref) in zip(pairs, ref):
            b, h = divmod(p, w.n_kv_heads)
            kq = kh[b, h].double()
            s_q = (q[b, h * R:(h + 1) * R].double() @ kq.T) * w.scale
            o_q = o[b, h * R:(h + 1) * R].double()
            for key, a_, e_ in (("k", kq, k_ref), ("s", s_q, s_ref), ("o", o_q, o_ref)):
                num[key] += float(((a_ - e_) ** 2).sum())
                den[key] += float((e_ ** 2).sum())
        for c in caches:
            c.check()
            c.close()
        err = {k: math.sqrt(num[k] / den[k]) for k in num}
        out.append({"combo": w.name.split("t2048-")[-1], "bits_k": w.bits_k, "bits_v": w.bits_v,
                    "group": w.group, "axis_k": "channel" if w.axis_k == 0 else "token",
                    "axis_v": "channel" if w.axis_v == 0 else "token",
                    "GB/s": gbs, "frac": gbs / peak, "bytes_per_launch": nb,
                    "median_ms": sp["median_ms"], "min_ms": sp["min_ms"], "max_ms": sp["max_ms"],
                    "key_rel_err": err["k"], "score_rel_err": err["s"], "output_rel_err": err["o"]})
    del K, V
    return {"workload": base.name, "error_pairs": len(pairs), "peak_source": f"hbm_gbs of {src}",
            "combos": out}


def quantize_leg(torch, kvq, dev, stream, case4, skip_cpu):
    """Prefill throughput of the long-context workload (131072 tokens, 8 KV
    heads), L2 flushed before each launch."""
    w4 = synth.WORKLOADS[4]
    K4 = torch.from_numpy(case4["K"]).to(dev)
    V4 = torch.from_numpy(case4["V"]).to(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    with make_cache(kvq, w4, w4.T) as c4:
        qt = flushed_launch_times(torch, stream, lambda: c4.prefill(K4, V4), 3 + 10, flush)[3:]
        c4.check()
    sp = spread(qt)
    qms = sp["median_ms"]
    qtok = w4.batch * w4.T
    peak, src = load_peaks()
    q_gbs = qtok * quantize_bytes_per_token(w4) / (qms * 1e-3) / 1e9
    t_cpu_tokens = 8192
    t_cpu = oracle_quantize_sample(w4, t_cpu_tokens) if not skip_cpu else None
    del K4, V4, flush
    return {"value": qtok / (qms * 1e-3) / 1e6, "unit": "Mtok/s", "workload": w4.name,
            "GB/s": q_gbs, "frac_of_hbm": q_gbs / peak, "peak_source": f"hbm_gbs of {src}",
            "l2": "flushed (512 MB written) before each launch",
            "cpu_oracle_Mtok_s": (t_cpu_tokens / w4.n_kv_heads / t_cpu / 1e6) if t_cpu else None,
            "cpu_oracle_cores": 1, **sp}


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, w):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from bit_kv_cache_11_gb300 import kvq

    dev = torch.device("cuda", torch.cuda.current_device())
    L = args.layers
    n_steps = args.warmup + args.steps
    caches, steps, qs0 = [], [], []
    for layer in range(L):
        seed = rank_seed(w.config_id, rank, layer)
        case = synth.make_case(w, seed=seed)
        c = make_cache(kvq, w, w.T + n_steps + 32)
        c.prefill(torch.from_numpy(case["K"]).to(dev), torch.from_numpy(case["V"]).to(dev))
        st = synth.make_decode_steps(w, n_steps, seed=seed + 500, outliers=case["outliers"])
        steps.append([{k: torch.from_numpy(v).to(dev) for k, v in s.items()} for s in st])
        qs0.append(torch.from_numpy(case["q"]).to(dev))
        caches.append(c)
        if layer == 0:
            case0 = case
    torch.cuda.synchronize()
    outs = [torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev) for _ in range(L)]
    stream = torch.cuda.current_stream()

    # ---- the decode kernel's roofline: regions of one decode per layer
    roof_bytes, roof = decode_roofline(torch, kvq, w, caches, qs0, outs, stream)

    # ---- the step: append one token + decode, per layer
    for i in range(args.warmup):
        for layer in range(L):
            s = steps[layer][i]
            caches[layer].append_decode(s["k"], s["v"], s["q"], outs[layer], w.scale)
    torch.cuda.synchronize()
    barrier(ws)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    nbytes = 0
    launches0 = kvq.kvq_launch_count()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(ws)
        t_start.record(stream)
        for i in range(args.warmup, n_steps):
            for layer in range(L):
                s = steps[layer][i]
                caches[layer].append_decode(s["k"], s["v"], s["q"], outs[layer], w.scale)
                tq, tt = caches[layer].state
                nbytes += decode_bytes(w, tq, tt)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    launches = kvq.kvq_launch_count() - launches0
    ms = t_start.elapsed_time(t_end)
    ms_max = reduce_max(ms, ws)
    job_bytes = reduce_sum(float(nbytes), ws)
    for c in caches:
        c.check()

    # end to end through the public API: every step copies its inputs (the new
    # k, v and q of every layer) from one pinned host buffer in one transfer,
    # runs kvq_append_decode per layer and reads all layers' outputs back in one
    # transfer; the wall clock covers the copies and a synchronize per step.
    e2e_steps = min(args.steps, 5)
    kv_n = w.batch * w.n_kv_heads * w.head_dim
    q_n = w.batch * w.n_q_heads * w.head_dim
    per_layer = 2 * kv_n + q_n
    host_in = torch.empty((e2e_steps, L * per_layer), dtype=torch.float16).pin_memory()
    for layer in range(L):
        st = synth.make_decode_steps(w, e2e_steps, seed=99 + layer, outliers=case0["outliers"])
        for i, sd in enumerate(st):
            o = layer * per_layer
            host_in[i, o:o + kv_n] = torch.from_numpy(sd["k"]).reshape(-1)
            host_in[i, o + kv_n:o + 2 * kv_n] = torch.from_numpy(sd["v"]).reshape(-1)
            host_in[i, o + 2 * kv_n:o + per_layer] = torch.from_numpy(sd["q"]).reshape(-1)
    dev_in = torch.empty(L * per_layer, dtype=torch.float16, device=dev)
    out_all = torch.empty((L,) + tuple(outs[0].shape), dtype=torch.float32, device=dev)
    host_out = torch.empty(out_all.shape, dtype=torch.float32).pin_memory()
    h2d = dev_in.numel() * 2
    d2h = out_all.numel() * 4
    kv_shape = (w.batch, w.n_kv_heads, 1, w.head_dim)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_bytes = 0
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        dev_in.copy_(host_in[i], non_blocking=True)
        for layer in range(L):
            o = layer * per_layer
            kd = dev_in[o:o + kv_n].view(kv_shape)
            vd = dev_in[o + kv_n:o + 2 * kv_n].view(kv_shape)
            qd = dev_in[o + 2 * kv_n:o + per_layer].view(w.batch, w.n_q_heads, w.head_dim)
            caches[layer].append_decode(kd, vd, qd, out_all[layer], w.scale)
            tq, tt = caches[layer].state
            e2e_bytes += decode_bytes(w, tq, tt)
        host_out.copy_(out_all, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, ws)
    e2e_job_bytes = reduce_sum(float(e2e_bytes), ws)
    for c in caches:
        c.check()
        c.close()
    del caches, steps

    legs = {}
    if rank == 0 and not args.skip_legs:
        case4 = synth.make_case(synth.WORKLOADS[4])
        if not args.skip_quantize:
            legs["quantize"] = quantize_leg(torch, kvq, dev, stream, case4, args.skip_cpu)
        legs["windows"] = variant_leg(torch, kvq, w, dev, stream, L, 16, n_sink=4, residual=128)
        legs["fp8"] = variant_leg(torch, kvq, w.with_(bits_k=8, bits_v=8), dev, stream, L, 16,
                                  fp8=True)
        rag = [int(x) for x in np.linspace(1024, w.T, w.batch)]
        legs["ragged"] = variant_leg(torch, kvq, w, dev, stream, L, 16, lengths=rag)
        legs["outliers"] = variant_leg(torch, kvq, w, dev, stream, L, 16, n_outliers=32)
        legs["rope"] = rope_leg(torch, kvq, dev, stream)
        legs["long_context"] = long_context_leg(torch, kvq, dev, stream, case4)
        legs["sweep"] = sweep_leg(torch, kvq, dev, stream)

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    value = job_bytes / (ms_max * 1e-3) / 1e9
    peak, src = load_peaks()
    achieved = roof_bytes / (roof["median_ms"] * 1e-3) / 1e9
    cpu = cpu_all = None
    if not args.skip_cpu:
        cpu, cpu_all = cpu_baselines(w, case0)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16x2 tensor-core products (hi/lo fp16 operands), fp32 accumulate; u2 codes",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": L, "batch": w.batch, "n_heads": w.n_q_heads,
                   "head_dim": w.head_dim, "context": w.T, "bits_k": w.bits_k, "bits_v": w.bits_v,
                   "group": w.group, "step": "per layer: append 1 token + decode attention (kvq_append_decode)",
                   "l2": f"inputs larger than L2: {L} layer caches of {decode_bytes(w, 4096, 17) / 1e6:.1f} MB read in turn"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": load_traffic(f"decode_mma_kernel<{w.head_dim}, {w.bits_k}, {w.bits_v}, {w.gqa}>"),
                     "kernel": "decode_mma_kernel (split-K decode, in-place merge: one launch per layer)",
                     "timing": f"{roof['samples']} regions of {L} back-to-back kvq_decode_attention launches "
                               "(one per layer cache), CUDA events per region; per-launch = region / "
                               f"{L}; achieved from the median",
                     "peak_source": f"hbm_gbs of {src}",
                     "bytes_per_launch": roof_bytes, "ms_per_launch": roof["median_ms"],
                     "ms_per_launch_min": roof["min_ms"], "ms_per_launch_max": roof["max_ms"]},
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": {"value": e2e_job_bytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "frac_of_8tbs_spec": achieved / 8000.0,
        **legs,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- profile case

def run_profile_case(args):
    """One workload's prefill and a few decode (or append, or prefill) calls
    through the C ABI, with the CUDA-event time of each call printed."""
    import torch
    from bit_kv_cache_11_gb300 import kvq
    w = synth.WORKLOADS[args.config]
    if args.bits:
        w = w.with_(bits_k=args.bits, bits_v=args.bits)
    if args.fp8:
        w = w.with_(bits_k=8, bits_v=8)
    if args.batch:
        w = w.with_(batch=args.batch)
    torch.cuda.set_device(0)
    case = synth.make_case(w)
    K = torch.from_numpy(case["K"]).cuda()
    V = torch.from_numpy(case["V"]).cuda()
    q = torch.from_numpy(case["q"]).cuda()
    steps = [{k: torch.from_numpy(v).cuda() for k, v in s.items()}
             for s in synth.make_decode_steps(w, args.iters, outliers=case["outliers"])]
    with make_cache(kvq, w, w.T + args.iters + 32, fp8=args.fp8, n_sink=args.n_sink,
                    residual=args.residual) as cache:
        out = torch.empty(w.batch, w.n_q_heads, w.head_dim, device="cuda")
        cache.prefill(K, V)
        times = []
        for i in range(args.iters):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            if args.what == "quantize":
                cache.prefill(K, V)
            elif args.what == "decode":
                cache.decode(q, out, w.scale)
            else:
                cache.append(steps[i]["k"], steps[i]["v"])
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        cache.check()
    tag = " fp8" if args.fp8 else (f" sink{args.n_sink} res{args.residual}" if args.n_sink or args.residual else "")
    print(f"{w.name}{tag} {args.what}: " + " ".join(f"{t * 1e3:.1f}us" for t in times))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-quantize", action="store_true")
    ap.add_argument("--skip-legs", action="store_true",
                    help="only the headline step, roofline, end-to-end and CPU baseline")
    ap.add_argument("--profile-case", action="store_true",
                    help="run one workload's prefill and a few calls (for profiler captures)")
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--bits", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--what", default="decode", choices=["decode", "quantize", "append"])
    ap.add_argument("--fp8", action="store_true")
    ap.add_argument("--n-sink", type=int, default=0)
    ap.add_argument("--residual", type=int, default=0)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = synth.WORKLOADS[2]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
