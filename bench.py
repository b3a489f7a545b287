"""Decode-step benchmark of the low-bit KV cache on one GB300 (or N, one
process per GPU, each rank an independent replica).

Workload: a Llama-2-7B-shaped attention layer at decode time — batch 8, 32
heads (MHA), head_dim 128, context 4096 + 17-token fp16 tail, 2-bit keys
(per channel) and values (per token), group 32 — synthetic seeded inputs.
A step runs the hot path once over a stack of L such layers (default 8, each
with its own cache, 825 MB in total, so every layer is read cold from HBM):
for each layer, append the step's new token and run split-K decode attention
— one kvq_append_decode call, a single launch unless the token completes a
group of 32 (then the flush kernel runs before the decode).

value = algorithmic decode bytes of all layers and ranks / step time (GB/s):
packed codes + fp16 metadata + fp16 tail + q in + out, per decode call.
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


def decode_bytes(w, T_q, T_t):
    """Algorithmic bytes of one decode call."""
    P = w.batch * w.n_kv_heads
    codes = P * T_q * w.head_dim * (w.bits_k + w.bits_v) // 8
    meta = 2 * P * (T_q * w.head_dim // w.group) * 4
    tail = P * T_t * w.head_dim * 2 * 2
    qo = w.batch * w.n_q_heads * w.head_dim * (2 + 4)
    return codes + meta + tail + qo


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


def variant_leg(w, dev, stream, n_layers, warmup, steps, n_sink=0, residual=0, fp8=False,
                lengths=None):
    """The same decode step on a variant of the cache: fp16 windows (the first
    n_sink tokens and `residual` recent tokens kept in fp16), the FP8 (E4M3)
    format (w with 8-bit sides), or a ragged batch (row b holds lengths[b]
    tokens).  Algorithmic bytes count sink rows like tail rows, per row; the
    single-launch steps are averaged, as for the main line."""
    import torch
    from bit_kv_cache_11_gb300 import kvq
    caches, steps_dev = [], []
    for layer in range(n_layers):
        seed = rank_seed(w.config_id, 0, layer) + 7
        case = synth.make_case(w, seed=seed)
        c = kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                        head_dim=w.head_dim, max_ctx=w.T + warmup + steps + 32, bits_k=w.bits_k,
                        bits_v=w.bits_v, group=w.group, axis_k=w.axis_k, axis_v=w.axis_v,
                        n_sink=n_sink, residual=residual, fp8=fp8)
        if lengths is None:
            c.prefill(torch.from_numpy(case["K"]).to(dev), torch.from_numpy(case["V"]).to(dev))
        else:
            c.prefill_ragged(torch.from_numpy(case["K"]).to(dev), torch.from_numpy(case["V"]).to(dev),
                             lengths)
        st = synth.make_decode_steps(w, warmup + steps, seed=seed + 500, outliers=case["outliers"])
        steps_dev.append([{k: torch.from_numpy(v).to(dev) for k, v in x.items()} for x in st])
        caches.append(c)
    outs = [torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev)
            for _ in range(n_layers)]
    for i in range(warmup):
        for layer in range(n_layers):
            s = steps_dev[layer][i]
            caches[layer].append_decode(s["k"], s["v"], s["q"], outs[layer], w.scale)
    torch.cuda.synchronize()
    # row lengths before the timed steps; the timed loop makes no host query
    # (it would let the GPU run dry and time the host)
    lens = [[list(caches[layer].row_state(b)[:3]) for b in range(w.batch)]
            for layer in range(n_layers)]
    ev = []
    for i in range(warmup, warmup + steps):
        for layer in range(n_layers):
            s = steps_dev[layer][i]
            a = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            caches[layer].append_decode(s["k"], s["v"], s["q"], outs[layer], w.scale)
            e.record(stream)
            ev.append((layer, a, e))
    torch.cuda.synchronize()
    # replay each row's lengths through the append rule (one token per row and
    # step): the step runs as one launch when every row's token goes to its
    # tail without a flush
    timed = []
    for layer, a, e in ev:
        rows = lens[layer]
        fused = all(ts == n_sink and tt + 1 < residual + w.group for ts, _, tt in rows)
        for i_r, r in enumerate(rows):
            rows[i_r] = append_one(r, n_sink, residual, w.group)
        nb = sum(decode_bytes(w.with_(batch=1), tq, tt + ts) for ts, tq, tt in rows)
        if fused:
            timed.append((a, e, nb))
    for layer in range(n_layers):
        assert [list(caches[layer].row_state(b)[:3]) for b in range(w.batch)] == lens[layer]
    for c in caches:
        c.check()
        c.close()
    ms = statistics.mean(a.elapsed_time(e) for a, e, _ in timed)
    nb = statistics.mean(b for _, _, b in timed)
    peak, src = load_peaks()
    gbs = nb / (ms * 1e-3) / 1e9
    if fp8:
        name = w.name.replace("-2bit", "-fp8")
    elif lengths is not None:
        name = w.name.replace("-t4113", f"-ragged-t{min(lengths)}..{max(lengths)}")
    else:
        name = f"{w.name}-sink{n_sink}-res{residual}"
    return {"workload": name, "n_sink": n_sink, "residual": residual, "fp8": fp8,
            "lengths": lengths, "GB/s": gbs, "frac": gbs / peak, "peak_source": f"hbm_gbs of {src}",
            "ms_per_launch": ms, "bytes_per_launch": nb, "launches_timed": len(timed)}


def quantize_bytes_per_token(w):
    Hkv, D = w.n_kv_heads, w.head_dim
    return 2 * Hkv * D * 2 + Hkv * D * (w.bits_k + w.bits_v) // 8 + 2 * Hkv * D // w.group * 4


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


# ---------------------------------------------------------------- CPU oracle arm

def oracle_decode_sample(w, case, pairs, T):
    """Oracle decode (dequantize + fp64 attention) of a few pairs; returns
    (seconds, algorithmic bytes of those pairs)."""
    import oracle
    states = []
    for p in pairs:
        b, h = divmod(p, w.n_kv_heads)
        states.append((b, h, oracle.build_pair(case["K"][b, h, :T], case["V"][b, h, :T], w.group,
                                               w.bits_k, w.bits_v, w.axis_k, w.axis_v)))
    R = w.gqa
    t0 = time.perf_counter()
    for b, h, st in states:
        oracle.decode_pair(st, case["q"][b, h * R:(h + 1) * R], w.scale, w.keys_pre_rope, w.rope_base)
    dt = time.perf_counter() - t0
    T_q = (T // w.group) * w.group
    one = w.with_(batch=1, n_kv_heads=1, n_q_heads=R)
    return dt, len(pairs) * decode_bytes(one, T_q, T - T_q)


def oracle_quantize_sample(w4, tokens):
    import oracle
    rng = np.random.default_rng(4242)
    K = rng.standard_normal((tokens, w4.head_dim), dtype=np.float32).astype(np.float16)
    V = rng.standard_normal((tokens, w4.head_dim), dtype=np.float32).astype(np.float16)
    t0 = time.perf_counter()
    oracle.pack_pair(oracle.build_pair(K, V, w4.group, w4.bits_k, w4.bits_v, w4.axis_k, w4.axis_v))
    return time.perf_counter() - t0


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    case = synth.make_case(w)
    pairs = [0, 1, 2, 3]
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
        "impl": "reference", "metric": "quantized decode-attention HBM GB/s", "value": value,
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": f"{len(pairs)} of {w.n_pairs} (batch, kv-head) pairs per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(pairs)} pairs of {w.n_pairs} per step, dequantize + fp64 attention"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


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
    caches, steps = [], []
    for layer in range(L):
        seed = rank_seed(w.config_id, rank, layer)
        case = synth.make_case(w, seed=seed)
        c = kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                        head_dim=w.head_dim, max_ctx=w.T + n_steps + 32, bits_k=w.bits_k,
                        bits_v=w.bits_v, group=w.group, axis_k=w.axis_k, axis_v=w.axis_v)
        c.prefill(torch.from_numpy(case["K"]).to(dev), torch.from_numpy(case["V"]).to(dev))
        st = synth.make_decode_steps(w, n_steps, seed=seed + 500, outliers=case["outliers"])
        steps.append([{k: torch.from_numpy(v).to(dev) for k, v in s.items()} for s in st])
        caches.append(c)
        if layer == 0:
            case0 = case
    torch.cuda.synchronize()
    outs = [torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev) for _ in range(L)]
    stream = torch.cuda.current_stream()

    def step_bytes(i):
        total = 0
        for c in caches:
            tq, tt = c.state
            total += decode_bytes(w, tq, tt)
        return total

    # warm-up
    for i in range(args.warmup):
        for layer in range(L):
            s = steps[layer][i]
            caches[layer].append_decode(s["k"], s["v"], s["q"], outs[layer], w.scale)
    torch.cuda.synchronize()
    barrier(ws)

    n_ev = args.steps * L
    fused = [False] * n_ev
    step_b = [0] * n_ev
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    nbytes = 0
    launches0 = kvq.kvq_launch_count()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(ws)
        t_start.record(stream)
        k = 0
        for i in range(args.warmup, n_steps):
            for layer in range(L):
                s = steps[layer][i]
                tq0, tt0 = caches[layer].state
                # one launch (append fused into the decode) unless the token
                # completes a group: then the flush and the decode run apart
                fused[k] = tt0 + 1 < w.group
                ev_a[k].record(stream)
                caches[layer].append_decode(s["k"], s["v"], s["q"], outs[layer], w.scale)
                ev_b[k].record(stream)
                tq, tt = caches[layer].state
                step_b[k] = decode_bytes(w, tq, tt)
                nbytes += step_b[k]
                k += 1
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    launches = kvq.kvq_launch_count() - launches0
    ms = t_start.elapsed_time(t_end)
    ms_max = reduce_max(ms, ws)
    job_bytes = reduce_sum(float(nbytes), ws)
    dec_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]
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

    # quantize throughput: prefill of the long-context workload (131072 tokens)
    q_line = None
    if rank == 0 and not args.skip_quantize:
        w4 = synth.WORKLOADS[4]
        case4 = synth.make_case(w4)
        K4 = torch.from_numpy(case4["K"]).to(dev)
        V4 = torch.from_numpy(case4["V"]).to(dev)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        with kvq.KVCache(batch=w4.batch, n_q_heads=w4.n_q_heads, n_kv_heads=w4.n_kv_heads,
                         head_dim=w4.head_dim, max_ctx=w4.T, bits_k=w4.bits_k, bits_v=w4.bits_v,
                         group=w4.group) as c4:
            qt = []
            for i in range(3 + 5):
                flush.fill_(i & 0xff)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                c4.prefill(K4, V4)
                b.record(stream)
                torch.cuda.synchronize()
                if i >= 3:
                    qt.append(a.elapsed_time(b))
            c4.check()
        qms = statistics.median(qt)
        qtok = w4.batch * w4.T
        peak, src = load_peaks()
        q_gbs = qtok * quantize_bytes_per_token(w4) / (qms * 1e-3) / 1e9
        t_cpu_tokens = 8192
        t_cpu = oracle_quantize_sample(w4, t_cpu_tokens) if not args.skip_cpu else None
        q_line = {"value": qtok / (qms * 1e-3) / 1e6, "unit": "Mtok/s", "workload": w4.name,
                  "ms": qms, "GB/s": q_gbs, "frac_of_hbm": q_gbs / peak,
                  "cpu_oracle_Mtok_s": (t_cpu_tokens / w4.n_kv_heads / t_cpu / 1e6) if t_cpu else None}
        del K4, V4, flush

    win_line = fp8_line = rag_line = None
    if rank == 0 and not args.skip_windows:
        win_line = variant_leg(w, dev, stream, L, 3, min(args.steps, 10), n_sink=4, residual=128)
        fp8_line = variant_leg(w.with_(bits_k=8, bits_v=8), dev, stream, L, 3, min(args.steps, 10),
                               fp8=True)
        rag = [int(x) for x in np.linspace(1024, w.T, w.batch)]
        rag_line = variant_leg(w, dev, stream, L, 3, min(args.steps, 10), lengths=rag)

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    value = job_bytes / (ms_max * 1e-3) / 1e9
    peak, src = load_peaks()
    # the decode kernel's launches: the fused single-launch steps (a step
    # whose token completes a group also runs the flush kernel)
    sel = [k for k in range(n_ev) if fused[k]] or list(range(n_ev))
    avg_dec = statistics.mean(dec_ms[k] for k in sel)
    per_launch = sum(step_b[k] for k in sel) / len(sel)
    achieved = per_launch / (avg_dec * 1e-3) / 1e9
    cpu = None
    if not args.skip_cpu:
        dt, b = oracle_decode_sample(w, case0, [0, 1, 2], w.T)
        cpu = {"value": b / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "3 of 256 (batch, kv-head) pairs of one layer: dequantize + fp64 attention"}
    line = {
        "metric": "quantized decode-attention HBM GB/s", "value": value, "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": L, "batch": w.batch, "n_heads": w.n_q_heads,
                   "head_dim": w.head_dim, "context": w.T, "bits_k": w.bits_k, "bits_v": w.bits_v,
                   "group": w.group, "step": "per layer: append 1 token + decode attention (kvq_append_decode)",
                   "l2": f"inputs larger than L2: {L} layer caches of {decode_bytes(w, 4096, 17) / 1e6:.1f} MB read in turn"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": load_traffic(f"decode_mma_kernel<{w.head_dim}, {w.bits_k}, {w.bits_v}, {w.gqa}>"),
                     "kernel": "decode_mma_kernel (split-K decode, token append fused in, in-place merge: one launch per step and layer)",
                     "launches_timed": len(sel),
                     "peak_source": f"hbm_gbs of {src}",
                     "ms_per_launch": avg_dec, "bytes_per_launch": per_launch},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_job_bytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "quantize": q_line,
        "windows": win_line,
        "fp8": fp8_line,
        "ragged": rag_line,
        "frac_of_8tbs_spec": achieved / 8000.0,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-quantize", action="store_true")
    ap.add_argument("--skip-windows", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = synth.WORKLOADS[2]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
