"""Runs one workload's prefill and a few decode (or append) calls through the C
ABI — the small, self-contained program that profiler captures wrap.

    python -m bit_kv_cache_11_gb300.profile_case --config 2 --iters 3
    python -m bit_kv_cache_11_gb300.profile_case --config 4 --what quantize
    python -m bit_kv_cache_11_gb300.profile_case --config 2 --fp8
    python -m bit_kv_cache_11_gb300.profile_case --config 2 --n-sink 4 --residual 128

Prints the CUDA-event time of each call.
"""
from __future__ import annotations

import argparse

import torch

from . import kvq, synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--bits", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--what", default="decode", choices=["decode", "quantize", "append"])
    ap.add_argument("--fp8", action="store_true", help="FP8 (E4M3) cache, 8-bit sides")
    ap.add_argument("--n-sink", type=int, default=0)
    ap.add_argument("--residual", type=int, default=0)
    args = ap.parse_args()
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
    with kvq.KVCache(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                     head_dim=w.head_dim, max_ctx=w.T + args.iters + 32, bits_k=w.bits_k,
                     bits_v=w.bits_v, group=w.group, axis_k=w.axis_k, axis_v=w.axis_v,
                     keys_pre_rope=w.keys_pre_rope, rope_base=w.rope_base, fp8=args.fp8,
                     n_sink=args.n_sink, residual=args.residual) as cache:
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


if __name__ == "__main__":
    main()
