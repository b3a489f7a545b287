"""Seeded synthetic KV-cache inputs.

This module only draws numbers: it holds none of the quantization or
attention arithmetic, and both the CUDA path and the CPU oracle take their
inputs from it.

The workloads stand in for the Llama-2-7B / Llama-2-13B layer caches the
pages discuss ("Your KV cache doesn't have a bit problem, it has a geometry
problem": KIVI ablation on Llama-2-13B at group size 32; "Keys: The Outliers
Live in Fixed Channels": fixed large-magnitude key channels and attention
sinks).  They match those caches in shape and in outlier structure only:

  * K, V ~ N(0, 1) (float32 draws rounded to fp16);
  * in K, a fixed set of outlier channels is scaled at every token
    (x50 on {3, 17} for the tiny case; x20..x100 otherwise);
  * sink tokens 0-3 get key 8 * q / |q| for the step's query (the first query
    head of each KV group under GQA);
  * queries ~ N(0, 1).

Seeds: ``seed = 1000 * config + replica`` unless given.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    T: int                      # tokens per pair at decode time
    bits_k: int = 2
    bits_v: int = 2
    group: int = 32
    axis_k: int = 0             # 0 = per channel, 1 = per token
    axis_v: int = 1
    keys_pre_rope: bool = False
    rope_base: float = 10000.0
    outlier_channels: tuple = ()      # fixed set; empty -> drawn per kv head
    outlier_scales: tuple = (20.0, 46.666666666666664, 73.33333333333333, 100.0)
    n_outliers: int = 4
    sinks: bool = True
    decode_steps: int = 0
    config_id: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def n_pairs(self) -> int:
        return self.batch * self.n_kv_heads

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads.  Sizes are those the decode benchmark and the parity
# tests use; the sweep (5) is expanded by ``sweep_workloads``.
WORKLOADS = {
    1: Workload("tiny-b1-h2-d64-t256-2bit", 1, 2, 2, 64, 256, 2, 2, 32,
                outlier_channels=(3, 17), outlier_scales=(50.0, 50.0), sinks=False, config_id=1),
    2: Workload("llama2-7b-layer-decode-b8-h32-d128-t4113-2bit", 8, 32, 32, 128, 4096 + 17,
                2, 2, 32, config_id=2),
    3: Workload("llama2-13b-layer-decode-b16-h40-d128-t8192-prerope", 16, 40, 40, 128, 8192,
                2, 2, 32, keys_pre_rope=True, config_id=3),
    4: Workload("long-context-b1-gqa32x8-d128-t131072", 1, 32, 8, 128, 131072, 2, 2, 32,
                outlier_channels=(0, 63, 64, 127), decode_steps=64, config_id=4),
    5: Workload("sweep-b64-gqa32x8-d128-t2048", 64, 32, 8, 128, 2048, 2, 2, 32, config_id=5),
}


def sweep_workloads():
    """The geometry and bit-width sweep: axis combos x bits x G, plus k8v4."""
    base = WORKLOADS[5]
    out = []
    for (ak, av) in ((0, 1), (1, 0), (0, 0), (1, 1)):
        for b in (2, 4, 8):
            for G in (32, 128):
                out.append(base.with_(axis_k=ak, axis_v=av, bits_k=b, bits_v=b, group=G,
                                      name=f"{base.name}-k{'ch' if ak == 0 else 'tok'}"
                                           f"-v{'ch' if av == 0 else 'tok'}-{b}bit-g{G}"))
    for G in (32, 128):
        out.append(base.with_(bits_k=8, bits_v=4, group=G, name=f"{base.name}-k8v4-g{G}"))
    return out


def _normal_f16(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)


def _outlier_sets(rng: np.random.Generator, w: Workload) -> np.ndarray:
    """[n_kv_heads][k] outlier channel indices."""
    if w.outlier_channels:
        return np.tile(np.asarray(w.outlier_channels, np.int64), (w.n_kv_heads, 1))
    return np.stack([rng.choice(w.head_dim, size=w.n_outliers, replace=False)
                     for _ in range(w.n_kv_heads)])


def _apply_outliers(K32: np.ndarray, sets: np.ndarray, scales) -> None:
    """Scale K's outlier channels in place; K32: float32 [B][Hkv][T][D]."""
    for h in range(sets.shape[0]):
        for ch, s in zip(sets[h], scales):
            K32[:, h, :, ch] *= np.float32(s)


def _sink_keys(q16: np.ndarray, w: Workload) -> np.ndarray:
    """Key of a sink token for every (b, kv head): 8 * q / |q| of the first
    query head of the group.  Returns float32 [B][Hkv][D]."""
    q = q16.astype(np.float32)[:, :: w.gqa, :]
    n = np.sqrt((q.astype(np.float64) ** 2).sum(-1, keepdims=True)).astype(np.float32)
    return 8.0 * q / n


def make_case(w: Workload, seed: int | None = None, T: int | None = None) -> dict:
    """K, V fp16 [B][Hkv][T][D], q fp16 [B][Hq][D] and the outlier sets."""
    if seed is None:
        seed = 1000 * w.config_id
    T = w.T if T is None else T
    rng = np.random.default_rng(seed)
    B, Hkv, Hq, D = w.batch, w.n_kv_heads, w.n_q_heads, w.head_dim
    sets = _outlier_sets(rng, w)
    q = _normal_f16(rng, (B, Hq, D))
    K = rng.standard_normal(size=(B, Hkv, T, D), dtype=np.float32)
    _apply_outliers(K, sets, w.outlier_scales)
    if w.sinks and T > 0:
        K[:, :, : min(4, T), :] = _sink_keys(q, w)[:, :, None, :]
    K = K.astype(np.float16)
    V = _normal_f16(rng, (B, Hkv, T, D))
    return dict(K=K, V=V, q=q, outliers=sets, seed=seed, workload=w)


def make_decode_steps(w: Workload, n_steps: int, seed: int | None = None,
                      outliers: np.ndarray | None = None) -> list:
    """Per step: one new key/value token per pair (same recipe, no sinks) and
    a fresh query.  Each entry: dict(k [B][Hkv][1][D], v, q [B][Hq][D])."""
    if seed is None:
        seed = 1000 * w.config_id + 500
    rng = np.random.default_rng(seed)
    B, Hkv, Hq, D = w.batch, w.n_kv_heads, w.n_q_heads, w.head_dim
    sets = _outlier_sets(rng, w) if outliers is None else outliers
    steps = []
    for _ in range(n_steps):
        k = rng.standard_normal(size=(B, Hkv, 1, D), dtype=np.float32)
        _apply_outliers(k, sets, w.outlier_scales)
        steps.append(dict(k=k.astype(np.float16), v=_normal_f16(rng, (B, Hkv, 1, D)),
                          q=_normal_f16(rng, (B, Hq, D))))
    return steps


def small(w: Workload, batch: int = 1, n_kv_heads: int | None = None, T: int | None = None) -> Workload:
    """A reduced copy of a workload (fewer pairs / tokens) for oracle-sized
    parity cases; head_dim, bits, G, axes and GQA ratio are kept."""
    hkv = w.n_kv_heads if n_kv_heads is None else n_kv_heads
    return w.with_(batch=batch, n_kv_heads=hkv, n_q_heads=hkv * w.gqa,
                   T=w.T if T is None else T, name=w.name + "-small",
                   outlier_channels=tuple(c for c in w.outlier_channels if c < w.head_dim))
