"""Thin Python binding of the C ABI in ``include/kvq.h`` (argument marshalling
only: every step of the path runs in the CUDA library ``libkvq.so``).

The functions carry the C names.  Device arguments are torch CUDA tensors (or
raw device addresses as ints); streams default to torch's current stream.
Importing this module raises if the library has not been built — there is no
CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"CUDA library not built: {LIB_PATH} is missing. Build it with "
        "`python -c \"import __graft_entry__ as g; g.build()\"` or "
        "`python -m bit_kv_cache_11_gb300.build`.")

_lib = ctypes.CDLL(LIB_PATH)

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_CAPACITY = 3
KVQ_ERR_OOM = 4
KVQ_ERR_CUDA = 5
KVQ_ERR_DEVICE_CHECK = 6
KVQ_AXIS_CHANNEL = 0
KVQ_AXIS_TOKEN = 1


class kvq_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_ctx", ctypes.c_int), ("bits_k", ctypes.c_int),
                ("bits_v", ctypes.c_int), ("group", ctypes.c_int), ("axis_k", ctypes.c_int),
                ("axis_v", ctypes.c_int), ("keys_pre_rope", ctypes.c_int), ("rope_base", ctypes.c_float),
                ("n_sink", ctypes.c_int), ("residual", ctypes.c_int), ("fp8", ctypes.c_int),
                ("n_outliers", ctypes.c_int)]


class kvq_buffers(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_void_p), ("k_tail", ctypes.c_void_p), ("v_tail", ctypes.c_void_p),
                ("block_bytes", ctypes.c_size_t), ("off_kc", ctypes.c_size_t),
                ("off_km", ctypes.c_size_t), ("off_vc", ctypes.c_size_t), ("off_vm", ctypes.c_size_t),
                ("blocks_per_pair", ctypes.c_int), ("n_pairs", ctypes.c_int), ("T_q", ctypes.c_int),
                ("T_tail", ctypes.c_int), ("code_order_k", ctypes.c_int), ("code_order_v", ctypes.c_int),
                ("k_sink", ctypes.c_void_p), ("v_sink", ctypes.c_void_p), ("T_sink", ctypes.c_int),
                ("tail_rows", ctypes.c_int), ("k_tail_buffer", ctypes.c_void_p * 2),
                ("v_tail_buffer", ctypes.c_void_p * 2), ("ragged", ctypes.c_int),
                ("off_ko", ctypes.c_size_t), ("off_vo", ctypes.c_size_t),
                ("n_outliers", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_S = ctypes.c_int  # kvq_status
_CFG = ctypes.POINTER(kvq_config)

_sigs = {
    "kvq_config_check": (_S, [_CFG]),
    "kvq_cache_bytes": (_S, [_CFG, ctypes.POINTER(ctypes.c_size_t)]),
    "kvq_create": (_S, [_CFG, ctypes.POINTER(_P)]),
    "kvq_destroy": (_S, [_P]),
    "kvq_quantize_prefill": (_S, [_P, _P, _P, _I, _P]),
    "kvq_append": (_S, [_P, _P, _P, _I, _P]),
    "kvq_quantize_prefill_ragged": (_S, [_P, _P, _P, ctypes.POINTER(_I), _I, _P]),
    "kvq_append_ragged": (_S, [_P, _P, _P, ctypes.POINTER(_I), _I, _P]),
    "kvq_get_row_state": (_S, [_P, _I] + [ctypes.POINTER(_I)] * 4),
    "kvq_decode_attention": (_S, [_P, _P, _P, ctypes.c_float, _P]),
    "kvq_append_decode": (_S, [_P, _P, _P, _I, _P, _P, ctypes.c_float, _P]),
    "kvq_dequantize": (_S, [_P, _P, _P, _P]),
    "kvq_decode_attention_noalloc": (_S, [_CFG, _P, _P, _P, _I, _I, _P, _P, ctypes.c_float, _P, _P]),
    "kvq_get_state": (_S, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "kvq_get_buffers": (_S, [_P, ctypes.POINTER(kvq_buffers)]),
    "kvq_check_device_error": (_S, [_P, _P]),
    "kvq_launch_count": (ctypes.c_uint64, []),
    "kvq_debug_fail_allocations": (_S, [_I, _I]),
    "kvq_debug_set_device_error": (_S, [_P, _I]),
    "kvq_debug_set_wait_limit": (_S, [_P, _I]),
    "kvq_status_string": (ctypes.c_char_p, [_S]),
}
for _name, (_res, _args) in _sigs.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class KvqError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {kvq_status_string(status)} (status {status})")


def _check(status: int, call: str) -> None:
    if status != KVQ_OK:
        raise KvqError(status, call)


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def make_config(batch, n_q_heads, n_kv_heads, head_dim, max_ctx, bits_k=2, bits_v=2, group=32,
                axis_k=KVQ_AXIS_CHANNEL, axis_v=KVQ_AXIS_TOKEN, keys_pre_rope=False,
                rope_base=10000.0, n_sink=0, residual=0, fp8=False, n_outliers=0) -> kvq_config:
    return kvq_config(int(batch), int(n_q_heads), int(n_kv_heads), int(head_dim), int(max_ctx),
                      int(bits_k), int(bits_v), int(group), int(axis_k), int(axis_v),
                      1 if keys_pre_rope else 0, float(rope_base), int(n_sink), int(residual),
                      1 if fp8 else 0, int(n_outliers))


# ---- the C calls, same names ------------------------------------------------

def kvq_status_string(status: int) -> str:
    return _lib.kvq_status_string(int(status)).decode()


def kvq_config_check(cfg: kvq_config) -> int:
    return _lib.kvq_config_check(ctypes.byref(cfg))


def kvq_cache_bytes(cfg: kvq_config) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.kvq_cache_bytes(ctypes.byref(cfg), ctypes.byref(n)), "kvq_cache_bytes")
    return n.value


def kvq_create(cfg: kvq_config) -> int:
    h = _P()
    _check(_lib.kvq_create(ctypes.byref(cfg), ctypes.byref(h)), "kvq_create")
    return h.value


def kvq_destroy(handle) -> None:
    _check(_lib.kvq_destroy(handle), "kvq_destroy")


def kvq_quantize_prefill(handle, k, v, T: int | None = None, stream=None) -> None:
    if T is None:
        T = k.shape[-2]
    _check(_lib.kvq_quantize_prefill(handle, _ptr(k), _ptr(v), int(T), _stream(stream)),
           "kvq_quantize_prefill")


def _ints(values):
    vals = [int(x) for x in values]
    return (_I * max(len(vals), 1))(*vals)


def kvq_quantize_prefill_ragged(handle, k, v, lengths, T_stride: int | None = None,
                                stream=None) -> None:
    """k, v: [batch][n_kv_heads][T_stride][head_dim]; row b holds lengths[b] tokens."""
    if T_stride is None:
        T_stride = k.shape[-2]
    _check(_lib.kvq_quantize_prefill_ragged(handle, _ptr(k), _ptr(v), _ints(lengths),
                                            int(T_stride), _stream(stream)),
           "kvq_quantize_prefill_ragged")


def kvq_append_ragged(handle, k, v, n_rows, n_stride: int | None = None, stream=None) -> None:
    """k, v: [batch][n_kv_heads][n_stride][head_dim]; row b appends n_rows[b] tokens."""
    if n_stride is None:
        n_stride = k.shape[-2]
    _check(_lib.kvq_append_ragged(handle, _ptr(k), _ptr(v), _ints(n_rows), int(n_stride),
                                  _stream(stream)), "kvq_append_ragged")


def kvq_get_row_state(handle, row: int) -> tuple[int, int, int, int]:
    """(T_sink, T_q, T_tail, tail_buffer) of batch row `row`."""
    vals = [_I(0) for _ in range(4)]
    _check(_lib.kvq_get_row_state(handle, int(row), *[ctypes.byref(x) for x in vals]),
           "kvq_get_row_state")
    return tuple(x.value for x in vals)


def kvq_append(handle, k, v, n: int | None = None, stream=None) -> None:
    if n is None:
        n = k.shape[-2]
    _check(_lib.kvq_append(handle, _ptr(k), _ptr(v), int(n), _stream(stream)), "kvq_append")


def kvq_decode_attention(handle, q, out, softmax_scale: float, stream=None) -> None:
    _check(_lib.kvq_decode_attention(handle, _ptr(q), _ptr(out), float(softmax_scale),
                                     _stream(stream)), "kvq_decode_attention")


def kvq_append_decode(handle, k, v, n: int, q, out, softmax_scale: float, stream=None) -> None:
    _check(_lib.kvq_append_decode(handle, _ptr(k) if n else None, _ptr(v) if n else None, int(n),
                                  _ptr(q), _ptr(out), float(softmax_scale), _stream(stream)),
           "kvq_append_decode")


def kvq_decode_attention_noalloc(cfg: kvq_config, blocks, k_tail, v_tail, T_q: int, T_tail: int,
                                 q, out, softmax_scale: float, device_error=None,
                                 stream=None) -> None:
    """Decode over a packed cache the caller owns, allocating no device memory
    (see include/kvq.h for who needs this and for the workspace limit)."""
    _check(_lib.kvq_decode_attention_noalloc(ctypes.byref(cfg), _ptr(blocks), _ptr(k_tail),
                                             _ptr(v_tail), int(T_q), int(T_tail), _ptr(q),
                                             _ptr(out), float(softmax_scale), _ptr(device_error),
                                             _stream(stream)), "kvq_decode_attention_noalloc")


def kvq_dequantize(handle, k_out, v_out, stream=None) -> None:
    _check(_lib.kvq_dequantize(handle, _ptr(k_out), _ptr(v_out), _stream(stream)), "kvq_dequantize")


def kvq_get_state(handle) -> tuple[int, int]:
    tq, tt = _I(0), _I(0)
    _check(_lib.kvq_get_state(handle, ctypes.byref(tq), ctypes.byref(tt)), "kvq_get_state")
    return tq.value, tt.value


def kvq_get_buffers(handle) -> kvq_buffers:
    b = kvq_buffers()
    _check(_lib.kvq_get_buffers(handle, ctypes.byref(b)), "kvq_get_buffers")
    return b


def kvq_check_device_error(handle, stream=None) -> int:
    return _lib.kvq_check_device_error(handle, _stream(stream))


def kvq_launch_count() -> int:
    return int(_lib.kvq_launch_count())


def kvq_debug_fail_allocations(after: int, n: int) -> None:
    _check(_lib.kvq_debug_fail_allocations(after, n), "kvq_debug_fail_allocations")


def kvq_debug_set_device_error(handle, value: int) -> None:
    _check(_lib.kvq_debug_set_device_error(handle, value), "kvq_debug_set_device_error")


def kvq_debug_set_wait_limit(handle, limit: int) -> None:
    _check(_lib.kvq_debug_set_wait_limit(handle, limit), "kvq_debug_set_wait_limit")


# ---- convenience -------------------------------------------------------------

class _DeviceArray:
    """Exposes a library-owned device range to torch without copying."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def device_view(ptr: int, shape, typestr: str = "|u1"):
    import torch
    return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")


class KVCache:
    """One layer's packed KV cache on the current CUDA device.

    Keyword arguments are those of ``make_config`` (the fields of
    ``kvq_config``): batch, n_q_heads, n_kv_heads, head_dim, max_ctx,
    bits_k / bits_v (2, 4, 8), group (32, 64, 128), axis_k / axis_v,
    keys_pre_rope / rope_base, n_sink and residual (fp16 windows), fp8 (E4M3
    codes, 8-bit sides), n_outliers (elements kept in fp16 per block and
    side).  A typical decode loop::

        cache = KVCache(batch=8, n_q_heads=32, n_kv_heads=32, head_dim=128,
                        max_ctx=8192, bits_k=2, bits_v=2)
        cache.prefill(k, v)                    # [B][Hkv][T][D] fp16 on the GPU
        for step in range(n):
            out = cache.append_decode(k1, v1, q)   # [B][Hkv][1][D], [B][Hq][D]

    ``prefill_ragged`` / ``append_ragged`` take per-row lengths (a serving
    batch of sequences of different lengths, batch <= 64); ``row_state``
    reports each row's sink, quantized and tail counts.
    """

    def __init__(self, **cfg_kw):
        self.cfg = make_config(**cfg_kw)
        self.handle = kvq_create(self.cfg)

    @property
    def gqa(self) -> int:
        return self.cfg.n_q_heads // self.cfg.n_kv_heads

    def close(self) -> None:
        if self.handle:
            kvq_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, k, v, stream=None):
        kvq_quantize_prefill(self.handle, k, v, k.shape[-2], stream)

    def prefill_ragged(self, k, v, lengths, stream=None):
        kvq_quantize_prefill_ragged(self.handle, k, v, lengths, k.shape[-2], stream)

    def append_ragged(self, k, v, n_rows, stream=None):
        kvq_append_ragged(self.handle, k, v, n_rows, k.shape[-2], stream)

    def row_state(self, row: int) -> tuple[int, int, int, int]:
        """(T_sink, T_q, T_tail, tail_buffer) of batch row `row`."""
        return kvq_get_row_state(self.handle, row)

    def append(self, k, v, stream=None):
        kvq_append(self.handle, k, v, k.shape[-2], stream)

    def decode(self, q, out=None, softmax_scale=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if softmax_scale is None:
            softmax_scale = self.cfg.head_dim ** -0.5
        kvq_decode_attention(self.handle, q, out, softmax_scale, stream)
        return out

    def append_decode(self, k, v, q, out=None, softmax_scale=None, stream=None):
        """Appends k, v ([batch][n_kv_heads][n][head_dim] fp16) and decodes q,
        in one launch when no group is completed."""
        import torch
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if softmax_scale is None:
            softmax_scale = self.cfg.head_dim ** -0.5
        n = 0 if k is None else k.shape[-2]
        kvq_append_decode(self.handle, k, v, n, q, out, softmax_scale, stream)
        return out

    def dequantize(self, stream=None):
        import torch
        tq, _ = self.state
        shape = (self.cfg.batch, self.cfg.n_kv_heads, tq, self.cfg.head_dim)
        k = torch.empty(shape, dtype=torch.float32, device="cuda")
        v = torch.empty(shape, dtype=torch.float32, device="cuda")
        kvq_dequantize(self.handle, k, v, stream)
        return k, v

    @property
    def state(self) -> tuple[int, int]:
        return kvq_get_state(self.handle)

    def buffers(self) -> kvq_buffers:
        return kvq_get_buffers(self.handle)

    def block_bytes_view(self):
        """uint8 [P][NB][block_bytes] view of the packed blocks (no copy)."""
        b = self.buffers()
        return device_view(b.blocks, (b.n_pairs, b.blocks_per_pair, b.block_bytes))

    def tail_views(self):
        """fp16 [P][tail_rows][D] views of the active K and V tails (no copy)."""
        b = self.buffers()
        shape = (b.n_pairs, b.tail_rows, self.cfg.head_dim)
        k = device_view(b.k_tail, shape, "<f2")
        v = device_view(b.v_tail, shape, "<f2")
        return k, v

    def row_tail_views(self, row: int):
        """fp16 [n_kv_heads][tail_rows][D] views of row `row`'s K and V tails."""
        b = self.buffers()
        buf = self.row_state(row)[3]
        shape = (b.n_pairs, b.tail_rows, self.cfg.head_dim)
        h = self.cfg.n_kv_heads
        k = device_view(b.k_tail_buffer[buf], shape, "<f2")[row * h:(row + 1) * h]
        v = device_view(b.v_tail_buffer[buf], shape, "<f2")[row * h:(row + 1) * h]
        return k, v

    def sink_views(self):
        """fp16 [P][n_sink][D] views of the K and V sink windows (no copy);
        None when the cache has no sink window."""
        b = self.buffers()
        if not b.k_sink:
            return None
        shape = (b.n_pairs, self.cfg.n_sink, self.cfg.head_dim)
        return device_view(b.k_sink, shape, "<f2"), device_view(b.v_sink, shape, "<f2")

    def check(self, stream=None) -> None:
        _check(kvq_check_device_error(self.handle, stream), "kvq_check_device_error")
