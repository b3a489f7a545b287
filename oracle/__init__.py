"""CPU oracle of the low-bit KV-cache path — TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``kvq_oracle.c`` (plain C, fp32 quantizer, fp64
attention); this module compiles it with gcc on first use and wraps it with
numpy.  Everything here works on one (batch, kv-head) pair at a time or loops
over pairs in plain Python.

Sources (page titles and sections):
  * quantizer: "Your KV cache doesn't have a bit problem, it has a geometry
    problem", "What Quantization Error Is Actually Made Of";
  * key/value grouping: same page, "Keys: The Outliers Live in Fixed Channels"
    and "Values: Where the Intuition Breaks";
  * fp16 residual tail: same page, "The Systems Tax, and Why It Is Not a
    Detail" — a cache built by any sequence of prefill/append calls equals the
    cache built from the whole token sequence at once, because full groups are
    always G-aligned; ``build_pair`` uses that definition;
  * RoPE after dequantization: same page, "Rotary Embeddings Complicate the
    Keys";
  * attention output and the error metrics (relative Frobenius norm, the
    plainest reading of the pages' unnamed error measures): same page, "Keys"
    and "Values" sections;
  * fp16 windows (``window_lengths``): the residual window from "The Systems
    Tax, and Why It Is Not a Detail" (a sliding window of recent tokens kept
    in full precision), the sink window from "Where the Work Is Headed"
    (high-precision windows for attention-sink tokens);
  * FP8 cache (``e4m3_value``, ``e4m3_encode``, ``quantize_group_fp8``):
    "Rotate, Then Round: The Geometry of KV-Cache Compression", "Key
    takeaway"; the E4M3 format as the OCP 8-bit floating-point specification
    defines it;
  * dense-and-sparse outlier isolation (``select_outliers``,
    ``quantize_tensor_sparse``, ``apply_outliers``): KVQuant's "isolating a
    small fraction of outliers" in "Why KV Cache Geometry Matters More Than
    Bit Precision", "KV Cache Size, GPU Memory Efficiency, and the Shift to
    Geometry-Aware Quantization"; the selection rule and the format are a
    reading (the pages give neither): the n largest-magnitude elements of
    every block side, kept in fp16 with their positions.
A batch of rows with different lengths is checked row by row: each row is
its own sequence (``build_pair`` of that row's tokens).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into liboracle.so (gcc); returns the path."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I = ctypes.c_int
    L = ctypes.c_long
    D = ctypes.c_double
    lib.kvo_h2f.restype = ctypes.c_float
    lib.kvo_h2f.argtypes = [ctypes.c_uint16]
    lib.kvo_f2h.restype = ctypes.c_uint16
    lib.kvo_f2h.argtypes = [ctypes.c_float]
    lib.kvo_h2f_array.argtypes = [P, P, L]
    lib.kvo_f2h_array.argtypes = [P, P, L]
    lib.kvo_quantize_group.argtypes = [P, L, I, I, P, P, P]
    lib.kvo_quantize_tensor.restype = I
    lib.kvo_quantize_tensor.argtypes = [I, I, I, I, I, I, P, P, P, P]
    lib.kvo_dequantize_tensor.argtypes = [I, I, I, I, I, P, P, P, P]
    lib.kvo_quantize_group_fp8.argtypes = [P, L, I, P, P, P]
    lib.kvo_e4m3_value.restype = ctypes.c_float
    lib.kvo_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.kvo_e4m3_encode.restype = ctypes.c_uint8
    lib.kvo_e4m3_encode.argtypes = [ctypes.c_float]
    lib.kvo_e4m3_value_array.argtypes = [P, P, L]
    lib.kvo_e4m3_encode_array.argtypes = [P, P, L]
    lib.kvo_block_bytes.restype = ctypes.c_size_t
    lib.kvo_code_order.argtypes = [I, I, I, I, I]
    lib.kvo_code_order.restype = I
    lib.kvo_block_bytes.argtypes = [I, I, I, I]
    lib.kvo_block_offsets.argtypes = [I, I, I, I, P]
    lib.kvo_pack_pair.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P]
    lib.kvo_unpack_pair.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P]
    lib.kvo_quantize_group_masked.argtypes = [P, L, I, I, P, L, P, P, P]
    lib.kvo_select_outliers.argtypes = [P, I, I, I, P]
    lib.kvo_quantize_tensor_sparse.restype = I
    lib.kvo_quantize_tensor_sparse.argtypes = [I, I, I, I, I, I, P, P, P, P, P]
    lib.kvo_apply_outliers.argtypes = [I, I, I, I, P, P]
    lib.kvo_block_bytes_n.restype = ctypes.c_size_t
    lib.kvo_block_bytes_n.argtypes = [I, I, I, I, I]
    lib.kvo_block_offsets_n.argtypes = [I, I, I, I, I, P]
    lib.kvo_pack_pair_n.argtypes = [I, I, I, I, I, I, I, I] + [P] * 9
    lib.kvo_unpack_pair_n.argtypes = [I, I, I, I, I, I, I, I] + [P] * 9
    lib.kvo_rope.argtypes = [P, I, L, D]
    lib.kvo_attention_pair.argtypes = [I, I, I, I, P, P, P, P, P, D, I, D, P, P]
    _lib = lib
    return lib


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- fp16 helpers -----------------------------------------------------------

def h2f(h_bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> float32 values."""
    h = _c(h_bits, np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().kvo_h2f_array(_p(h), _p(out), h.size)
    return out


def f2h(f: np.ndarray) -> np.ndarray:
    """float32 values -> fp16 bit patterns (round to nearest even)."""
    x = _c(f, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().kvo_f2h_array(_p(x), _p(out), x.size)
    return out


def bits_of(x: np.ndarray) -> np.ndarray:
    """np.float16 array -> its uint16 bit patterns."""
    return _c(x, np.float16).view(np.uint16)


# ---- quantizer ----------------------------------------------------------------

def quantize_group(x_f16: np.ndarray, bits: int):
    """One group: returns (scale fp16 bits, zero fp16 bits, codes uint8[n])."""
    x = bits_of(x_f16).reshape(-1)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(x.size, np.uint8)
    _load().kvo_quantize_group(_p(x), 1, x.size, bits, _p(s), _p(z), _p(codes))
    return int(s[0]), int(z[0]), codes


def e4m3_value(codes) -> np.ndarray:
    """fp32 values of E4M3 codes (NaN for 0x7F and 0xFF)."""
    c = _c(np.asarray(codes, np.uint8).reshape(-1), np.uint8)
    out = np.zeros(c.size, np.float32)
    _load().kvo_e4m3_value_array(_p(c), _p(out), c.size)
    return out.reshape(np.shape(codes))


def e4m3_encode(y) -> np.ndarray:
    """Nearest E4M3 codes of fp32 values (ties to even, saturating at 448)."""
    f = _c(np.asarray(y, np.float32).reshape(-1), np.float32)
    out = np.zeros(f.size, np.uint8)
    _load().kvo_e4m3_encode_array(_p(f), _p(out), f.size)
    return out.reshape(np.shape(y))


def quantize_group_fp8(x_f16: np.ndarray):
    """One FP8 group: returns (scale fp16 bits, zero fp16 bits, E4M3 codes)."""
    x = bits_of(x_f16).reshape(-1)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(x.size, np.uint8)
    _load().kvo_quantize_group_fp8(_p(x), 1, x.size, _p(s), _p(z), _p(codes))
    return int(s[0]), int(z[0]), codes


def quantize_tensor(X_f16: np.ndarray, G: int, bits: int, axis: int, fp8: bool = False):
    """X: fp16 [T][D].  Returns (Tq, codes [Tq][D], scale bits, zero bits) with
    scale/zero shaped [Tq/G][D] (channel axis) or [Tq][D/G] (token axis).
    fp8: E4M3 codes with absmax scales (bits must be 8)."""
    T, D = X_f16.shape
    Tq = (T // G) * G
    x = bits_of(X_f16)
    codes = np.zeros((Tq, D), np.uint8)
    mshape = (Tq // G, D) if axis == 0 else (Tq, D // G)
    scale = np.zeros(mshape, np.uint16)
    zero = np.zeros(mshape, np.uint16)
    got = _load().kvo_quantize_tensor(T, D, G, bits, 1 if fp8 else 0, axis, _p(x), _p(codes),
                                      _p(scale), _p(zero))
    assert got == Tq
    return Tq, codes, scale, zero


def select_outliers(tile_f16: np.ndarray, n: int) -> np.ndarray:
    """Positions j*D + d (ascending) of the n elements of largest magnitude in
    a G x D fp16 tile (ties: lower position)."""
    G, D = tile_f16.shape
    assert 0 <= n <= G * D
    x = bits_of(tile_f16)
    pos = np.zeros(max(n, 1), np.int32)
    _load().kvo_select_outliers(_p(x), G, D, n, _p(pos))
    return pos[:n]


def quantize_group_masked(x_f16: np.ndarray, bits: int, skip: np.ndarray):
    """One group over its elements with skip == 0: (scale bits, zero bits,
    codes); skipped elements get code 0."""
    x = bits_of(x_f16).reshape(-1)
    m = _c(skip, np.uint8).reshape(-1)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(x.size, np.uint8)
    _load().kvo_quantize_group_masked(_p(x), 1, x.size, bits, _p(m), 1, _p(s), _p(z), _p(codes))
    return int(s[0]), int(z[0]), codes


def quantize_tensor_sparse(X_f16: np.ndarray, G: int, bits: int, axis: int, n_out: int):
    """quantize_tensor with n_out outliers isolated per G-token block.
    Returns (Tq, codes, scale bits, zero bits, outliers uint32 [Tq/G][n_out]):
    each outlier entry holds the kept fp16 value in bits 0-15 and its
    position j*D + d in the block in bits 16-31."""
    T, D = X_f16.shape
    assert 0 <= n_out <= G * D
    Tq = (T // G) * G
    x = bits_of(X_f16)
    codes = np.zeros((Tq, D), np.uint8)
    mshape = (Tq // G, D) if axis == 0 else (Tq, D // G)
    scale = np.zeros(mshape, np.uint16)
    zero = np.zeros(mshape, np.uint16)
    outl = np.zeros((Tq // G, max(n_out, 1)), np.uint32)
    got = _load().kvo_quantize_tensor_sparse(T, D, G, bits, axis, n_out, _p(x), _p(codes),
                                             _p(scale), _p(zero), _p(outl))
    assert got == Tq
    return Tq, codes, scale, zero, outl[:, :n_out]


def dequantize_tensor(codes, scale, zero, G: int, axis: int, fp8: bool = False) -> np.ndarray:
    Tq, D = codes.shape
    out = np.zeros((Tq, D), np.float32)
    c, s, z = _c(codes, np.uint8), _c(scale, np.uint16), _c(zero, np.uint16)
    _load().kvo_dequantize_tensor(Tq, D, G, axis, 1 if fp8 else 0, _p(c), _p(s), _p(z), _p(out))
    return out


# ---- layout -----------------------------------------------------------------

def code_order(D: int, G: int, bits: int, ak: int, av: int) -> int:
    """1 when a side's codes are stored in fragment order, 0 for sequential."""
    return int(_load().kvo_code_order(D, G, bits, ak, av))


def block_bytes(D: int, G: int, bk: int, bv: int, n_out: int = 0) -> int:
    return int(_load().kvo_block_bytes_n(D, G, bk, bv, n_out))


def block_offsets(D: int, G: int, bk: int, bv: int, n_out: int | None = None):
    """[K codes, K meta, V codes, V meta] offsets; with n_out given, the six
    offsets [K codes, K meta, K outliers, V codes, V meta, V outliers]."""
    if n_out is None:
        off = np.zeros(4, np.uint64)
        _load().kvo_block_offsets(D, G, bk, bv, _p(off))
    else:
        off = np.zeros(6, np.uint64)
        _load().kvo_block_offsets_n(D, G, bk, bv, n_out, _p(off))
    return [int(v) for v in off]


def pack_pair(st: dict) -> np.ndarray:
    """Packs one pair's quantized state into its blocks: uint8 [Tq/G][block_bytes]."""
    Tq, D = st["kcodes"].shape
    G, bk, bv, ak, av = st["G"], st["bk"], st["bv"], st["ak"], st["av"]
    n = st.get("n_out", 0)
    bb = block_bytes(D, G, bk, bv, n)
    out = np.zeros((Tq // G, bb), np.uint8)
    arrs = [_c(st["kcodes"], np.uint8), _c(st["kscale"], np.uint16), _c(st["kzero"], np.uint16),
            _c(st["vcodes"], np.uint8), _c(st["vscale"], np.uint16), _c(st["vzero"], np.uint16)]
    empty = np.zeros((max(Tq // G, 1), 1), np.uint32)
    kout = _c(st["kout"], np.uint32) if n else empty
    vout = _c(st["vout"], np.uint32) if n else empty
    _load().kvo_pack_pair_n(Tq, D, G, bk, bv, ak, av, n, *[_p(a) for a in arrs], _p(kout),
                            _p(vout), _p(out))
    return out


def unpack_pair(blocks: np.ndarray, D: int, G: int, bk: int, bv: int, ak: int, av: int,
                n_out: int = 0) -> dict:
    nb = blocks.shape[0]
    Tq = nb * G
    km = (nb, D) if ak == 0 else (Tq, D // G)
    vm = (nb, D) if av == 0 else (Tq, D // G)
    st = dict(G=G, bk=bk, bv=bv, ak=ak, av=av, n_out=n_out,
              kcodes=np.zeros((Tq, D), np.uint8), kscale=np.zeros(km, np.uint16),
              kzero=np.zeros(km, np.uint16), vcodes=np.zeros((Tq, D), np.uint8),
              vscale=np.zeros(vm, np.uint16), vzero=np.zeros(vm, np.uint16),
              kout=np.zeros((nb, max(n_out, 1)), np.uint32),
              vout=np.zeros((nb, max(n_out, 1)), np.uint32))
    blk = _c(blocks, np.uint8)
    _load().kvo_unpack_pair_n(Tq, D, G, bk, bv, ak, av, n_out, _p(blk),
                              _p(st["kcodes"]), _p(st["kscale"]), _p(st["kzero"]),
                              _p(st["vcodes"]), _p(st["vscale"]), _p(st["vzero"]),
                              _p(st["kout"]), _p(st["vout"]))
    st["kout"] = st["kout"][:, :n_out]
    st["vout"] = st["vout"][:, :n_out]
    return st


# ---- one pair's cache -------------------------------------------------------

def window_lengths(T: int, G: int, n_sink: int = 0, residual: int = 0):
    """Token counts (Ts, Tq, Tt) of a pair holding T tokens.

    Sinks: the first n_sink tokens stay fp16 (the high-precision sink window
    of "Your KV cache doesn't have a bit problem, it has a geometry problem",
    section "Where the Work Is Headed").  Residual window: the most recent
    tokens stay fp16 and a group of G is quantized only when it leaves a
    window of at least `residual` recent tokens behind (section "The Systems
    Tax, and Why It Is Not a Detail": a full-precision window of recently
    produced tokens, groups quantized once enough have accumulated).  With
    n_sink = residual = 0 this is the plain rule: the G-aligned prefix is
    quantized and fewer than G tokens stay in the tail."""
    Ts = min(T, n_sink)
    rest = T - Ts
    Tq = (rest - residual) // G * G if rest >= residual else 0
    return Ts, Tq, rest - Tq


def build_pair(K_f16: np.ndarray, V_f16: np.ndarray, G: int, bk: int, bv: int,
               ak: int = 0, av: int = 1, n_sink: int = 0, residual: int = 0,
               fp8: bool = False, n_outliers: int = 0) -> dict:
    """The cache state of one pair after its T tokens arrived (any mix of
    prefill and appends): the sink tokens in fp16, then the quantized groups,
    then the fp16 tail (window_lengths gives the three counts).  The state
    does not depend on how the tokens were split into calls, because every
    flush leaves the same G-aligned boundary.  fp8: both sides stored as E4M3
    with absmax scales (bk = bv = 8).  n_outliers: the elements of largest
    magnitude kept apart in every block of each side (dense-and-sparse
    isolation, quantize_tensor_sparse)."""
    T, D = K_f16.shape
    assert not fp8 or bk == bv == 8
    assert not (fp8 and n_outliers)
    Ts, Tq, Tt = window_lengths(T, G, n_sink, residual)
    kout = vout = np.zeros((Tq // G, 0), np.uint32)
    if n_outliers:
        Tq_, kc, ks, kz, kout = quantize_tensor_sparse(K_f16[Ts:Ts + Tq], G, bk, ak, n_outliers)
        _, vc, vs, vz, vout = quantize_tensor_sparse(V_f16[Ts:Ts + Tq], G, bv, av, n_outliers)
    else:
        Tq_, kc, ks, kz = quantize_tensor(K_f16[Ts:Ts + Tq], G, bk, ak, fp8)
        _, vc, vs, vz = quantize_tensor(V_f16[Ts:Ts + Tq], G, bv, av, fp8)
    assert Tq_ == Tq
    return dict(G=G, bk=bk, bv=bv, ak=ak, av=av, fp8=fp8, Ts=Ts, Tq=Tq, Tt=Tt,
                n_out=n_outliers, kout=kout, vout=vout,
                kcodes=kc, kscale=ks, kzero=kz, vcodes=vc, vscale=vs, vzero=vz,
                ksink=np.ascontiguousarray(K_f16[:Ts], np.float16),
                vsink=np.ascontiguousarray(V_f16[:Ts], np.float16),
                ktail=np.ascontiguousarray(K_f16[Ts + Tq:], np.float16),
                vtail=np.ascontiguousarray(V_f16[Ts + Tq:], np.float16))


def apply_outliers(xhat: np.ndarray, outliers: np.ndarray, G: int) -> np.ndarray:
    """Dequantized values with every block's kept outliers put back."""
    Tq, D = xhat.shape
    out = np.array(xhat, np.float32, copy=True)
    o = _c(outliers, np.uint32)
    _load().kvo_apply_outliers(Tq, D, G, o.shape[1] if o.ndim == 2 else 0, _p(o), _p(out))
    return out


def dequantize_pair(st: dict):
    f8 = st.get("fp8", False)
    kh = dequantize_tensor(st["kcodes"], st["kscale"], st["kzero"], st["G"], st["ak"], f8)
    vh = dequantize_tensor(st["vcodes"], st["vscale"], st["vzero"], st["G"], st["av"], f8)
    if st.get("n_out", 0):
        kh = apply_outliers(kh, st["kout"], st["G"])
        vh = apply_outliers(vh, st["vout"], st["G"])
    return kh, vh


# ---- RoPE and attention -----------------------------------------------------

def rope(x: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate-half RoPE of one vector, fp64."""
    v = np.array(x, dtype=np.float64, copy=True)
    _load().kvo_rope(_p(v), v.size, int(pos), float(base))
    return v


def attention_pair(q_f16: np.ndarray, khat: np.ndarray, vhat: np.ndarray,
                   ktail_f16: np.ndarray, vtail_f16: np.ndarray, scale: float,
                   rope_on: bool = False, base: float = 10000.0, want_scores: bool = False):
    """fp64 attention of R query heads over one pair's keys/values.
    q: fp16 [R][D]; khat/vhat: fp32 [Tq][D]; tails: fp16 [Tt][D]."""
    R, D = q_f16.shape
    khat = _c(khat, np.float32).reshape(-1, D)
    vhat = _c(vhat, np.float32).reshape(-1, D)
    kt = bits_of(ktail_f16).reshape(-1, D)
    vt = bits_of(vtail_f16).reshape(-1, D)
    Tq, Tt = khat.shape[0], kt.shape[0]
    out = np.zeros((R, D), np.float64)
    scores = np.zeros((R, Tq + Tt), np.float64) if want_scores else None
    qb = bits_of(q_f16)
    _load().kvo_attention_pair(R, D, Tq, Tt, _p(qb), _p(khat), _p(vhat), _p(kt), _p(vt),
                               float(scale), 1 if rope_on else 0, float(base), _p(out),
                               _p(scores) if want_scores else None)
    return (out, scores) if want_scores else out


def decode_pair(st: dict, q_f16: np.ndarray, scale: float, rope_on: bool = False,
                base: float = 10000.0, want_scores: bool = False):
    """Decode attention of one pair's cache: the fp16 sink tokens, the
    dequantized tokens and the fp16 tail, in token order (positions 0..T-1
    for RoPE).  Sink rows are fp16 values, exact in fp32, so they join the
    dequantized rows ahead of them."""
    kh, vh = dequantize_pair(st)
    D = kh.shape[1]
    if st.get("Ts", 0):
        kh = np.concatenate([st["ksink"].astype(np.float32).reshape(-1, D), kh])
        vh = np.concatenate([st["vsink"].astype(np.float32).reshape(-1, D), vh])
    return attention_pair(q_f16, kh, vh, st["ktail"], st["vtail"], scale, rope_on, base, want_scores)


def reference_pair(K_f16, V_f16, q_f16, scale, rope_on=False, base=10000.0, want_scores=False):
    """fp64 attention over the unquantized fp16 keys/values (the error
    metrics' reference)."""
    D = K_f16.shape[1]
    empty = np.zeros((0, D), np.float32)
    return attention_pair(q_f16, empty, empty, K_f16, V_f16, scale, rope_on, base, want_scores)


def rel_fro(approx: np.ndarray, exact: np.ndarray) -> float:
    """Relative Frobenius error ||approx - exact|| / ||exact||."""
    a = np.asarray(approx, np.float64)
    e = np.asarray(exact, np.float64)
    return float(np.linalg.norm(a - e) / np.linalg.norm(e))
