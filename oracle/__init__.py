"""CPU oracle for paged-KV attention with asymmetric K/V head dims.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package.  The product
path (``paged_kv_asymmetric_gb300``) never imports it and shares no code with
it.  The arithmetic lives in ``pkv_oracle.c`` (plain C, compiled with gcc);
this module only builds it, loads it and marshals numpy arrays.

Functions and the passages they follow are documented in ``pkv_oracle.c``:

* ``e4m3_encode`` / ``e4m3_decode`` -- OCP FP8 E4M3 with RNE and saturation.
* ``kv_cache_write`` -- vLLM PR #64064, "Details": K and V scattered by
  slot_mapping into one packed (head_size + head_size_v) row per KV head.
* ``paged_attn`` -- causal (bottom-right) paged attention, whole rows or one
  split-KV segment.
* ``splitkv_reduce`` -- LSE merge; rows with no visible key give 0
  (MiMo-V2.6-Flash 2x RTX PRO 6000 model card, "Update 2026-10-01").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

DT_BF16, DT_FP8 = 0, 1
NHD, HND = 0, 1
SCALE_NONE, SCALE_TENSOR, SCALE_HEAD = 0, 1, 2


class CacheDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "dtype", "layout", "num_blocks", "block_size", "num_kv_heads",
        "row_elems", "k_off", "head_size", "v_off", "head_size_v",
        "scale_mode")]


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into a shared library (gcc, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call([
            "gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_kv_cache_write.argtypes = [
            P, i64, i64, P, i64, i64, P, i32, P, ctypes.POINTER(CacheDesc), P, P]
        lib.oracle_kv_cache_write.restype = i32
        lib.oracle_paged_attn.argtypes = [
            P, i32, i32, P, ctypes.POINTER(CacheDesc), P, i32, P, P, i32,
            ctypes.c_float, P, P, P, i32, i32, i32, i32, P, P, P]
        lib.oracle_paged_attn.restype = i32
        lib.oracle_splitkv_reduce.argtypes = [P, P, i32, i64, i32, P, P, P, i32]
        lib.oracle_splitkv_reduce.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def desc(dtype=DT_BF16, layout=NHD, num_blocks=1, block_size=16,
         num_kv_heads=4, row_elems=320, k_off=0, head_size=192, v_off=192,
         head_size_v=128, scale_mode=SCALE_NONE) -> CacheDesc:
    return CacheDesc(dtype, layout, num_blocks, block_size, num_kv_heads,
                     row_elems, k_off, head_size, v_off, head_size_v,
                     scale_mode)


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(_load().oracle_e4m3_decode(int(c) & 0xFF))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in flat],
                    dtype=np.uint8).reshape(np.shape(x))


def kv_cache_write(key_bits, value_bits, slot_mapping, cache, d: CacheDesc,
                   k_scale=None, v_scale=None, key_strides=None,
                   value_strides=None):
    """In-place write into ``cache`` (a numpy uint8 array holding the raw
    cache bytes).  ``key_bits`` / ``value_bits`` are uint16 arrays of bf16
    bits with shape [T, Hkv, D] (or any array plus explicit element strides
    (token, head)).  ``value_bits=None`` writes K only."""
    lib = _load()
    key_bits = np.asarray(key_bits)
    assert key_bits.dtype == np.uint16
    ks = key_strides or (key_bits.strides[0] // 2, key_bits.strides[1] // 2)
    if value_bits is not None:
        value_bits = np.asarray(value_bits)
        assert value_bits.dtype == np.uint16
        vs = value_strides or (value_bits.strides[0] // 2,
                               value_bits.strides[1] // 2)
    else:
        vs = (0, 0)
    slots = _c(slot_mapping, np.int64)
    kscale = None if k_scale is None else _c(k_scale, np.float32)
    vscale = None if v_scale is None else _c(v_scale, np.float32)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    rc = lib.oracle_kv_cache_write(
        _ptr(key_bits), ks[0], ks[1], _ptr(value_bits), vs[0], vs[1],
        _ptr(slots), int(slots.shape[0]), _ptr(cache), ctypes.byref(d),
        _ptr(kscale), _ptr(vscale))
    if rc != 0:
        raise ValueError("oracle_kv_cache_write rejected its arguments")


def paged_attn(q_bits, num_q_heads, cache, d: CacheDesc, block_table,
               seq_lens, query_start_loc, softmax_scale, k_scale=None,
               v_scale=None, tokens=None, num_splits=0, split=-1,
               threads=1, sinks=None, split_ranges=0):
    """Returns (out [n, Hq, dv] float64, lse [n, Hq] float64) for the query
    tokens listed in ``tokens`` (all tokens when None).  ``split`` >= 0 gives
    the partial of that segment: equal segments of ``num_splits``, or, with
    ``split_ranges`` = W > 0, the balanced ranges of W (see segment_pages in
    pkv_oracle.c).  ``threads`` > 1
    splits the token list over Python threads (the C call releases the
    GIL); the arithmetic of each row is unchanged.  ``sinks`` (float32 [Hq],
    or None): one attention-sink logit per query head, for whole rows
    (split < 0) only."""
    lib = _load()
    q_bits = _c(q_bits, np.uint16)
    T = q_bits.shape[0]
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    kscale = None if k_scale is None else _c(k_scale, np.float32)
    vscale = None if v_scale is None else _c(v_scale, np.float32)
    toks = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    snk = None if sinks is None else _c(sinks, np.float32)
    assert snk is None or snk.shape == (num_q_heads,)
    n = int(toks.shape[0])
    out = np.zeros((n, num_q_heads, d.head_size_v), dtype=np.float64)
    lse = np.zeros((n, num_q_heads), dtype=np.float64)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    max_blocks = int(bt.shape[1]) if bt.ndim == 2 else 0

    def run(lo, hi):
        if hi <= lo:
            return 0
        sub = np.ascontiguousarray(toks[lo:hi])
        o = out[lo:hi]
        ls = lse[lo:hi]
        return lib.oracle_paged_attn(
            _ptr(q_bits), num_q_heads, T, _ptr(cache), ctypes.byref(d),
            _ptr(bt), max_blocks, _ptr(sl), _ptr(qsl), int(sl.shape[0]),
            float(softmax_scale), _ptr(kscale), _ptr(vscale), _ptr(sub),
            hi - lo, int(num_splits), int(split), int(split_ranges), _ptr(o),
            _ptr(ls), _ptr(snk))

    if threads <= 1 or n < 2:
        rcs = [run(0, n)]
    else:
        bounds = np.linspace(0, n, min(threads, n) + 1).astype(int)
        rcs = [None] * (len(bounds) - 1)

        def worker(k):
            rcs[k] = run(int(bounds[k]), int(bounds[k + 1]))
        ths = [threading.Thread(target=worker, args=(k,))
               for k in range(len(bounds) - 1)]
        for th in ths:
            th.start()
        for th in ths:
            th.join()
    if any(rc != 0 for rc in rcs):
        raise ValueError("oracle_paged_attn: a token lies outside every sequence")
    return out, lse


def splitkv_reduce(partial_o, partial_lse, sinks=None, num_q_heads=1):
    """partial_o [S, rows, dv] float32, partial_lse [S, rows] float32 ->
    (out [rows, dv] float64, lse [rows] float64).  ``sinks`` (float32
    [num_q_heads], or None): row r's sink logit is sinks[r % num_q_heads]."""
    lib = _load()
    po = _c(partial_o, np.float32)
    pl = _c(partial_lse, np.float32)
    S, rows, dv = po.shape
    snk = None if sinks is None else _c(sinks, np.float32)
    assert snk is None or snk.shape == (num_q_heads,)
    out = np.zeros((rows, dv), dtype=np.float64)
    lse = np.zeros((rows,), dtype=np.float64)
    lib.oracle_splitkv_reduce(_ptr(po), _ptr(pl), S, rows, dv, _ptr(out),
                              _ptr(lse), _ptr(snk), int(num_q_heads))
    return out, lse
