"""Paged-KV attention with asymmetric K/V head sizes for GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/pkv.h`` (libpkv.so, built
from ``csrc/`` by ``_build.py``).  It only marshals arguments: every step of
the computation runs in the library's CUDA kernels.  Tensors are torch CUDA
tensors (device memory and the current stream come from torch); nothing here
falls back to another implementation -- if the library is missing, every call
raises.

Functions (same names as the C entry points, without the ``pkv_`` prefix):
``kv_cache_write``, ``paged_attn_prefill``, ``paged_attn_decode``,
``paged_attn_decode_balanced``, ``splitkv_reduce``,
``decode_suggest_splits``, ``decode_balanced_ranges``, ``supports``,
``get_device_error``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

# constants mirrored from include/pkv.h
OK, EINVAL, EUNSUPPORTED, ECUDA = 0, -1, -2, -3
EDEV_NONE, EDEV_RANGE, EDEV_TIMEOUT = 0, 1, 2
BF16, FP8_E4M3 = 0, 1
NHD, HND = 0, 1
SCALE_NONE, SCALE_TENSOR, SCALE_HEAD = 0, 1, 2

EXPORTED = (
    "pkv_kv_cache_write", "pkv_paged_attn_prefill", "pkv_paged_attn_decode",
    "pkv_paged_attn_decode_fused", "pkv_paged_attn_decode_fused_noalloc",
    "pkv_decode_workspace_bytes", "pkv_splitkv_reduce", "pkv_splitkv_reduce_sink",
    "pkv_paged_attn_prefill_sink", "pkv_prefill_fp8_workspace_bytes",
    "pkv_paged_attn_prefill_fp8", "pkv_decode_suggest_splits",
    "pkv_paged_attn_decode_balanced", "pkv_decode_balanced_ranges",
    "pkv_paged_attn_decode_balanced_fused",
    "pkv_supports",
    "pkv_get_device_error", "pkv_selftest_bounded_wait", "pkv_last_cuda_error",
    "pkv_status_string",
)


class PkvError(RuntimeError):
    def __init__(self, fn, status, cuda_error=0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{fn} failed with status {status}"
        try:
            msg += f" ({_lib().pkv_status_string(status).decode()})"
        except Exception:  # pragma: no cover
            pass
        if status == ECUDA:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


class CacheDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "dtype", "layout", "num_blocks", "block_size", "num_kv_heads",
        "row_elems", "k_off", "head_size", "v_off", "head_size_v",
        "scale_mode")]


@dataclasses.dataclass
class Cache:
    """A block-paged cache: its storage (a CUDA tensor of bytes, or of bf16)
    and its description."""
    data: torch.Tensor
    desc: CacheDesc


_lock = threading.Lock()
_handle = None


def _lib():
    global _handle
    with _lock:
        if _handle is not None:
            return _handle
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libpkv.so is not built ({LIB_PATH}); run "
                "`python -m paged_kv_asymmetric_gb300._build` first")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, I64, F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                        ctypes.c_float)
        D = ctypes.POINTER(CacheDesc)
        lib.pkv_kv_cache_write.argtypes = [P, I64, I64, P, I64, I64, P, I, P,
                                           D, P, P, P]
        lib.pkv_paged_attn_prefill.argtypes = [P, I, I, P, D, P, I, P, P, I,
                                               F, P, P, P, P]
        lib.pkv_paged_attn_decode.argtypes = [P, I, I, P, D, P, I, P, P, I, I,
                                              F, P, P, I, P, P, P]
        lib.pkv_paged_attn_decode_fused.argtypes = [P, I, I, P, D, P, I, P, P, I,
                                                    I, F, P, P, I, P, P, P,
                                                    ctypes.c_size_t, P, P, P]
        lib.pkv_paged_attn_decode_fused_noalloc.argtypes = [
            P, I, I, P, D, P, I, P, P, I, I, F, P, P, I, P, P, P, P, P]
        lib.pkv_paged_attn_decode_balanced.argtypes = [P, I, I, P, D, P, I, P, P, I, I,
                                                       F, P, P, I, I, P, P, P]
        lib.pkv_decode_balanced_ranges.argtypes = [D]
        lib.pkv_paged_attn_decode_balanced_fused.argtypes = [
            P, I, I, P, D, P, I, P, P, I, I, F, P, P, I, I, P, P, P, ctypes.c_size_t, P, P, P]
        lib.pkv_prefill_fp8_workspace_bytes.argtypes = [I, I, D]
        lib.pkv_prefill_fp8_workspace_bytes.restype = ctypes.c_size_t
        lib.pkv_paged_attn_prefill_fp8.argtypes = [P, I, I, P, D, P, I, P, P, I, F, P, P,
                                                   P, P, ctypes.c_size_t, P, P]
        lib.pkv_decode_workspace_bytes.argtypes = [I, I, I, I]
        lib.pkv_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.pkv_splitkv_reduce.argtypes = [P, P, I, I, I, P, P, P]
        lib.pkv_splitkv_reduce_sink.argtypes = [P, P, I, I, I, P, I, P, P, P]
        lib.pkv_paged_attn_prefill_sink.argtypes = [P, I, I, P, D, P, I, P, P, I,
                                                    F, P, P, P, P, P]
        lib.pkv_decode_suggest_splits.argtypes = [I, I, I, I, I, I]
        lib.pkv_supports.argtypes = [I, I, I]
        lib.pkv_get_device_error.argtypes = [ctypes.POINTER(I), P]
        lib.pkv_selftest_bounded_wait.argtypes = [I, P]
        lib.pkv_last_cuda_error.argtypes = []
        lib.pkv_status_string.argtypes = [I]
        lib.pkv_status_string.restype = ctypes.c_char_p
        for name in EXPORTED:
            if name not in ("pkv_status_string", "pkv_decode_workspace_bytes",
                            "pkv_prefill_fp8_workspace_bytes"):
                getattr(lib, name).restype = ctypes.c_int
        _handle = lib
        return lib


def library_path() -> str:
    return LIB_PATH


def load():
    """Loads the library (raises ImportError when it is not built)."""
    return _lib()


def _check(fn, status):
    if status != OK:
        raise PkvError(fn, status, _lib().pkv_last_cuda_error()
                       if status == ECUDA else 0)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()  # ctypes passes the int as the c_void_p argument


# The current device's current stream without the device lookups of
# torch.cuda.current_stream(), which cost a few microseconds a call; torch's
# public call is the fallback.
_cuda_get_device = getattr(torch._C, "_cuda_getDevice", None)
_cuda_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is not None:
        return stream.cuda_stream
    if _cuda_get_device is not None and _cuda_raw_stream is not None and \
            torch.cuda.is_initialized():
        return _cuda_raw_stream(_cuda_get_device())
    return torch.cuda.current_stream().cuda_stream


def make_desc(*, dtype=BF16, layout=NHD, num_blocks, block_size=16,
              num_kv_heads=4, row_elems=320, k_off=0, head_size=192,
              v_off=192, head_size_v=128, scale_mode=SCALE_NONE) -> CacheDesc:
    return CacheDesc(dtype, layout, num_blocks, block_size, num_kv_heads,
                     row_elems, k_off, head_size, v_off, head_size_v,
                     scale_mode)


def cache_nbytes(d: CacheDesc) -> int:
    e = 1 if d.dtype == FP8_E4M3 else 2
    return d.num_blocks * d.block_size * d.num_kv_heads * d.row_elems * e


def kv_cache_write(key, value, slot_mapping, cache: Cache, k_scale=None,
                   v_scale=None, stream=None):
    """key: bf16 [T, Hkv, dk] (any token/head strides, unit element stride),
    value: bf16 [T, Hkv, dv] or None, slot_mapping: int64 [T]."""
    assert key.dtype == torch.bfloat16 and key.stride(2) == 1
    assert slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous()
    if value is not None:
        assert value.dtype == torch.bfloat16 and value.stride(2) == 1
    vs = (value.stride(0), value.stride(1)) if value is not None else (0, 0)
    _check("pkv_kv_cache_write", _lib().pkv_kv_cache_write(
        _ptr(key), key.stride(0), key.stride(1), _ptr(value), vs[0], vs[1],
        _ptr(slot_mapping), int(slot_mapping.shape[0]), _ptr(cache.data),
        ctypes.byref(cache.desc), _ptr(k_scale), _ptr(v_scale),
        _stream(stream)))


def _attn_common(q, block_table, seq_lens, query_start_loc):
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3
    for t in (block_table, seq_lens, query_start_loc):
        assert t.dtype == torch.int32 and t.is_contiguous()
    assert block_table.dim() == 2


def prefill_fp8_workspace_bytes(num_seqs, max_blocks_per_seq, cache: Cache) -> int:
    return int(_lib().pkv_prefill_fp8_workspace_bytes(int(num_seqs), int(max_blocks_per_seq),
                                                      ctypes.byref(cache.desc)))


def paged_attn_prefill(q, cache: Cache, block_table, seq_lens,
                       query_start_loc, softmax_scale, out=None,
                       k_scale=None, v_scale=None, stream=None, sinks=None,
                       workspace=None):
    """q: bf16 [T, Hq, dk]; returns out bf16 [T, Hq, dv].  ``sinks``: float32
    [Hq] CUDA tensor of attention-sink logits, or None.  An FP8 cache takes
    k_scale / v_scale (float32 CUDA tensors); with ``workspace`` None its
    codes are widened in the kernel (pkv_paged_attn_prefill), with a uint8
    CUDA tensor of at least prefill_fp8_workspace_bytes(...) bytes the
    two-pass form runs (pkv_paged_attn_prefill_fp8)."""
    _attn_common(q, block_table, seq_lens, query_start_loc)
    T, Hq, _ = q.shape
    if out is None:
        out = torch.empty(T, Hq, cache.desc.head_size_v, dtype=torch.bfloat16,
                          device=q.device)
    args = (_ptr(q), Hq, T, _ptr(cache.data), ctypes.byref(cache.desc),
            _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
            _ptr(query_start_loc), int(seq_lens.shape[0]), float(softmax_scale),
            _ptr(k_scale), _ptr(v_scale))
    if sinks is not None:
        assert sinks.dtype == torch.float32 and sinks.is_contiguous()
        assert tuple(sinks.shape) == (Hq,)
    if workspace is not None:
        nb = workspace.numel() * workspace.element_size()
        _check("pkv_paged_attn_prefill_fp8", _lib().pkv_paged_attn_prefill_fp8(
            *args, _ptr(sinks), _ptr(workspace), nb, _ptr(out), _stream(stream)))
    elif sinks is None:
        _check("pkv_paged_attn_prefill", _lib().pkv_paged_attn_prefill(
            *args, _ptr(out), _stream(stream)))
    else:
        _check("pkv_paged_attn_prefill_sink", _lib().pkv_paged_attn_prefill_sink(
            *args, _ptr(sinks), _ptr(out), _stream(stream)))
    return out


def paged_attn_decode(q, cache: Cache, block_table, seq_lens,
                      query_start_loc, softmax_scale, max_query_len,
                      num_splits, partial_o=None, partial_lse=None,
                      k_scale=None, v_scale=None, stream=None):
    """Returns (partial_o [S, T, Hq, dv] f32, partial_lse [S, T, Hq] f32)."""
    _attn_common(q, block_table, seq_lens, query_start_loc)
    T, Hq, _ = q.shape
    dv = cache.desc.head_size_v
    if partial_o is None:
        partial_o = torch.empty(num_splits, T, Hq, dv, dtype=torch.float32,
                                device=q.device)
    if partial_lse is None:
        partial_lse = torch.empty(num_splits, T, Hq, dtype=torch.float32,
                                  device=q.device)
    _check("pkv_paged_attn_decode", _lib().pkv_paged_attn_decode(
        _ptr(q), Hq, T, _ptr(cache.data), ctypes.byref(cache.desc),
        _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
        _ptr(query_start_loc), int(seq_lens.shape[0]), int(max_query_len),
        float(softmax_scale), _ptr(k_scale), _ptr(v_scale), int(num_splits),
        _ptr(partial_o), _ptr(partial_lse), _stream(stream)))
    return partial_o, partial_lse


def paged_attn_decode_balanced(q, cache: Cache, block_table, seq_lens,
                               query_start_loc, softmax_scale, max_query_len,
                               max_splits, num_ranges=0, partial_o=None,
                               partial_lse=None, k_scale=None, v_scale=None,
                               stream=None):
    """Split-KV decode with balanced ranges (pkv_paged_attn_decode_balanced):
    the segments are cut on the device from seq_lens so that every range of
    the batch's pages is the same size.  Returns (partial_o [max_splits, T,
    Hq, dv] f32, partial_lse [max_splits, T, Hq] f32)."""
    _attn_common(q, block_table, seq_lens, query_start_loc)
    T, Hq, _ = q.shape
    dv = cache.desc.head_size_v
    if partial_o is None:
        partial_o = torch.empty(max_splits, T, Hq, dv, dtype=torch.float32,
                                device=q.device)
    if partial_lse is None:
        partial_lse = torch.empty(max_splits, T, Hq, dtype=torch.float32,
                                  device=q.device)
    _check("pkv_paged_attn_decode_balanced", _lib().pkv_paged_attn_decode_balanced(
        _ptr(q), Hq, T, _ptr(cache.data), ctypes.byref(cache.desc),
        _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
        _ptr(query_start_loc), int(seq_lens.shape[0]), int(max_query_len),
        float(softmax_scale), _ptr(k_scale), _ptr(v_scale), int(max_splits),
        int(num_ranges), _ptr(partial_o), _ptr(partial_lse), _stream(stream)))
    return partial_o, partial_lse


def paged_attn_decode_balanced_fused(q, cache: Cache, block_table, seq_lens,
                                     query_start_loc, softmax_scale, max_query_len,
                                     max_splits, workspace, num_ranges=0, out=None,
                                     lse_out=None, partial_o=None, partial_lse=None,
                                     k_scale=None, v_scale=None, stream=None):
    """Balanced-range decode and split merge in one launch
    (pkv_paged_attn_decode_balanced_fused).  `workspace`: a zero-filled int32
    CUDA tensor of at least decode_workspace_bytes(...) bytes, left zero by
    every call.  Returns (out [T, Hq, dv] bf16, lse_out or None)."""
    _attn_common(q, block_table, seq_lens, query_start_loc)
    T, Hq, _ = q.shape
    dv = cache.desc.head_size_v
    if partial_o is None:
        partial_o = torch.empty(max_splits, T, Hq, dv, dtype=torch.float32,
                                device=q.device)
    if partial_lse is None:
        partial_lse = torch.empty(max_splits, T, Hq, dtype=torch.float32,
                                  device=q.device)
    if out is None:
        out = torch.empty(T, Hq, dv, dtype=torch.bfloat16, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("pkv_paged_attn_decode_balanced_fused",
           _lib().pkv_paged_attn_decode_balanced_fused(
               _ptr(q), Hq, T, _ptr(cache.data), ctypes.byref(cache.desc),
               _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
               _ptr(query_start_loc), int(seq_lens.shape[0]), int(max_query_len),
               float(softmax_scale), _ptr(k_scale), _ptr(v_scale), int(max_splits),
               int(num_ranges), _ptr(partial_o), _ptr(partial_lse), _ptr(workspace),
               ws_bytes, _ptr(out), _ptr(lse_out), _stream(stream)))
    return out, lse_out


def decode_balanced_ranges(cache: Cache) -> int:
    """The range count pkv_paged_attn_decode_balanced uses for num_ranges=0."""
    r = _lib().pkv_decode_balanced_ranges(ctypes.byref(cache.desc))
    if r < 1:
        raise PkvError("pkv_decode_balanced_ranges", r)
    return r


def decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, max_query_len) -> int:
    return int(_lib().pkv_decode_workspace_bytes(int(num_seqs), int(num_q_heads),
                                                 int(num_kv_heads), int(max_query_len)))


def paged_attn_decode_fused(q, cache: Cache, block_table, seq_lens,
                            query_start_loc, softmax_scale, max_query_len,
                            num_splits, workspace, out=None, lse_out=None,
                            partial_o=None, partial_lse=None, k_scale=None,
                            v_scale=None, stream=None):
    """Decode and split merge in one launch (pkv_paged_attn_decode_fused).
    `workspace`: a zero-filled int32 (or byte) CUDA tensor of at least
    decode_workspace_bytes(...) bytes, left zero by every call.  Returns
    (out [T, Hq, dv] bf16, lse_out or None)."""
    _attn_common(q, block_table, seq_lens, query_start_loc)
    T, Hq, _ = q.shape
    dv = cache.desc.head_size_v
    if partial_o is None:
        partial_o = torch.empty(num_splits, T, Hq, dv, dtype=torch.float32,
                                device=q.device)
    if partial_lse is None:
        partial_lse = torch.empty(num_splits, T, Hq, dtype=torch.float32,
                                  device=q.device)
    if out is None:
        out = torch.empty(T, Hq, dv, dtype=torch.bfloat16, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("pkv_paged_attn_decode_fused", _lib().pkv_paged_attn_decode_fused(
        _ptr(q), Hq, T, _ptr(cache.data), ctypes.byref(cache.desc),
        _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
        _ptr(query_start_loc), int(seq_lens.shape[0]), int(max_query_len),
        float(softmax_scale), _ptr(k_scale), _ptr(v_scale), int(num_splits),
        _ptr(partial_o), _ptr(partial_lse), _ptr(workspace), ws_bytes,
        _ptr(out), _ptr(lse_out), _stream(stream)))
    return out, lse_out


NOALLOC_MAX_COUNTERS = 65536


def paged_attn_decode_fused_noalloc(q, cache: Cache, block_table, seq_lens,
                                    query_start_loc, softmax_scale, max_query_len,
                                    num_splits, out=None, lse_out=None,
                                    partial_o=None, partial_lse=None,
                                    k_scale=None, v_scale=None, stream=None):
    """paged_attn_decode_fused with the library's own fixed counter array
    (pkv_paged_attn_decode_fused_noalloc): no workspace argument, at most
    NOALLOC_MAX_COUNTERS counters, and calls that overlap in time race.
    Returns (out [T, Hq, dv] bf16, lse_out or None)."""
    _attn_common(q, block_table, seq_lens, query_start_loc)
    T, Hq, _ = q.shape
    dv = cache.desc.head_size_v
    if partial_o is None:
        partial_o = torch.empty(num_splits, T, Hq, dv, dtype=torch.float32,
                                device=q.device)
    if partial_lse is None:
        partial_lse = torch.empty(num_splits, T, Hq, dtype=torch.float32,
                                  device=q.device)
    if out is None:
        out = torch.empty(T, Hq, dv, dtype=torch.bfloat16, device=q.device)
    _check("pkv_paged_attn_decode_fused_noalloc",
           _lib().pkv_paged_attn_decode_fused_noalloc(
               _ptr(q), Hq, T, _ptr(cache.data), ctypes.byref(cache.desc),
               _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
               _ptr(query_start_loc), int(seq_lens.shape[0]), int(max_query_len),
               float(softmax_scale), _ptr(k_scale), _ptr(v_scale), int(num_splits),
               _ptr(partial_o), _ptr(partial_lse), _ptr(out), _ptr(lse_out),
               _stream(stream)))
    return out, lse_out


def splitkv_reduce(partial_o, partial_lse, out=None, lse_out=None,
                   stream=None, sinks=None):
    """partial_o [S, ..., dv] f32, partial_lse [S, ...] f32 -> out bf16
    [..., dv] (and lse_out f32 [...] when given).  ``sinks``: float32 [Hq]
    CUDA tensor of attention-sink logits, Hq the last dimension of the rows
    (pkv_splitkv_reduce_sink), or None."""
    assert partial_o.dtype == torch.float32 and partial_o.is_contiguous()
    assert partial_lse.dtype == torch.float32 and partial_lse.is_contiguous()
    S = partial_o.shape[0]
    dv = partial_o.shape[-1]
    rows = 1
    for n in partial_lse.shape[1:]:
        rows *= int(n)
    if out is None:
        out = torch.empty(*partial_o.shape[1:], dtype=torch.bfloat16,
                          device=partial_o.device)
    if sinks is None:
        _check("pkv_splitkv_reduce", _lib().pkv_splitkv_reduce(
            _ptr(partial_o), _ptr(partial_lse), S, rows, dv, _ptr(out),
            _ptr(lse_out), _stream(stream)))
    else:
        assert sinks.dtype == torch.float32 and sinks.is_contiguous()
        hq = int(sinks.shape[0])
        assert partial_lse.shape[-1] == hq
        _check("pkv_splitkv_reduce_sink", _lib().pkv_splitkv_reduce_sink(
            _ptr(partial_o), _ptr(partial_lse), S, rows, dv, _ptr(sinks), hq,
            _ptr(out), _ptr(lse_out), _stream(stream)))
    return out


def decode_suggest_splits(num_seqs, num_q_heads, num_kv_heads, max_query_len,
                          max_seq_len, block_size) -> int:
    r = _lib().pkv_decode_suggest_splits(num_seqs, num_q_heads, num_kv_heads,
                                         max_query_len, max_seq_len,
                                         block_size)
    if r < 1:
        raise PkvError("pkv_decode_suggest_splits", r)
    return r


def supports(head_size, head_size_v, dtype=BF16) -> int:
    return int(_lib().pkv_supports(head_size, head_size_v, dtype))


def get_device_error(stream=None) -> int:
    code = ctypes.c_int(0)
    _check("pkv_get_device_error",
           _lib().pkv_get_device_error(ctypes.byref(code), _stream(stream)))
    return code.value


def selftest_bounded_wait(limit_us: int, stream=None) -> None:
    """Runs the bounded-wait check (see pkv_selftest_bounded_wait); read
    the outcome with get_device_error()."""
    _check("pkv_selftest_bounded_wait",
           _lib().pkv_selftest_bounded_wait(int(limit_us), _stream(stream)))
