"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/pkv.h declares, and rejects bad arguments on the host before
anything is launched (the checks below never reach a CUDA call)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("pkv_kv_cache_write", "pkv_paged_attn_prefill",
              "pkv_paged_attn_decode", "pkv_splitkv_reduce"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) <= set(pkv.EXPORTED) | {"pkv_status_string"}


def test_supports_mirrors_v_le_k(lib):
    assert pkv.supports(192, 128) == 7
    assert pkv.supports(192, 128, pkv.FP8_E4M3) == 7   # FP8 prefill widens in the kernel
    assert pkv.supports(576, 512) == 5
    assert pkv.supports(128, 192) == 0                  # V wider than K
    assert pkv.supports(64, 64) == 1                    # write only


def _desc(**kw):
    base = dict(num_blocks=4)
    base.update(kw)
    return pkv.make_desc(**base)


DUMMY = ctypes.c_void_p(256)   # never dereferenced: validation fails first


def _write(lib, d, key=DUMMY, slots=DUMMY, cache=DUMMY, T=1, ks=None, vs=None,
           value=DUMMY):
    return lib.pkv_kv_cache_write(key, 192, 192 * 0 + 192, value, 128, 128,
                                  slots, T, cache,
                                  None if d is None else ctypes.byref(d),
                                  ks, vs, None)


def test_write_rejects_bad_arguments(lib):
    assert _write(lib, None) == pkv.EINVAL
    assert _write(lib, _desc(), key=None) == pkv.EINVAL
    assert _write(lib, _desc(), slots=None) == pkv.EINVAL
    assert _write(lib, _desc(), T=-1) == pkv.EINVAL
    assert _write(lib, _desc(dtype=7)) == pkv.EUNSUPPORTED
    assert _write(lib, _desc(layout=5)) == pkv.EUNSUPPORTED
    assert _write(lib, _desc(v_off=250)) == pkv.EINVAL        # V past the row
    assert _write(lib, _desc(dtype=pkv.FP8_E4M3,
                             scale_mode=pkv.SCALE_HEAD)) == pkv.EINVAL  # no scales
    assert _write(lib, _desc(scale_mode=pkv.SCALE_TENSOR)) == pkv.EINVAL
    assert _write(lib, _desc(), T=0) == pkv.OK                # nothing to do


def _decode(lib, d, **kw):
    a = dict(q=DUMMY, Hq=16, T=4, cache=DUMMY, bt=DUMMY, mb=4, sl=DUMMY,
             qsl=DUMMY, B=2, mq=1, scale=0.1, ks=None, vs=None, S=4,
             po=DUMMY, pl=DUMMY)
    a.update(kw)
    return lib.pkv_paged_attn_decode(
        a["q"], a["Hq"], a["T"], a["cache"],
        None if d is None else ctypes.byref(d), a["bt"], a["mb"], a["sl"],
        a["qsl"], a["B"], a["mq"], ctypes.c_float(a["scale"]), a["ks"],
        a["vs"], a["S"], a["po"], a["pl"], None)


def test_decode_rejects_bad_arguments(lib):
    d = _desc()
    assert _decode(lib, None) == pkv.EINVAL
    assert _decode(lib, _desc(head_size=128, head_size_v=192, v_off=128,
                              row_elems=320)) == pkv.EUNSUPPORTED  # v > k
    assert _decode(lib, d, Hq=15) == pkv.EINVAL          # Hq % Hkv
    assert _decode(lib, d, S=0) == pkv.EINVAL
    assert _decode(lib, d, mq=0) == pkv.EINVAL
    assert _decode(lib, d, mq=65) == pkv.EINVAL
    assert _decode(lib, d, po=None) == pkv.EINVAL
    assert _decode(lib, d, bt=None) == pkv.EINVAL
    assert _decode(lib, d, scale=float("nan")) == pkv.EINVAL
    assert _decode(lib, _desc(head_size=64, head_size_v=64, row_elems=128,
                              v_off=64)) == pkv.EUNSUPPORTED
    assert _decode(lib, _desc(dtype=pkv.FP8_E4M3,
                              scale_mode=pkv.SCALE_TENSOR)) == pkv.EINVAL
    assert _decode(lib, d, T=0) == pkv.OK


def _fused(lib, d, **kw):
    a = dict(q=DUMMY, Hq=16, T=4, cache=DUMMY, bt=DUMMY, mb=4, sl=DUMMY,
             qsl=DUMMY, B=2, mq=1, scale=0.1, ks=None, vs=None, S=4,
             po=DUMMY, pl=DUMMY, ws=DUMMY, nws=1 << 20, out=DUMMY)
    a.update(kw)
    return lib.pkv_paged_attn_decode_fused(
        a["q"], a["Hq"], a["T"], a["cache"], ctypes.byref(d), a["bt"], a["mb"], a["sl"],
        a["qsl"], a["B"], a["mq"], ctypes.c_float(a["scale"]), a["ks"], a["vs"], a["S"],
        a["po"], a["pl"], a["ws"], ctypes.c_size_t(a["nws"]), a["out"], None, None)


def test_decode_rejects_misaligned_partials(lib):
    d = _desc()
    odd4 = ctypes.c_void_p(256 + 2)    # not even float-aligned
    assert _decode(lib, d, po=odd4) == pkv.EINVAL
    assert _decode(lib, d, pl=odd4) == pkv.EINVAL
    # the fused merge reads the partials 16 bytes at a time and stores 4 bf16
    # at a time; with no sequence the call stops after these checks
    assert _fused(lib, d, B=0, po=ctypes.c_void_p(256 + 4)) == pkv.EINVAL
    assert _fused(lib, d, B=0, out=ctypes.c_void_p(256 + 4)) == pkv.EINVAL
    assert _fused(lib, d, B=0) == pkv.OK
    assert _fused(lib, d, B=0, T=1 << 28, Hq=16) == pkv.EINVAL   # rows past int


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="a valid call would launch on the dummy pointers")
def test_valid_shapes_pass_the_host_checks(lib):
    """The shapes the GPU tests and the bench launch pass every host check:
    without a GPU they end at the device query (PKV_ECUDA), not at a
    rejection."""
    bf = _desc(num_blocks=4096)
    f8 = _desc(num_blocks=4096, block_size=64, dtype=pkv.FP8_E4M3,
               scale_mode=pkv.SCALE_HEAD)
    mla = _desc(num_blocks=4096, block_size=64, num_kv_heads=1, row_elems=576,
                head_size=576, v_off=0, head_size_v=512)
    assert _decode(lib, bf, T=32, B=32, mb=512, S=16) == pkv.ECUDA      # batched decode
    assert _decode(lib, f8, T=96, B=24, mb=800, mq=4, S=16, ks=DUMMY,
                   vs=DUMMY) == pkv.ECUDA                                # FP8 verify
    assert _decode(lib, mla, Hq=16, T=1, B=1, mb=1600, S=304) == pkv.ECUDA   # MLA
    assert _fused(lib, bf, T=32, B=32, mb=512, S=16) == pkv.ECUDA


def _balanced(lib, d, W=0, **kw):
    a = dict(q=DUMMY, Hq=16, T=4, cache=DUMMY, bt=DUMMY, mb=4, sl=DUMMY, qsl=DUMMY,
             B=1, mq=1, scale=0.1, ks=None, vs=None, S=4, po=DUMMY, pl=DUMMY)
    a.update(kw)
    return lib.pkv_paged_attn_decode_balanced(
        a["q"], a["Hq"], a["T"], a["cache"], ctypes.byref(d), a["bt"], a["mb"], a["sl"],
        a["qsl"], a["B"], a["mq"], ctypes.c_float(a["scale"]), a["ks"], a["vs"], a["S"],
        W, a["po"], a["pl"], None)


def test_balanced_decode_rejects_bad_arguments(lib):
    d = _desc()
    assert _balanced(lib, d, W=-1) == pkv.EINVAL
    assert _balanced(lib, d, W=(1 << 24) + 1) == pkv.EINVAL
    assert _balanced(lib, d, B=16385) == pkv.EUNSUPPORTED    # more than 128 x 128 sequences
    assert _balanced(lib, d, B=64, mb=1 << 26) == pkv.EINVAL  # page line past int
    assert _balanced(lib, d, S=0) == pkv.EINVAL
    assert _balanced(lib, d, po=None) == pkv.EINVAL
    assert _balanced(lib, d, T=0) == pkv.OK
    assert lib.pkv_decode_balanced_ranges(None) == pkv.EINVAL
    assert lib.pkv_decode_balanced_ranges(ctypes.byref(_desc(
        head_size=64, head_size_v=64, row_elems=128, v_off=64))) == pkv.EUNSUPPORTED


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="a valid call would launch on the dummy pointers")
def test_balanced_shapes_pass_the_host_checks(lib):
    bf = _desc(num_blocks=4096)
    assert _balanced(lib, bf, T=32, B=32, mb=512, S=16) == pkv.ECUDA
    assert _balanced(lib, bf, W=152, T=128, B=128, mb=512, S=16) == pkv.ECUDA
    assert _balanced(lib, bf, T=16384, B=16384, mb=8, S=16) == pkv.ECUDA   # wide batch


def test_prefill_rejects_bad_arguments(lib):
    def call(d, **kw):
        a = dict(q=DUMMY, Hq=16, T=4, scale=0.1, out=DUMMY)
        a.update(kw)
        return lib.pkv_paged_attn_prefill(
            a["q"], a["Hq"], a["T"], DUMMY, ctypes.byref(d), DUMMY, 4, DUMMY,
            DUMMY, 1, ctypes.c_float(a["scale"]), None, None, a["out"], None)
    assert call(_desc(), scale=-1.0) == pkv.EINVAL
    assert call(_desc(), out=None) == pkv.EINVAL
    assert call(_desc(block_size=12)) == pkv.EUNSUPPORTED
    assert call(_desc(), Hq=12 * 4 * 3) in (pkv.EUNSUPPORTED,)  # G = 36
    assert call(_desc(dtype=pkv.FP8_E4M3, scale_mode=pkv.SCALE_HEAD)) == \
        pkv.EINVAL   # scales missing


def test_reduce_rejects_bad_arguments(lib):
    f = lib.pkv_splitkv_reduce
    assert f(DUMMY, DUMMY, -1, 4, 128, DUMMY, None, None) == pkv.EINVAL
    assert f(DUMMY, DUMMY, 2, 4, 0, DUMMY, None, None) == pkv.EINVAL
    assert f(None, DUMMY, 2, 4, 128, DUMMY, None, None) == pkv.EINVAL
    assert f(DUMMY, DUMMY, 2, 4, 128, None, None, None) == pkv.EINVAL
    assert f(DUMMY, DUMMY, 2, 0, 128, None, None, None) == pkv.OK


def test_reduce_sink_rejects_bad_arguments(lib):
    f = lib.pkv_splitkv_reduce_sink
    # rows (6) not a multiple of the query heads (4); no query heads
    assert f(DUMMY, DUMMY, 2, 6, 128, DUMMY, 4, DUMMY, None, None) == pkv.EINVAL
    assert f(DUMMY, DUMMY, 2, 8, 128, DUMMY, 0, DUMMY, None, None) == pkv.EINVAL
    assert f(DUMMY, DUMMY, -1, 8, 128, DUMMY, 4, DUMMY, None, None) == pkv.EINVAL
    assert f(None, DUMMY, 2, 8, 128, DUMMY, 4, DUMMY, None, None) == pkv.EINVAL
    assert f(DUMMY, DUMMY, 2, 8, 128, DUMMY, 4, None, None, None) == pkv.EINVAL
    assert f(DUMMY, DUMMY, 2, 0, 128, DUMMY, 4, None, None, None) == pkv.OK


def test_prefill_fp8_rejects_bad_arguments(lib):
    d8 = _desc(dtype=pkv.FP8_E4M3, scale_mode=pkv.SCALE_HEAD)

    def call(d, ks=DUMMY, vs=DUMMY, **kw):
        a = dict(q=DUMMY, Hq=16, T=4, scale=0.1, out=DUMMY)
        a.update(kw)
        return lib.pkv_paged_attn_prefill(
            a["q"], a["Hq"], a["T"], DUMMY, ctypes.byref(d), DUMMY, 4, DUMMY,
            DUMMY, 1, ctypes.c_float(a["scale"]), ks, vs, a["out"], None)
    assert call(d8, ks=None) == pkv.EINVAL                   # scales missing
    assert call(d8, vs=None) == pkv.EINVAL
    assert call(d8, scale=-1.0) == pkv.EINVAL
    assert call(d8, out=None) == pkv.EINVAL
    assert call(_desc(dtype=pkv.FP8_E4M3, scale_mode=pkv.SCALE_HEAD,
                      v_off=200, row_elems=328)) == pkv.EUNSUPPORTED  # V not on 16 bytes
    assert call(d8, T=0) == pkv.OK                           # nothing to do


def test_prefill_fp8_workspace_size(lib):
    d8 = _desc(dtype=pkv.FP8_E4M3, scale_mode=pkv.SCALE_HEAD)   # block 16, 4 heads, row 320
    f = lib.pkv_prefill_fp8_workspace_bytes
    f.restype = ctypes.c_size_t
    page = 16 * 4 * 320 * 2
    n = f(3, 5, ctypes.byref(d8))
    pages = (3 * 5 * page + 255) // 256 * 256
    assert n == pages + 3 * 5 * 4       # widened pages, then the remapped table
    assert f(3, 0, ctypes.byref(d8)) == 0
    assert f(-1, 5, ctypes.byref(d8)) == 0
    assert f(3, 5, None) == 0


def test_prefill_fp8_two_pass_rejects_bad_arguments(lib):
    d8 = _desc(dtype=pkv.FP8_E4M3, scale_mode=pkv.SCALE_HEAD)
    f = lib.pkv_prefill_fp8_workspace_bytes
    f.restype = ctypes.c_size_t
    need = f(1, 4, ctypes.byref(d8))
    WS = ctypes.c_void_p(1 << 20)       # 256-byte aligned, never dereferenced

    def call(d, ws=WS, nbytes=need, ks=DUMMY, vs=DUMMY, **kw):
        a = dict(q=DUMMY, Hq=16, T=4, scale=0.1, out=DUMMY)
        a.update(kw)
        return lib.pkv_paged_attn_prefill_fp8(
            a["q"], a["Hq"], a["T"], DUMMY, ctypes.byref(d), DUMMY, 4, DUMMY,
            DUMMY, 1, ctypes.c_float(a["scale"]), ks, vs, None, ws,
            ctypes.c_size_t(nbytes), a["out"], None)
    assert call(_desc()) == pkv.EINVAL                       # a bf16 cache
    assert call(d8, ks=None) == pkv.EINVAL                   # scales missing
    assert call(d8, ws=None) == pkv.EINVAL                   # no workspace
    assert call(d8, nbytes=need - 1) == pkv.EINVAL           # too small
    assert call(d8, ws=ctypes.c_void_p((1 << 20) + 16)) == pkv.EINVAL  # misaligned
    assert call(d8, scale=-1.0) == pkv.EINVAL
    assert call(d8, out=None) == pkv.EINVAL
    assert call(d8, T=0) == pkv.OK                           # nothing to do


def test_status_strings(lib):
    for s in (pkv.OK, pkv.EINVAL, pkv.EUNSUPPORTED, pkv.ECUDA):
        assert lib.pkv_status_string(s)
