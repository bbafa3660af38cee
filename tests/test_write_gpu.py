"""Cache write on the GPU against the oracle: bit-exact, FP8 quantisation
included (vLLM PR #64064 "Tests": MiMo geometry, block sizes 16 and 64, both
layouts, bf16 and fp8 caches, per-tensor and per-head scales, slack past the
cache)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs

pytestmark = pytest.mark.gpu


def _case(layout, kv_dtype, scale_mode, block_size, T, seed=1):
    w = wl.make_workload("write", seq_lens=[T], q_lens=[T], layout=layout,
                         kv_dtype=kv_dtype, scale_mode=scale_mode,
                         block_size=block_size, extra_blocks=2, seed=seed)
    slots = w.slot_mapping_all().copy()
    if T > 3:
        slots[3] = -1   # a skipped (padding) token
    return w, slots


def _oracle_bytes(w, slots, fill=0xFF):
    exp = np.full(w.cache_bytes(), fill, dtype=np.uint8)
    oracle.kv_cache_write(refs.bf16_bits(w.k_ctx),
                          None if w.v_ctx is None else refs.bf16_bits(w.v_ctx),
                          slots, exp, refs.oracle_desc(w), w.k_scale, w.v_scale)
    return exp


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("block_size", [16, 64])
@pytest.mark.parametrize("kv", [(wl.BF16, wl.SCALE_NONE),
                                (wl.FP8, wl.SCALE_TENSOR),
                                (wl.FP8, wl.SCALE_HEAD)])
@pytest.mark.parametrize("T", [1, 29, 300])
def test_write_bit_exact_with_slack(layout, block_size, kv, T):
    w, slots = _case(layout, kv[0], kv[1], block_size, T)
    dw = wl.to_device(w)
    s = torch.from_numpy(slots).cuda()
    pkv.kv_cache_write(dw.k_ctx, dw.v_ctx, s, dw.cache, dw.k_scale, dw.v_scale)
    got = dw.cache_buf.cpu().numpy()
    exp = _oracle_bytes(w, slots)
    assert (got[:dw.slack] == 0xFF).all() and (got[-dw.slack:] == 0xFF).all()
    core = got[dw.slack:-dw.slack]
    bad = np.nonzero(core != exp)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_write_strided_sources_and_k_only():
    """K and V slices of a fused activation (own token and head strides), and
    the MLA form (value NULL: K only, V being a prefix of K)."""
    w, slots = _case(wl.NHD, wl.BF16, wl.SCALE_NONE, 16, 40)
    T = w.k_ctx.shape[0]
    g = torch.Generator().manual_seed(2)
    fused = torch.randn(T, 4 * 320 + 64, generator=g).to(torch.bfloat16)
    k = fused[:, :768].reshape(T, 4, 192)
    v = fused[:, 768 + 64:].reshape(T, 4, 128)
    w.k_ctx, w.v_ctx = k.contiguous(), v.contiguous()
    dw = wl.to_device(w)
    fd = fused.cuda()
    s = torch.from_numpy(slots).cuda()
    pkv.kv_cache_write(fd[:, :768].view(T, 4, 192), fd[:, 832:].view(T, 4, 128),
                       s, dw.cache)
    assert (dw.cache.data.cpu().numpy() == _oracle_bytes(w, slots)).all()
    # K only
    dw2 = wl.to_device(w)
    pkv.kv_cache_write(dw2.k_ctx, None, s, dw2.cache)
    exp = np.full(w.cache_bytes(), 0xFF, dtype=np.uint8)
    oracle.kv_cache_write(refs.bf16_bits(w.k_ctx), None, slots, exp,
                          refs.oracle_desc(w))
    assert (dw2.cache.data.cpu().numpy() == exp).all()


# Scales with exact and inexact reciprocals, the largest binary32
# significand below 2, powers of two at the ends of the range where the
# write divides through the corrected reciprocal (2^-60, 2^60), and scales
# outside it, where it divides directly (1e-30, 1e30).
@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.7e-3, 1.0 / 3.0, 0.3, 7.0,
                                   float(np.float32(1.9999999)), 2.0 ** -60,
                                   2.0 ** 60, 1e-30, 1e30])
def test_fp8_encode_every_bf16_pattern(scale):
    """All 65,536 bf16 bit patterns through the fp8 write, bit-exact against
    the oracle's E4M3 encoder (x / s divided in binary32); NaN inputs must
    give a NaN code on both sides (either sign)."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    H, dk, dv = 4, 192, 128
    per_tok = H * (dk + dv)
    T = (65536 + per_tok - 1) // per_tok
    flat = np.resize(pats, T * per_tok)
    kb = flat[:T * H * dk].reshape(T, H, dk)
    vb = flat[T * H * dk:].reshape(T, H, dv)
    w = wl.make_workload("enc", seq_lens=[T], q_lens=[T], kv_dtype=wl.FP8,
                         scale_mode=wl.SCALE_TENSOR, block_size=16, seed=3)
    w.k_ctx = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16)
    w.v_ctx = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16)
    w.k_scale = np.array([scale], np.float32)
    w.v_scale = np.array([scale], np.float32)
    slots = w.slot_mapping_all()
    dw = wl.to_device(w)
    pkv.kv_cache_write(dw.k_ctx, dw.v_ctx, dw.slots_all, dw.cache,
                       dw.k_scale, dw.v_scale)
    got = dw.cache.data.cpu().numpy()
    exp = _oracle_bytes(w, slots)
    nan_g = (got & 0x7F) == 0x7F
    nan_e = (exp & 0x7F) == 0x7F
    assert (nan_g == nan_e).all()
    assert (got[~nan_e] == exp[~nan_e]).all()


def test_write_full_size_32k():
    """The long-prefill write: 32,768 tokens, 4 KV heads, block 16."""
    w = wl.long_prefill(32768)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    exp = _oracle_bytes(w, w.slot_mapping_all())
    assert (dw.cache.data.cpu().numpy() == exp).all()


def test_out_of_range_slot_is_skipped_and_reported():
    w, slots = _case(wl.NHD, wl.BF16, wl.SCALE_NONE, 16, 20)
    slots[5] = w.num_blocks * w.block_size + 7     # past the cache
    dw = wl.to_device(w)
    gpu_path.device_error()                        # clear
    pkv.kv_cache_write(dw.k_ctx, dw.v_ctx, torch.from_numpy(slots).cuda(),
                       dw.cache)
    assert gpu_path.device_error() == pkv.EDEV_RANGE
    got = dw.cache_buf.cpu().numpy()
    assert (got[-dw.slack:] == 0xFF).all()
    slots2 = slots.copy()
    slots2[5] = -1
    exp = _oracle_bytes(w, slots2)
    assert (got[dw.slack:-dw.slack] == exp).all()


@pytest.mark.parametrize("kv", [(wl.BF16, wl.SCALE_NONE), (wl.FP8, wl.SCALE_HEAD),
                                (wl.FP8, wl.SCALE_TENSOR)])
def test_write_many_tokens_per_warp(kv):
    """More tokens than the launch has warps, so each warp strides over
    several tokens and loads the next one while it stores the current one;
    skipped (negative) slots sit among them.  Bit-exact with the oracle."""
    T = 20011
    w, slots = _case(wl.NHD, kv[0], kv[1], 16, T, seed=3)
    slots = slots.copy()
    slots[::7] = -1
    dw = wl.to_device(w)
    s = torch.from_numpy(slots).cuda()
    pkv.kv_cache_write(dw.k_ctx, dw.v_ctx, s, dw.cache, dw.k_scale, dw.v_scale)
    got = dw.cache_buf.cpu().numpy()
    exp = _oracle_bytes(w, slots)
    assert (got[:dw.slack] == 0xFF).all() and (got[-dw.slack:] == 0xFF).all()
    bad = np.nonzero(got[dw.slack:-dw.slack] != exp)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"
    assert gpu_path.device_error() == pkv.EDEV_NONE
