"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- the E4M3 format definition and torch's own float8 conversion, a
per-slot closed form of the cache write, a dense brute-force softmax
attention in numpy, closed-form special cases, and invariants.  A plausible
mistake anywhere in the oracle (a dropped term, a wrong sign, a wrong index,
a transposed operand, the pre-fix V addressing) fails at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import refs


# ------------------------------------------------------------------ E4M3 --

def test_e4m3_decode_spot_values():
    # From the E4M3 definition: bias 7, 3 mantissa bits, no inf, S.1111.111
    # is NaN, max 448, subnormal step 2^-9.
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x40) == 2.0
    assert oracle.e4m3_decode(0x3C) == 1.5
    assert oracle.e4m3_decode(0x00) == 0.0
    assert math.copysign(1.0, oracle.e4m3_decode(0x80)) == -1.0
    assert math.isnan(oracle.e4m3_decode(0x7F))
    assert math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_e4m3_roundtrip_every_code():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_e4m3_midpoints_round_to_even():
    for c in range(0, 0x7E):   # positive finite neighbours (c, c+1)
        a, b = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((a + b) / 2)        # exact in binary32
        assert float(mid) == (a + b) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == even, hex(c)
        assert oracle.e4m3_encode(-float(mid)) == 0x80 | even
        # a hair either side of the midpoint goes to the nearer code
        lo = np.nextafter(mid, np.float32(-np.inf))
        hi = np.nextafter(mid, np.float32(np.inf))
        assert oracle.e4m3_encode(float(lo)) == c
        assert oracle.e4m3_encode(float(hi)) == c + 1


def test_e4m3_saturation_and_nan():
    assert oracle.e4m3_encode(448.0 * (1 + 2.0 ** -4)) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(-500.0) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00     # below half the step
    assert oracle.e4m3_encode(-2.0 ** -11) == 0x80


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([
        torch.randn(4000, generator=g) * 100,
        torch.randn(2000, generator=g) * 1e-2,        # subnormal range
        (torch.rand(2000, generator=g) * 2 - 1) * 464,
    ]).float()
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(x.numpy())
    assert (got == ref).all()


# ----------------------------------------------------------- cache write --

def _write_case(layout, kv_dtype, scale_mode, block_size, T=29, seed=1):
    w = wl.make_workload("write", seq_lens=[T], q_lens=[T], layout=layout,
                         kv_dtype=kv_dtype, scale_mode=scale_mode,
                         block_size=block_size, extra_blocks=2, seed=seed)
    slots = w.slot_mapping_all().copy()
    slots[3] = -1          # a skipped (padding) token
    return w, slots


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("block_size", [16, 64])
def test_write_bf16_closed_form(layout, block_size):
    w, slots = _write_case(layout, wl.BF16, wl.SCALE_NONE, block_size)
    kb, vb = refs.bf16_bits(w.k_ctx), refs.bf16_bits(w.v_ctx)
    base = np.full(w.cache_bytes(), refs.SENTINEL, dtype=np.uint8)
    got = base.copy()
    oracle.kv_cache_write(kb, vb, slots, got, refs.oracle_desc(w))
    exp = refs.expected_cache_closed_form(w, kb, vb, slots, base)
    assert (got == exp).all()
    # V occupies columns [192, 320) of each written row
    rows = got.view(np.uint16).reshape(-1, w.row_elems)
    t = 5
    blk, off = divmod(int(slots[t]), block_size)
    for h in range(w.num_kv_heads):
        r = (blk * block_size + off) * 4 + h if layout == wl.NHD else \
            (blk * 4 + h) * block_size + off
        assert (rows[r, 192:320] == vb[t, h]).all()
        assert (rows[r, 0:192] == kb[t, h]).all()


def test_write_strided_sources():
    """K and V read with their own token and head strides (e.g. slices of a
    fused QKV activation)."""
    w, slots = _write_case(wl.NHD, wl.BF16, wl.SCALE_NONE, 16)
    T = w.k_ctx.shape[0]
    fused = torch.randn(T, 4 * (192 + 128) + 40, generator=torch.Generator()
                        .manual_seed(9)).to(torch.bfloat16)
    fb = refs.bf16_bits(fused)
    kview = fb[:, :4 * 192].reshape(T, 4, 192)
    vview = fb[:, 4 * 192 + 40:].reshape(T, 4, 128)
    got = np.full(w.cache_bytes(), refs.SENTINEL, dtype=np.uint8)
    oracle.kv_cache_write(fb, fb[:, 4 * 192 + 40:], slots, got,
                          refs.oracle_desc(w),
                          key_strides=(fb.shape[1], 192),
                          value_strides=(fb.shape[1], 128))
    base = np.full(w.cache_bytes(), refs.SENTINEL, dtype=np.uint8)
    exp = refs.expected_cache_closed_form(w, kview, vview, slots, base)
    assert (got == exp).all()


def test_write_detects_prefix_v_addressing():
    """Plant the pre-fix addressing of vLLM PR #64064 "Details" (V read and
    written with K's head stride and K's width) in a CPU writer and check
    that the byte comparison with slack past the cache catches it."""
    w, slots = _write_case(wl.NHD, wl.BF16, wl.SCALE_NONE, 16)
    kb, vb = refs.bf16_bits(w.k_ctx), refs.bf16_bits(w.v_ctx)
    slack = 4096
    base = np.full(w.cache_bytes() + slack, refs.SENTINEL, dtype=np.uint8)
    good = base.copy()
    oracle.kv_cache_write(kb, vb, slots, good[:w.cache_bytes()],
                          refs.oracle_desc(w))
    bad = base.copy().view(np.uint16)
    vflat = np.concatenate([vb.reshape(-1),
                            np.zeros(vb.size, np.uint16)])  # reads past V
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), 16)
        for h in range(4):
            row = ((blk * 16 + off) * 4 + h) * 320
            bad[row:row + 192] = kb[t, h]
            src = (t * 4 + h) * 192             # K's head stride for V
            bad[row + 192: row + 192 + 192] = vflat[src:src + 192]  # K's width
    assert not (bad.view(np.uint8) == good).all()
    # the last slot's overrun reaches the slack past the cache
    last = max(int(s) for s in slots)
    if last == w.num_blocks * 16 - 1:
        assert (bad.view(np.uint8)[w.cache_bytes():] != refs.SENTINEL).any()


@pytest.mark.parametrize("scale_mode", [wl.SCALE_TENSOR, wl.SCALE_HEAD])
@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
def test_write_fp8_matches_torch_conversion(scale_mode, layout):
    w, slots = _write_case(layout, wl.FP8, scale_mode, 64)
    kb, vb = refs.bf16_bits(w.k_ctx), refs.bf16_bits(w.v_ctx)
    got = np.full(w.cache_bytes(), refs.SENTINEL, dtype=np.uint8)
    oracle.kv_cache_write(kb, vb, slots, got, refs.oracle_desc(w),
                          w.k_scale, w.v_scale)
    per_head = scale_mode == wl.SCALE_HEAD
    ks = torch.from_numpy(w.k_scale).view(1, -1, 1) if per_head else \
        torch.from_numpy(w.k_scale).view(1, 1, 1)
    vs = torch.from_numpy(w.v_scale).view(1, -1, 1) if per_head else \
        torch.from_numpy(w.v_scale).view(1, 1, 1)
    kc = (w.k_ctx.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (w.v_ctx.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
    exp = np.full(w.cache_bytes(), refs.SENTINEL, dtype=np.uint8)
    R, bs = w.row_elems, w.block_size
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        for h in range(4):
            row = (((blk * bs + off) * 4 + h) if layout == wl.NHD else
                   ((blk * 4 + h) * bs + off)) * R
            exp[row:row + 192] = kc[t, h].numpy()
            exp[row + 192:row + 320] = vc[t, h].numpy()
    assert (got == exp).all()


# -------------------------------------------------------------- attention --

def _cases():
    yield wl.tiny("decode")
    yield wl.tiny("prefill")
    yield wl.tiny("prefill", layout=wl.HND)
    yield wl.make_workload("verify-small", seq_lens=[70, 0, 130, 3],
                           q_lens=[4, 4, 4, 4], block_size=64,
                           kv_dtype=wl.FP8, scale_mode=wl.SCALE_HEAD, seed=4)
    yield wl.make_workload("mla-small", seq_lens=[90, 33], q_lens=[1, 1],
                           num_q_heads=12, num_kv_heads=1, head_size=576,
                           head_size_v=512, block_size=64, v_aliases_k=True,
                           softmax_scale=1 / 24, seed=5)
    yield wl.make_workload("chunked", seq_lens=[50, 40], q_lens=[20, 3],
                           block_size=16, seed=6)


@pytest.mark.parametrize("w", list(_cases()), ids=lambda w: w.name)
def test_attention_matches_dense_bruteforce(w):
    cache = refs.oracle_cache(w)
    got, lse = refs.oracle_attn(w, cache)
    ref, rlse = refs.dense_attention(w)
    assert np.allclose(got, ref, atol=1e-11, rtol=1e-9)
    fin = np.isfinite(rlse)
    assert (np.isfinite(lse) == fin).all()
    assert np.allclose(lse[fin], rlse[fin], atol=1e-10)
    assert (got[~fin] == 0).all()


def test_single_visible_key_returns_that_value():
    w = wl.make_workload("one", seq_lens=[1, 1], q_lens=[1, 1], seed=7)
    cache = refs.oracle_cache(w)
    got, _ = refs.oracle_attn(w, cache)
    V = w.v_ctx.double().numpy()
    for b in range(2):
        for h in range(16):
            assert (got[b, h] == V[b, h // 4]).all()


def test_zero_query_gives_mean_of_visible_values():
    w = wl.make_workload("zq", seq_lens=[41], q_lens=[3], seed=8)
    w.q.zero_()
    cache = refs.oracle_cache(w)
    got, lse = refs.oracle_attn(w, cache)
    V = w.v_ctx.double().numpy()
    for i in range(3):
        n_vis = 41 - 3 + i + 1
        for h in range(16):
            assert np.allclose(got[i, h], V[:n_vis, h // 4].mean(0),
                               atol=1e-14, rtol=1e-12)
            assert abs(lse[i, h] - math.log(n_vis)) < 1e-12


def test_shared_value_rows_give_that_value():
    w = wl.make_workload("shv", seq_lens=[77], q_lens=[2], seed=9)
    w.v_ctx[:] = w.v_ctx[0:1]
    cache = refs.oracle_cache(w)
    got, _ = refs.oracle_attn(w, cache)
    V0 = w.v_ctx[0].double().numpy()
    for h in range(16):
        assert np.allclose(got[:, h], V0[h // 4][None], atol=1e-14)


def test_score_shift_invariance():
    """A constant key column makes q[d0] add the same amount to every score of
    the row; the output must not change."""
    w = wl.make_workload("shift", seq_lens=[60], q_lens=[5], seed=10)
    w.k_ctx[:, :, 7] = 1.0
    w.q[:, :, 7] = 0.0
    cache = refs.oracle_cache(w)
    a, la = refs.oracle_attn(w, cache)
    w.q[:, :, 7] = 3.0
    b, lb = refs.oracle_attn(w, cache)
    assert np.allclose(a, b, atol=1e-12)
    assert np.allclose(lb - la, 3.0 * float(np.float32(w.softmax_scale)),
                       atol=1e-12)


def test_page_permutation_bit_identical():
    w = wl.make_workload("perm", seq_lens=[70, 33], q_lens=[2, 1],
                         extra_blocks=5, seed=11)
    cache = refs.oracle_cache(w)
    a, la = refs.oracle_attn(w, cache)
    rng = np.random.default_rng(0)
    newpos = rng.permutation(w.num_blocks)
    w2 = wl.make_workload("perm", seq_lens=[70, 33], q_lens=[2, 1],
                          extra_blocks=5, seed=11)
    w2.block_table = np.where(w.block_table >= 0,
                              newpos[np.maximum(w.block_table, 0)], -1
                              ).astype(np.int32)
    cache2 = refs.oracle_cache(w2)
    b, lb = refs.oracle_attn(w2, cache2)
    assert (a == b).all() and (la == lb).all()


def test_gqa_head_mapping():
    """Query head h reads KV head h // G: changing KV head 2 changes exactly
    query heads 8..11."""
    w = wl.make_workload("gqa", seq_lens=[30], q_lens=[1], seed=12)
    a, _ = refs.oracle_attn(w, refs.oracle_cache(w))
    w.v_ctx[:, 2] += 1.0
    b, _ = refs.oracle_attn(w, refs.oracle_cache(w))
    changed = np.abs(a - b).max(axis=2)[0] > 0
    assert list(np.nonzero(changed)[0]) == [8, 9, 10, 11]


def test_zero_padded_heads_leave_real_heads_unchanged():
    """vLLM PR #50371 "Purpose": 12 query heads padded to 16 with zero heads;
    the first 12 outputs must be those of the 12-head run."""
    kw = dict(seq_lens=[150, 64], q_lens=[1, 1], num_kv_heads=1,
              head_size=576, head_size_v=512, block_size=64,
              v_aliases_k=True, softmax_scale=1 / 24, seed=13)
    w12 = wl.make_workload("m12", num_q_heads=12, **kw)
    w16 = wl.make_workload("m16", num_q_heads=12, pad_q_heads=4, **kw)
    assert w16.num_q_heads == 16 and (w16.q[:, 12:] == 0).all()
    a, la = refs.oracle_attn(w12, refs.oracle_cache(w12))
    b, lb = refs.oracle_attn(w16, refs.oracle_cache(w16))
    assert (a == b[:, :12]).all() and (la == lb[:, :12]).all()
    # the padded heads see a zero query: mean of the visible values
    V = w16.k_ctx.double().numpy()[:, 0, :512]
    assert np.allclose(b[0, 12], V[:150].mean(0), atol=1e-13)


def test_rows_without_keys_are_zero_not_nan():
    """MiMo model card "Update 2026-10-01": padded CUDA-graph rows (no visible
    key) give 0."""
    w = wl.verify_fp8(n_real=2, n_pad=3, ctx=200)
    cache = refs.oracle_cache(w)
    got, lse = refs.oracle_attn(w, cache)
    pad_rows = slice(8, 20)
    assert (got[pad_rows] == 0).all()
    assert np.isneginf(lse[pad_rows]).all()
    assert np.isfinite(got).all()


# --------------------------------------------------- split-KV and the merge --

@pytest.mark.parametrize("S", [1, 2, 3, 16, 96])
def test_split_partials_merge_to_whole(S):
    w = wl.make_workload("split", seq_lens=[300, 17, 0], q_lens=[4, 4, 4],
                         block_size=16, seed=14)
    cache = refs.oracle_cache(w)
    whole, wl_lse = refs.oracle_attn(w, cache)
    po = np.zeros((S,) + whole.shape, np.float32)
    pl = np.zeros((S,) + wl_lse.shape, np.float32)
    for s in range(S):
        o, l = refs.oracle_attn(w, cache, num_splits=S, split=s)
        po[s], pl[s] = o, l
        assert np.isfinite(o).all()
    T, H, dv = whole.shape
    out, lse = oracle.splitkv_reduce(po.reshape(S, T * H, dv),
                                     pl.reshape(S, T * H))
    assert np.allclose(out.reshape(whole.shape), whole, atol=1e-6, rtol=1e-6)
    fin = np.isfinite(wl_lse.reshape(-1))
    assert (np.isfinite(lse) == fin).all()
    assert np.allclose(lse[fin], wl_lse.reshape(-1)[fin], atol=1e-5)
    assert (out[~fin] == 0).all()


def test_split_segments_partition_the_keys():
    """Segment s covers pages [s*pps, min((s+1)*pps, P)): the segments'
    visible-key counts sum to the row's n_vis (checked via exp(lse) with a
    zero query, where lse = log(count))."""
    w = wl.make_workload("cnt", seq_lens=[211], q_lens=[3], block_size=16,
                         seed=15)
    w.q.zero_()
    cache = refs.oracle_cache(w)
    for S in (1, 4, 5, 14, 20):
        tot = np.zeros(3)
        for s in range(S):
            _, l = refs.oracle_attn(w, cache, num_splits=S, split=s)
            tot += np.where(np.isfinite(l[:, 0]), np.exp(l[:, 0]), 0)
        assert np.allclose(tot, [209, 210, 211])


def test_reduce_closed_forms():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((3, 5, 8)).astype(np.float32)
    # one split: identity
    out, lse = oracle.splitkv_reduce(o[:1], np.full((1, 5), 0.5, np.float32))
    assert np.allclose(out, o[0]) and np.allclose(lse, 0.5)
    # equal lse: arithmetic mean, lse + log(S)
    out, lse = oracle.splitkv_reduce(o, np.zeros((3, 5), np.float32))
    assert np.allclose(out, o.mean(0), atol=1e-7)
    assert np.allclose(lse, math.log(3))
    # weights exp(lse): split 1 dominates by e^30
    pl = np.array([[0.0] * 5, [30.0] * 5, [-np.inf] * 5], np.float32)
    o2 = o.copy()
    o2[2] = np.nan          # an empty segment's o is never read
    out, lse = oracle.splitkv_reduce(o2, pl)
    w0, w1 = math.exp(-30), 1.0
    assert np.allclose(out, (w0 * o[0] + w1 * o[1]) / (w0 + w1), atol=1e-7)
    # every segment empty: 0, lse -inf, no NaN
    out, lse = oracle.splitkv_reduce(o2, np.full((3, 5), -np.inf, np.float32))
    assert (out == 0).all() and np.isneginf(lse).all()


# ------------------------------------------ segment boundaries, by example --

def _segment_key_counts(w, S, W=0):
    """Visible keys of each segment for each query row: with a zero query
    every score is 0 and a segment's lse is log(its key count) exactly."""
    w.q.zero_()
    cache = refs.oracle_cache(w)
    rows = []
    for s in range(S):
        _, l = refs.oracle_attn(w, cache, num_splits=S, split=s, split_ranges=W)
        c = np.where(np.isfinite(l[:, 0]), np.exp(l[:, 0]), 0.0)
        rows.append(np.rint(c).astype(int))
        assert np.allclose(c, rows[-1], atol=1e-9)
    return np.stack(rows, 1)   # [token, segment]


def test_equal_segments_closed_form():
    """211 keys in pages of 16 are 14 pages; 5 segments of ceil(14 / 5) = 3
    pages hold 3, 3, 3, 3 and 2 pages, i.e. 48, 48, 48, 48 and the last 19
    keys.  50 keys (4 pages) over 8 segments: one page each, then 4 empty
    ones."""
    w = wl.make_workload("seg", seq_lens=[211], q_lens=[1], seed=30)
    assert _segment_key_counts(w, 5).tolist() == [[48, 48, 48, 48, 19]]
    w = wl.make_workload("seg", seq_lens=[50], q_lens=[1], seed=30)
    assert _segment_key_counts(w, 8).tolist() == [[16, 16, 16, 2, 0, 0, 0, 0]]


def test_balanced_ranges_closed_forms():
    """Balanced ranges, worked by hand.  Keys 100, 50, 30 in pages of 10 are
    10, 5 and 3 pages, laid end to end at global pages 0, 10 and 15 (18 in
    all)."""
    kw = dict(seq_lens=[100, 50, 30], q_lens=[1, 1, 1], block_size=10, seed=31)
    # W = 4: R = ceil(18 / 4) = 5 (Rmin = floor(8 / 3) + 1 = 3); ranges
    # [0,5) [5,10) [10,15) [15,18): sequence 0 is two ranges of 50 keys,
    # sequences 1 and 2 one range each
    w = wl.make_workload("bal", **kw)
    assert _segment_key_counts(w, 4, W=4).tolist() == [
        [50, 50, 0, 0], [50, 0, 0, 0], [30, 0, 0, 0]]
    # W = 3: R = 6; ranges [0,6) [6,12) [12,18): sequence 0 takes 6 + 4
    # pages, sequence 1 (pages 10..14) 2 pages of range 1 and 3 of range 2,
    # sequence 2 the last 3 pages of range 2
    w = wl.make_workload("bal", **kw)
    assert _segment_key_counts(w, 4, W=3).tolist() == [
        [60, 40, 0, 0], [20, 30, 0, 0], [30, 0, 0, 0]]
    # W = 1: one range, one segment per sequence
    w = wl.make_workload("bal", **kw)
    assert _segment_key_counts(w, 4, W=1).tolist() == [
        [100, 0, 0, 0], [50, 0, 0, 0], [30, 0, 0, 0]]


def test_balanced_ranges_keep_within_max_splits():
    """One long and one short sequence with many ranges asked for: keys 1000
    and 10 in pages of 10 are 100 + 1 pages.  W = 101 would give R = 1, but
    with at most 4 segments per sequence R grows to Rmin = floor(98 / 3) + 1
    = 33: ranges [0,33) [33,66) [66,99) [99,132).  The short sequence (global
    page 100) lies in range 3, its segment 0.  With 1 segment allowed, R is
    the whole line."""
    kw = dict(seq_lens=[1000, 10], q_lens=[1, 1], block_size=10, seed=32)
    w = wl.make_workload("cap", **kw)
    assert _segment_key_counts(w, 4, W=101).tolist() == [
        [330, 330, 330, 10], [10, 0, 0, 0]]
    w = wl.make_workload("cap", **kw)
    assert _segment_key_counts(w, 1, W=101).tolist() == [[1000], [10]]


def test_balanced_ranges_causal_rows_and_empty_sequences():
    """Rows of a 3-token query see 209, 210 and 211 keys; empty sequences
    (seq_len 0) hold no page and have no segment.  Keys 211 (14 pages of 16),
    0, 40 (3 pages), 0: 17 pages; W = 4 gives R = 5 (Rmin = floor(12 / 4) + 1
    = 4).  Sequence 0: ranges [0,5) [5,10) [10,15) -> 80, 80 and the rest
    (4 pages: 51, 50, 49 keys for its three rows); sequence 2 (global pages
    14..16): 1 page in range 2, 2 pages in range 3 -> 16 and 24 keys."""
    w = wl.make_workload("cz", seq_lens=[211, 0, 40, 0], q_lens=[3, 2, 1, 1],
                         block_size=16, seed=33)
    got = _segment_key_counts(w, 5, W=4)
    assert got.tolist() == [[80, 80, 49, 0, 0], [80, 80, 50, 0, 0],
                            [80, 80, 51, 0, 0], [0] * 5, [0] * 5,
                            [16, 24, 0, 0, 0], [0] * 5]


@pytest.mark.parametrize("W", [1, 3, 7, 152, 1000])
def test_balanced_partials_merge_to_whole(W):
    """Whatever the cut, the merged segments are the whole row."""
    w = wl.make_workload("bm", seq_lens=[300, 17, 0, 129, 64], q_lens=[4, 4, 4, 1, 2],
                         block_size=16, seed=34)
    cache = refs.oracle_cache(w)
    whole, wl_lse = refs.oracle_attn(w, cache)
    S = 8
    po = np.zeros((S,) + whole.shape, np.float32)
    pl = np.zeros((S,) + wl_lse.shape, np.float32)
    for s in range(S):
        po[s], pl[s] = refs.oracle_attn(w, cache, num_splits=S, split=s,
                                        split_ranges=W)
    T, H, dv = whole.shape
    out, lse = oracle.splitkv_reduce(po.reshape(S, T * H, dv), pl.reshape(S, T * H))
    assert np.allclose(out.reshape(whole.shape), whole, atol=1e-6, rtol=1e-6)
    fin = np.isfinite(wl_lse.reshape(-1))
    assert (np.isfinite(lse) == fin).all()
    assert np.allclose(lse[fin], wl_lse.reshape(-1)[fin], atol=1e-5)
