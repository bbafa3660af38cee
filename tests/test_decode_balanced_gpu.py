"""Split-KV decode with balanced ranges (pkv_paged_attn_decode_balanced) on
the GPU against the oracle: the segments the device cuts from seq_lens are
the oracle's balanced ranges for the same W, partial by partial (lse within
2e-3 / 1e-4, o within the path's tolerance: bf16 1e-2 / 1e-2, FP8 KV 3e-2),
and the merged rows equal whole-row attention."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs
from tests.test_decode_gpu import SMALL, _check_out

pytestmark = pytest.mark.gpu


def _decode(dw, S, W):
    w = dw.w
    po, pl = pkv.paged_attn_decode_balanced(
        dw.q, dw.cache, dw.block_table, dw.seq_lens, dw.query_start_loc,
        w.softmax_scale, max(1, w.max_query_len), S, W,
        k_scale=dw.k_scale, v_scale=dw.v_scale)
    lse = torch.empty(pl.shape[1:], dtype=torch.float32, device=pl.device)
    out = pkv.splitkv_reduce(po, pl, lse_out=lse)
    torch.cuda.synchronize()
    return po, pl, out, lse


def _check_partials(w, po, pl, S, W, tokens=None, seqs=None, splits=None):
    sel = slice(None) if tokens is None else torch.from_numpy(
        np.asarray(tokens, dtype=np.int64)).cuda()
    po, pl = po[:, sel], pl[:, sel]
    for s in (range(S) if splits is None else splits):
        o, l = gpu_path.oracle_rows(w, tokens=tokens, seqs=seqs, num_splits=S,
                                    split=s, split_ranges=W)
        gl = gpu_path.host(pl[s])
        fin = np.isfinite(l)
        assert (np.isneginf(gl) == ~fin).all(), f"segment {s}: empty pattern"
        assert not np.isnan(gl).any()
        refs.assert_close(gl[fin], l[fin], atol=2e-3, rtol=1e-4, what=f"lse {s}")
        go = gpu_path.host(po[s])
        refs.assert_close(go[fin], o[fin], **gpu_path.tol(w), what=f"o {s}")


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("S,W", [(1, 0), (4, 3), (8, 0), (16, 7), (16, 1000)])
def test_balanced_small(name, S, W):
    w = SMALL[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    We = W or pkv.decode_balanced_ranges(dw.cache)
    po, pl, out, lse = _decode(dw, S, W)
    _check_partials(w, po, pl, S, We)
    _check_out(w, out, lse)
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_balanced_mixed_lengths_and_empty_sequences():
    """One long sequence among short and empty ones: the ranges cut the long
    one into many segments and leave the padded rows at -inf everywhere."""
    w = wl.make_workload("mix", seq_lens=[5000, 3, 0, 40, 0, 700, 17],
                         q_lens=[1, 1, 4, 2, 1, 4, 1], block_size=16, seed=21)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    for S, W in ((16, 0), (32, 5), (3, 152)):
        We = W or pkv.decode_balanced_ranges(dw.cache)
        po, pl, out, lse = _decode(dw, S, W)
        _check_partials(w, po, pl, S, We)
        _check_out(w, out, lse)
        empty = gpu_path.tokens_of(w, [2, 4])
        assert np.isneginf(gpu_path.host(pl)[:, empty]).all()
        assert (gpu_path.host(out)[empty] == 0).all()
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_balanced_repeatable_and_many_ranges_per_cta():
    """Two calls give the same bits; W above the resident CTAs (so a CTA
    takes several ranges) matches the oracle."""
    w = SMALL["verify-bf16"]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    W = 3 * pkv.decode_balanced_ranges(dw.cache)
    a = [t.clone() for t in _decode(dw, 64, W)]
    b = _decode(dw, 64, W)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    written = torch.isfinite(b[1])   # an empty segment's o is left unwritten
    assert torch.equal(a[0][written], b[0][written])
    _check_partials(w, b[0], b[1], 64, W)


def _wide(name, n, seed, *, empty_chunk=False, **kw):
    """n sequences (more than the 128 a CTA holds at once): lengths U[0, 300]
    with every eleventh empty, q_len 1..4; with empty_chunk, sequences
    128..255 (a whole chunk) are empty."""
    g = np.random.default_rng(seed)
    L = g.integers(0, 300, size=n, endpoint=True)
    L[::11] = 0
    if empty_chunk:
        L[128:256] = 0
    q = np.minimum(g.integers(1, 4, size=n, endpoint=True), np.maximum(L, 1))
    return wl.make_workload(name, seq_lens=list(L), q_lens=list(q), seed=seed, **kw)


WIDE = {
    "129": lambda: _wide("w129", 129, 31),
    "300-empty-chunk": lambda: _wide("w300", 300, 32, empty_chunk=True),
    "256-fp8-b64": lambda: _wide("w256", 256, 33, kv_dtype=wl.FP8,
                                 scale_mode=wl.SCALE_HEAD, block_size=64),
    # V before K in the row: the FP8 warp-MMA form
    "200-fp8-vfirst": lambda: _wide("w200", 200, 34, kv_dtype=wl.FP8,
                                    scale_mode=wl.SCALE_TENSOR, k_off=128, v_off=0,
                                    row_elems=320),
    # the MLA head (bf16, two CTAs per SM)
    "150-mla": lambda: _wide("w150", 150, 35, num_q_heads=16, num_kv_heads=1,
                             head_size=576, head_size_v=512, block_size=64,
                             v_aliases_k=True, softmax_scale=1 / 24),
}


@pytest.mark.parametrize("name", list(WIDE))
@pytest.mark.parametrize("S,W", [(16, 0), (16, 7), (4, 1000)])
def test_balanced_wide_batches(name, S, W):
    """More than 128 sequences: each CTA counts the pages chunk by chunk and
    walks a window of 128 sequences; the segments are still the oracle's
    balanced ranges (few ranges spanning many sequences and chunks, the
    default, and more ranges than CTAs)."""
    w = WIDE[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    We = W or pkv.decode_balanced_ranges(dw.cache)
    po, pl, out, lse = _decode(dw, S, W)
    _check_partials(w, po, pl, S, We)
    _check_out(w, out, lse)
    empty = gpu_path.tokens_of(w, [b for b in range(w.num_seqs) if w.seq_lens[b] == 0])
    assert np.isneginf(gpu_path.host(pl)[:, empty]).all()
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_balanced_rejects_bad_ranges():
    w = WIDE["129"]()
    dw = wl.to_device(w)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attn_decode_balanced(
            dw.q, dw.cache, dw.block_table, dw.seq_lens, dw.query_start_loc,
            w.softmax_scale, 1, 4, -1)
    assert e.value.status == pkv.EINVAL


# ----------------------------------------------------------- full sizes ----

def test_balanced_batched_decode_full():
    """The batched-decode workload in the bench's launch shape (16 segments
    at most, one range per resident CTA): every merged row, and the
    partials of every sequence for four of the segments."""
    w = wl.batched_decode()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    W = pkv.decode_balanced_ranges(dw.cache)
    po, pl, out, lse = _decode(dw, w.max_splits, W)
    _check_out(w, out, lse)
    _check_partials(w, po, pl, w.max_splits, W, splits=[0, 1, 4, 15])


def test_balanced_verify_fp8_full():
    """16 x ~46K keys, q_len 4, FP8 per-head scales, block 64, 8 padded
    rows: every row of every sequence."""
    w = wl.verify_fp8()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    _, pl, out, lse = _decode(dw, 16, 0)
    _check_out(w, out, lse)
    assert np.isneginf(gpu_path.host(pl)[:, 64:]).all()


# ------------------------------------------- balanced ranges, fused merge ----

def _fused(dw, S, W, ws):
    w = dw.w
    T, Hq = w.num_tokens, w.num_q_heads
    lse = torch.empty(T, Hq, dtype=torch.float32, device=dw.q.device)
    out, _ = pkv.paged_attn_decode_balanced_fused(
        dw.q, dw.cache, dw.block_table, dw.seq_lens, dw.query_start_loc, w.softmax_scale,
        max(1, w.max_query_len), S, ws, num_ranges=W, lse_out=lse,
        k_scale=dw.k_scale, v_scale=dw.v_scale)
    torch.cuda.synchronize()
    return out, lse


def _workspace(w):
    n = pkv.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                   max(1, w.max_query_len))
    return torch.zeros(max(1, n // 4), dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("S,W", [(4, 3), (16, 0), (8, 1000), (40, 0)])
def test_balanced_fused_small(name, S, W):
    """The merge inside the launch gives the whole rows (the oracle), twice in
    a row with the same workspace (every counter is left at zero); past 32
    segments the merge runs as a second launch."""
    w = SMALL[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    ws = _workspace(w)
    out, lse = _fused(dw, S, W, ws)
    assert int(ws.abs().sum()) == 0
    out2, lse2 = _fused(dw, S, W, ws)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    _check_out(w, out, lse)
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_balanced_fused_mixed_lengths_and_empty_sequences():
    w = wl.make_workload("mixf", seq_lens=[5000, 3, 0, 40, 0, 700, 17],
                         q_lens=[1, 1, 4, 2, 1, 4, 1], block_size=16, seed=23)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    ws = _workspace(w)
    for S, W in ((16, 0), (32, 5), (3, 152)):
        out, lse = _fused(dw, S, W, ws)
        _check_out(w, out, lse)
        empty = gpu_path.tokens_of(w, [2, 4])
        assert (gpu_path.host(out)[empty] == 0).all()
        assert np.isneginf(gpu_path.host(lse)[empty]).all()
    assert int(ws.abs().sum()) == 0
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_balanced_fused_wide_batch():
    """300 sequences with an empty chunk, merged in the launch: every row,
    empty sequences 0 with lse -inf."""
    w = WIDE["300-empty-chunk"]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    ws = _workspace(w)
    for S, W in ((16, 0), (8, 7)):
        out, lse = _fused(dw, S, W, ws)
        _check_out(w, out, lse)
        empty = gpu_path.tokens_of(w, [b for b in range(w.num_seqs) if w.seq_lens[b] == 0])
        assert (gpu_path.host(out)[empty] == 0).all()
        assert np.isneginf(gpu_path.host(lse)[empty]).all()
    assert int(ws.abs().sum()) == 0
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_balanced_fused_batched_decode_full():
    """The headline batched decode in one launch: every row against the oracle."""
    w = wl.batched_decode()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    out, lse = _fused(dw, w.max_splits, 0, _workspace(w))
    _check_out(w, out, lse)
