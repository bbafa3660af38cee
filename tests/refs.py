"""Test-side helpers: marshalling between workloads and the oracle, and the
independent references the oracle is pinned against (a dense brute-force
softmax attention in numpy binary64, and a per-slot closed form of the cache
write).  None of this is used by the library."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_asymmetric_gb300 import workloads as wl

SENTINEL = 0xA5


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def oracle_desc(w: wl.Workload) -> oracle.CacheDesc:
    return oracle.desc(
        dtype=oracle.DT_BF16 if w.kv_dtype == wl.BF16 else oracle.DT_FP8,
        layout=oracle.NHD if w.layout == wl.NHD else oracle.HND,
        num_blocks=w.num_blocks, block_size=w.block_size,
        num_kv_heads=w.num_kv_heads, row_elems=w.row_elems, k_off=w.k_off,
        head_size=w.head_size, v_off=w.v_off, head_size_v=w.head_size_v,
        scale_mode={wl.SCALE_NONE: 0, wl.SCALE_TENSOR: 1,
                    wl.SCALE_HEAD: 2}[w.scale_mode])


def oracle_cache(w: wl.Workload, seqs=None) -> np.ndarray:
    """The cache bytes the oracle writes for every context token of the
    listed sequences (all when None); other bytes hold SENTINEL."""
    cache = np.full(w.cache_bytes(), SENTINEL, dtype=np.uint8)
    if seqs is None:
        seqs = range(w.num_seqs)
    kb = bf16_bits(w.k_ctx)
    vb = None if w.v_ctx is None else bf16_bits(w.v_ctx)
    d = oracle_desc(w)
    for b in seqs:
        lo, hi = int(w.ctx_start[b]), int(w.ctx_start[b + 1])
        if hi <= lo:
            continue
        slots = wl.slot_mapping_for(w, [b], new_only=False)
        oracle.kv_cache_write(kb[lo:hi], None if vb is None else vb[lo:hi],
                              slots, cache, d, w.k_scale, w.v_scale)
    return cache


def oracle_attn(w: wl.Workload, cache: np.ndarray, tokens=None,
                num_splits=0, split=-1, threads=1, sinks=None, split_ranges=0):
    return oracle.paged_attn(
        bf16_bits(w.q), w.num_q_heads, cache, oracle_desc(w), w.block_table,
        w.seq_lens, w.query_start_loc, w.softmax_scale, w.k_scale, w.v_scale,
        tokens=tokens, num_splits=num_splits, split=split, threads=threads,
        sinks=sinks, split_ranges=split_ranges)


# ------------------------------------------------------------ references --

def torch_fp8_dequant(x: torch.Tensor, scale: np.ndarray, per_head: bool):
    """Quantise through torch's own float8_e4m3fn conversion (a library
    routine, independent of the oracle) and dequantise: x/s -> e4m3 -> *s.
    Valid while |x/s| <= 448, which absmax/448 scales guarantee."""
    xf = x.float()
    s = torch.from_numpy(np.asarray(scale, dtype=np.float32))
    if per_head:
        s = s.view(1, -1, 1)
    else:
        s = s.view(1, 1, 1)
    y = (xf / s).to(torch.float8_e4m3fn).to(torch.float64)
    return (y * s.double()).numpy()


def dense_kv(w: wl.Workload):
    """K and V of every context token as the cache holds them (dequantised),
    binary64, computed without the oracle."""
    if w.kv_dtype == wl.BF16:
        K = w.k_ctx.double().numpy()
        V = None if w.v_ctx is None else w.v_ctx.double().numpy()
    else:
        per_head = w.scale_mode == wl.SCALE_HEAD
        K = torch_fp8_dequant(w.k_ctx, w.k_scale, per_head)
        V = None if w.v_ctx is None else torch_fp8_dequant(w.v_ctx, w.v_scale,
                                                            per_head)
    if V is None:  # V is the first head_size_v columns of the latent K row
        if w.kv_dtype == wl.BF16:
            V = K[:, :, w.v_off:w.v_off + w.head_size_v]
        else:
            V = torch_fp8_dequant(w.k_ctx, w.v_scale,
                                  w.scale_mode == wl.SCALE_HEAD)[
                :, :, w.v_off:w.v_off + w.head_size_v]
    return K, V


def dense_attention(w: wl.Workload, K=None, V=None):
    """Brute force: per sequence, the full score matrix scale * Q K^T with an
    explicit causal mask (-inf above the bottom-right diagonal), a row
    softmax in binary64, times V.  Rows with no visible key are 0 with
    lse -inf.  Returns (out [T, Hq, dv], lse [T, Hq])."""
    if K is None:
        K, V = dense_kv(w)
    Q = w.q.double().numpy()
    T, Hq, dk = Q.shape
    G = Hq // w.num_kv_heads
    out = np.zeros((T, Hq, w.head_size_v))
    lse = np.full((T, Hq), -np.inf)
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        q0, q1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
        ql = q1 - q0
        if ql == 0:
            continue
        c0 = int(w.ctx_start[b])
        Kb, Vb = K[c0:c0 + L], V[c0:c0 + L]
        pos = L - ql + np.arange(ql)
        mask = np.arange(L)[None, :] > pos[:, None]          # [ql, L]
        for h in range(Hq):
            g = h // G
            # the softmax scale crosses the ABI as a binary32 value
            s = float(np.float32(w.softmax_scale)) * (Q[q0:q1, h, :] @ Kb[:, g, :].T)
            s = np.where(mask, -np.inf, s)
            m = s.max(axis=1, initial=-np.inf)
            ok = np.isfinite(m)
            e = np.zeros_like(s)
            e[ok] = np.exp(s[ok] - m[ok, None])
            l = e.sum(axis=1)
            o = np.zeros((ql, w.head_size_v))
            o[ok] = (e[ok] @ Vb[:, g, :]) / l[ok, None]
            out[q0:q1, h] = o
            lse[q0:q1, h] = np.where(ok, m + np.log(np.where(ok, l, 1.0)),
                                     -np.inf)
    return out, lse


def expected_cache_closed_form(w: wl.Workload, kb, vb, slots, base: np.ndarray):
    """Per-slot closed form of the write for a bf16 cache: the K bits go to
    columns [k_off, k_off+dk) and the V bits to [v_off, v_off+dv) of the
    (block, offset, head) row; nothing else changes."""
    exp = base.copy().view(np.uint16).reshape(-1)
    R, H, bs = w.row_elems, w.num_kv_heads, w.block_size
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        for h in range(H):
            if w.layout == wl.NHD:
                row = ((blk * bs + off) * H + h) * R
            else:
                row = ((blk * H + h) * bs + off) * R
            exp[row + w.k_off: row + w.k_off + w.head_size] = kb[t, h]
            if vb is not None:
                exp[row + w.v_off: row + w.v_off + w.head_size_v] = vb[t, h]
    return exp.view(np.uint8)


def assert_close(got, ref, atol, rtol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))),
                             err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of "
            f"tolerance (atol={atol}, rtol={rtol}); worst at {i}: got "
            f"{got[i]!r} ref {ref[i]!r}; max abs err {err.max():.3e}")
