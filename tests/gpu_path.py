"""Helpers for the GPU parity tests: run the library path on a device
workload, and the oracle on the same (host) inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import refs

BF16_TOL = dict(atol=1e-2, rtol=1e-2)
FP8_TOL = dict(atol=3e-2, rtol=0.0)
THREADS = max(1, min(16, os.cpu_count() or 1))


def tol(w):
    return FP8_TOL if w.kv_dtype == wl.FP8 else BF16_TOL


def write_all(dw):
    pkv.kv_cache_write(dw.k_ctx, dw.v_ctx, dw.slots_all, dw.cache,
                       dw.k_scale, dw.v_scale)


def decode(dw, num_splits, reduce=True):
    w = dw.w
    po, pl = pkv.paged_attn_decode(
        dw.q, dw.cache, dw.block_table, dw.seq_lens, dw.query_start_loc,
        w.softmax_scale, max(1, w.max_query_len), num_splits,
        k_scale=dw.k_scale, v_scale=dw.v_scale)
    if not reduce:
        return po, pl, None, None
    lse = torch.empty(pl.shape[1:], dtype=torch.float32, device=pl.device)
    out = pkv.splitkv_reduce(po, pl, lse_out=lse)
    return po, pl, out, lse


def prefill(dw):
    w = dw.w
    return pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                                  dw.query_start_loc, w.softmax_scale,
                                  k_scale=dw.k_scale, v_scale=dw.v_scale)


def host(t):
    return t.detach().float().cpu().numpy()


def oracle_rows(w, tokens=None, seqs=None, num_splits=0, split=-1, sinks=None,
                split_ranges=0):
    cache = refs.oracle_cache(w, seqs=seqs)
    return refs.oracle_attn(w, cache, tokens=tokens, num_splits=num_splits,
                            split=split, threads=THREADS, sinks=sinks,
                            split_ranges=split_ranges)


def tokens_of(w, seqs):
    out = []
    for b in seqs:
        out.extend(range(int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])))
    return np.asarray(out, dtype=np.int32)


def device_error():
    return pkv.get_device_error()
