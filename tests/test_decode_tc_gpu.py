"""The FP8 decode's tensor-core form on the GPU against the oracle.

The form covers rows with K before V. The cases below are the ones its
design singles out:
- one query token (rows 4..15 of the 16-row group are padding);
- several 16-row groups per head;
- block sizes that give 8, 16 or 32-row TMA boxes;
- both layouts and both scale modes;
- keys whose scores keep rising along the sequence, so the lazily moved row
  reference is raised again and again and O^T in TMEM is rescaled.

A row with V before K takes the warp-MMA form, checked here as well.
FP8-KV tolerance: atol 3e-2 on outputs; lse within 2e-3."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path
from tests.test_decode_gpu import _check_out, _check_partials

pytestmark = pytest.mark.gpu

CASES = {
    "q1-b16-nhd-head": lambda: wl.make_workload(
        "t1", seq_lens=[37, 300, 1000], q_lens=[1, 1, 1], block_size=16,
        kv_dtype=wl.FP8, scale_mode=wl.SCALE_HEAD, seed=31),
    "q1-b8-hnd-tensor": lambda: wl.make_workload(
        "t2", seq_lens=[129, 8, 513], q_lens=[1, 1, 1], block_size=8,
        kv_dtype=wl.FP8, scale_mode=wl.SCALE_TENSOR, layout=wl.HND, seed=32),
    "q9-three-row-groups-b32": lambda: wl.make_workload(
        "t3", seq_lens=[500, 260], q_lens=[9, 5], block_size=32,
        kv_dtype=wl.FP8, scale_mode=wl.SCALE_HEAD, seed=33),
    "q3-gqa8-b64": lambda: wl.make_workload(
        "t4", seq_lens=[1100, 77], q_lens=[3, 2], num_q_heads=16,
        num_kv_heads=2, block_size=64, kv_dtype=wl.FP8,
        scale_mode=wl.SCALE_HEAD, seed=34),
    "v-before-k-warp-mma": lambda: wl.make_workload(
        "t5", seq_lens=[300, 45], q_lens=[4, 1], block_size=16, k_off=128,
        v_off=0, row_elems=320, kv_dtype=wl.FP8, scale_mode=wl.SCALE_HEAD,
        seed=35),
}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("S", [1, 5])
def test_fp8_decode_cases(name, S):
    w = CASES[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    po, pl, out, lse = gpu_path.decode(dw, S)
    torch.cuda.synchronize()
    _check_partials(w, po, pl, S)
    _check_out(w, out, lse)
    assert gpu_path.device_error() == pkv.EDEV_NONE


def _rising(seed):
    """Keys scaled by 1 + j / 40 at position j of their sequence: every
    128-key chunk raises the row maxima by more than 2^8 (log2 units), so
    the reference moves at nearly every chunk."""
    w = wl.make_workload("rise", seq_lens=[2000, 700], q_lens=[4, 1],
                         block_size=64, kv_dtype=wl.FP8,
                         scale_mode=wl.SCALE_HEAD, seed=seed)
    k = w.k_ctx.clone().float()
    for b in range(len(w.seq_lens)):
        c0, L = int(w.ctx_start[b]), int(w.seq_lens[b])
        ramp = 1.0 + torch.arange(L, dtype=torch.float32) / 40.0
        k[c0:c0 + L] *= ramp[:, None, None]
    k = k.to(w.k_ctx.dtype)
    return dataclasses.replace(w, k_ctx=k,
                               k_scale=wl._choose_scales(k, w.scale_mode))


@pytest.mark.parametrize("S", [1, 3])
def test_fp8_decode_rising_scores(S):
    w = _rising(36)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    po, pl, out, lse = gpu_path.decode(dw, S)
    torch.cuda.synchronize()
    _check_partials(w, po, pl, S)
    _check_out(w, out, lse)
    # the scores did rise: the merged lse of the long sequence's last row is
    # far above what unscaled keys give
    assert float(gpu_path.host(lse)[3].max()) > 20.0


def test_fp8_fused_rising_scores():
    w = _rising(37)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    n = pkv.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                   w.max_query_len)
    ws = torch.zeros(max(1, n // 4), dtype=torch.int32, device=dw.q.device)
    lse = torch.empty(w.num_tokens, w.num_q_heads, dtype=torch.float32,
                      device=dw.q.device)
    out, _ = pkv.paged_attn_decode_fused(
        dw.q, dw.cache, dw.block_table, dw.seq_lens, dw.query_start_loc,
        w.softmax_scale, w.max_query_len, 4, ws, lse_out=lse,
        k_scale=dw.k_scale, v_scale=dw.v_scale)
    torch.cuda.synchronize()
    _check_out(w, out, lse)
    assert int(ws.abs().sum()) == 0
