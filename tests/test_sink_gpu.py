"""Attention sink on the GPU (MiMo-V2.6 model card, "Update 2026-10-01": one
extra logit per head in the softmax denominator, vLLM #58235), against the
oracle's whole-row sink attention:
- decode / verify: sink-free partials, then pkv_splitkv_reduce_sink;
- prefill: pkv_paged_attn_prefill_sink.
Rows without a visible key (padded sequences) are 0 with lse = sink.  Sinks
of -inf give the sink-free results bit for bit.  Tolerances as elsewhere:
bf16 atol / rtol 1e-2, FP8 KV atol 3e-2, lse 2e-3."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs

pytestmark = pytest.mark.gpu


def _sinks(Hq, seed, scale=3.0):
    g = np.random.default_rng(seed)
    return (g.standard_normal(Hq) * scale).astype(np.float32)


DECODE = {
    "bf16-decode-padded": lambda: wl.make_workload(
        "s1", seq_lens=[300, 0, 77, 1000], q_lens=[1, 1, 1, 1], seed=51),
    "bf16-verify": lambda: wl.make_workload(
        "s2", seq_lens=[129, 1000, 4], q_lens=[4, 3, 4], block_size=64, seed=52),
    "fp8-verify-padded": lambda: wl.make_workload(
        "s3", seq_lens=[700, 0, 130], q_lens=[4, 4, 2], block_size=64,
        kv_dtype=wl.FP8, scale_mode=wl.SCALE_HEAD, seed=53),
    "mla-12": lambda: wl.make_workload(
        "s4", seq_lens=[300, 65], q_lens=[1, 1], num_q_heads=12, num_kv_heads=1,
        head_size=576, head_size_v=512, block_size=64, v_aliases_k=True,
        softmax_scale=1 / 24, seed=54),
}


def _decode_sink(dw, S, sinks_t):
    w = dw.w
    po, pl, _, _ = gpu_path.decode(dw, S, reduce=False)
    lse = torch.empty(pl.shape[1:], dtype=torch.float32, device=pl.device)
    out = pkv.splitkv_reduce(po, pl, lse_out=lse, sinks=sinks_t)
    return out, lse


@pytest.mark.parametrize("name", list(DECODE))
@pytest.mark.parametrize("S", [1, 3])
def test_decode_with_sinks(name, S):
    w = DECODE[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    sinks = _sinks(w.num_q_heads, 7 + S)
    out, lse = _decode_sink(dw, S, torch.from_numpy(sinks).cuda())
    torch.cuda.synchronize()
    o, l = gpu_path.oracle_rows(w, sinks=sinks)
    go, gl = gpu_path.host(out), gpu_path.host(lse)
    refs.assert_close(go, o, **gpu_path.tol(w), what="sink decode output")
    refs.assert_close(gl, l, atol=2e-3, rtol=1e-4, what="sink decode lse")
    # padded sequences: no key, so 0 and lse = sink
    for b in range(w.num_seqs):
        if int(w.seq_lens[b]) == 0:
            t0, t1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
            assert (go[t0:t1] == 0).all()
            # lse = sink up to the rounding of sink * log2(e) in the merge
            assert np.allclose(gl[t0:t1], np.broadcast_to(sinks, gl[t0:t1].shape),
                               rtol=1e-6, atol=1e-6)
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_minus_inf_sinks_match_plain_merge():
    w = DECODE["bf16-verify"]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    po, pl, out0, lse0 = gpu_path.decode(dw, 3)
    ninf = torch.full((w.num_q_heads,), float("-inf"), dtype=torch.float32, device="cuda")
    lse1 = torch.empty_like(lse0)
    out1 = pkv.splitkv_reduce(po, pl, lse_out=lse1, sinks=ninf)
    torch.cuda.synchronize()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


PREFILL = {
    "tiny-prefill": lambda: wl.tiny("prefill"),
    "chunked-hnd": lambda: wl.make_workload(
        "p2", seq_lens=[400, 150], q_lens=[130, 150], block_size=32,
        layout=wl.HND, seed=55),
}


@pytest.mark.parametrize("name", list(PREFILL))
def test_prefill_with_sinks(name):
    w = PREFILL[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    sinks = _sinks(w.num_q_heads, 11)
    out = pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                                 dw.query_start_loc, w.softmax_scale,
                                 sinks=torch.from_numpy(sinks).cuda())
    torch.cuda.synchronize()
    o, _ = gpu_path.oracle_rows(w, sinks=sinks)
    refs.assert_close(gpu_path.host(out), o, **gpu_path.tol(w), what="sink prefill")
    # -inf sinks: the sink-free kernel result exactly
    ninf = torch.full((w.num_q_heads,), float("-inf"), dtype=torch.float32, device="cuda")
    a = gpu_path.prefill(dw)
    b = pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                               dw.query_start_loc, w.softmax_scale, sinks=ninf)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_sink_entry_points_reject_bad_sizes():
    po = torch.zeros(2, 6, 8, dtype=torch.float32, device="cuda")
    pl = torch.zeros(2, 6, dtype=torch.float32, device="cuda")
    out = torch.empty(6, 8, dtype=torch.bfloat16, device="cuda")
    sk = torch.zeros(4, dtype=torch.float32, device="cuda")
    lib = pkv.load()
    # 6 rows are not a multiple of 4 query heads
    rc = lib.pkv_splitkv_reduce_sink(po.data_ptr(), pl.data_ptr(), 2, 6, 8, sk.data_ptr(),
                                     4, out.data_ptr(), None, None)
    assert rc == pkv.EINVAL
    rc = lib.pkv_splitkv_reduce_sink(po.data_ptr(), pl.data_ptr(), 2, 6, 8, sk.data_ptr(),
                                     0, out.data_ptr(), None, None)
    assert rc == pkv.EINVAL
