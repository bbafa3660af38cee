"""The prefill over an FP8 E4M3 cache against the oracle, which reads the
same cache through its own E4M3 decoder, in both forms: pkv_paged_attn_prefill
(the E4M3 codes widened to bf16 in shared memory between the TMA load and
the tcgen05 MMAs, no workspace) and pkv_paged_attn_prefill_fp8 (the pages
widened into a workspace first); the scales fold in.  FP8-KV tolerance:
atol 3e-2.  Unwritten cache bytes hold NaN codes, so the partly filled last
page of a sequence exercises the tail masking."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs

pytestmark = pytest.mark.gpu

H, T_ = wl.SCALE_HEAD, wl.SCALE_TENSOR
CASES = {
    "tiny-head": lambda: wl.tiny("prefill", kv_dtype=wl.FP8, scale_mode=H),
    "tiny-hnd-tensor": lambda: wl.tiny("prefill", layout=wl.HND, kv_dtype=wl.FP8,
                                       scale_mode=T_),
    "ragged-varlen": lambda: wl.make_workload(
        "rag8", seq_lens=[1, 33, 129, 300], q_lens=[1, 33, 129, 300],
        kv_dtype=wl.FP8, scale_mode=H, seed=61),
    "chunked-with-context-b64": lambda: wl.make_workload(
        "chunk8", seq_lens=[700, 95, 260], q_lens=[150, 31, 1], block_size=64,
        kv_dtype=wl.FP8, scale_mode=H, seed=62),
    "block8-hnd": lambda: wl.make_workload(
        "b8f", seq_lens=[150], q_lens=[150], block_size=8, layout=wl.HND,
        kv_dtype=wl.FP8, scale_mode=T_, seed=63),
    "gqa-8": lambda: wl.make_workload(
        "g8f", seq_lens=[200], q_lens=[200], num_q_heads=16, num_kv_heads=2,
        kv_dtype=wl.FP8, scale_mode=H, seed=64),
}


def _run(w, tokens=None, seqs=None, sinks=None, two_pass=False):
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    gpu_path.device_error()
    st = None if sinks is None else torch.from_numpy(sinks).cuda()
    ws = None
    if two_pass:
        n = pkv.prefill_fp8_workspace_bytes(w.num_seqs, dw.block_table.shape[1], dw.cache)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                                 dw.query_start_loc, w.softmax_scale,
                                 k_scale=dw.k_scale, v_scale=dw.v_scale, sinks=st,
                                 workspace=ws)
    torch.cuda.synchronize()
    assert gpu_path.device_error() == pkv.EDEV_NONE
    o, _ = gpu_path.oracle_rows(w, tokens=tokens, seqs=seqs, sinks=sinks)
    got = gpu_path.host(out)
    if tokens is not None:
        got = got[tokens]
    refs.assert_close(got, o, **gpu_path.FP8_TOL, what=w.name)
    return dw, out


@pytest.mark.parametrize("two_pass", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_fp8_prefill_small(name, two_pass):
    _run(CASES[name](), two_pass=two_pass)


def test_fp8_prefill_two_forms_agree():
    """Both forms run the same tensor-core prefill on the same bf16 values
    (exact widening), so their outputs are identical bits."""
    w = CASES["chunked-with-context-b64"]()
    sinks = np.linspace(-3, 3, w.num_q_heads).astype(np.float32)
    _, a = _run(w, sinks=sinks)
    _, b = _run(w, sinks=sinks, two_pass=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_fp8_prefill_two_pass_workspace_checks():
    w = CASES["ragged-varlen"]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    n = pkv.prefill_fp8_workspace_bytes(w.num_seqs, dw.block_table.shape[1], dw.cache)
    assert n > 0
    small = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                               dw.query_start_loc, w.softmax_scale,
                               k_scale=dw.k_scale, v_scale=dw.v_scale, workspace=small)
    assert e.value.status == pkv.EINVAL
    big = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:  # not 256-byte aligned
        pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                               dw.query_start_loc, w.softmax_scale,
                               k_scale=dw.k_scale, v_scale=dw.v_scale, workspace=big[16:])
    assert e.value.status == pkv.EINVAL


def test_fp8_prefill_with_sinks():
    w = CASES["chunked-with-context-b64"]()
    sinks = np.linspace(-3, 3, w.num_q_heads).astype(np.float32)
    _run(w, sinks=sinks)


def test_fp8_prefill_repeatable():
    w = CASES["ragged-varlen"]()
    dw, a = _run(w)
    b = pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                               dw.query_start_loc, w.softmax_scale,
                               k_scale=dw.k_scale, v_scale=dw.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_fp8_prefill_matches_bf16_prefill_of_the_widened_codes():
    """The in-kernel widening is exact: the FP8 prefill equals, bit for bit,
    the bf16 prefill over a bf16 cache holding the same codes widened on the
    host (torch's float8_e4m3fn -> bfloat16), with the scales applied to
    q and the output the way the kernel folds them (here: unit scales)."""
    w = CASES["chunked-with-context-b64"]()
    w.k_scale = np.ones_like(w.k_scale)
    w.v_scale = np.ones_like(w.v_scale)
    dw, a = _run(w)
    codes = dw.cache.data.view(torch.float8_e4m3fn)
    wide = codes.to(torch.bfloat16)
    desc = pkv.make_desc(dtype=pkv.BF16, layout=dw.cache.desc.layout,
                         num_blocks=dw.cache.desc.num_blocks,
                         block_size=dw.cache.desc.block_size,
                         num_kv_heads=dw.cache.desc.num_kv_heads,
                         row_elems=dw.cache.desc.row_elems, k_off=dw.cache.desc.k_off,
                         head_size=dw.cache.desc.head_size, v_off=dw.cache.desc.v_off,
                         head_size_v=dw.cache.desc.head_size_v)
    b = pkv.paged_attn_prefill(dw.q, pkv.Cache(wide, desc), dw.block_table, dw.seq_lens,
                               dw.query_start_loc, w.softmax_scale)
    torch.cuda.synchronize()
    fin = torch.isfinite(b.float()).all(dim=-1).all(dim=-1)
    assert fin.all()
    assert torch.equal(a, b)


def test_fp8_prefill_32k_sampled():
    """32,768 tokens, FP8 cache with per-head scales, in the bench's launch
    shape: the tokens of the bf16 32K test's choice (first and last dealt
    units, both CTAs and both tiles of each, tile edges) and a random
    spread, every head, against the oracle."""
    from tests.test_prefill_gpu import prefill_sample_tokens
    w = wl.make_workload("prefill-32768-fp8", seq_lens=[32768], q_lens=[32768],
                         kv_dtype=wl.FP8, scale_mode=H, seed=0)
    units = [0, 1, 2, 8, 9, 63, 64, 100, 127, 128, 200, 236, 237, 254, 255]
    toks = prefill_sample_tokens(32768, units, 24, seed=1)
    assert len(toks) * 16 >= 2048
    _run(w, tokens=toks, seqs=[0])
    _run(w, tokens=toks, seqs=[0], two_pass=True)


def test_fp8_prefill_131k_sampled():
    """The 131,072-token prefill over an FP8 cache with per-head scales, both
    forms (widened in the kernel, and two-pass through the workspace): the
    first and last dealt units, the middle ones, tile edges and a random
    spread, every head, against the oracle.  Sampled rows are gathered on
    the device, so only they come back to the host."""
    from tests.test_prefill_gpu import prefill_sample_tokens
    n = 131072
    w = wl.make_workload(f"prefill-{n}-fp8", seq_lens=[n], q_lens=[n],
                         kv_dtype=wl.FP8, scale_mode=H, seed=0)
    units = [0, 1, 2, 511, 512, 1000, 1021, 1022, 1023]
    toks = prefill_sample_tokens(n, units, 16, seed=2)
    assert len(toks) * 16 >= 1024
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    gpu_path.device_error()
    idx = torch.from_numpy(toks.astype(np.int64)).cuda()
    n_ws = pkv.prefill_fp8_workspace_bytes(w.num_seqs, dw.block_table.shape[1], dw.cache)
    got = []
    for ws in (None, torch.empty(n_ws, dtype=torch.uint8, device="cuda")):
        out = pkv.paged_attn_prefill(dw.q, dw.cache, dw.block_table, dw.seq_lens,
                                     dw.query_start_loc, w.softmax_scale,
                                     k_scale=dw.k_scale, v_scale=dw.v_scale, workspace=ws)
        got.append(gpu_path.host(out[idx]))
        del out
    torch.cuda.synchronize()
    assert gpu_path.device_error() == pkv.EDEV_NONE
    o, _ = gpu_path.oracle_rows(w, tokens=toks, seqs=[0])
    for g in got:
        refs.assert_close(g, o, **gpu_path.FP8_TOL, what=w.name)
