"""Causal varlen prefill on the GPU (tcgen05 kernel) against the oracle,
bf16 within atol/rtol 1e-2.  Unwritten cache bytes hold NaN patterns, so the
partly filled last page of a sequence exercises the tail masking."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs

pytestmark = pytest.mark.gpu


def _run_and_check(w, tokens=None, seqs=None):
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    gpu_path.device_error()
    out = gpu_path.prefill(dw)
    torch.cuda.synchronize()
    assert gpu_path.device_error() == pkv.EDEV_NONE
    o, _ = gpu_path.oracle_rows(w, tokens=tokens, seqs=seqs)
    got = gpu_path.host(out)
    if tokens is not None:
        got = got[tokens]
    refs.assert_close(got, o, **gpu_path.BF16_TOL, what=w.name)
    return got


CASES = {
    "tiny-prefill": lambda: wl.tiny("prefill"),
    "tiny-prefill-hnd": lambda: wl.tiny("prefill", layout=wl.HND),
    "one-token": lambda: wl.make_workload("one", seq_lens=[1], q_lens=[1], seed=1),
    "ragged-varlen": lambda: wl.make_workload(
        "rag", seq_lens=[1, 33, 129, 300, 257], q_lens=[1, 33, 129, 300, 257],
        seed=2),
    "chunked-with-context": lambda: wl.make_workload(
        "chunk", seq_lens=[700, 95, 260], q_lens=[150, 31, 1], seed=3),
    "block64": lambda: wl.make_workload(
        "b64", seq_lens=[513, 77], q_lens=[513, 40], block_size=64, seed=4),
    "block8-hnd": lambda: wl.make_workload(
        "b8", seq_lens=[150], q_lens=[150], block_size=8, layout=wl.HND,
        seed=5),
    "block256": lambda: wl.make_workload(
        "b256", seq_lens=[600], q_lens=[300], block_size=256, seed=6),
    "gqa-8": lambda: wl.make_workload(
        "g8", seq_lens=[200], q_lens=[200], num_q_heads=16, num_kv_heads=2,
        seed=7),
    "gqa-1": lambda: wl.make_workload(
        "g1", seq_lens=[170], q_lens=[170], num_q_heads=4, num_kv_heads=4,
        seed=8),
    "scaled-scores": lambda: wl.make_workload(
        "hot", seq_lens=[400], q_lens=[400], softmax_scale=0.5, seed=9),
    # page-grouped fills with other geometries: 8-key pages in NHD (8-key
    # boxes), 32-key pages (two 16-key boxes a page), V ahead of K in the row
    "block8-nhd": lambda: wl.make_workload(
        "b8n", seq_lens=[150, 40], q_lens=[150, 17], block_size=8, seed=10),
    "block32": lambda: wl.make_workload(
        "b32", seq_lens=[333], q_lens=[333], block_size=32, seed=11),
    "v-first-row": lambda: wl.make_workload(
        "vf", seq_lens=[260, 31], q_lens=[260, 31], k_off=128, v_off=0, seed=12),
    # rows that do not split into 64-column slabs (V at column 200 of 328):
    # one box per 64-column slab and page
    "padded-row": lambda: wl.make_workload(
        "pad", seq_lens=[300, 45], q_lens=[300, 45], row_elems=328, v_off=200, seed=13),
    "padded-row-hnd-b64": lambda: wl.make_workload(
        "padh", seq_lens=[200], q_lens=[200], row_elems=336, v_off=200, block_size=64,
        layout=wl.HND, seed=14),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_small(name):
    _run_and_check(CASES[name]())


def test_prefill_rows_without_keys_are_zero():
    """seq_lens < q_len leaves the first rows without a key: they are 0."""
    w = wl.make_workload("short", seq_lens=[40], q_lens=[40], seed=10)
    w.seq_lens = np.array([30], np.int32)     # 10 rows see nothing
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    out = gpu_path.prefill(dw)
    o, _ = gpu_path.oracle_rows(w)
    got = gpu_path.host(out)
    assert (got[:10] == 0).all()
    refs.assert_close(got, o, **gpu_path.BF16_TOL)


def test_prefill_repeatable():
    w = wl.make_workload("rep", seq_lens=[1000], q_lens=[1000], seed=11)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    a = gpu_path.prefill(dw).clone()
    b = gpu_path.prefill(dw)
    assert torch.equal(a, b)


def prefill_sample_tokens(n_tokens, units, n_random, seed=0, G=4, kv_heads=4):
    """Query tokens to check in a long single-sequence prefill, chosen from
    the kernel's work numbering: a query tile is 128 / G tokens of the G
    query heads of one KV head; unit u of a KV head holds tiles 4u .. 4u + 3
    (tiles 4u, 4u + 1 -- a work item's tiles A and B -- go to the first CTA
    of a 2-CTA cluster, 4u + 2 and 4u + 3 to the second); units are numbered
    from the last (longest) one and dealt to the clusters in rounds.  For
    each listed unit the first and last token of each of its four tiles is
    taken (every query head of those tokens is compared, so every KV head's
    unit is covered), plus the first and last token of the sequence and a
    random spread."""
    tq = 128 // G
    toks = [0, n_tokens - 1]
    for u in units:
        for tile in range(4):
            t0 = (4 * u + tile) * tq
            toks += [t0, t0 + tq - 1]
    rng = np.random.default_rng(seed)
    toks += list(rng.integers(0, n_tokens, n_random))
    return np.unique(np.asarray(toks, dtype=np.int64)).astype(np.int32)


def _long_prefill_check(n_tokens, units, n_random):
    w = wl.long_prefill(n_tokens)
    toks = prefill_sample_tokens(n_tokens, units, n_random)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    gpu_path.device_error()
    out = gpu_path.prefill(dw)
    got = gpu_path.host(out[torch.from_numpy(toks.astype(np.int64)).cuda()])
    torch.cuda.synchronize()
    assert gpu_path.device_error() == pkv.EDEV_NONE
    o, _ = gpu_path.oracle_rows(w, tokens=toks, seqs=[0])
    refs.assert_close(got, o, **gpu_path.BF16_TOL, what=w.name)
    return toks


def test_prefill_32k_sampled():
    """The long-prefill workload: 32,768 tokens, causal, in the bench's launch
    shape.  1,024 tiles of 32 tokens make 256 units per KV head (1,024 in
    all, 76 clusters on 152 SMs): the units dealt first (255 .. 237), last
    (0 .. 8) and between, both CTAs and both tiles of each, every head."""
    units = [0, 1, 2, 8, 9, 63, 64, 100, 127, 128, 200, 236, 237, 254, 255]
    toks = _long_prefill_check(32768, units, 24)
    assert len(toks) * 16 >= 2048


def test_prefill_131k_sampled():
    """The 131,072-token prefill (the long-prefill workload's larger run):
    4,096 units per KV head; the first and last dealt units, the middle
    ones, tile edges and a random spread, every head."""
    units = [0, 1, 2, 511, 512, 1000, 1021, 1022, 1023]
    toks = _long_prefill_check(131072, units, 16)
    assert len(toks) * 16 >= 1024


def _raw_prefill(q_ptr, cache_ptr, out_ptr, dw):
    """pkv_paged_attn_prefill through the C ABI with the given raw pointers
    (the binding itself takes CUDA tensors only)."""
    import ctypes
    w = dw.w
    return pkv.load().pkv_paged_attn_prefill(
        ctypes.c_void_p(q_ptr), w.num_q_heads, w.num_tokens, ctypes.c_void_p(cache_ptr),
        ctypes.byref(dw.cache.desc), ctypes.c_void_p(dw.block_table.data_ptr()),
        int(dw.block_table.shape[1]), ctypes.c_void_p(dw.seq_lens.data_ptr()),
        ctypes.c_void_p(dw.query_start_loc.data_ptr()), w.num_seqs,
        float(w.softmax_scale), None, None, ctypes.c_void_p(out_ptr),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_prefill_rejects_memory_of_other_kinds():
    """The prefill's tensor maps (K/V tiles multicast to the two CTAs of a
    cluster) must cover this GPU's own memory: a pinned host buffer passed
    as the cache, q or out is refused with PKV_EINVAL and nothing runs."""
    w = wl.tiny("prefill")
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    T, Hq = w.num_tokens, w.num_q_heads
    out = torch.full((T, Hq, w.head_size_v), 7.0, dtype=torch.bfloat16, device="cuda")
    nbytes = dw.cache.data.numel() * dw.cache.data.element_size()
    host_cache = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host_cache.copy_(dw.cache.data.cpu())
    host_q = dw.q.cpu().pin_memory()
    host_out = torch.zeros(T, Hq, w.head_size_v, dtype=torch.bfloat16, pin_memory=True)
    torch.cuda.synchronize()
    q, c, o = dw.q.data_ptr(), dw.cache.data.data_ptr(), out.data_ptr()
    for args in ((q, host_cache.data_ptr(), o), (host_q.data_ptr(), c, o),
                 (q, c, host_out.data_ptr())):
        assert _raw_prefill(*args, dw) == pkv.EINVAL
    torch.cuda.synchronize()
    assert (out.float() == 7.0).all()           # nothing was launched
    assert (host_out.float() == 0.0).all()
    assert gpu_path.device_error() == pkv.EDEV_NONE
    # the same call on device memory runs
    assert _raw_prefill(q, c, o, dw) == pkv.OK
    torch.cuda.synchronize()
    ref, _ = gpu_path.oracle_rows(w)
    refs.assert_close(gpu_path.host(out), ref, **gpu_path.BF16_TOL)
