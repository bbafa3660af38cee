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


def test_prefill_32k_sampled():
    """The long-prefill workload: 32,768 tokens, causal, in the bench's launch
    shape; rows checked against the oracle: the first, the last, and a spread
    between them, every head."""
    w = wl.long_prefill(32768)
    rng = np.random.default_rng(0)
    toks = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 32767],
                                     rng.integers(0, 32768, 10)])).astype(np.int32)
    _run_and_check(w, tokens=toks, seqs=[0])
