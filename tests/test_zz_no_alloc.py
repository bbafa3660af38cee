"""The no-allocation fused decode (pkv_paged_attn_decode_fused_noalloc): its
counters live in the library's own fixed device array, so it takes no
workspace.  Two calls in a row give, bit for bit, what the workspace entry
pkv_paged_attn_decode_fused gives on the same inputs, and, when the merge
runs inside the decode kernel (up to 32 splits), sizes needing more than
65536 counters are rejected before anything is launched.  The file is
named to be collected last, so it also runs after every other GPU test has
used the library in the same process."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs
from tests.test_decode_gpu import SMALL

pytestmark = pytest.mark.gpu

CASES = ["tiny-decode", "verify-fp8-head", "verify-bf16", "mla-12",
         "long-query-rows"]


def _call(dw, S, ws=None):
    w = dw.w
    T, Hq = w.num_tokens, w.num_q_heads
    lse = torch.empty(T, Hq, dtype=torch.float32, device=dw.q.device)
    args = (dw.q, dw.cache, dw.block_table, dw.seq_lens, dw.query_start_loc,
            w.softmax_scale, max(1, w.max_query_len), S)
    kw = dict(lse_out=lse, k_scale=dw.k_scale, v_scale=dw.v_scale)
    if ws is None:
        out, _ = pkv.paged_attn_decode_fused_noalloc(*args, **kw)
    else:
        out, _ = pkv.paged_attn_decode_fused(*args, ws, **kw)
    return gpu_path.host(out), gpu_path.host(lse)


@pytest.mark.parametrize("name", CASES)
@pytest.mark.parametrize("S", [3, 16, 40])
def test_two_noalloc_calls_match_workspace_entry(name, S):
    w = SMALL[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    n = pkv.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                   max(1, w.max_query_len))
    ws = torch.zeros(max(1, n // 4), dtype=torch.int32, device=dw.q.device)
    ref_o, ref_l = _call(dw, S, ws)
    for _ in range(2):
        o, l = _call(dw, S)
        torch.cuda.synchronize()
        # same kernel, same merge order: identical bits, lse -inf included
        assert np.array_equal(o, ref_o)
        assert np.array_equal(l, ref_l)
    assert gpu_path.device_error() == pkv.EDEV_NONE
    # and the merged rows are the attention the oracle computes
    oo, ol = gpu_path.oracle_rows(w)
    refs.assert_close(o, oo, **gpu_path.tol(w), what="no-alloc vs oracle")
    assert (o[~np.isfinite(ol)] == 0).all()


def test_noalloc_interleaved_shapes():
    """Calls of different shapes in turn reuse the one counter array."""
    dws = [wl.to_device(SMALL[n]()) for n in ("verify-bf16", "mla-12")]
    for dw in dws:
        gpu_path.write_all(dw)
    first = [_call(dw, 16)[0] for dw in dws]
    again = [_call(dw, 16)[0] for dw in reversed(dws)][::-1]
    torch.cuda.synchronize()
    for a, b in zip(first, again):
        assert np.array_equal(a, b)
    assert gpu_path.device_error() == pkv.EDEV_NONE


def _empty_batch(dw, num_seqs):
    """A batch of `num_seqs` sequences with no tokens and no keys."""
    w = dw.w
    dev = dw.q.device
    q = torch.empty(0, w.num_q_heads, w.head_size, dtype=torch.bfloat16,
                    device=dev)
    bt = torch.zeros(num_seqs, 1, dtype=torch.int32, device=dev)
    sl = torch.zeros(num_seqs, dtype=torch.int32, device=dev)
    qsl = torch.zeros(num_seqs + 1, dtype=torch.int32, device=dev)
    return q, bt, sl, qsl


def test_noalloc_rejects_more_than_65536_counters():
    w = SMALL["tiny-decode"]()
    dw = wl.to_device(w)
    per_seq = pkv.decode_workspace_bytes(1, w.num_q_heads, w.num_kv_heads, 1) // 4
    assert per_seq >= 1
    fit = pkv.NOALLOC_MAX_COUNTERS // per_seq
    for n, ok in ((fit, True), (fit + 1, False)):
        q, bt, sl, qsl = _empty_batch(dw, n)
        call = lambda: pkv.paged_attn_decode_fused_noalloc(
            q, dw.cache, bt, sl, qsl, w.softmax_scale, 1, 4,
            k_scale=dw.k_scale, v_scale=dw.v_scale)
        if ok:
            call()
        else:
            with pytest.raises(pkv.PkvError) as e:
                call()
            assert e.value.status == pkv.EINVAL
            # the same batch is valid for the entry with a caller workspace
            ws = torch.zeros(n * per_seq, dtype=torch.int32, device=q.device)
            pkv.paged_attn_decode_fused(
                q, dw.cache, bt, sl, qsl, w.softmax_scale, 1, 4, ws,
                k_scale=dw.k_scale, v_scale=dw.v_scale)
    # past 32 splits the merge is a second launch that uses no counter: the
    # same oversized batch is taken
    q, bt, sl, qsl = _empty_batch(dw, fit + 1)
    pkv.paged_attn_decode_fused_noalloc(q, dw.cache, bt, sl, qsl, w.softmax_scale,
                                        1, 40, k_scale=dw.k_scale, v_scale=dw.v_scale)
    torch.cuda.synchronize()
    assert gpu_path.device_error() == pkv.EDEV_NONE
