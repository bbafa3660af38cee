"""The fused decode (decode + split merge in one launch) on the GPU: its
merged output and lse match the two-launch path and the oracle, the
workspace is left zero by every call (so it is reusable), repeated calls
agree, and more than 32 splits fall back to a second launch."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs
from tests.test_decode_gpu import SMALL

pytestmark = pytest.mark.gpu


def _fused(dw, S, ws):
    w = dw.w
    T, Hq, dv = w.num_tokens, w.num_q_heads, w.head_size_v
    lse = torch.empty(T, Hq, dtype=torch.float32, device=dw.q.device)
    out, _ = pkv.paged_attn_decode_fused(
        dw.q, dw.cache, dw.block_table, dw.seq_lens, dw.query_start_loc,
        w.softmax_scale, max(1, w.max_query_len), S, ws, lse_out=lse,
        k_scale=dw.k_scale, v_scale=dw.v_scale)
    return out, lse


def _workspace(w, dev):
    n = pkv.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                   max(1, w.max_query_len))
    return torch.zeros(max(1, n // 4), dtype=torch.int32, device=dev)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("S", [1, 3, 16, 40])
def test_fused_matches_two_launches_and_oracle(name, S):
    w = SMALL[name]()
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    ws = _workspace(w, dw.q.device)
    out, lse = _fused(dw, S, ws)
    _, _, out2, lse2 = gpu_path.decode(dw, S)
    torch.cuda.synchronize()
    assert int(ws.abs().sum()) == 0, "workspace left non-zero"
    go, go2 = gpu_path.host(out), gpu_path.host(out2)
    # same merge arithmetic up to summation order: at most a bf16 rounding step
    refs.assert_close(go, go2, atol=1e-3, rtol=8e-3, what="fused vs two launches")
    gl, gl2 = gpu_path.host(lse), gpu_path.host(lse2)
    assert (np.isneginf(gl) == np.isneginf(gl2)).all()
    fin = np.isfinite(gl2)
    refs.assert_close(gl[fin], gl2[fin], atol=1e-5, rtol=1e-5, what="fused lse")
    o, l = gpu_path.oracle_rows(w)
    refs.assert_close(go, o, **gpu_path.tol(w), what="fused vs oracle")
    assert (go[~np.isfinite(l)] == 0).all()
    assert gpu_path.device_error() == pkv.EDEV_NONE


def test_fused_repeated_calls_reuse_the_workspace():
    w = wl.batched_decode()
    w = wl.make_workload("r", seq_lens=w.seq_lens[:8], q_lens=[1] * 8, seed=3)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    ws = _workspace(w, dw.q.device)
    outs = [gpu_path.host(_fused(dw, 16, ws)[0]) for _ in range(3)]
    torch.cuda.synchronize()
    assert int(ws.abs().sum()) == 0
    assert (outs[0] == outs[1]).all() and (outs[1] == outs[2]).all()


def test_fused_padded_rows_are_zero():
    w = wl.verify_fp8(n_real=2, n_pad=8, ctx=3000)
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    ws = _workspace(w, dw.q.device)
    out, lse = _fused(dw, 16, ws)
    o = gpu_path.host(out)
    assert np.isfinite(o).all()
    assert (o[8:] == 0).all()
    assert np.isneginf(gpu_path.host(lse)[8:]).all()


def test_fused_rejects_small_workspace():
    w = SMALL["tiny-decode"]()
    dw = wl.to_device(w)
    ws = torch.zeros(1, dtype=torch.int32, device=dw.q.device)
    need = pkv.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, 1)
    assert need > 4
    with pytest.raises(pkv.PkvError):
        _fused(dw, 3, ws)
