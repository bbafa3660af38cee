"""Pins of the oracle's attention sink (MiMo-V2.6 model card, "Update
2026-10-01": the vision encoder's sink taken as one extra logit in the
softmax denominator, vLLM #58235) to facts outside the oracle:
- sink = -inf is no sink, bit for bit;
- one visible key gives v * sigmoid(s - sink) in closed form, from scores
  computed here with numpy;
- a row without visible keys is 0 with lse = sink;
- for any row, out_sink = out * sigmoid(lse - sink) and
  lse_sink = logaddexp(lse, sink);
- split-KV partials (sink-free) merged with the sink equal the whole row
  with the sink, which fails if the sink is counted once per segment."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import refs


def _w(**kw):
    args = dict(seq_lens=[37, 80, 5], q_lens=[1, 3, 2], block_size=16, seed=41)
    args.update(kw)
    return wl.make_workload("sink", **args)


def _sinks(w, seed=0, scale=3.0):
    g = np.random.default_rng(seed)
    return (g.standard_normal(w.num_q_heads) * scale).astype(np.float32)


@pytest.mark.parametrize("kv", [wl.BF16, wl.FP8])
def test_minus_inf_sink_is_no_sink(kv):
    w = _w(kv_dtype=kv, scale_mode=wl.SCALE_HEAD if kv == wl.FP8 else wl.SCALE_NONE)
    cache = refs.oracle_cache(w)
    o0, l0 = refs.oracle_attn(w, cache)
    o1, l1 = refs.oracle_attn(w, cache, sinks=np.full(w.num_q_heads, -np.inf, np.float32))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_single_key_closed_form():
    w = wl.make_workload("one", seq_lens=[1, 1], q_lens=[1, 1], block_size=16, seed=42)
    sinks = _sinks(w, 1, scale=1.5)
    o, l = refs.oracle_attn(w, refs.oracle_cache(w), sinks=sinks)
    K, V = refs.dense_kv(w)
    Q = w.q.double().numpy()
    G = w.num_q_heads // w.num_kv_heads
    scale = float(np.float32(w.softmax_scale))
    for t in range(2):  # token t is sequence t's only query and key t its key
        for h in range(w.num_q_heads):
            s = scale * float(Q[t, h] @ K[t, h // G])
            sig = 1.0 / (1.0 + np.exp(float(sinks[h]) - s))
            assert np.allclose(o[t, h], V[t, h // G] * sig, rtol=1e-12, atol=1e-14)
            assert np.isclose(l[t, h], np.logaddexp(s, float(sinks[h])), rtol=1e-13)


def test_row_without_keys_is_zero_with_lse_sink():
    w = _w(seq_lens=[0, 40], q_lens=[2, 1])
    sinks = _sinks(w, 2)
    o, l = refs.oracle_attn(w, refs.oracle_cache(w), sinks=sinks)
    assert (o[:2] == 0).all()
    assert np.array_equal(l[:2], np.broadcast_to(sinks.astype(np.float64), (2, w.num_q_heads)))
    # the merge: a row whose segments are all empty
    po = np.zeros((3, 4, 8), np.float32)
    pl = np.full((3, 4), -np.inf, np.float32)
    s4 = np.array([0.5, -2.0], np.float32)
    mo, ml = oracle.splitkv_reduce(po, pl, sinks=s4, num_q_heads=2)
    assert (mo == 0).all() and np.array_equal(ml, np.array([0.5, -2.0, 0.5, -2.0]))


@pytest.mark.parametrize("kv", [wl.BF16, wl.FP8])
def test_sink_scales_rows_by_sigmoid(kv):
    w = _w(kv_dtype=kv, scale_mode=wl.SCALE_TENSOR if kv == wl.FP8 else wl.SCALE_NONE)
    cache = refs.oracle_cache(w)
    sinks = _sinks(w, 3)
    o0, l0 = refs.oracle_attn(w, cache)
    o1, l1 = refs.oracle_attn(w, cache, sinks=sinks)
    sig = 1.0 / (1.0 + np.exp(sinks[None, :].astype(np.float64) - l0))
    assert np.allclose(o1, o0 * sig[..., None], rtol=1e-11, atol=1e-14)
    assert np.allclose(l1, np.logaddexp(l0, sinks[None, :].astype(np.float64)),
                       rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("S", [1, 3, 7])
def test_merge_with_sink_equals_whole_row(S):
    w = _w(seq_lens=[130, 66, 300], q_lens=[1, 4, 2], seed=43)
    cache = refs.oracle_cache(w)
    sinks = _sinks(w, 4)
    T, Hq, dv = w.num_tokens, w.num_q_heads, w.head_size_v
    po = np.zeros((S, T, Hq, dv), np.float32)
    pl = np.zeros((S, T, Hq), np.float32)
    for s in range(S):
        o, l = refs.oracle_attn(w, cache, num_splits=S, split=s)
        po[s], pl[s] = o, l
    mo, ml = oracle.splitkv_reduce(po.reshape(S, T * Hq, dv), pl.reshape(S, T * Hq),
                                   sinks=sinks, num_q_heads=Hq)
    wo, wlse = refs.oracle_attn(w, cache, sinks=sinks)
    # the partials cross the merge in binary32
    assert np.allclose(mo.reshape(T, Hq, dv), wo, rtol=1e-5, atol=1e-6)
    assert np.allclose(ml.reshape(T, Hq), wlse, rtol=1e-6, atol=1e-6)
