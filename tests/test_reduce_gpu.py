"""Split-KV merge on the GPU against the oracle, with empty segments and
rows whose segments are all empty (MiMo model card, "Update 2026-10-01").
The cases span the merge's three forms: up to 32 splits (one warp per row
and 128 columns, in its 8-, 16- and 32-split instantiations, dv 512 as four
column blocks), more than 32 splits (a CTA per row and column block), and
dv not a multiple of 4 (one warp per row)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_asymmetric_gb300 as pkv
from tests import refs

pytestmark = pytest.mark.gpu


CASES = [(1, 7, 128), (16, 300, 128), (96, 33, 512), (5, 10, 24), (3, 4, 6),
         (8, 5, 128), (9, 13, 128), (17, 21, 128), (32, 64, 128), (19, 30, 512),
         (33, 11, 128), (32, 3, 36), (16, 1536, 128), (40, 2, 6),
         # > 512 splits: a thread of the CTA-per-row form takes more than one
         # step of eight splits and rescales to a later, larger maximum
         (600, 3, 128), (1100, 4, 512), (304, 16, 512),
         # column pieces that do not divide the CTA's 512 threads (the last
         # threads belong to no group), and a single piece per row
         (40, 5, 24), (33, 7, 4)]


@pytest.mark.parametrize("S,rows,dv", CASES)
def test_reduce_matches_oracle(S, rows, dv):
    rng = np.random.default_rng(S * 1000 + rows)
    po = rng.standard_normal((S, rows, dv)).astype(np.float32)
    pl = (rng.standard_normal((S, rows)) * 4).astype(np.float32)
    pl[rng.random((S, rows)) < 0.3] = -np.inf       # empty segments
    pl[:, rows // 2] = -np.inf                      # a row with no key at all
    po[np.isneginf(pl)] = np.nan                    # never read
    ref, rlse = oracle.splitkv_reduce(po, pl)
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    out = pkv.splitkv_reduce(torch.from_numpy(po).cuda(),
                             torch.from_numpy(pl).cuda(), lse_out=lse)
    got = out.float().cpu().numpy()
    gl = lse.cpu().numpy()
    assert np.isfinite(got).all()
    refs.assert_close(got, ref, atol=1e-2, rtol=1e-2, what="reduce")
    fin = np.isfinite(rlse)
    assert (np.isneginf(gl) == ~fin).all()
    refs.assert_close(gl[fin], rlse[fin], atol=1e-5, rtol=1e-5)
    assert (got[~fin] == 0).all()


def test_reduce_zero_splits_gives_zero():
    po = torch.empty(0, 4, 128, device="cuda")
    pl = torch.empty(0, 4, device="cuda")
    out = torch.full((4, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    pkv.splitkv_reduce(po, pl, out=out)
    assert (out == 0).all()


@pytest.mark.parametrize("S,rows,dv", [(4, 12, 128), (19, 32, 512), (32, 8, 128),
                                       (48, 8, 128), (6, 8, 10), (700, 4, 128)])
def test_reduce_with_sinks_matches_oracle(S, rows, dv):
    """The sink joins each row's merge once (4 query heads: row r takes
    sink r % 4); head 1's sink is -inf (no sink).  A row with no visible
    key but a sink has output 0 and lse = the sink."""
    hq = 4
    rng = np.random.default_rng(S * 7 + rows)
    po = rng.standard_normal((S, rows, dv)).astype(np.float32)
    pl = (rng.standard_normal((S, rows)) * 4).astype(np.float32)
    pl[rng.random((S, rows)) < 0.3] = -np.inf
    pl[:, 1] = -np.inf   # no key and no sink (head 1): 0, lse -inf
    pl[:, 2] = -np.inf   # no key, sink 3.0: 0, lse 3.0
    po[np.isneginf(pl)] = np.nan
    sinks = np.array([0.5, -np.inf, 3.0, -2.0], np.float32)
    ref, rlse = oracle.splitkv_reduce(po, pl, sinks=sinks, num_q_heads=hq)
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    # rows as [tokens, query heads]: the binding takes Hq from the last axis
    out = pkv.splitkv_reduce(torch.from_numpy(po.reshape(S, rows // hq, hq, dv)).cuda(),
                             torch.from_numpy(pl.reshape(S, rows // hq, hq)).cuda(),
                             lse_out=lse, sinks=torch.from_numpy(sinks).cuda())
    got = out.reshape(rows, dv).float().cpu().numpy()
    gl = lse.cpu().numpy()
    assert np.isfinite(got).all()
    refs.assert_close(got, ref, atol=1e-2, rtol=1e-2, what="reduce with sinks")
    fin = np.isfinite(rlse)
    assert (np.isneginf(gl) == ~fin).all()
    refs.assert_close(gl[fin], rlse[fin], atol=1e-5, rtol=1e-5)
    assert (got[1] == 0).all() and np.isneginf(gl[1])
    assert (got[2] == 0).all() and abs(gl[2] - 3.0) < 1e-5
