"""Split-KV merge on the GPU against the oracle, with empty segments and
rows whose segments are all empty (MiMo model card, "Update 2026-10-01")."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_asymmetric_gb300 as pkv
from tests import refs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S,rows,dv", [(1, 7, 128), (16, 300, 128),
                                       (96, 33, 512), (5, 10, 24), (3, 4, 6)])
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
