"""The benchmark's reference arm on CPU (it times the oracle, so it runs
without a GPU): one JSON line with the contract's keys, the same metric,
unit and workload as the GPU arm's headline, and an e2e entry that moves no
bytes between host and device."""
from __future__ import annotations

import json


def test_reference_arm_line():
    import bench
    args = type("A", (), dict(steps=1, warmup=0, ref_seconds=0.0))()
    res = bench.reference_arm(args, 1, 0)
    json.dumps(res)  # one JSON line
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "impl", "cpu_baseline", "e2e"):
        assert k in res, k
    assert res["metric"] == bench.METRIC   # the GPU arm's metric
    assert res["impl"] == "reference"
    assert res["unit"] == "GB/s" and res["higher_is_better"] is True
    assert res["value"] > 0 and res["steps"] == 1 and res["n_gpus"] == 1
    assert res["config"]["workload"].startswith("batched-decode")
    cb = res["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == res["value"]
    e2e = res["e2e"]
    assert e2e["value"] == res["value"] and e2e["unit"] == res["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _args(**kw):
    base = dict(no_sub=False, skip_prefill=False)
    base.update(kw)
    return type("A", (), base)()


def test_multi_rank_plan_has_no_prefill():
    """The prefill multicasts K/V tiles between the CTAs of a cluster, which
    is for single-GPU jobs only: a job of two or more ranks plans no prefill
    measurement, and the prefill measurements refuse to run there."""
    import bench
    one = [k for k, _, _ in bench.sub_plan(_args(), 1)]
    assert "prefill" in one and "prefill_fp8" in one
    assert ("prefill", "prefill_128k", 131072) in bench.sub_plan(_args(), 1)
    for ws in (2, 4, 8):
        kinds = [k for k, _, _ in bench.sub_plan(_args(), ws)]
        assert not set(kinds) & set(bench.PREFILL_KINDS)
        assert "verify" in kinds and "mla" in kinds
        import pytest
        with pytest.raises(RuntimeError):
            bench.require_single_gpu(ws, "prefill")
    bench.require_single_gpu(1, "prefill")
    assert bench.sub_plan(_args(no_sub=True), 1) == []


def test_prefill_runs_only_through_the_plan():
    """Every call of the prefill measurements in the GPU arm goes through
    the plan's dispatch (so the world-size filter above covers them all),
    and each of them starts with the single-GPU guard."""
    import inspect

    import bench
    src = inspect.getsource(bench.gpu_arm)
    for fn in ("prefill_sub", "prefill_fp8_sub"):
        calls = [ln.strip() for ln in src.splitlines()
                 if f"{fn}(" in ln and not ln.strip().startswith("def ")]
        assert calls, fn
        for c in calls:  # the plan's dispatch, or the guarded --only path
            assert c.startswith(f"{fn}(name, size)") or "args.prefill_tokens" in c, c
        body = src[src.index(f"def {fn}("):]
        first = [ln.strip() for ln in body.splitlines()[1:]
                 if ln.strip() and not ln.strip().startswith("#")][0]
        assert first.startswith("require_single_gpu(ws"), first


def test_gpus_flag_must_match_world_size(monkeypatch, capsys):
    import pytest

    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "8"])
    assert e.value.code == 2
    assert "world size 1" in capsys.readouterr().err
