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
