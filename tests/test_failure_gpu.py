"""The failure path on the GPU, without faulting or hanging it: every kernel
waits on mbarriers with a bound; pkv_selftest_bounded_wait runs that wait on
a barrier nothing arrives on.  The wait must give up, the device error word
must read PKV_EDEV_TIMEOUT (once: reading clears it), and the context must
stay usable for a normal decode checked against the oracle."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import paged_kv_asymmetric_gb300 as pkv
from paged_kv_asymmetric_gb300 import workloads as wl
from tests import gpu_path, refs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert pkv.get_device_error() == pkv.EDEV_NONE
    t0 = time.perf_counter()
    pkv.selftest_bounded_wait(20_000)  # 20 ms
    code = pkv.get_device_error()  # synchronises
    dt = time.perf_counter() - t0
    assert code == pkv.EDEV_TIMEOUT
    assert 0.015 < dt < 5.0
    assert pkv.get_device_error() == pkv.EDEV_NONE  # reading cleared it
    # the context is still usable: a tiny decode matches the oracle
    w = wl.tiny("decode")
    dw = wl.to_device(w)
    gpu_path.write_all(dw)
    _, _, out, _ = gpu_path.decode(dw, 3)
    o, _ = gpu_path.oracle_rows(w)
    refs.assert_close(gpu_path.host(out), o, **gpu_path.tol(w), what="decode after timeout")
    assert pkv.get_device_error() == pkv.EDEV_NONE


def test_selftest_rejects_bad_limits():
    for bad in (0, -5, 2_000_001):
        with pytest.raises(pkv.PkvError):
            pkv.selftest_bounded_wait(bad)
