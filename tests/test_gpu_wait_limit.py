"""The library's bounded waits end: a wait on an mbarrier that nothing
completes gives up after its limit, reports PA_ERR_TIMEOUT through the error
word, and the context keeps working (no fault, no hang)."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _gpu import TOL, max_err, oracle_pools, run_gpu

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    import paged_kv_cache_writes_gb300 as pa
    assert pa.pa_get_device_error() == 0
    t0 = time.monotonic()
    pa.pa_selftest_wait_timeout()
    code = pa.pa_get_device_error()          # synchronises
    waited = time.monotonic() - t0
    assert code == 5                          # PA_ERR_TIMEOUT
    assert 0.5 < waited < 30.0
    # the same context decodes correctly afterwards
    b = W.decode_batch("after-timeout", [1, 40, 333], 8, 2, 128, 16, "bf16", seed=61)
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    assert max_err(dev.out, oracle.decode_batch(b, kp, vp)) <= TOL["bf16"]
