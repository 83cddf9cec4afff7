"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The attention kernels wait on shared-memory barriers for their staged K/V copies; every
such wait gives up after a limit, sets PKV_DEVERR_PIPELINE_TIMEOUT and leaves.  The
self-test entry point runs that wait on a barrier that nothing completes, with a short
limit: the host must read the bit, and the context must stay usable (a decode step right
after still matches the oracle).
"""
import time

import pytest
import torch

import paged_kv_cache_275_gb300 as pkv
from gpu_util import assert_close, device_errors, gpu_step, oracle_step
from workloads import make_decode_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [20_000, 2_000_000])
def test_wait_that_runs_out_is_reported_and_context_survives(limit_ns):
    assert device_errors() == 0
    t0 = time.perf_counter()
    pkv.selftest_wait_timeout(limit_ns)
    bits = pkv.get_and_clear_device_error()
    elapsed = time.perf_counter() - t0
    assert bits == pkv.DEVERR_PIPELINE_TIMEOUT
    assert elapsed >= limit_ns * 1e-9  # it waited at least the limit ...
    assert elapsed < 5.0               # ... and then gave up
    # The context is usable: a full decode step right after is correct and flags nothing.
    c = make_decode_case("qwen3_0.6b", seed=3)
    ref, _, _ = oracle_step(c)
    g = c.to("cuda")
    out = gpu_step(g, 0)
    torch.cuda.synchronize()
    assert_close(out, ref, "decode after a timed-out wait")
    assert device_errors() == 0

