"""Failure handling on the device without a fault: the bounded wait that
guards every barrier in the kernels gives up on a phase that nothing
completes, reports a timeout, and leaves the context usable; a call after it
still matches the oracle."""
import time

import pytest
import torch

from paged_fp8_kv_decode_gb300 import workloads as W
from test_gpu_parity import B, run_and_compare  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable(B):
    r = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    B.pfkv_selftest_bounded_wait(r)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(r.item()) == B.PFKV_FLAG_DEVICE_TIMEOUT | 0x100
    assert 0.09 < elapsed < 10.0      # the 100 ms limit, not a hang
    run_and_compare(W.spec_tiny(), label="after the timed-out wait")
