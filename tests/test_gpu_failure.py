"""The device-side failure path, exercised without a fault: a kernel's wait that nothing will
satisfy gives up after its limit, records the timeout in the device status word and returns; the
host reads and clears the word and the context keeps working."""
import time

import pytest
import torch

from ulysses_sequence_all_gb300 import binding as B
from ulysses_sequence_all_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared():
    assert torch.cuda.is_available()
    assert B.ulysses_device_status() == 0, "status word not clean before the test"
    t0 = time.perf_counter()
    B.ulysses_selftest_wait_timeout(20_000)  # 20 ms limit
    status = B.ulysses_device_status()       # synchronises
    elapsed = time.perf_counter() - t0
    assert status == 1, f"expected the timeout bit, got {status:#x}"
    assert 0.015 < elapsed < 5.0, elapsed
    assert B.ulysses_device_status() == 0, "reading the word must clear it"

    # the context is still usable: a relayout afterwards is exact and reports no timeout
    cfg = wl.TINY
    plan = B.ulysses_plan(cfg.W, cfg.b, cfg.seq_splits, cfg.head_splits, cfg.d, cfg.dtype)
    x = [t.cuda() for t in wl.seq_side_inputs(cfg, "cpu")]
    y = [torch.empty(cfg.head_side_shape(r), dtype=torch.bfloat16, device="cuda") for r in range(cfg.W)]
    z = [torch.empty_like(t) for t in x]
    B.ulysses_a2a_4d(plan, 0, x, y)
    B.ulysses_a2a_4d(plan, 1, y, z)
    assert B.ulysses_device_status() == 0
    for a, b in zip(z, x):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_selftest_rejects_bad_limits():
    for bad in (0, 2_000_000):
        with pytest.raises(B.UlyssesError) as ei:
            B.ulysses_selftest_wait_timeout(bad)
        assert ei.value.status == B.ULY_EINVAL
