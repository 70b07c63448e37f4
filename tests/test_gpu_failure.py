"""Failure detection without a GPU fault: a bounded wait that nothing ends
gives up, reports DSPARK_ERR_TIMEOUT through the workspace status block, and
leaves the context usable for the next call."""
import time

import pytest

from serving_draft_verify_gb300 import workloads as wl
from tests.gpu_harness import gpu_draft

pytestmark = pytest.mark.gpu

DSPARK_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def dsv():
    import serving_draft_verify_gb300 as m
    m.load()
    return m


def test_bounded_wait_times_out(dsv):
    t0 = time.perf_counter()
    ws = dsv._binding.bounded_wait(2_000_000)             # 2 ms
    assert dsv.workspace_status(ws) == DSPARK_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the context still runs work: a small draft block completes with status 0
    cfg = wl.scaled(wl.QWEN3_8B, B=4, gamma=2, V=1024, H=16)
    out = gpu_draft(dsv, wl.make_draft_inputs(cfg))
    assert out["x"].shape == (4, 2)


def test_bounded_wait_rejects_long_limits(dsv):
    with pytest.raises(Exception):
        dsv._binding.bounded_wait(10_000_000_000)         # 10 s: refused on the host
