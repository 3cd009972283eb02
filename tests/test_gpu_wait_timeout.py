"""Failure detection on the GPU without a fault: a cooperative merger's
bounded wait for arrivals is made to run out, and the call must return with
PD_DEV_WAIT_TIMEOUT in the device status word, merge the groups that were
not affected, leave the affected group's output untouched, keep every later
call on that scratch in bounds (reporting PD_DEV_BAD_SCRATCH) and give
correct results again once the scratch is initialised anew.

The wait is made to run out from the host: the arrival counter of one group
is set to -1 before the call, so the count stops one short of the segments
and the group's mergers wait for an arrival that never comes; a test-only
option shortens their wait to 2 ms."""

import time

import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W
from gpu_helpers import check, run, scratch_for

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    pd.build()
    pd.paged_decode_device_status(reset=True)
    yield
    assert pd.paged_decode_device_status(reset=True) == 0


def _rows_of_other_heads(case, skip_heads):
    return [(t, h) for t in range(case.q.shape[0]) for h in range(case.num_q_heads)
            if h not in skip_heads]


def _timed_call(g, sc, opts):
    out = torch.full_like(g.q, SENTINEL)
    t0 = time.time()
    run(g, scratch=sc, opts=opts, out=out)
    return out, time.time() - t0


@pytest.mark.parametrize("merge", [2, 1])
def test_merge_gives_up_and_scratch_recovers(merge):
    case = W.spec_decode_hnd(4, 4096, seed=71)
    g = case.to("cuda")
    sc = scratch_for(case)
    opts = pd.options(merge=merge, segments=8, wait_limit_us=2000)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, g.block_table.shape[1], sms,
                                scratch=sc, opts=opts)
    assert plan["merge"] == merge and plan["row_groups"] == 1 and plan["max_segments"] == 8
    G = case.num_q_heads // case.num_kv_heads
    group0 = set(range(G))            # q heads of kv head 0 (group 0)
    ref_rows = _rows_of_other_heads(case, group0)
    ref = oracle.attention(case, rows=ref_rows)
    pd.paged_decode_device_status(reset=True)

    # group 0's arrival count starts at -1 (cooperative merge: its mergers
    # wait for an arrival that never comes) or at the segment count (last
    # arriver: no arrival is the last one)
    sc.counters()[0] = -1 if merge == 2 else 8
    out, dt = _timed_call(g, sc, opts)
    assert dt < 5.0
    st = pd.paged_decode_device_status(reset=True)
    assert st & pd.DEV_BAD_SCRATCH
    if merge == 2:
        assert st & pd.DEV_WAIT_TIMEOUT
    check(case, out, rows=ref_rows, ref=ref)          # the other groups were merged
    assert torch.all(out[:, :G] == SENTINEL)           # group 0 was not written

    # the same scratch without a new initialisation: group 0 is skipped and
    # reported, nothing waits, every other group is still right
    out, dt = _timed_call(g, sc, opts)
    assert dt < 5.0
    st = pd.paged_decode_device_status(reset=True)
    assert st & pd.DEV_BAD_SCRATCH and not st & pd.DEV_WAIT_TIMEOUT
    check(case, out, rows=ref_rows, ref=ref)
    assert torch.all(out[:, :G] == SENTINEL)

    # initialised again: the whole call is right and the counters end at zero
    sc.reinit()
    out, _ = _timed_call(g, sc, opts)
    assert pd.paged_decode_device_status(reset=True) == 0
    check(case, out)
    assert int(sc.counters().abs().sum()) == 0
