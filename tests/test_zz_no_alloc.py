"""paged_decode_attn_static: the decode call for callers that cannot allocate
device memory (a host framework that owns every device allocation, a
runtime that forbids allocating after start-up), which uses the library's
own fixed scratch array instead of a caller buffer.

It must give the same outputs as paged_decode_attn with a caller scratch,
within the dtype's tolerance, on two calls in a row (the second one reuses
the array the first one left behind), and both must match the oracle.  The
calls after the first one (which looks up the array's address) must not
change the device's free memory.  This file is collected last; it passes on
its own in a fresh process and after the other tests.
"""

import pytest
import torch

import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W
from gpu_helpers import TOL, check, scratch_for

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20          # PD_STATIC_SCRATCH_BYTES
STATIC_COUNTER_BYTES = 512 << 10  # PD_STATIC_COUNTER_BYTES


def _static(g, out=None):
    out = torch.empty_like(g.q) if out is None else out
    pd.paged_decode_attn_static(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, out,
                                g.num_q_heads, g.num_kv_heads, g.head_size, g.page_size,
                                g.max_query_len, g.window, g.scale, g.layout)
    return out


def _static_plan(c):
    """The plan a static call makes: the library's array as the scratch."""
    d = pd.PdScratch()
    d.data = 1 << 30
    d.bytes = STATIC_BYTES
    d.counter_slots = c.num_seqs * c.num_kv_heads * pd.COUNTERS_PER_PAIR
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return pd.paged_decode_plan(c.num_seqs, c.num_q_heads, c.num_kv_heads, c.head_size,
                                c.page_size, c.max_query_len, c.window, c.block_table.shape[1],
                                sms, scratch_desc=d)


def test_static_scratch_matches_caller_scratch_on_two_calls():
    pd.build()
    text = open(pd.HEADER).read()
    assert "#define PD_STATIC_SCRATCH_BYTES (16u << 20)" in text
    assert "#define PD_STATIC_COUNTER_BYTES (512u << 10)" in text
    cases = [
        # one long sequence: split over many segments, merged in the kernel
        W.spec_decode_hnd(4, 8192, seed=31),
        # a batch of uneven lengths with an empty slot
        W.make_case("static_batch", seed=32, dtype=torch.float16, head_size=256,
                    num_q_heads=16, num_kv_heads=2, page_size=32, max_query_len=3,
                    seq_lens=[2500, 0, 37, 900], layout=W.NHD),
    ]
    # the long sequence really takes the split-KV path with the array
    p0 = _static_plan(cases[0])
    assert p0["max_parts"] > 1 and p0["merge"] > 0 and p0["scratch_needed"] <= STATIC_BYTES
    gpu = [c.to("cuda") for c in cases]
    refs = [pd.decode_case(g, scratch=scratch_for(c)) for g, c in zip(gpu, cases)]
    outs = [torch.empty_like(g.q) for g in gpu]
    again = torch.empty_like(gpu[0].q)
    torch.cuda.synchronize()
    _static(gpu[0], again)  # the first call looks up the array's address
    torch.cuda.synchronize()
    # (every output buffer exists before this point, and the comparisons,
    # which allocate through torch, come after the last measurement)
    free0 = torch.cuda.mem_get_info()[0]
    for g, out in zip(gpu, outs):  # two calls in a row
        _static(g, out)
    # and the first case again, on the array the first two calls left
    _static(gpu[0], again)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "a static call changed the free device memory"
    for c, ref, out in zip(cases + cases[:1], refs + refs[:1], outs + [again]):
        assert torch.isfinite(out.float()).all()
        err = float((out.double() - ref.double()).abs().max())
        assert err <= TOL[c.dtype], f"{c.name}: max abs difference {err:.3g}"
        check(c, out)  # and against the oracle
    assert pd.paged_decode_device_status(reset=True) == 0
