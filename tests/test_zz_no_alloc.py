"""paged_decode_attn_static: the decode call for callers that cannot allocate
device memory (a host framework that owns every device allocation, a
runtime that forbids allocating after start-up), which uses the library's
own fixed scratch array instead of a caller buffer.

It must give the same outputs as paged_decode_attn with a caller scratch,
within the dtype's tolerance, on two calls in a row (the second one reuses
the array the first one left behind).  This file is collected last; it
passes on its own in a fresh process and after the other tests.
"""

import pytest
import torch

import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W
from gpu_helpers import TOL, scratch_for

pytestmark = pytest.mark.gpu


def _static(g):
    out = torch.empty_like(g.q)
    pd.paged_decode_attn_static(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, out,
                                g.num_q_heads, g.num_kv_heads, g.head_size, g.page_size,
                                g.max_query_len, g.window, g.scale, g.layout)
    return out


def test_static_scratch_matches_caller_scratch_on_two_calls():
    pd.build()
    cases = [
        # one long sequence: split over many segments, merged in the kernel
        W.spec_decode_hnd(4, 8192, seed=31),
        # a batch of uneven lengths with an empty slot
        W.make_case("static_batch", seed=32, dtype=torch.float16, head_size=256,
                    num_q_heads=16, num_kv_heads=2, page_size=32, max_query_len=3,
                    seq_lens=[2500, 0, 37, 900], layout=W.NHD),
    ]
    gpu = [c.to("cuda") for c in cases]
    refs = [pd.decode_case(g, scratch=scratch_for(c)) for g, c in zip(gpu, cases)]
    torch.cuda.synchronize()
    outs = [_static(g) for g in gpu]  # two calls in a row
    torch.cuda.synchronize()
    for c, ref, out in zip(cases, refs, outs):
        assert torch.isfinite(out.float()).all()
        err = float((out.double() - ref.double()).abs().max())
        assert err <= TOL[c.dtype], f"{c.name}: max abs difference {err:.3g}"
    # and again in the other order, on the array the first two calls left
    again = _static(gpu[0])
    torch.cuda.synchronize()
    assert float((again.double() - refs[0].double()).abs().max()) <= TOL[cases[0].dtype]
    assert pd.paged_decode_device_status(reset=True) == 0
