"""The outputs of the benchmark's timed pattern, checked: bench.py's sweep
builds replicas of each case, captures one CUDA graph per step (one call per
case, replicas alternating between graphs, one shared scratch, calls
overlapping through programmatic dependent launch) and replays the graphs
back to back.  Here the same pattern runs on a reduced sweep, and after the
replays every call's output is checked on sampled rows against the oracle,
with the counters left at zero; both with the bench's early reads (a call
reads its block table, seq_lens and older pages while the previous call
finishes) and with every call waiting first."""

import pytest
import torch

import bench
import paged_split_kv_02_gb300 as pd
from gpu_helpers import check, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("early", [0, 1])
def test_bench_step_graph_replays_match_the_oracle(early):
    pd.build()
    device = "cuda"
    l2 = int(torch.cuda.get_device_properties(0).L2_cache_size)
    # (1024 keys: a cooperative launch under early reads; 4096 and 16384: a
    # plain one)
    only = {(1, 4096), (4, 4096), (2, 128), (3, 16384), (2, 1024)}
    opts = pd.options(early_reads=1) if early else None
    # (two replicas per case are enough here: the check is of the outputs)
    cases = bench.build_sweep(device, l2, only=only, rep_factor=0.0)
    first = next(iter(cases.values()))[0]
    scratch = pd.Scratch(1, first.num_q_heads, first.num_kv_heads, first.head_size,
                         max(bench.MS), max_splits=256, device=device)
    outs = {k: [torch.empty_like(r.q) for r in reps] for k, reps in cases.items()}
    stream = torch.cuda.Stream(device=device)
    keys = sorted(cases)

    def call(k, r):
        pd.decode_case(cases[k][r], out=outs[k][r], scratch=scratch, stream=stream, opts=opts)

    with torch.cuda.stream(stream):
        for k in keys:
            for r in range(len(cases[k])):
                call(k, r)
    torch.cuda.synchronize()
    graphs = []
    for gi in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in keys:
                call(k, gi % len(cases[k]))
        graphs.append(g)
    for o in (o for lst in outs.values() for o in lst):
        o.fill_(7.0)  # every output below comes from a replay
    with torch.cuda.stream(stream):
        for i in range(6):
            graphs[i % 2].replay()
    torch.cuda.synchronize()
    assert pd.paged_decode_device_status(reset=True) == 0
    assert int(scratch.counters().abs().sum()) == 0, "counters not left at zero"
    for k in keys:
        for r in range(min(2, len(cases[k]))):
            c = cases[k][r].to("cpu")
            check(c, outs[k][r], rows=sample_rows(c, 24, seed=k[0] + k[1] + r))
