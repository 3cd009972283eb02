"""Calls issued back to back on one stream, with no host synchronisation in
between, all sharing one scratch buffer, checked against the oracle after a
single synchronisation at the end.

Consecutive launches overlap through programmatic dependent launch (a grid
sets up while the previous one finishes), and every call relies on the
previous one leaving the split-KV counters at zero: these tests exercise
both.  Between calls some inputs change on the device (seq_lens, block-table
entries), ordered by the stream only.  The graph test replays a captured
sequence of calls with inputs changed between replays (the "graph replay"
case of the pages' test plan, ROCm/vllm PR #1330, "Test plan"; counters
zeroed once and left zeroed by every launch, as make_scratch on the
vllm.v1.attention.ops.rocm_rdna_hip page describes)."""

import dataclasses

import pytest
import torch

import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W
from gpu_helpers import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pd.build()
    yield
    assert pd.paged_decode_device_status(reset=True) == 0


def _cases():
    """(cpu case, launch options) of a mixed sequence of calls."""
    return [
        (W.spec_decode_hnd(4, 4096, seed=61), None),                          # cooperative merge
        (W.spec_decode_hnd(1, 2048, seed=62), pd.options(merge=1, segments=8)),  # last arriver
        (W.sliding_window(torch.float16, 4, 4096, seed=63), None),
        (W.wide_head(8, 2048, seed=64), None),                                # row groups
        (W.batched_hybrid_pages(seed=65, num_seqs=8, max_len=3000), None),    # a batch
        (W.make_varlen_case("b2b_varlen", seed=66, q_lens=[3, 1, 0, 4], pad_tokens=2,
                            dtype=torch.bfloat16, head_size=128, num_q_heads=32,
                            num_kv_heads=8, page_size=16, seq_lens=[2100, 700, 50, 1500]),
         pd.options(segments=6)),
        (W.spec_decode_hnd(3, 1024, seed=67), pd.options(cluster=4, segments=8)),  # clusters
        (W.spec_decode_hnd(2, 2048, seed=68), pd.options(path=3, segments=4)),     # tcgen05
    ]


def _shared_scratch(cases):
    nbytes = max(pd.paged_decode_scratch_bytes(c.num_seqs, c.num_q_heads, c.num_kv_heads,
                                               c.head_size, c.max_query_len, 256)
                 for c, _ in cases)
    pairs = max(c.num_seqs * c.num_kv_heads for c, _ in cases)
    # counters for `pairs` (sequence, kv head) pairs (one kv head per
    # "sequence"), in front of the largest partial area any case asks for
    return pd.Scratch(pairs, 1, 1, 64, 1, nbytes=nbytes + pairs * 4 * pd.COUNTERS_PER_PAIR + 256)


def _mutated(case, new_len, swap):
    """The case with seq_lens[0] = new_len and block-table entries swap[0],
    swap[1] of sequence 0 exchanged (both on the host copy)."""
    bt = case.block_table.clone()
    a, b = swap
    bt[0, a], bt[0, b] = case.block_table[0, b], case.block_table[0, a]
    sl = case.seq_lens.clone()
    sl[0] = new_len
    lens = list(case.seq_lens_host)
    lens[0] = new_len
    return dataclasses.replace(case, seq_lens=sl, seq_lens_host=lens, block_table=bt)


def test_back_to_back_calls_share_one_scratch():
    cases = _cases()
    sc = _shared_scratch(cases)
    gpu = [(c.to("cuda"), o) for c, o in cases]
    stream = torch.cuda.Stream()
    outs = []
    changed = _mutated(cases[0][0], 3001, (0, 5))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for g, o in gpu:
            outs.append(pd.decode_case(g, scratch=sc, opts=o, stream=stream))
        # the first case again, its seq_lens and two block-table entries
        # changed on the device by the stream (no host sync before or after)
        g0 = gpu[0][0]
        g0.seq_lens.copy_(changed.seq_lens.to("cuda", non_blocking=True))
        g0.block_table.copy_(changed.block_table.to("cuda", non_blocking=True))
        outs.append(pd.decode_case(g0, scratch=sc, stream=stream))
        # and every case once more, in reverse order, on the same scratch
        for g, o in reversed(gpu[1:]):
            outs.append(pd.decode_case(g, scratch=sc, opts=o, stream=stream))
    torch.cuda.synchronize()
    expected = [c for c, _ in cases] + [changed] + [c for c, _ in reversed(cases[1:])]
    assert len(outs) == len(expected)
    for c, out in zip(expected, outs):
        check(c, out)
    assert int(sc.counters().abs().sum()) == 0, "counters not left at zero"
    assert pd.paged_decode_device_status(reset=True) == 0


def _early(o):
    """The launch options `o` with early reads on."""
    d = {n: getattr(o, n) for n, _ in o._fields_} if o is not None else {}
    d["early_reads"] = 1
    return pd.options(**d)


def test_back_to_back_calls_with_early_reads():
    """Every call reads its block table, seq_lens and older pages while the
    previous call finishes (its own inputs were written before that call
    started); outputs, q and the scratch wait for it."""
    cases = _cases()
    sc = _shared_scratch(cases)
    gpu = [(c.to("cuda"), _early(o)) for c, o in cases]
    stream = torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(2):
            for g, o in gpu:
                outs.append(pd.decode_case(g, scratch=sc, opts=o, stream=stream))
    torch.cuda.synchronize()
    expected = [c for c, _ in cases] * 2
    for c, out in zip(expected, outs):
        check(c, out)
    assert int(sc.counters().abs().sum()) == 0, "counters not left at zero"
    assert pd.paged_decode_device_status(reset=True) == 0


def test_graph_replays_with_inputs_changed_between_replays():
    cases = [_cases()[i] for i in (0, 1, 4, 6)]
    sc = _shared_scratch(cases)
    gpu = [(c.to("cuda"), o) for c, o in cases]
    outs = [torch.empty_like(g.q) for g, _ in gpu]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for (g, o), out in zip(gpu, outs):   # outside capture: tensor maps, attributes
            pd.decode_case(g, out=out, scratch=sc, opts=o, stream=stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for (g, o), out in zip(gpu, outs):
            pd.decode_case(g, out=out, scratch=sc, opts=o, stream=stream)
    # replay 1: the inputs as captured
    versions = [[c for c, _ in cases]]
    # replay 2: the first sequence shorter and two of its pages exchanged,
    # the batch's first sequence shorter by a few keys
    v2 = list(versions[0])
    v2[0] = _mutated(cases[0][0], 2500, (1, 7))
    # (shorter only: slots past a sequence's last key hold NaN)
    v2[2] = _mutated(cases[2][0], max(0, int(cases[2][0].seq_lens_host[0]) - 5), (0, 0))
    versions.append(v2)
    # replay 3: back to the originals
    versions.append(versions[0])
    for vers in versions:
        with torch.cuda.stream(stream):
            for (g, _), c in zip(gpu, vers):
                g.seq_lens.copy_(c.seq_lens.to("cuda", non_blocking=True))
                g.block_table.copy_(c.block_table.to("cuda", non_blocking=True))
            graph.replay()
        torch.cuda.synchronize()
        for c, out in zip(vers, outs):
            check(c, out)
        assert int(sc.counters().abs().sum()) == 0, "counters not left at zero"
    assert pd.paged_decode_device_status(reset=True) == 0
