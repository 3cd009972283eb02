"""The CUDA path against the fp64 oracle, element by element, on the same
seeded inputs (through the C ABI).

Sizes here are ones the oracle finishes in seconds; they span several
stages, several segments and a ragged last page.  Tolerances: max-abs
2e-3 (fp16) and 1e-2 (bf16) on O(1)-scaled outputs."""

import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W
from gpu_helpers import TOL, check, run, sample_rows, scratch_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pd.build()
    yield
    assert pd.paged_decode_device_status(reset=True) == 0


def _parity(case, splits=256, opts=None):
    g = case.to("cuda")
    sc = scratch_for(case, splits)
    out = run(g, scratch=sc, opts=opts)
    err = check(case, out)
    assert int(sc.counters().abs().sum()) == 0, "counters not left at zero"
    return out, err


def test_single_seq_nhd():
    _parity(W.single_seq_nhd())


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [128, 1024, 4096])
def test_spec_decode_hnd(M, L):
    _parity(W.spec_decode_hnd(M, L))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("L", [1024, 4096])
def test_sliding_window(dtype, M, L):
    _parity(W.sliding_window(dtype, M, L))


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_wide_head(M):
    _parity(W.wide_head(M, 4096))


def test_batched_hybrid_pages_small():
    _parity(W.batched_hybrid_pages(num_seqs=16, max_len=3000))


@pytest.mark.parametrize("segments,cluster", [(1, 1), (2, 1), (3, 1), (7, 1), (16, 1),
                                              (2, 2), (4, 4), (8, 8), (16, 8), (24, 8), (12, 4)])
def test_forced_splits_agree(segments, cluster):
    case = W.spec_decode_hnd(4, 4096, seed=3)
    out, _ = _parity(case, opts=pd.options(segments=segments, cluster=cluster))


@pytest.mark.parametrize("merge", [1, 2])
@pytest.mark.parametrize("M,L,seg", [(1, 4096, 19), (4, 4096, 5), (4, 16384, 19), (2, 1024, 16),
                                     (3, 2048, 3)])
def test_merge_modes(merge, M, L, seg):
    """Last-arriving CTA vs the last K arrivals of a cooperative grid."""
    _parity(W.spec_decode_hnd(M, L, seed=14), opts=pd.options(segments=seg, merge=merge))


@pytest.mark.parametrize("k", [1, 2, 4, 16])
@pytest.mark.parametrize("early", [0, 1])
def test_merger_counts(k, early):
    """The cooperative merge with 1..16 mergers (each a D/K slice of every
    part), launched cooperatively and, with early reads, plainly."""
    _parity(W.spec_decode_hnd(4, 4096, seed=17),
            opts=pd.options(segments=19, merge=2, mergers=k, early_reads=early))


def test_cooperative_merge_refused_when_grid_does_not_fit():
    case = W.spec_decode_hnd(2, 1024, seed=15)
    g = case.to("cuda")
    rc = pd.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens,
                              torch.empty_like(g.q), g.num_q_heads, g.num_kv_heads,
                              g.head_size, g.page_size, g.max_query_len, g.window, g.scale,
                              g.layout, scratch_for(case), opts=pd.options(segments=64, merge=2),
                              check=False)
    assert rc == -1


@pytest.mark.parametrize("merge", [1, 2])
def test_batched_uneven_segments(merge):
    """A batch whose sequences split into different numbers of segments (some
    fewer than the cooperative mergers, some unsplit, one empty)."""
    case = W.make_case("uneven", seed=16, dtype=torch.bfloat16, head_size=128, num_q_heads=16,
                       num_kv_heads=2, page_size=16, max_query_len=3,
                       seq_lens=[3000, 200, 40, 0, 1, 1100, 600], layout=W.HND)
    # 7 sequences x 2 kv heads x 1 row group x 10 segments = 140 CTAs: one
    # wave, so the cooperative merge is allowed
    _parity(case, opts=pd.options(segments=10, merge=merge, row_groups=1))


@pytest.mark.parametrize("kg,ns", [(1, 2), (1, 5), (2, 2), (2, 6), (3, 6), (4, 4)])
def test_warp_groups_and_stages(kg, ns):
    _parity(W.spec_decode_hnd(2, 1024, seed=4), opts=pd.options(key_groups=kg, stages=ns))


@pytest.mark.parametrize("rg", [2, 4])
def test_row_groups(rg):
    _parity(W.wide_head(8, 1024, seed=5), opts=pd.options(row_groups=rg))


@pytest.mark.parametrize("layout", [W.NHD, W.HND])
@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_layouts_and_head_sizes(layout, packed, D):
    case = W.make_case("layouts", seed=6, dtype=torch.bfloat16, head_size=D, num_q_heads=8,
                       num_kv_heads=2, page_size=32, max_query_len=3, seq_lens=[300, 77, 1],
                       layout=layout, packed=packed, window=0)
    _parity(case)


@pytest.mark.parametrize("P", [16, 32, 528, 544, 784, 1056])
def test_page_sizes(P):
    case = W.make_case("pages", seed=7, dtype=torch.float16, head_size=128, num_q_heads=16,
                       num_kv_heads=2, page_size=P, max_query_len=4,
                       seq_lens=[2 * P + 5, P, 3], layout=W.HND)
    _parity(case)


@pytest.mark.parametrize("Hq,Hkv,M,lens", [
    (12, 4, 3, [2500, 700, 33]),   # G = 3: packed rows -> tokens by division
    (10, 2, 4, [2500, 700, 33]),   # G = 5, 20 rows: three 8-row n-tiles in a batch
    (24, 4, 2, [6000]),            # G = 6, one sequence: many segments, cooperative merge
    (6, 6, 5, [1800, 5]),          # G = 1 (no grouping), M = 5
])
def test_head_ratios_not_powers_of_two(Hq, Hkv, M, lens):
    case = W.make_case("ratios", seed=17, dtype=torch.bfloat16, head_size=128, num_q_heads=Hq,
                       num_kv_heads=Hkv, page_size=16, max_query_len=M, seq_lens=lens,
                       layout=W.HND)
    _parity(case)


def test_one_scratch_across_merge_kinds():
    """One scratch serves calls whose merges differ (cooperative, last
    arriver, cluster partials, a batch, unsplit) and whose partial layouts
    overlap: every call must be right whatever the previous one left in the
    partial area, and leave the counters at zero."""
    cases = [
        (W.spec_decode_hnd(4, 4096, seed=21), None),                        # cooperative
        (W.wide_head(1, 8192, seed=22), None),                              # many parts
        (W.spec_decode_hnd(2, 4096, seed=23), pd.options(merge=1)),         # last arriver
        (W.spec_decode_hnd(4, 4096, seed=24), pd.options(cluster=4, segments=16)),
        (W.batched_hybrid_pages(num_seqs=8, max_len=3000, seed=25), None),  # a batch
        (W.spec_decode_hnd(1, 1024, seed=26), pd.options(merge=2, key_groups=1, stages=2)),
        (W.spec_decode_hnd(3, 128, seed=27), None),                         # unsplit
        (W.spec_decode_hnd(4, 4096, seed=21), None),
    ]
    sc = pd.Scratch(8, 16, 2, 512, 4, max_splits=64)
    for case, opts in cases:
        g = case.to("cuda")
        out = run(g, scratch=sc, opts=opts)
        check(case, out)
        assert int(sc.counters().abs().sum()) == 0, case.name


def test_empty_and_short_sequences():
    case = W.make_case("edge", seed=8, dtype=torch.bfloat16, head_size=128, num_q_heads=8,
                       num_kv_heads=1, page_size=16, max_query_len=4,
                       seq_lens=[0, 1, 2, 3, 4, 5, 16, 17, 0], layout=W.HND, window=3)
    out, _ = _parity(case)
    assert torch.all(out[0:4] == 0) and torch.all(out[-4:] == 0)


def test_windows():
    for w in (1, 2, 15, 16, 17, 100, 5000):
        case = W.make_case("win", seed=9, dtype=torch.float16, head_size=256, num_q_heads=8,
                           num_kv_heads=1, page_size=32, max_query_len=4, seq_lens=[1500, 40],
                           layout=W.HND, window=w, window_pages_only=True)
        _parity(case)


def test_outputs_stay_order_one_with_shifted_values():
    """V = N(0,1) + 1 keeps the outputs near 1 at long contexts, where a
    plain N(0,1) output shrinks like 1/sqrt(keys)."""
    case = W.make_case("shifted", seed=10, dtype=torch.bfloat16, head_size=128, num_q_heads=32,
                       num_kv_heads=8, page_size=16, max_query_len=4, seq_lens=[8192],
                       layout=W.HND, v_mean=1.0)
    out, (err, rel) = _parity(case)
    assert out.float().abs().mean() > 0.5


def test_negative_control_detects_a_wrong_page():
    """A block-table entry pointing at another page of the sequence (one
    page read twice, one never) on the GPU side only must break parity."""
    case = W.spec_decode_hnd(2, 1024, seed=11)
    g = case.to("cuda")
    bt = g.block_table.clone()
    bt[0, 3] = g.block_table[0, 40]
    g.block_table = bt
    out = run(g, scratch=scratch_for(case))
    with pytest.raises(AssertionError):
        check(case, out)


def test_negative_control_detects_a_wrong_scale():
    case = W.spec_decode_hnd(1, 1024, seed=12)
    g = case.to("cuda")
    g.scale = case.scale * 2.0
    out = run(g, scratch=scratch_for(case))
    with pytest.raises(AssertionError):
        check(case, out)


@pytest.mark.parametrize("M,L,D,layout,dtype,window,seqs", [
    (1, 40, 128, W.HND, torch.bfloat16, 0, None),
    (4, 300, 128, W.HND, torch.bfloat16, 0, None),
    (4, 4100, 128, W.HND, torch.bfloat16, 0, None),
    (2, 1037, 128, W.NHD, torch.float16, 0, None),
    (3, 2048, 64, W.HND, torch.float16, 300, None),
    (4, 2000, 256, W.HND, torch.float16, 512, None),
    (2, 700, 256, W.NHD, torch.bfloat16, 0, None),
    (3, 0, 128, W.HND, torch.bfloat16, 0, [900, 0, 17, 2500, 1]),
])
def test_tensor_memory_path(M, L, D, layout, dtype, window, seqs):
    """The tcgen05 / tensor-memory consumer (path 3) against the oracle."""
    case = W.make_case("tensor_memory", seed=60 + M, dtype=dtype, head_size=D, num_q_heads=16,
                       num_kv_heads=4, page_size=16, max_query_len=M,
                       seq_lens=seqs if seqs else [L], layout=layout, window=window,
                       window_pages_only=bool(window))
    _parity(case, opts=pd.options(path=3))


@pytest.mark.parametrize("seg,merge", [(1, 0), (5, 1), (19, 2), (16, 1)])
def test_tensor_memory_path_splits(seg, merge):
    case = W.spec_decode_hnd(4, 8192, seed=70)
    _parity(case, opts=pd.options(path=3, segments=seg, merge=merge))


def test_tensor_memory_path_refused_for_d512():
    case = W.make_case("tm_d512", seed=71, dtype=torch.float16, head_size=512, num_q_heads=8,
                       num_kv_heads=1, page_size=16, max_query_len=1, seq_lens=[100], layout=W.HND)
    g = case.to("cuda")
    rc = pd.paged_decode_attn(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens,
                              torch.empty_like(g.q), g.num_q_heads, g.num_kv_heads,
                              g.head_size, g.page_size, g.max_query_len, g.window, g.scale,
                              g.layout, scratch_for(case), opts=pd.options(path=3), check=False)
    assert rc == -1


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.3])
def test_scales_of_any_sign(scale):
    """The scale is as passed: zero (uniform weights), negative, or larger."""
    case = W.make_case("scales", seed=80, dtype=torch.bfloat16, head_size=128, num_q_heads=16,
                       num_kv_heads=4, page_size=16, max_query_len=3, seq_lens=[1500, 40],
                       layout=W.HND, scale=scale)
    _parity(case)


# ---- decode batches with a query length per request (query_start) ----------

@pytest.mark.parametrize("q_lens,lens,pad,D,layout,dtype,window,P,opts", [
    # mixed lengths with an empty request and padding tokens (a batch)
    ([1, 4, 2, 0, 3, 8, 5, 1], [900, 37, 2000, 15, 1, 700, 64, 3], 5, 128, W.HND,
     torch.bfloat16, 0, 16, None),
    # the same, merges forced: last arriver, cooperative
    ([1, 4, 2, 0, 3, 8, 5, 1], [900, 37, 2000, 15, 1, 700, 64, 3], 5, 128, W.HND,
     torch.bfloat16, 0, 16, "merge1"),
    ([2, 3, 1, 4], [3000, 1200, 40, 2500], 0, 128, W.HND, torch.bfloat16, 0, 16, "merge2"),
    # sliding window, wide heads, NHD, small heads
    ([4, 1, 3], [1500, 600, 2100], 2, 256, W.HND, torch.float16, 100, 32, None),
    ([2, 7, 1], [300, 77, 9], 1, 64, W.NHD, torch.bfloat16, 0, 16, None),
    ([5, 2], [2200, 48], 0, 512, W.HND, torch.float16, 0, 16, None),
    # one request shorter than the planned M: many segments, cooperative merge
    ([3], [9000], 4, 128, W.HND, torch.bfloat16, 0, 16, None),
    # seq_len below q_len: the first tokens of those requests see no key
    ([5, 4, 2], [3, 1, 700], 1, 128, W.HND, torch.bfloat16, 0, 16, None),
])
def test_varlen(q_lens, lens, pad, D, layout, dtype, window, P, opts):
    G = 4 if D <= 256 else 8
    case = W.make_varlen_case("varlen", seed=40 + len(q_lens), q_lens=q_lens, pad_tokens=pad,
                              dtype=dtype, head_size=D, num_q_heads=2 * G, num_kv_heads=2,
                              page_size=P, seq_lens=lens, layout=layout, window=window,
                              max_query_len=8 if len(q_lens) == 1 else None)
    o = {None: None, "merge1": pd.options(merge=1),
         "merge2": pd.options(merge=2, row_groups=1, segments=16)}[opts]
    out, _ = _parity(case, opts=o)
    t_end = case.query_start_host[-1]
    assert torch.all(out[t_end:] == 0), "padding rows not zero"


def test_varlen_window_pages_only():
    """A windowed batch whose block table holds only the pages the window
    reaches for the longest query (earlier entries point at a NaN page):
    shorter requests must not read before their own window either."""
    for w in (1, 17, 300):
        case = W.make_varlen_case("varlen_win", seed=52, q_lens=[1, 4, 2, 3], pad_tokens=2,
                                  dtype=torch.float16, head_size=256, num_q_heads=8,
                                  num_kv_heads=1, page_size=32, seq_lens=[1500, 900, 40, 2600],
                                  layout=W.HND, window=w, window_pages_only=True)
        _parity(case)


def test_varlen_rejects_tensor_memory_path_and_bad_shapes():
    case = W.make_varlen_case("varlen_args", seed=50, q_lens=[2, 1], dtype=torch.bfloat16,
                              head_size=128, num_q_heads=8, num_kv_heads=2, page_size=16,
                              seq_lens=[100, 20])
    g = case.to("cuda")
    out = torch.empty_like(g.q)
    args = (g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens)
    tail = (g.num_q_heads, g.num_kv_heads, g.head_size, g.page_size, g.max_query_len, g.window,
            g.scale, g.layout, scratch_for(case))
    assert pd.paged_decode_attn_varlen(*args, g.query_start, out, *tail,
                                       opts=pd.options(path=3), check=False) == -1
    assert pd.paged_decode_attn_varlen(*args, g.query_start[:2], out, *tail, check=False) == -1
    assert pd.paged_decode_attn_varlen(*args, g.query_start.to(torch.int64), out, *tail,
                                       check=False) < 0
    torch.cuda.synchronize()
    assert pd.paged_decode_device_status(reset=True) == 0


def test_varlen_out_of_order_query_start_is_clamped_and_reported():
    """A decreasing query_start and one past the rows are clamped on the
    device (no access outside q and out) and reported as PD_DEV_BAD_QSTART."""
    case = W.make_varlen_case("varlen_bad", seed=51, q_lens=[3, 2, 2], dtype=torch.bfloat16,
                              head_size=128, num_q_heads=8, num_kv_heads=2, page_size=16,
                              seq_lens=[300, 90, 40])
    g = case.to("cuda")
    g.query_start = torch.tensor([0, 5, 2, 40], dtype=torch.int32, device="cuda")
    sentinel = torch.full((4, g.q.shape[1], g.q.shape[2]), 7.0, dtype=g.q.dtype, device="cuda")
    out_full = torch.cat([torch.empty_like(g.q), sentinel])
    out = out_full[: g.q.shape[0]]
    pd.decode_case(g, out=out, scratch=scratch_for(case))
    torch.cuda.synchronize()
    assert torch.all(out_full[g.q.shape[0]:] == 7.0), "a row past out was written"
    assert torch.isfinite(out.float()).all()
    assert pd.paged_decode_device_status(reset=True) == pd.DEV_BAD_QSTART


# ---- the warp dot-product consumer (path 2) --------------------------------

def _dot(case, **kw):
    return _parity(case, opts=pd.options(path=2, **kw))


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [128, 1024, 4096])
def test_warp_dot_spec_decode(M, L):
    """bf16 D=128 32/8: 4 and 8 packed rows in one CTA, 12 and 16 in two
    row groups."""
    _dot(W.spec_decode_hnd(M, L, seed=40 + M))


def test_warp_dot_single_seq_nhd():
    _dot(W.single_seq_nhd(seed=41))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("M", [1, 4])
def test_warp_dot_sliding_window(dtype, M):
    _dot(W.sliding_window(dtype, M, 4096, seed=42))


@pytest.mark.parametrize("D", [64, 256])
def test_warp_dot_head_sizes(D):
    _dot(W.make_case(f"dot_d{D}", seed=43, dtype=torch.float16, head_size=D, num_q_heads=8,
                     num_kv_heads=2, page_size=32, max_query_len=2, seq_lens=[1777],
                     layout=W.NHD))


def test_warp_dot_batch_varlen_and_splits():
    _dot(W.batched_hybrid_pages(seed=44, num_seqs=8, max_len=3000))
    _dot(W.make_varlen_case("dot_varlen", seed=45, q_lens=[2, 1, 0, 2], pad_tokens=3,
                            dtype=torch.bfloat16, head_size=128, num_q_heads=16,
                            num_kv_heads=4, page_size=16, seq_lens=[900, 50, 7, 2100]))
    _dot(W.spec_decode_hnd(2, 4096, seed=46), segments=7, merge=1)
    _dot(W.spec_decode_hnd(1, 8192, seed=47, v_mean=1.0))
