"""Paged prefill (paged_prefill_plan + paged_prefill_attn) against the fp64
oracle through the C ABI: requests of any query length over the paged
cache, the work list made on the host, split tiles merged in the kernel.
The oracle is the same definition as for decode (each token t of request r
sees seq_len - q_len + (t - query_start[r]) + 1 keys).  Bounds as for
decode: max-abs 2e-3 (fp16) / 1e-2 (bf16) and, row by row, 2^-10 / 2^-7 of
the row's largest oracle value."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W
from gpu_helpers import check, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pd.build()
    pd.paged_decode_device_status(reset=True)
    yield
    assert pd.paged_decode_device_status(reset=True) == 0


def _run(case, num_sms=0, rows=None, expect_split=None):
    g = case.to("cuda")
    items, info = pd.paged_prefill_plan(case.query_start_host, case.seq_lens_host,
                                        case.num_q_heads, case.num_kv_heads, case.head_size,
                                        case.window, num_sms)
    if expect_split is not None:
        assert (info.num_split_tiles > 0) == expect_split
    sms = num_sms or torch.cuda.get_device_properties(0).multi_processor_count
    sc = pd.prefill_scratch(case.num_kv_heads, case.head_size, sms)
    out = torch.full_like(g.q, 3.0)
    pd.prefill_case(g, out=out, scratch=sc, plan=(items, info))
    torch.cuda.synchronize()
    assert pd.paged_decode_device_status(reset=True) == 0
    assert int(sc.counters().abs().sum()) == 0, "counters not left at zero"
    check(case, out, rows=rows)
    return out, info


def test_single_long_request():
    c = W.make_prefill_case("pf_single", seed=1, q_lens=[300], contexts=[700])
    _run(c)


def test_mixed_batch_with_empty_request_and_padding():
    c = W.make_prefill_case("pf_mixed", seed=2, q_lens=[1, 40, 257, 0, 100],
                            contexts=[0, 1000, 60, 500, 2000], pad_tokens=5)
    out, _ = _run(c)
    assert torch.all(out[c.query_start_host[-1]:] == 0)


def test_forced_splits_merge_in_kernel():
    # a large resident-CTA target lowers the load: most tiles are split
    c = W.make_prefill_case("pf_split", seed=3, q_lens=[64, 200], contexts=[3000, 1500])
    _, info = _run(c, num_sms=4000, expect_split=True)
    assert info.num_split_tiles >= 4


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_sliding_window(dtype):
    c = W.make_prefill_case("pf_window", seed=4, q_lens=[400, 33], contexts=[2000, 0],
                            dtype=dtype, head_size=256, num_q_heads=8, num_kv_heads=1,
                            page_size=32, window=256)
    _run(c)


@pytest.mark.parametrize("D,Hq,Hkv,P,layout", [(64, 16, 2, 16, W.HND), (128, 8, 8, 32, W.NHD),
                                                (512, 8, 1, 16, W.HND), (256, 16, 2, 1056, W.HND)])
def test_head_sizes_layouts_pages(D, Hq, Hkv, P, layout):
    c = W.make_prefill_case(f"pf_d{D}", seed=5 + D, q_lens=[97, 130], contexts=[500, 1200],
                            dtype=torch.float16 if D == 512 else torch.bfloat16, head_size=D,
                            num_q_heads=Hq, num_kv_heads=Hkv, page_size=P, layout=layout,
                            v_mean=1.0 if D == 512 else 0.0)
    _run(c)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 1), (16, 16), (12, 4)])
def test_tensor_memory_tiles_d128(dtype, Hq, Hkv):
    # head size 128 runs 256-row tiles (two halves of 128) on the tensor
    # cores: G = 4, 8, 1 and 3 (a tile then ends inside a token), ragged query
    # lengths, a request with no context and one shorter than a half; values
    # shifted so the outputs are O(1)
    c = W.make_prefill_case(f"pf_tp_{Hq}_{Hkv}", seed=11 + Hq + Hkv, q_lens=[131, 7, 300, 64],
                            contexts=[500, 33, 0, 1999], dtype=dtype, head_size=128,
                            num_q_heads=Hq, num_kv_heads=Hkv, page_size=16, v_mean=1.0)
    _, info = _run(c)
    assert info.tile_rows == 256


@pytest.mark.parametrize("window", [1, 100, 129])
def test_tensor_memory_tiles_d128_windows(window):
    c = W.make_prefill_case(f"pf_tp_w{window}", seed=21 + window, q_lens=[200, 45],
                            contexts=[700, 0], head_size=128, num_q_heads=16, num_kv_heads=4,
                            page_size=32, window=window)
    _run(c)


def test_tensor_memory_tiles_d128_split_nhd():
    # split tiles (a large resident-CTA target) merged in the kernel, NHD pages
    c = W.make_prefill_case("pf_tp_split", seed=31, q_lens=[256, 100], contexts=[4000, 900],
                            head_size=128, num_q_heads=32, num_kv_heads=8, page_size=16,
                            layout=W.NHD, v_mean=1.0)
    _, info = _run(c, num_sms=4000, expect_split=True)
    assert info.num_split_tiles >= 4


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("scale", [12.0, -10.0, 0.0])
def test_tensor_memory_tiles_d128_large_scores(scale, dtype):
    # q, K, V of std 0.4 and scores of std |scale| 0.16 sqrt(D) log2(e) (~30):
    # a row's max often grows by more than 8 (log2 units) past its reference
    # on an unmasked stage, so the rescale of O and the stage's exponentials
    # taken again are exercised (fp16 P then overflows before the retake); a
    # negative scale takes the smallest raw score as the max; zero gives
    # uniform weights.  The outputs stay below ~2, where the max-abs bound
    # is above the output's own rounding.
    c = W.make_prefill_case(f"pf_tp_scale{scale}", seed=41, q_lens=[300, 64],
                            contexts=[1500, 700], dtype=dtype, head_size=128, num_q_heads=32,
                            num_kv_heads=8, page_size=16, std=0.4)
    _run(dataclasses.replace(c, scale=scale))


def test_prefill_sized_batch_sampled_rows():
    # 4 requests x 1024 new tokens after 4k of context: sampled rows
    c = W.make_prefill_case("pf_big", seed=6, q_lens=[1024] * 4, contexts=[4096] * 4,
                            v_mean=1.0)
    rows = sample_rows(c, 96, seed=6)
    _run(c, rows=rows)


def test_bad_work_item_is_skipped_and_reported():
    c = W.make_prefill_case("pf_bad", seed=7, q_lens=[70], contexts=[100])
    g = c.to("cuda")
    items, info = pd.paged_prefill_plan(c.query_start_host, c.seq_lens_host, c.num_q_heads,
                                        c.num_kv_heads, c.head_size, c.window, 0)
    bad = items.clone()
    bad[0, 0] = 5          # a request that does not exist
    out = torch.full_like(g.q, 3.0)
    pd.paged_prefill_attn(g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.query_start,
                          bad.cuda(), info, out, c.num_q_heads, c.num_kv_heads, c.head_size,
                          c.page_size, c.window, c.scale, c.layout, None)
    torch.cuda.synchronize()
    assert pd.paged_decode_device_status(reset=True) & pd.DEV_BAD_WORK
    # the other items ran: rows outside the skipped tile match the oracle
    tile, TR = int(items[0, 1]), info.tile_rows
    G = c.num_q_heads // c.num_kv_heads
    rows = [(t, h) for t in range(70) for h in range(c.num_q_heads)
            if not (tile * TR <= t * G + h % G < (tile + 1) * TR)]
    check(c, out, rows=rows)
