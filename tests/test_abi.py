"""The C ABI on the CPU: the library loads, exports every declared symbol,
and its host-side logic (argument checks, plan, scratch sizing) behaves,
all without a GPU."""

import ctypes

import pytest
import torch

import paged_split_kv_02_gb300 as pd
from paged_split_kv_02_gb300 import workloads as W


@pytest.fixture(scope="module")
def lib():
    pd.build()
    return pd.lib()


def test_exports_every_declared_symbol(lib):
    names = pd.declared_symbols()
    assert len(names) == 14 and "paged_rope_cache_write" in names
    assert {"paged_prefill_plan", "paged_prefill_scratch_bytes", "paged_prefill_attn"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strerror(lib):
    assert pd.paged_decode_version() == 10300
    for code in range(0, -9, -1):
        assert lib.paged_decode_strerror(code)
    assert b"unknown" in lib.paged_decode_strerror(-99)


def test_scratch_bytes():
    a = pd.paged_decode_scratch_bytes(1, 32, 8, 128, 4, 16)
    b = pd.paged_decode_scratch_bytes(1, 32, 8, 128, 4, 32)
    c = pd.paged_decode_scratch_bytes(2, 32, 8, 128, 4, 16)
    assert 0 < a < b and a < c
    # acc (rows * D) + m, l (2 * rows), per partial: rows = 16 at G=4, M=4
    assert b - a == pytest.approx(16 * 8 * 16 * (128 + 2) * 4, abs=1024)
    assert pd.paged_decode_scratch_bytes(1, 32, 8, 96, 4, 16) == 0      # head size
    assert pd.paged_decode_scratch_bytes(1, 32, 8, 128, 9, 16) == 0     # M > 8
    assert pd.paged_decode_scratch_bytes(1, 30, 8, 128, 1, 16) == 0     # Hq % Hkv


def _fake_scratch(S, Hq, Hkv, D, M, splits):
    d = pd.PdScratch()
    d.data = 1 << 30
    d.bytes = pd.paged_decode_scratch_bytes(S, Hq, Hkv, D, M, splits)
    d.counter_slots = S * Hkv * pd.COUNTERS_PER_PAIR
    return d


@pytest.mark.parametrize("shape", [
    (1, 8, 2, 128, 16, 1, 0, 19),       # single sequence, NHD test case
    (1, 32, 8, 128, 16, 4, 0, 2048),    # spec decode, 32k
    (1, 8, 1, 256, 32, 4, 512, 1024),   # sliding window
    (1, 8, 1, 512, 16, 8, 0, 2048),     # wide head, 64 packed rows
    (64, 16, 2, 256, 1056, 4, 0, 16),   # batched, hybrid pages
])
def test_plan_invariants(shape):
    S, Hq, Hkv, D, P, M, w, Wd = shape
    sd = _fake_scratch(S, Hq, Hkv, D, M, 256)
    p = pd.paged_decode_plan(S, Hq, Hkv, D, P, M, w, Wd, 152, scratch_desc=sd)
    G = Hq // Hkv
    assert p["rows"] == G * M
    assert p["rows_per_cta"] * p["row_groups"] >= G * M
    assert p["n_tiles"] * 8 >= p["rows_per_cta"]
    assert p["n_tiles"] * p["key_groups"] <= 8
    assert p["stages"] % p["key_groups"] == 0          # slot -> warp group is static
    assert p["max_segments"] % p["cluster"] == 0
    assert p["grid_x"] == Hkv * p["row_groups"] * p["max_segments"]
    assert p["grid_y"] == S
    assert p["block_threads"] == 32 * (p["n_tiles"] * p["key_groups"] + 1)
    assert p["smem_bytes"] <= 232448
    assert p["scratch_needed"] <= sd.bytes
    # the segments cover every 16-key block a row can see
    nb_max = -(-Wd * P // 16)
    if w:
        nb_max = min(nb_max, -(-(w + M - 1) // 16) + 1)
    assert p["seg_blocks"] * p["max_segments"] >= nb_max
    if S == 1 and Wd * P >= 32768 and not w:
        assert p["grid_x"] >= 128                      # a long sequence fills the SMs


def test_plan_segments_grow_with_the_context():
    # one sequence, 8 kv heads, D=128, M=4: with 1-8 MiB of K and V per kv
    # head the CTAs are capped at (12 + 7/3 log2(MiB)) / 19 of the SMs
    # (fewer, longer segments: fewer parts to merge), below and above that
    # the SM count and the segment floor decide
    want = {1024: 6, 2048: 12, 4096: 14, 8192: 16, 16384: 19, 32768: 19}
    for L, nseg in want.items():
        sd = _fake_scratch(1, 32, 8, 128, 4, 256)
        p = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, L // 16, 152, scratch_desc=sd)
        assert p["max_segments"] == nseg, (L, p["max_segments"])
    # the cap is a fraction of the resident CTAs, shared by the units: two
    # kv heads at 8k keys (4 MiB each) get (12 + 14/3) / 19 x 152 / 2 = 66
    # segments (the SM share alone gives 76, the floor 512 / 6 = 85)
    sd = _fake_scratch(1, 8, 2, 128, 4, 256)
    p = pd.paged_decode_plan(1, 8, 2, 128, 16, 4, 0, 8192 // 16, 152, scratch_desc=sd)
    assert p["max_segments"] == 66


def test_counters_per_pair_matches_header():
    text = open(pd.HEADER).read()
    assert f"#define PD_COUNTERS_PER_PAIR {pd.COUNTERS_PER_PAIR}" in text
    # the counter area of scratch_bytes: PD_COUNTERS_PER_PAIR int32 per pair
    # (no partials with max_splits = 0), rounded to 256 bytes, plus 256
    n = pd.paged_decode_scratch_bytes(1000, 32, 8, 128, 4, 0)
    assert n == -(-1000 * 8 * pd.COUNTERS_PER_PAIR * 4 // 256) * 256 + 256


def test_plan_splits_with_eight_row_groups():
    # one sequence with G * M = 128 packed rows takes 8 row groups, i.e. 16
    # counters per (sequence, kv head): a scratch sized and initialised by
    # the library must still let it split
    S, Hq, Hkv, D, M = 1, 16, 1, 128, 8
    sd = _fake_scratch(S, Hq, Hkv, D, M, 256)
    p = pd.paged_decode_plan(S, Hq, Hkv, D, 16, M, 0, 2048, 148, scratch_desc=sd)
    assert p["row_groups"] == 8
    assert p["max_parts"] > 1 and p["max_segments"] > 1 and p["merge"] > 0
    assert p["scratch_needed"] <= sd.bytes
    # the same with 64 q heads over 4 kv heads
    sd = _fake_scratch(S, 64, 4, D, M, 256)
    p = pd.paged_decode_plan(S, 64, 4, D, 16, M, 0, 2048, 148, scratch_desc=sd)
    assert p["row_groups"] == 8 and p["max_parts"] > 1


def test_scratch_bytes_covers_single_sequence_row_groups():
    # R = 20 packed rows: a batch plan keeps one row group of 24 padded rows,
    # a single-sequence plan two groups of 16; the size covers the larger
    for Hq, Hkv, M in [(20, 4, 4), (40, 8, 4), (12, 2, 3)]:
        sd = _fake_scratch(1, Hq, Hkv, 128, M, 8)
        p = pd.paged_decode_plan(1, Hq, Hkv, 128, 16, M, 0, 2048, 152, scratch_desc=sd,
                                 opts=pd.options(segments=8))
        assert p["max_parts"] == 8 and p["scratch_needed"] <= sd.bytes


def test_static_entry_refuses_too_many_pairs_before_the_device(lib):
    # more sequence x kv-head pairs than the static counter area holds:
    # PD_ESCRATCH from the host checks, with no device touched
    def call(num_seqs, hkv):
        sl = pd.PdTensor()
        sl.data, sl.dtype, sl.ndim = 1 << 20, 2, 1
        sl.shape[0], sl.stride[0] = num_seqs, 1
        d = pd.PdTensor()
        return lib.paged_decode_attn_static(*[ctypes.byref(x) for x in (d, d, d, d, sl, d)],
                                            8 * hkv, hkv, 128, 16, 1, 0, 0.1, 1, None)
    pairs = (512 << 10) // (4 * pd.COUNTERS_PER_PAIR)
    assert pairs == 8192
    assert call(pairs // 2 + 1, 2) == -6
    assert call(pairs + 1, 1) == -6
    if not torch.cuda.is_available():
        # at the limit the call goes on to the device, which is missing here
        assert call(pairs, 1) == -8


def test_wait_limit_option_checked():
    with pytest.raises(pd.PagedDecodeError):
        pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 256, 152,
                             opts=pd.options(wait_limit_us=-1))


def test_early_reads_option_checked():
    for v in (-1, 2):
        with pytest.raises(pd.PagedDecodeError):
            pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 256, 152,
                                 opts=pd.options(early_reads=v))
    # the option does not change the plan
    a = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 2048, 152,
                             scratch_desc=_fake_scratch(1, 32, 8, 128, 4, 64))
    b = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 2048, 152,
                             scratch_desc=_fake_scratch(1, 32, 8, 128, 4, 64),
                             opts=pd.options(early_reads=1))
    assert a == b


def test_merger_count_rule():
    """K of the cooperative merge: the largest power of two <= min(D / 8, 64,
    segments, W), W the smallest power of two >= 4 with W x 8192 >= segments x
    rows per CTA x D; capped by pd_options.mergers."""
    sc = _fake_scratch(1, 32, 8, 128, 4, 64)

    def plan(M, **kw):
        return pd.paged_decode_plan(1, 32, 8, 128, 16, M, 0, 1024, 152, scratch_desc=sc,
                                    opts=pd.options(**kw) if kw else None)
    # 16k keys, 19 segments: 4, 8 and 12 rows -> 4 mergers, 16 -> 8 (19 x 16
    # x 128 = 38912 > 4 x 8192)
    assert [plan(M)["mergers"] for M in (1, 2, 3, 4)] == [4, 4, 4, 8]
    assert all(plan(M)["merge"] == 2 for M in (1, 2, 3, 4))
    assert plan(4, mergers=2)["mergers"] == 2
    assert plan(4, mergers=1)["mergers"] == 1
    assert plan(1, mergers=16)["mergers"] == 4       # a cap, not a request
    for bad in (-1, 3, 6):
        with pytest.raises(pd.PagedDecodeError):
            plan(1, mergers=bad)
    # the wide head (D = 512, M = 8: 64 rows, 16 per CTA in 4 row groups) and
    # few segments: the segments bound K
    p = pd.paged_decode_plan(1, 8, 1, 512, 16, 8, 0, 2048, 152,
                             scratch_desc=_fake_scratch(1, 8, 1, 512, 8, 64))
    assert p["merge"] == 2 and p["mergers"] == min(32, 1 << (p["max_segments"].bit_length() - 1))
    # 4k keys, 14 segments: 14 x 16 x 128 = 28672 <= 4 x 8192 -> 4 mergers
    p = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 256, 152, scratch_desc=sc)
    assert p["max_segments"] == 14 and p["mergers"] == 4
    # D = 512, M = 1: 152 segments of 8 rows -> the D / 8 = 64 bound
    p = pd.paged_decode_plan(1, 8, 1, 512, 16, 1, 0, 2048, 152,
                             scratch_desc=_fake_scratch(1, 8, 1, 512, 8, 256))
    assert p["max_segments"] == 152 and p["mergers"] == 64


def test_plan_without_scratch_does_not_split():
    p = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 2048, 152)
    assert p["max_parts"] == 0 and p["scratch_needed"] == 0
    assert p["max_segments"] == 1


def test_plan_shrinks_to_small_scratch():
    small = _fake_scratch(1, 32, 8, 128, 4, 3)
    p = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 2048, 152, scratch_desc=small)
    assert 0 < p["scratch_needed"] <= small.bytes
    assert p["max_parts"] <= 3


def test_plan_forced_knobs_and_errors():
    sd = _fake_scratch(1, 32, 8, 128, 4, 64)
    p = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 256, 152, scratch_desc=sd,
                             opts=pd.options(segments=16, cluster=4, key_groups=2, stages=4))
    assert (p["max_segments"], p["cluster"], p["key_groups"], p["stages"]) == (16, 4, 2, 4)
    assert p["max_parts"] == 4
    with pytest.raises(pd.PagedDecodeError):   # stages not a multiple of the warp groups
        pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 256, 152, scratch_desc=sd,
                             opts=pd.options(key_groups=4, stages=6))
    with pytest.raises(pd.PagedDecodeError):   # segments not a multiple of the cluster
        pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 256, 152, scratch_desc=sd,
                             opts=pd.options(segments=6, cluster=4))
    with pytest.raises(pd.PagedDecodeError) as e:
        pd.paged_decode_plan(1, 32, 8, 96, 16, 4, 0, 256, 152)
    assert e.value.code == -3
    with pytest.raises(pd.PagedDecodeError) as e:
        pd.paged_decode_plan(1, 32, 8, 128, 16, 9, 0, 256, 152)
    assert e.value.code == -4
    with pytest.raises(pd.PagedDecodeError) as e:
        pd.paged_decode_plan(1, 32, 8, 128, 24, 4, 0, 256, 152)   # page size % 16
    assert e.value.code == -1
    big = _fake_scratch(1, 32, 8, 128, 4, 1)
    with pytest.raises(pd.PagedDecodeError) as e:  # forced split that the scratch cannot hold
        pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 2048, 152, scratch_desc=big,
                             opts=pd.options(segments=64))
    assert e.value.code == -6


def _cpu_case(**kw):
    base = dict(seed=0, dtype=torch.float16, head_size=128, num_q_heads=8, num_kv_heads=2,
                page_size=16, max_query_len=2, seq_lens=[40, 7], layout=W.HND)
    base.update(kw)
    return W.make_case("abi", **base)


def _call(case, **over):
    args = dict(q=case.q, k_cache=case.k_cache, v_cache=case.v_cache,
                block_table=case.block_table, seq_lens=case.seq_lens, out=torch.empty_like(case.q),
                num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                head_size=case.head_size, page_size=case.page_size,
                max_query_len=case.max_query_len, window=case.window, scale=case.scale,
                layout=case.layout)
    args.update(over)
    return pd.paged_decode_attn(**args, stream=0, check=False)


def test_argument_checks_on_host():
    """Every malformed call is refused before any CUDA call (these run on a
    machine without a GPU)."""
    c = _cpu_case()
    assert _call(c, head_size=96) == -3
    assert _call(c, max_query_len=0) == -4
    assert _call(c, max_query_len=9) == -4
    assert _call(c, num_q_heads=6) == -1              # Hq % Hkv, and q's shape
    assert _call(c, page_size=8) == -1
    assert _call(c, window=-1) == -1
    assert _call(c, layout=3) == -1
    assert _call(c, scale=float("nan")) == -1
    assert _call(c, out=torch.empty_like(c.q, dtype=torch.bfloat16)) == -2
    assert _call(c, q=c.q.float()) == -2
    assert _call(c, seq_lens=c.seq_lens.long()) == -2
    assert _call(c, block_table=c.block_table[:1]) == -1
    assert _call(c, q=c.q[:, :, :64]) == -1
    q_odd = torch.empty(c.q.shape[0], c.q.shape[1], 129, dtype=c.q.dtype)[:, :, 1:]
    assert _call(c, q=q_odd) == -5                    # rows not 16-byte aligned
    assert _call(c, k_cache=c.k_cache.transpose(1, 2)) == -1
    # a well-formed call on a machine without an sm_103 device
    if not torch.cuda.is_available():
        assert _call(c) == -8


def test_varlen_argument_checks_on_host():
    """The variable-length call refuses a missing or malformed query_start
    and rows that do not match before any CUDA call."""
    c = W.make_varlen_case("abi_varlen", seed=1, q_lens=[2, 0, 3], pad_tokens=1,
                           dtype=torch.float16, head_size=128, num_q_heads=8, num_kv_heads=2,
                           page_size=16, seq_lens=[40, 7, 19])

    def call(**over):
        a = dict(q=c.q, k_cache=c.k_cache, v_cache=c.v_cache, block_table=c.block_table,
                 seq_lens=c.seq_lens, query_start=c.query_start, out=torch.empty_like(c.q),
                 num_q_heads=8, num_kv_heads=2, head_size=128, page_size=16,
                 max_query_len=c.max_query_len, window=0, scale=c.scale, layout=c.layout)
        a.update(over)
        return pd.paged_decode_attn_varlen(**a, stream=0, check=False)

    assert call(query_start=c.query_start[:3]) == -1          # S + 1 entries
    assert call(query_start=c.query_start.long()) == -2       # int32
    assert call(query_start=c.query_start.view(1, -1)) == -1
    assert call(out=torch.empty(c.q.shape[0] + 1, 8, 128, dtype=c.q.dtype)) == -1
    assert call(max_query_len=9) == -4
    assert pd.lib().paged_decode_attn_varlen(*([None] * 7), 8, 2, 128, 16, 3, 0, 1.0, 1,
                                             None, None, None) == -1
    if not torch.cuda.is_available():
        assert call() == -8


def test_plan_small_calls_unsplit_and_batch_segments_capped():
    """A single sequence whose K+V per kv head is at most 256 KiB is one CTA
    per head; a batch's segments hold at most 384 blocks (6144 keys)."""
    def plan(S, Hq, Hkv, D, P, M, W_):
        sd = _fake_scratch(S, Hq, Hkv, D, M, 256)
        return pd.paged_decode_plan(S, Hq, Hkv, D, P, M, 0, W_, 152, scratch_desc=sd)

    p = plan(1, 8, 2, 128, 16, 1, 19)        # 300 keys, D=128: 152 KiB per head
    assert p["max_segments"] == 1 and p["merge"] == 0
    p = plan(1, 32, 8, 128, 16, 4, 64)       # 1k keys: 512 KiB per head, split
    assert p["max_segments"] > 1
    p = plan(32, 32, 8, 128, 16, 4, 1013)    # 32 requests of up to 16k keys
    assert p["seg_blocks"] <= 384 and p["max_segments"] >= 3
    p = plan(8, 32, 8, 128, 16, 4, 1008)     # fewer groups: the estimate rules
    assert p["seg_blocks"] < 384


def test_plan_windowed_segments():
    """A windowed single-sequence call split into row groups takes segments
    of two blocks; with one row group the usual floor holds."""
    def plan(M):
        sd = _fake_scratch(1, 8, 1, 256, M, 256)
        return pd.paged_decode_plan(1, 8, 1, 256, 32, M, 512, 1024, 152, scratch_desc=sd)

    p4, p1 = plan(4), plan(1)
    assert p4["row_groups"] == 2 and p4["max_segments"] == 17
    assert p1["row_groups"] == 1 and p1["max_segments"] == 8


def test_plan_tensor_memory_path():
    """path 3: 4 softmax warps + 1 MMA warp + the producer, 16 packed rows
    per CTA (four copies fill the M = 64 side), four partial states."""
    sd = _fake_scratch(1, 32, 8, 128, 4, 64)
    p = pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 2048, 152, scratch_desc=sd,
                             opts=pd.options(path=3))
    assert p["path"] == 3 and p["block_threads"] == 192 and p["key_groups"] == 4
    assert p["rows_per_cta"] <= 16 and p["cluster"] == 1
    wide = _fake_scratch(1, 64, 8, 128, 8, 64)   # 64 packed rows -> 4 row groups
    p = pd.paged_decode_plan(1, 64, 8, 128, 16, 8, 0, 256, 152, scratch_desc=wide,
                             opts=pd.options(path=3))
    assert p["row_groups"] == 4 and p["rows_per_cta"] == 16
    assert pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 2048, 152,
                                scratch_desc=sd)["path"] == 1  # the default is mma.sync
    with pytest.raises(pd.PagedDecodeError):   # D = 512 does not fit tensor memory
        pd.paged_decode_plan(1, 8, 1, 512, 16, 1, 0, 64, 152, opts=pd.options(path=3))
    with pytest.raises(pd.PagedDecodeError):   # no clusters on this path
        pd.paged_decode_plan(1, 32, 8, 128, 16, 4, 0, 256, 152, scratch_desc=sd,
                             opts=pd.options(path=3, cluster=2, segments=4))


def test_plan_warp_dot_path():
    """path 2: one 8-row n-tile per CTA (more rows in row groups), warp
    groups of one warp, shared memory for fp32 Q rows and the P buffers."""
    sd = _fake_scratch(1, 32, 8, 128, 4, 256)
    for M, rg in [(1, 1), (2, 1), (3, 2), (4, 2)]:
        p = pd.paged_decode_plan(1, 32, 8, 128, 16, M, 0, 2048, 152, scratch_desc=sd,
                                 opts=pd.options(path=2))
        assert p["path"] == 2 and p["n_tiles"] == 1 and p["row_groups"] == rg
        assert p["rows_per_cta"] <= 8 and p["cluster"] == 1
        KG, NS = p["key_groups"], p["stages"]
        stage_keys = 32768 // 2 // (16 * 128 * 2) * 16
        base = 1024 + NS * 32768 + 128 * 16 + 2 * NS * 8 + 16 + 4 * 512
        assert p["smem_bytes"] == base + 16 + 8 * 128 * 4 + KG * stage_keys * 8 * 4
        assert p["smem_bytes"] <= 232448
    for D in (64, 256):
        p = pd.paged_decode_plan(1, 8, 1, D, 16, 1, 0, 512, 152, scratch_desc=sd,
                                 opts=pd.options(path=2))
        assert p["path"] == 2 and p["smem_bytes"] <= 232448
    with pytest.raises(pd.PagedDecodeError):   # head size 512 is not served
        pd.paged_decode_plan(1, 8, 1, 512, 16, 1, 0, 64, 152, opts=pd.options(path=2))
    with pytest.raises(pd.PagedDecodeError):   # no clusters on this path
        pd.paged_decode_plan(1, 32, 8, 128, 16, 1, 0, 256, 152, scratch_desc=sd,
                             opts=pd.options(path=2, cluster=2, segments=4))


def test_rope_argument_checks_on_host(lib):
    """paged_rope_cache_write's argument checks run before any device call."""
    c = W.make_rope_case("abi", seed=1, dtype=torch.bfloat16, num_tokens=6, num_q_heads=4,
                         num_kv_heads=2, head_size=64, rot_dim=32, page_size=16, num_pages=2)

    def call(**over):
        a = dict(q=c.q, k=c.k, v=c.v, positions=c.positions, slot_mapping=c.slot_mapping,
                 cos_sin_cache=c.cos_sin, q_out=c.q, k_cache=c.k_cache, v_cache=c.v_cache,
                 num_q_heads=4, num_kv_heads=2, head_size=64, rot_dim=32, page_size=16,
                 layout=W.HND, is_neox=True)
        a.update(over)
        return pd.paged_rope_cache_write(**a, check=False)

    assert call(head_size=96) == -3                       # head size
    assert call(rot_dim=24) == -1                         # NeoX: rot_dim % 16
    assert call(rot_dim=80) == -1                         # rot_dim > D
    assert call(rot_dim=0) == -1
    assert call(positions=c.positions.to(torch.int64)) == -2          # int32 only
    assert call(slot_mapping=c.slot_mapping[:5]) == -1                # length
    assert call(cos_sin_cache=c.cos_sin.to(torch.float16)) == -2      # fp32 table
    assert call(cos_sin_cache=c.cos_sin[:, :16]) == -1                # narrower than rot_dim
    assert call(k=c.k.to(torch.float16)) == -2                        # mixed dtypes
    assert call(q_out=torch.empty(6, 4, 64, dtype=torch.float16)) == -2
    assert call(num_kv_heads=1) == -1                                 # k shape
    assert call(layout=W.NHD) == -1                                   # pool shape vs layout
    assert call(page_size=8) == -1
    odd = torch.empty(6, 4, 72, dtype=torch.bfloat16)[..., 4:68]      # 8-byte aligned rows
    assert call(q=odd) == -5
    empty = W.make_rope_case("abi0", seed=1, dtype=torch.bfloat16, num_tokens=0, num_q_heads=4,
                             num_kv_heads=2, head_size=64, rot_dim=32, page_size=16,
                             num_pages=2)
    assert pd.paged_rope_cache_write(empty.q, empty.k, empty.v, empty.positions,
                                     empty.slot_mapping, empty.cos_sin, empty.q, empty.k_cache,
                                     empty.v_cache, 4, 2, 64, 32, 16, W.HND, True,
                                     check=False) == 0            # nothing to do, no device
    if not torch.cuda.is_available():
        assert call() == -8                                           # a valid call needs the GPU


def test_prefill_argument_checks_on_host(lib):
    """paged_prefill_attn's checks run before any device call."""
    c = W.make_prefill_case("abi_pf", seed=1, q_lens=[70, 20], contexts=[30, 0],
                            num_q_heads=8, num_kv_heads=2)
    items, info = pd.paged_prefill_plan(c.query_start_host, c.seq_lens_host, 8, 2, 128, 0, 152)

    def call(**over):
        a = dict(q=c.q, k_cache=c.k_cache, v_cache=c.v_cache, block_table=c.block_table,
                 seq_lens=c.seq_lens, query_start=c.query_start, work=items, info=info,
                 out=c.q, num_q_heads=8, num_kv_heads=2, head_size=128, page_size=16,
                 window=0, scale=0.1, layout=W.HND, scratch=None)
        a.update(over)
        return pd.paged_prefill_attn(**a, check=False)

    assert call(head_size=96) == -3
    assert call(num_q_heads=7) == -1
    assert call(work=items[:-1]) == -1                      # rows != info.num_items
    assert call(work=items[:, :4].contiguous()) == -1       # 8 int32 per item
    assert call(query_start=c.query_start[:-1]) == -1
    assert call(query_start=c.query_start.to(torch.int64)) == -2
    assert call(page_size=24) == -1
    bad = pd.PdPrefillPlanInfo.from_buffer_copy(info)
    bad.tile_rows = 32
    assert call(info=bad) == -1
    # a plan made for another head size (64-row tiles) does not fit head size 128
    items64, info64 = pd.paged_prefill_plan(c.query_start_host, c.seq_lens_host, 8, 2, 64, 0, 152)
    assert info64.tile_rows == 64 and info.tile_rows == 256
    assert call(work=items64, info=info64) == -1
    if not torch.cuda.is_available():
        assert call() == -8                                  # a valid call needs the GPU
