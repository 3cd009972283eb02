"""The prefill work-list planner on the CPU (host code of the C ABI, no
device): the rules of plan_prefill and prefill_target_workgroups on the
vllm.v1.attention.ops.rocm_rdna_hip page, restated for this kernel (64
packed rows per tile, 256 at head size 128; 16-key blocks, one CTA per SM):

* a request's tiles cover its q_len x G packed rows, token-major;
* a tile's keys run from its window start, rounded down to a 16-key block,
  to the last key its last token sees;
* the load is the larger of (kv heads x all blocks / resident CTAs) and a
  floor; a tile above it is cut into min(ceil(blocks / load), blocks /
  floor, 32) segments;
* items are ordered by blocks per segment, heaviest first, stably;
* fewer than target / kv heads tiles are split, into fewer than 2 x target
  / kv heads slots (what paged_prefill_scratch_bytes provides)."""

import math

import numpy as np
import pytest

import paged_split_kv_02_gb300 as pd

FLOOR, MAX_SEG, BLOCK = 8, 32, 16


def rows_for(D):
    return 256 if D == 128 else 64


def _plan(q_lens, ctx, Hq=32, Hkv=8, window=0, sms=152, D=64):
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    lens = (np.asarray(ctx) + np.asarray(q_lens)).astype(np.int32)
    items, info = pd.paged_prefill_plan(qs, lens, Hq, Hkv, D, window, sms)
    return items.numpy(), info, qs, lens


def _expected_tiles(q_lens, ctx, G, window, ROWS):
    """(seq, tile) -> (first token, last token, key_begin, key_end, blocks)."""
    out = {}
    for s, (m, c) in enumerate(zip(q_lens, ctx)):
        for t in range(-(-m * G // ROWS)):
            first, last = t * ROWS // G, min(m - 1, ((t + 1) * ROWS - 1) // G)
            end = c + last + 1
            begin = (max(0, c + first - window + 1) // BLOCK * BLOCK) if window else 0
            out[(s, t)] = (first, last, begin, end, -(-(end - begin) // BLOCK))
    return out


def test_hand_worked_single_request():
    # 512 new tokens, no context, G = 4: 32 tiles, tile t sees 16 (t + 1)
    # keys = t + 1 blocks; 528 blocks x 8 kv heads / 152 = 27.8 per CTA;
    # tiles of 28 .. 32 blocks split in two; 27 + 5 x 2 = 37 items, the
    # unsplit 27-block tile first
    items, info, _, _ = _plan([512], [0])
    assert info.num_items == 37 and info.num_split_tiles == 5 and info.num_slots == 10
    assert info.total_blocks == 528
    assert info.load_blocks == pytest.approx(8 * 528 / 152)
    assert tuple(items[0, :4]) == (0, 26, 0, 1) and items[0, 6] == 27
    split = items[items[:, 3] > 1]
    assert sorted(set(split[:, 1].tolist())) == [27, 28, 29, 30, 31]
    assert np.all(split[:, 3] == 2)


def test_hand_worked_single_request_256_row_tiles():
    # the same request at head size 128: 8 tiles of 64 tokens, tile t sees
    # 64 (t + 1) keys = 4 (t + 1) blocks; 144 blocks x 8 / 152 = 7.6 per CTA,
    # below the floor of 8; a tile of b > 8 blocks is cut into
    # min(ceil(b / 8), b // 8) segments: 12 -> 1, 16 -> 2, 20 -> 2, 24 -> 3,
    # 28 -> 3, 32 -> 4; 3 + 14 = 17 items.  Heaviest per segment first: the
    # unsplit 12-block tile, the 20-block tile's halves (10), the 28-block
    # tile's thirds (9.3), then the 8-block segments in tile order
    items, info, _, _ = _plan([512], [0], D=128)
    assert info.tile_rows == 256 and info.total_blocks == 144
    assert info.load_blocks == pytest.approx(8)
    assert info.num_items == 17 and info.num_split_tiles == 5 and info.num_slots == 14
    assert [tuple(r) for r in items[:6, :4]] == [(0, 2, 0, 1), (0, 4, 0, 2), (0, 4, 1, 2),
                                                 (0, 6, 0, 3), (0, 6, 1, 3), (0, 6, 2, 3)]
    assert [int(t) for t in items[6:, 1]] == [7] * 4 + [5] * 3 + [3] * 2 + [1, 0]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("q_lens,ctx,Hq,Hkv,window,sms", [
    ([512], [0], 32, 8, 0, 152),
    ([1, 40, 257, 0, 100], [0, 1000, 60, 500, 3000], 32, 8, 0, 152),
    ([400], [2000], 8, 1, 256, 152),
    ([3000, 17, 900], [100, 20000, 0], 16, 2, 0, 148),
    ([64, 64, 64, 64], [8000, 8000, 8000, 8000], 8, 8, 0, 2000),   # many splits
    ([5, 9, 1], [0, 0, 0], 4, 4, 0, 152),                           # tiny
    ([2048], [30000], 64, 8, 4096, 152),
])
def test_plan_rules(q_lens, ctx, Hq, Hkv, window, sms, D):
    G = Hq // Hkv
    ROWS = rows_for(D)
    items, info, qs, lens = _plan(q_lens, ctx, Hq, Hkv, window, sms, D)
    exp = _expected_tiles(q_lens, ctx, G, window, ROWS)
    total = sum(v[4] for v in exp.values())
    assert info.total_blocks == total and info.tile_rows == ROWS and info.target_ctas == sms
    load = max(Hkv * total / sms, FLOOR)
    assert info.load_blocks == pytest.approx(load)
    # every tile once, with all of its segments, in order
    seen = {}
    for it in items:
        s, t, g, n, split, slot, blocks, res = (int(x) for x in it)
        assert res == 0 and 0 <= g < n
        key = (s, t)
        assert blocks == exp[key][4]
        want_n = 1
        if blocks > load:
            want_n = max(1, min(math.ceil(blocks / load), blocks // FLOOR, MAX_SEG))
        assert n == want_n, (key, blocks, load)
        if n == 1:
            assert split == -1 and slot == -1
        seen.setdefault(key, []).append((g, split, slot))
    assert set(seen) == set(exp)
    splits, slots = set(), set()
    for key, segs in seen.items():
        assert [g for g, _, _ in segs] == list(range(len(segs)))
        if len(segs) > 1:
            assert len({sp for _, sp, _ in segs}) == 1 and len({sl for _, _, sl in segs}) == 1
            splits.add(segs[0][1])
            slots.update(range(segs[0][2], segs[0][2] + len(segs)))
    # split indices 0..n-1, slots consecutive and disjoint
    assert splits == set(range(info.num_split_tiles))
    assert slots == set(range(info.num_slots))
    assert info.num_split_tiles * Hkv < sms and info.num_slots * Hkv < 2 * sms
    # heaviest per segment first, stable
    per = items[:, 6] / items[:, 3]
    assert np.all(np.diff(per) <= 1e-12)
    # the tiles' rows cover every (token, q head) of every request once
    for s, m in enumerate(q_lens):
        rows = sorted(r for (ss, t) in exp if ss == s for r in range(t * ROWS, (t + 1) * ROWS)
                      if r < m * G)
        assert rows == list(range(m * G))


def test_plan_size_query_and_capacity():
    items, info, qs, lens = _plan([300, 20], [100, 0])
    info2 = pd.PdPrefillPlanInfo()
    import ctypes
    L = pd.lib()
    assert L.paged_prefill_plan(qs.ctypes.data, lens.ctypes.data, 2, 32, 8, 64, 0, 152, None, 0,
                                ctypes.byref(info2)) == 0
    assert info2.num_items == info.num_items
    buf = (pd.PdPrefillItem * max(1, int(info.num_items) - 1))()
    assert L.paged_prefill_plan(qs.ctypes.data, lens.ctypes.data, 2, 32, 8, 64, 0, 152, buf,
                                int(info.num_items) - 1, ctypes.byref(info2)) == -1
    # a head size the kernels do not serve
    assert L.paged_prefill_plan(qs.ctypes.data, lens.ctypes.data, 2, 32, 8, 96, 0, 152, None, 0,
                                ctypes.byref(info2)) == -3


def test_plan_rejects_malformed_query_start():
    with pytest.raises(pd.PagedDecodeError):
        pd.paged_prefill_plan([0, 10, 5], [10, 10], 32, 8, 128, 0, 152)   # decreasing
    with pytest.raises(pd.PagedDecodeError):
        pd.paged_prefill_plan([0, 10], [10], 30, 8, 128, 0, 152)          # Hq % Hkv
    items, info = pd.paged_prefill_plan([0, 0, 0], [5, 0], 32, 8, 128, 0, 152)
    assert info.num_items == 0 and items.shape == (0, 8)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_prefill_scratch_bytes_cover_every_plan(D):
    Hkv, sms = 8, 152
    ROWS = rows_for(D)
    n = pd.paged_prefill_scratch_bytes(Hkv, D, sms)
    counters = -(-sms * pd.COUNTERS_PER_PAIR * 4 // 256) * 256
    acc = -(-2 * sms * ROWS * D * 4 // 256) * 256
    ml = -(-2 * sms * ROWS * 2 * 4 // 256) * 256
    assert n == counters + acc + ml
    # a plan's split tiles and slots fit: (tiles x kv heads) counters in
    # pairs, (slots x kv heads) partials
    for q_lens, ctx in [([512], [0]), ([64] * 8, [8000] * 8), ([2048], [30000])]:
        _, info, _, _ = _plan(q_lens, ctx, Hkv=Hkv, sms=sms, D=D)
        assert 2 * info.num_split_tiles * Hkv <= sms * pd.COUNTERS_PER_PAIR
        assert info.num_slots * Hkv <= 2 * sms
    assert pd.paged_prefill_scratch_bytes(8, 96, 152) == 0
