"""Pins of the fp64 oracle against facts fixed by the decode semantics and
by mathematics, not by the oracle itself.

Every function takes ``lib`` (a loaded oracle library, or None for the
built one) and raises AssertionError when the pin fails, so the same pins
also run against planted mistakes (``test_oracle_mutants.py``).

Sources of the facts:
* key length of query i: seq_len - q_len + i + 1, padding queries get 0
  (rocm_octave_attn, ``RocmOctaveMetadataBuilder._fill_query_maps``);
* window in keys, 0 = full causal (rocm_rdna_hip, ``KernelVariant``), the
  window's first key of query ``first`` is ``context + first - window + 1``
  (rocm_rdna_hip, ``plan_prefill``);
* rows of a kv head = gqa * M (rocm_rdna_hip, ``KernelVariant.rows_padded``);
* NHD / HND / packed K|V are stride orders of one cache
  (rocm_rdna_hip, ``KernelVariant.layout``, ``expected_kv_cache_strides``);
* split-KV partials (acc, m, l) merged in-kernel
  (rocm_rdna_hip, ``KernelVariant.scratch_shapes``).
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from paged_split_kv_02_gb300 import workloads as W


def _case(**kw):
    base = dict(seed=1, dtype=torch.float16, head_size=16, num_q_heads=4, num_kv_heads=2,
                page_size=4, max_query_len=1, seq_lens=[11], layout=W.HND)
    base.update(kw)
    return W.make_case("pin", **base)


def _visible(L, M, i, window):
    n = max(L - M + i + 1, 0)
    lo = max(0, n - window) if window else 0
    return lo, n


def _logical_rows(case, which, s, h):
    """fp64 rows [L_s, D] of K or V of kv head h in logical order (a gather
    written independently of the oracle, with torch indexing)."""
    t = case.k_cache if which == "k" else case.v_cache
    L = int(case.seq_lens[s])
    pos = torch.arange(L)
    phys = case.block_table[s, pos // case.page_size].long()
    tok = pos % case.page_size
    if case.layout == W.NHD:
        rows = t[phys, tok, h]
    else:
        rows = t[phys, h, tok]
    return rows.double().numpy()


def pin_single_key(lib=None):
    """One key, one query: the output is that key's V row, exactly."""
    for dt in (torch.float16, torch.bfloat16):
        c = _case(dtype=dt, seq_lens=[1], page_size=4)
        o = oracle.attention(c, lib=lib)
        for hq in range(c.num_q_heads):
            h = hq // (c.num_q_heads // c.num_kv_heads)
            v0 = _logical_rows(c, "v", 0, h)[0]
            assert np.array_equal(o[0, hq], v0), (dt, hq)


def pin_identical_keys_mean(lib=None):
    """All keys equal: softmax is uniform, the output is the mean of the
    visible V rows (checked per row, with M = 3 causal rows)."""
    c = _case(seq_lens=[13], max_query_len=3, num_q_heads=6, num_kv_heads=3, page_size=4)
    # overwrite every K slot of the pool with one row
    c.k_cache[:] = c.k_cache.new_tensor(np.linspace(-1, 1, c.head_size))
    o = oracle.attention(c, lib=lib)
    G = c.num_q_heads // c.num_kv_heads
    for i in range(3):
        lo, hi = _visible(13, 3, i, 0)
        for hq in range(c.num_q_heads):
            v = _logical_rows(c, "v", 0, hq // G)
            np.testing.assert_allclose(o[i, hq], v[lo:hi].mean(axis=0), rtol=0, atol=1e-12)


def pin_zero_query_mean(lib=None):
    """q = 0: every logit is 0, the output is the mean of the visible V rows."""
    c = _case(seq_lens=[21], max_query_len=2, page_size=8, window=5)
    c.q.zero_()
    o = oracle.attention(c, lib=lib)
    for i in range(2):
        lo, hi = _visible(21, 2, i, 5)
        assert hi - lo == 5
        for hq in range(c.num_q_heads):
            v = _logical_rows(c, "v", 0, hq // 2)
            np.testing.assert_allclose(o[i, hq], v[lo:hi].mean(axis=0), rtol=0, atol=1e-12)


def pin_position_mean(lib=None):
    """q = 0 and V[k] = k (every element): the output is the mean of the
    visible positions, (lo + hi - 1) / 2, for each causal row and window."""
    for window in (0, 1, 3, 7, 100):
        c = _case(seq_lens=[37, 5, 0, 2], max_query_len=4, page_size=4, window=window,
                  num_q_heads=2, num_kv_heads=1, head_size=8)
        c.q.zero_()
        for s, L in enumerate(c.seq_lens.tolist()):
            for k in range(L):
                phys = int(c.block_table[s, k // c.page_size])
                c.v_cache[phys, :, k % c.page_size, :] = float(k)
        o = oracle.attention(c, lib=lib)
        for s, L in enumerate(c.seq_lens.tolist()):
            for i in range(4):
                lo, hi = _visible(L, 4, i, window)
                want = (lo + hi - 1) / 2.0 if hi > lo else 0.0
                assert np.all(o[s * 4 + i] == want), (window, s, L, i, o[s * 4 + i, 0, 0], want)


def pin_window_one(lib=None):
    """Window 1: each row sees only its own position n_i - 1."""
    c = _case(seq_lens=[19], max_query_len=4, page_size=4, window=1)
    o = oracle.attention(c, lib=lib)
    for i in range(4):
        n = 19 - 4 + i + 1
        for hq in range(c.num_q_heads):
            v = _logical_rows(c, "v", 0, hq // 2)
            assert np.array_equal(o[i, hq], v[n - 1])


def pin_wide_window_is_full(lib=None):
    """A window at least as long as the sequence is no window."""
    a = oracle.attention(_case(seq_lens=[23], max_query_len=2, window=0), lib=lib)
    for w in (23, 24, 1000):
        b = oracle.attention(_case(seq_lens=[23], max_query_len=2, window=w), lib=lib)
        assert np.array_equal(a, b)


def pin_page_permutation(lib=None):
    """Moving pages in the pool and the block table with them changes nothing."""
    c = _case(seq_lens=[30], page_size=4, max_query_len=2, pool_pages=12)
    a = oracle.attention(c, lib=lib)
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(5))
    inv = torch.argsort(perm)
    c.k_cache = c.k_cache[perm].contiguous()
    c.v_cache = c.v_cache[perm].contiguous()
    c.block_table = inv[c.block_table.long()].to(torch.int32)
    b = oracle.attention(c, lib=lib)
    assert np.array_equal(a, b)


def pin_layouts(lib=None):
    """NHD, HND and the packed K|V cache give bit-identical outputs."""
    kw = dict(seq_lens=[29, 7], page_size=4, max_query_len=3, window=9, seed=3)
    outs = []
    for layout in (W.NHD, W.HND):
        for packed in (False, True):
            outs.append(oracle.attention(_case(layout=layout, packed=packed, **kw), lib=lib))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def pin_split_merge(lib=None):
    """Merging partials over any segmentation of the keys (empty segments
    included) equals the unsplit result."""
    c = _case(seq_lens=[45, 17, 0], max_query_len=3, page_size=8, window=20)
    full = oracle.attention(c, lib=lib)
    for cuts in ([0, 45], [0, 5, 5, 30, 45], [0, 1, 2, 3, 44, 45], list(range(0, 46, 7)) + [45]):
        parts = [oracle.partial(c, a, b, lib=lib) for a, b in zip(cuts[:-1], cuts[1:])]
        np.testing.assert_allclose(oracle.merge(parts), full, rtol=0, atol=1e-12)


def pin_causal_rows(lib=None):
    """Row i of an M-row call equals a one-row call whose sequence ends at
    the row's own position, L' = L - M + i + 1, on the same cache."""
    M, L = 4, 26
    c = _case(seq_lens=[L], max_query_len=M, page_size=4, window=6)
    o = oracle.attention(c, lib=lib)
    for i in range(M):
        c1 = _case(seq_lens=[L], max_query_len=M, page_size=4, window=6)
        c1.max_query_len = 1
        c1.q = c.q[i:i + 1].clone()
        c1.seq_lens = torch.tensor([L - M + i + 1], dtype=torch.int32)
        o1 = oracle.attention(c1, lib=lib)
        assert np.array_equal(o[i], o1[0])


def pin_gqa_is_repeated_mha(lib=None):
    """GQA equals MHA whose kv heads are each kv head repeated G times."""
    c = _case(seq_lens=[14], num_q_heads=6, num_kv_heads=2, page_size=4, max_query_len=2,
              layout=W.NHD)
    a = oracle.attention(c, lib=lib)
    G = 3
    c.k_cache = c.k_cache.repeat_interleave(G, dim=2).contiguous()
    c.v_cache = c.v_cache.repeat_interleave(G, dim=2).contiguous()
    c.num_kv_heads = 6
    b = oracle.attention(c, lib=lib)
    assert np.array_equal(a, b)


def pin_gqa_group_of_head(lib=None):
    """q head hq reads kv head hq // G: with V of kv head h constant h + 1,
    the output of q head hq is hq // G + 1 (up to rounding of the weights)."""
    c = _case(seq_lens=[9], num_q_heads=8, num_kv_heads=4, page_size=4, layout=W.HND)
    for h in range(4):
        c.v_cache[:, h] = float(h + 1)
    o = oracle.attention(c, lib=lib)
    for hq in range(8):
        np.testing.assert_allclose(o[0, hq], hq // 2 + 1, rtol=0, atol=1e-12)


def pin_one_hot_logit(lib=None):
    """A key aligned with q at a large norm dominates: |o - V_j| is bounded by
    the softmax mass of the other keys, sum_k e^(x_k - x_j)."""
    c = _case(seq_lens=[10], num_q_heads=1, num_kv_heads=1, head_size=8, page_size=4)
    c.q.zero_()
    c.q[0, 0, 0] = 8.0
    c.k_cache.zero_()
    j = 6
    phys = int(c.block_table[0, j // 4])
    c.k_cache[phys, 0, j % 4, 0] = 8.0
    c.scale = 1.0 / 4.0
    o = oracle.attention(c, lib=lib)[0, 0]
    v = _logical_rows(c, "v", 0, 0)
    x_j = c.scale * 64.0
    bound = 9 * math.exp(-x_j) * (np.abs(v).max() * 2)
    assert np.max(np.abs(o - v[j])) <= bound
    assert np.max(np.abs(o - v[j])) > 0  # the other keys still carry mass


def pin_two_keys_logistic(lib=None):
    """Two keys: the weight of key 0 is the logistic function of the logit
    difference, sigma(x0 - x1) = 1 / (1 + e^(x1 - x0))."""
    c = _case(seq_lens=[2], num_q_heads=1, num_kv_heads=1, head_size=4, page_size=4)
    c.q[0, 0] = torch.tensor([1.0, 0.5, -2.0, 0.25], dtype=torch.float16)
    kk = torch.tensor([[0.5, 1.0, 0.25, 2.0], [-1.0, 0.75, 0.5, 0.0]], dtype=torch.float16)
    vv = torch.tensor([[1.0, 0.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0]], dtype=torch.float16)
    phys = int(c.block_table[0, 0])
    c.k_cache[phys, 0, :2] = kk
    c.v_cache[phys, 0, :2] = vv
    c.scale = 0.5
    o = oracle.attention(c, lib=lib)[0, 0]
    q = c.q[0, 0].double()
    x0 = 0.5 * float(q @ kk[0].double())
    x1 = 0.5 * float(q @ kk[1].double())
    w0 = 1.0 / (1.0 + math.exp(x1 - x0))
    np.testing.assert_allclose(o, [w0, 1 - w0, 0, 0], rtol=0, atol=1e-15)


def pin_empty_rows_zero(lib=None):
    """Rows that see no key (an empty slot, or L < M) output zeros."""
    c = _case(seq_lens=[0, 2, 5], max_query_len=4, page_size=4)
    o = oracle.attention(c, lib=lib)
    assert np.all(o[0:4] == 0)
    assert np.all(o[4:6] == 0)      # L=2, M=4: rows 0, 1 see nothing
    assert np.all(np.isfinite(o))
    assert np.any(o[6:8] != 0)


def pin_poison_never_read(lib=None):
    """NaN in every slot no row may see (partial last page, pages before a
    window, slack pages) never reaches the output."""
    c = W.make_case("poison", seed=2, dtype=torch.bfloat16, head_size=32, num_q_heads=4,
                    num_kv_heads=1, page_size=8, max_query_len=4, seq_lens=[77, 3],
                    layout=W.HND, window=10, window_pages_only=True, pool_pages=20)
    o = oracle.attention(c, lib=lib)
    assert np.all(np.isfinite(o))


def pin_library_sdpa(lib=None):
    """Against torch's scaled_dot_product_attention (fp64) on the densely
    gathered keys with an explicit causal/window mask and repeated kv heads."""
    for window, M, layout, dt in ((0, 1, W.NHD, torch.float16), (0, 4, W.HND, torch.bfloat16),
                                  (7, 3, W.HND, torch.float16), (2, 8, W.NHD, torch.bfloat16)):
        c = _case(seq_lens=[40, 13, 9], max_query_len=M, page_size=8, window=window,
                  num_q_heads=8, num_kv_heads=2, head_size=32, layout=layout, dtype=dt, seed=9)
        o = oracle.attention(c, lib=lib)
        G = 4
        for s, L in enumerate(c.seq_lens.tolist()):
            K = np.stack([_logical_rows(c, "k", s, h) for h in range(2)])  # [Hkv, L, D]
            V = np.stack([_logical_rows(c, "v", s, h) for h in range(2)])
            Kt = torch.from_numpy(K).repeat_interleave(G, dim=0)
            Vt = torch.from_numpy(V).repeat_interleave(G, dim=0)
            Q = c.q[s * M:(s + 1) * M].double().permute(1, 0, 2)  # [Hq, M, D]
            mask = torch.zeros((M, L), dtype=torch.bool)
            for i in range(M):
                lo, hi = _visible(L, M, i, window)
                mask[i, lo:hi] = True
            ref = torch.nn.functional.scaled_dot_product_attention(
                Q, Kt, Vt, attn_mask=mask, scale=c.scale).permute(1, 0, 2).numpy()
            for i in range(M):
                lo, hi = _visible(L, M, i, window)
                if hi > lo:
                    np.testing.assert_allclose(o[s * M + i], ref[i], rtol=0, atol=1e-12)


def pin_widen_exact(lib=None):
    """The oracle widens every fp16 and bf16 word exactly like torch does."""
    lib_ = lib or oracle._load()
    words = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    for dt, flag in ((torch.float16, 0), (torch.bfloat16, 1)):
        ref = words.view(dt).double().numpy()
        step = 97 if lib is not None else 1
        for w in range(0, 65536, step):
            got = lib_.pdo_widen(w, flag)
            r = ref[w]
            assert (math.isnan(got) and math.isnan(r)) or got == r, (dt, hex(w), got, r)


def _varlen_case(q_lens, seq_lens, pad=0, **kw):
    base = dict(seed=4, dtype=torch.float16, head_size=16, num_q_heads=4, num_kv_heads=2,
                page_size=4, seq_lens=seq_lens, layout=W.HND)
    base.update(kw)
    return W.make_varlen_case("pin_varlen", q_lens=q_lens, pad_tokens=pad, **base)


def pin_varlen_uniform(lib=None):
    """Equal query lengths M with query_start = [0, M, 2M, ...] are the
    uniform batch: the same outputs, bit for bit."""
    M = 3
    c = _case(seq_lens=[17, 5, 9], max_query_len=M, window=4, seed=6)
    o = oracle.attention(c, lib=lib)
    qsl = [M * s for s in range(4)]
    v = W.DecodeCase(**{**c.__dict__, "query_start": torch.tensor(qsl, dtype=torch.int32),
                        "query_start_host": qsl})
    assert np.array_equal(oracle.attention(v, lib=lib), o)


def pin_varlen_request_alone(lib=None):
    """Each request of a mixed batch (lengths 3, 0, 1, 5, 2, a window) gives
    the outputs of a uniform call of that request alone with M = its q_len,
    on the same cache and block-table row."""
    q_lens, lens = [3, 0, 1, 5, 2], [14, 6, 1, 23, 2]
    c = _varlen_case(q_lens, lens, pad=2, window=6)
    o = oracle.attention(c, lib=lib)
    qsl = c.query_start_host
    for s, m in enumerate(q_lens):
        if m == 0:
            continue
        c1 = W.DecodeCase(**{**c.__dict__, "q": c.q[qsl[s]:qsl[s + 1]].clone(),
                             "block_table": c.block_table[s:s + 1].clone(),
                             "seq_lens": c.seq_lens[s:s + 1].clone(), "seq_lens_host": None,
                             "max_query_len": m, "query_start": None, "query_start_host": None})
        assert np.array_equal(oracle.attention(c1, lib=lib), o[qsl[s]:qsl[s + 1]])


def pin_varlen_padding_zero(lib=None):
    """Tokens at and past query_start[S] belong to no request: zeros; the
    rows of the requests are not all zero."""
    c = _varlen_case([2, 1], [9, 4], pad=3)
    o = oracle.attention(c, lib=lib)
    assert np.all(o[3:] == 0.0) and np.abs(o[:3]).max() > 0


def pin_varlen_library_sdpa(lib=None, q_lens=(2, 4, 0, 1, 3), lens=(19, 8, 5, 1, 30), window=5):
    """Against torch's scaled_dot_product_attention (fp64) on densely
    gathered keys, each token's request found with numpy's right-sided
    searchsorted over query_start[1:] and its key length seq_len - q_len +
    (t - query_start[r]) + 1 (the query maps of the pages)."""
    q_lens, lens = list(q_lens), list(lens)
    c = _varlen_case(q_lens, lens, pad=1, window=window, num_q_heads=8, head_size=32,
                     page_size=8, dtype=torch.bfloat16, seed=12)
    o = oracle.attention(c, lib=lib)
    qsl = np.asarray(c.query_start_host)
    T = c.q.shape[0]
    req = np.searchsorted(qsl[1:], np.arange(T), side="right")
    G = 4
    for t in range(T):
        r = int(req[t])
        if r >= len(q_lens):
            assert np.all(o[t] == 0.0)
            continue
        L = lens[r]
        klen = max(L - q_lens[r] + (t - int(qsl[r])) + 1, 0)
        lo = max(0, klen - window) if window else 0
        if klen <= lo:
            assert np.all(o[t] == 0.0)
            continue
        K = np.stack([_logical_rows(c, "k", r, h) for h in range(2)])
        V = np.stack([_logical_rows(c, "v", r, h) for h in range(2)])
        Kt = torch.from_numpy(K).repeat_interleave(G, dim=0)[:, lo:klen]
        Vt = torch.from_numpy(V).repeat_interleave(G, dim=0)[:, lo:klen]
        Q = c.q[t:t + 1].double().permute(1, 0, 2)  # [Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, scale=c.scale)
        np.testing.assert_allclose(o[t], ref.permute(1, 0, 2)[0].numpy(), rtol=0, atol=1e-12)


def pin_prefill_library_sdpa(lib=None):
    """Prefill-sized requests (query lengths past 8, one without context,
    the new tokens' keys included in seq_len) against SDPA the same way,
    with and without a window; the plan_prefill tiles of a request are the
    rows of this one definition."""
    pin_varlen_library_sdpa(lib, q_lens=(37, 1, 20, 0), lens=(60, 9, 20, 3), window=0)
    pin_varlen_library_sdpa(lib, q_lens=(37, 1, 20, 0), lens=(60, 9, 20, 3), window=13)


ALL_PINS = [
    pin_single_key, pin_identical_keys_mean, pin_zero_query_mean, pin_position_mean,
    pin_window_one, pin_wide_window_is_full, pin_page_permutation, pin_layouts,
    pin_split_merge, pin_causal_rows, pin_gqa_is_repeated_mha, pin_gqa_group_of_head,
    pin_one_hot_logit, pin_two_keys_logistic, pin_empty_rows_zero, pin_poison_never_read,
    pin_library_sdpa, pin_widen_exact, pin_varlen_uniform, pin_varlen_request_alone,
    pin_varlen_padding_zero, pin_varlen_library_sdpa, pin_prefill_library_sdpa,
]
