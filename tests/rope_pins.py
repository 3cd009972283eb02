"""Pins of the rotary-embedding + cache-write oracle (``oracle/rope_cache.py``)
against facts fixed by mathematics and by the cache's slot convention, not
by the oracle itself.

Every pin takes ``R`` (the oracle module, or a copy of it with a planted
mistake: ``test_rope_oracle_mutants.py``) and raises AssertionError when it
fails.

Sources of the facts:
* slot -> (page, token in the page) = (slot // page_size, slot % page_size),
  -1 = no write (the cache store of vllm.v1.attention.backends.
  rocm_octave_attn, ``do_kv_cache_update`` with ``slot_mapping``);
* rotary dims: a leading part of the head (the Octave backend's
  ``rope_dim`` of ``head_size``), the rest passes through;
* a rotation by angle theta of each pair: the identity at theta = 0, norm
  preserving, R(a) R(b) = R(a + b), and <R(m) q, R(n) k> depends on m - n
  only (the defining property of a rotary position embedding).
"""

from __future__ import annotations

import math

import numpy as np
import torch

from paged_split_kv_02_gb300 import workloads as W


def _x(shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape)


def _table(max_pos, rot):
    return W.rope_cos_sin_table(max_pos, rot).double().numpy()


def pin_position_zero_is_identity(R):
    x = _x((3, 2, 16))
    for neox in (True, False):
        out = R.rope(x, np.zeros(3, dtype=np.int64), _table(8, 16), 16, neox)
        assert np.array_equal(out, x)


def pin_quarter_turn(R):
    # a table row with cos = 0, sin = 1 exactly: (x1, x2) -> (-x2, x1)
    rot = 8
    tab = np.zeros((1, rot))
    tab[0, rot // 2:] = 1.0
    x = _x((1, 1, rot), 1)
    out = R.rope(x, np.zeros(1, dtype=np.int64), tab, rot, True)
    exp = np.concatenate([-x[0, 0, 4:], x[0, 0, :4]])
    assert np.array_equal(out[0, 0], exp)
    out = R.rope(x, np.zeros(1, dtype=np.int64), tab, rot, False)
    exp = np.empty(rot)
    exp[0::2], exp[1::2] = -x[0, 0, 1::2], x[0, 0, 0::2]
    assert np.array_equal(out[0, 0], exp)


def pin_brute_force_tiny(R):
    # D = rot = 4, one row [c0, c1, s0, s1], expanded by hand
    a, b, c, d = 0.5, -1.25, 2.0, 0.75
    c0, c1, s0, s1 = 0.6, -0.8, 0.8, 0.6
    x = np.array([[[a, b, c, d]]])
    tab = np.array([[c0, c1, s0, s1]])
    pos = np.zeros(1, dtype=np.int64)
    neox = R.rope(x, pos, tab, 4, True)[0, 0]
    assert np.allclose(neox, [a * c0 - c * s0, b * c1 - d * s1, c * c0 + a * s0, d * c1 + b * s1],
                       rtol=0, atol=1e-15)
    gptj = R.rope(x, pos, tab, 4, False)[0, 0]
    assert np.allclose(gptj, [a * c0 - b * s0, b * c0 + a * s0, c * c1 - d * s1, d * c1 + c * s1],
                       rtol=0, atol=1e-15)


def pin_norm_preserved(R):
    rot = 32
    tab = _table(64, rot)
    x = _x((5, 3, 48), 2)
    pos = np.array([0, 1, 7, 33, 63])
    for neox in (True, False):
        out = R.rope(x, pos, tab, rot, neox)
        n_in = np.linalg.norm(x, axis=-1)
        n_out = np.linalg.norm(out, axis=-1)
        # the fp32 table's cos^2 + sin^2 is 1 to ~1e-7
        assert np.allclose(n_out, n_in, rtol=1e-6, atol=0)


def pin_relative_position(R):
    rot = 64
    tab = _table(256, rot)
    q = _x((1, 1, 64), 3)
    k = _x((1, 1, 64), 4)
    for neox in (True, False):
        for m, n in [(5, 2), (100, 37), (200, 200), (255, 0)]:
            lhs = float(np.sum(R.rope(q, np.array([m]), tab, rot, neox) *
                               R.rope(k, np.array([n]), tab, rot, neox)))
            rhs = float(np.sum(R.rope(q, np.array([m - n]), tab, rot, neox) * k))
            assert abs(lhs - rhs) <= 1e-4 * (1 + abs(rhs)), (m, n, lhs, rhs)
        # and it does depend on m - n
        a = float(np.sum(R.rope(q, np.array([9]), tab, rot, neox) * k))
        b = float(np.sum(R.rope(q, np.array([3]), tab, rot, neox) * k))
        assert abs(a - b) > 1e-3


def pin_composition(R):
    rot = 16
    tab = _table(64, rot)
    x = _x((1, 2, 16), 5)
    for neox in (True, False):
        twice = R.rope(R.rope(x, np.array([11]), tab, rot, neox), np.array([20]), tab, rot, neox)
        once = R.rope(x, np.array([31]), tab, rot, neox)
        assert np.allclose(twice, once, rtol=0, atol=1e-5)


def pin_neox_is_interleaved_gptj(R):
    # NeoX on x equals GPT-J on the interleaved x, mapped back
    rot, D = 16, 24
    tab = _table(32, rot)
    x = _x((4, 2, D), 6)
    pos = np.array([0, 3, 17, 31])
    perm = np.arange(D)
    half = rot // 2
    perm[0:rot:2], perm[1:rot:2] = np.arange(half), np.arange(half) + half
    neox = R.rope(x, pos, tab, rot, True)
    gptj = R.rope(x[..., perm], pos, tab, rot, False)
    back = np.empty_like(gptj)
    back[..., perm] = gptj
    assert np.array_equal(neox, back)


def pin_partial_rotary_passthrough(R):
    x = _x((3, 2, 64), 7)
    tab = _table(16, 16)
    for neox in (True, False):
        out = R.rope(x, np.array([1, 5, 15]), tab, 16, neox)
        assert np.array_equal(out[..., 16:], x[..., 16:])
        assert not np.allclose(out[1:, :, :16], x[1:, :, :16])


def _write_case(layout, neox=True, rot=32, pad=2):
    return W.make_rope_case("pin", seed=3, dtype=torch.bfloat16, num_tokens=12, num_q_heads=4,
                            num_kv_heads=2, head_size=64, rot_dim=rot, page_size=16,
                            num_pages=5, layout=layout, is_neox=neox, max_pos=64,
                            pad_tokens=pad)


def _pool_at(pool, layout, page, off, h):
    return pool[page, off, h] if layout == W.NHD else pool[page, h, off]


def pin_cache_write_roundtrip(R):
    for layout in (W.NHD, W.HND):
        c = _write_case(layout)
        q_out, k_pool, v_pool, written = R.rope_cache_write(
            c.q, c.k, c.v, c.positions, c.slot_mapping, c.cos_sin, c.k_cache, c.v_cache,
            layout, c.rot_dim, c.is_neox)
        tab = c.cos_sin.double().numpy()
        pos = c.positions.numpy().astype(np.int64)
        k_rot = R.rope(c.k.double().numpy(), pos, tab, c.rot_dim, c.is_neox)
        assert np.array_equal(q_out, R.rope(c.q.double().numpy(), pos, tab, c.rot_dim, c.is_neox))
        slots = c.slot_mapping.numpy()
        live = [t for t in range(len(slots)) if slots[t] >= 0]
        assert len(written) == len(live) == 10
        touched = set()
        for t in live:
            page, off = int(slots[t]) // 16, int(slots[t]) % 16
            touched.add((page, off))
            for h in range(2):
                assert np.array_equal(_pool_at(k_pool, layout, page, off, h), k_rot[t, h])
                assert np.array_equal(_pool_at(v_pool, layout, page, off, h),
                                      c.v.double().numpy()[t, h])
        k0, v0 = c.k_cache.double().numpy(), c.v_cache.double().numpy()
        for page in range(5):
            for off in range(16):
                if (page, off) in touched:
                    continue
                for h in range(2):
                    assert np.array_equal(_pool_at(k_pool, layout, page, off, h),
                                          _pool_at(k0, layout, page, off, h))
                    assert np.array_equal(_pool_at(v_pool, layout, page, off, h),
                                          _pool_at(v0, layout, page, off, h))


def pin_layouts_agree(R):
    out = {}
    for layout in (W.NHD, W.HND):
        c = _write_case(layout, neox=False, rot=64, pad=0)
        _, k_pool, v_pool, written = R.rope_cache_write(
            c.q, c.k, c.v, c.positions, c.slot_mapping, c.cos_sin, c.k_cache, c.v_cache,
            layout, c.rot_dim, c.is_neox)
        out[layout] = {(t, h): (_pool_at(k_pool, layout, p, o, h), _pool_at(v_pool, layout, p, o, h))
                       for t, p, o in written for h in range(2)}
    assert out[W.NHD].keys() == out[W.HND].keys()
    for key in out[W.NHD]:
        assert np.array_equal(out[W.NHD][key][0], out[W.HND][key][0])
        assert np.array_equal(out[W.NHD][key][1], out[W.HND][key][1])


def pin_table_is_the_closed_form(R):
    # the generated table (an input, checked here so the other pins stand on
    # a real rotation table): cos / sin of position x base^(-2i/rot)
    tab = _table(50, 16)
    for p in (0, 1, 49):
        for i in (0, 3, 7):
            th = p * 10000.0 ** (-2.0 * i / 16)
            assert abs(tab[p, i] - math.cos(th)) < 1e-7
            assert abs(tab[p, 8 + i] - math.sin(th)) < 1e-7


ALL_PINS = [pin_position_zero_is_identity, pin_quarter_turn, pin_brute_force_tiny,
            pin_norm_preserved, pin_relative_position, pin_composition,
            pin_neox_is_interleaved_gptj, pin_partial_rotary_passthrough,
            pin_cache_write_roundtrip, pin_layouts_agree, pin_table_is_the_closed_form]
