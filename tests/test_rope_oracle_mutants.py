"""Planted mistakes in the rotary-embedding + cache-write oracle must fail
at least one pin.

Each mutant is a copy of ``oracle/rope_cache.py`` with one plausible
mistake (a flipped sign, cos and sin exchanged, the wrong pairing, a
position off by one, page and in-page offset exchanged, v rotated, the
pass-through dims dropped, padding tokens written), loaded as a separate
module.  The real oracle is never modified."""

import os
import types

import pytest

import rope_pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rope_cache.py")

MUTANTS = {
    "first_sign": ("out[t, h, a] = x1 * c - x2 * s", "out[t, h, a] = x1 * c + x2 * s"),
    "second_sign": ("out[t, h, b] = x2 * c + x1 * s", "out[t, h, b] = x2 * c - x1 * s"),
    "cos_sin_swapped": ("c, s = row[:half], row[half:rot_dim]", "s, c = row[:half], row[half:rot_dim]"),
    "neox_pairs_interleaved": ("        return i, i + half", "        return 2 * i, 2 * i + 1"),
    "gptj_pairs_halves": ("    return 2 * i, 2 * i + 1", "    return i, i + half"),
    "position_off_by_one": ("row = cos_sin[int(positions[t])]", "row = cos_sin[int(positions[t]) + 1]"),
    "page_offset_swapped": ("return slot // page_size, slot % page_size",
                            "return slot % page_size, slot // page_size"),
    "v_rotated_nhd": ("v_pool[page, off, h] = vv[t, h]", "v_pool[page, off, h] = k_rot[t, h]"),
    "v_rotated_hnd": ("v_pool[page, h, off] = vv[t, h]", "v_pool[page, h, off] = k_rot[t, h]"),
    "passthrough_dropped": ("out = np.array(x, dtype=np.float64, copy=True)",
                            "out = np.zeros_like(x, dtype=np.float64)"),
    "padding_written": ("if slots[t] < 0:\n            continue", "if slots[t] < -1:\n            continue"),
    "layouts_swapped": ("P = k_cache.shape[1] if layout == 0 else k_cache.shape[2]",
                        "P = k_cache.shape[2] if layout == 0 else k_cache.shape[1]"),
    "q_unrotated": ("q_out = rope(widen(q), pos, table, rot_dim, is_neox)", "q_out = widen(q)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found exactly once: {old}"
    mod = types.ModuleType(f"rope_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    failed = []
    for pin in rope_pins.ALL_PINS:
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
