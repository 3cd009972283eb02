"""fp64 CPU oracle of the rotary embedding and the paged KV-cache write that
run ahead of decode attention (test infrastructure only: only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import it;
the product path never does).

The pages only name this step: the fused RoPE / KV-cache write was split
out of ROCm/vllm PR #1330 into a draft PR of its own (#1342; "Summary") and
its text is not given.  What they do show fixes the data it works on:

* the cache store of the vLLM ROCm Octave backend
  (``RocmOctaveAttentionImpl.do_kv_cache_update(layer, key, value,
  kv_cache, slot_mapping)``): token t's key and value go to the cache slot
  ``slot_mapping[t]`` (page ``slot // page_size``, token ``slot %
  page_size``), for the first ``len(slot_mapping)`` tokens;
* a rotary part of the head (``rope_dim`` of ``head_size``; the Octave
  backend registers 64 rotary dims of 256), so the rotation may cover only
  the leading ``rot_dim`` dims of a head.

The reading taken here (the plainest one the rest supports): the standard
rotary position embedding of q and k, with angles from a precomputed
``cos_sin_cache[position]`` row (cos in its first ``rot_dim / 2`` columns,
sin in the rest), in the "rotate half" pairing (dim i with dim i +
rot_dim/2, the NeoX form) or the interleaved pairing (dims 2i, 2i+1, the
GPT-J form); dims at and past ``rot_dim`` pass through; v is stored
unrotated; a slot of -1 is a padding token and writes nothing.  For a pair
(x1, x2) and angle (c, s):

    x1' = x1 c - x2 s,    x2' = x2 c + x1 s.

Everything here is fp64 on the exactly widened fp16/bf16 inputs and the
fp32 table.
"""

from __future__ import annotations

import numpy as np
import torch


def widen(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 values of an fp16 / bf16 / fp32 tensor."""
    return t.detach().cpu().double().numpy()


def pair_index(rot_dim: int, is_neox: bool):
    """(first, second) dim of every rotated pair, in angle order i =
    0 .. rot_dim/2 - 1: (i, i + rot_dim/2) for NeoX, (2i, 2i + 1) for GPT-J."""
    half = rot_dim // 2
    i = np.arange(half)
    if is_neox:
        return i, i + half
    return 2 * i, 2 * i + 1


def rope(x: np.ndarray, positions: np.ndarray, cos_sin: np.ndarray, rot_dim: int,
         is_neox: bool) -> np.ndarray:
    """Rotate every head of every token: x [T, H, D] (fp64), positions [T],
    cos_sin [max_pos, rot_dim]; dims >= rot_dim are copied."""
    out = np.array(x, dtype=np.float64, copy=True)
    half = rot_dim // 2
    a, b = pair_index(rot_dim, is_neox)
    for t in range(x.shape[0]):
        row = cos_sin[int(positions[t])]
        c, s = row[:half], row[half:rot_dim]
        for h in range(x.shape[1]):
            x1, x2 = x[t, h, a], x[t, h, b]
            out[t, h, a] = x1 * c - x2 * s
            out[t, h, b] = x2 * c + x1 * s
    return out


def cache_slot_index(slot: int, page_size: int):
    """(page, token within the page) of a cache slot."""
    return slot // page_size, slot % page_size


def rope_cache_write(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                     positions: torch.Tensor, slot_mapping: torch.Tensor,
                     cos_sin_cache: torch.Tensor, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, layout: int, rot_dim: int, is_neox: bool):
    """The expected results of one call.

    q [T, Hq, D], k / v [T, Hkv, D]; positions, slot_mapping [T] (slot -1:
    nothing written); k_cache / v_cache the pools before the call, NHD
    [NB, P, Hkv, D] (layout 0) or HND [NB, Hkv, P, D] (layout 1).

    Returns (q_out [T, Hq, D], k_pool, v_pool, written) in fp64, the pools in
    the caches' own index order, and ``written`` the list of (token, page,
    in-page slot) the call writes.  The slots of one call are distinct (a
    slot named twice has no defined result)."""
    pos = positions.cpu().numpy().astype(np.int64)
    slots = slot_mapping.cpu().numpy().astype(np.int64)
    table = widen(cos_sin_cache)
    q_out = rope(widen(q), pos, table, rot_dim, is_neox)
    k_rot = rope(widen(k), pos, table, rot_dim, is_neox)
    vv = widen(v)
    k_pool, v_pool = widen(k_cache), widen(v_cache)
    P = k_cache.shape[1] if layout == 0 else k_cache.shape[2]
    written = []
    for t in range(k.shape[0]):
        if slots[t] < 0:
            continue
        page, off = cache_slot_index(int(slots[t]), P)
        for h in range(k.shape[1]):
            if layout == 0:
                k_pool[page, off, h] = k_rot[t, h]
                v_pool[page, off, h] = vv[t, h]
            else:
                k_pool[page, h, off] = k_rot[t, h]
                v_pool[page, h, off] = vv[t, h]
        written.append((t, page, off))
    return q_out, k_pool, v_pool, written
