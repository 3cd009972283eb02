"""fp64 CPU oracle for paged decode attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never does: it fails loudly
when its CUDA library is missing instead of falling back to anything here.

The arithmetic lives in ``paged_decode_oracle.c`` (plain C, fp64, one thread
per slice of output rows).  This wrapper only hands it raw 16-bit words and
element strides; it shares no code with the CUDA path.

* ``attention(case, rows=None)``: outputs ``[S*M, Hq, D]`` (fp64), or the
  selected output rows ``[(t, hq), ...]`` as ``[len(rows), D]``.  A case
  with ``query_start`` (variable query lengths) gives ``[T, Hq, D]`` over
  its T token rows.
* ``partial(case, key_lo, key_hi)``: unnormalised ``(acc, m, l)`` over a key
  sub-range, for the split-KV pins.
* ``merge(parts)``: the split-KV merge of partials, written from its
  definition: ``m* = max m_j``, ``L = sum l_j e^(m_j - m*)``,
  ``o = sum acc_j e^(m_j - m*) / L`` (a segment with ``l = 0`` adds nothing).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_decode_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

NHD = 0
HND = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no GPU code)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its entry points."""
    lib = ctypes.CDLL(path)
    i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    common = [vp, i64, i64, i64, vp, vp, i64, i64, i64, i64, vp, i64, i64, vp,
              i32, i32, i32, i32, i32, i32, i32, i32, dbl]
    lib.pdo_attention.argtypes = common + [vp, i64, vp, i32]
    lib.pdo_attention.restype = i32
    lib.pdo_attention_varlen.argtypes = common + [vp, i64, vp, i64, vp, i32]
    lib.pdo_attention_varlen.restype = i32
    lib.pdo_partial.argtypes = common + [i64, i64, vp, vp, vp, i32]
    lib.pdo_partial.restype = i32
    lib.pdo_widen.argtypes = [ctypes.c_uint16, i32]
    lib.pdo_widen.restype = dbl
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = load_library(_LIB_PATH)
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _raw(t: torch.Tensor):
    """(pointer, element strides) of a CPU fp16/bf16 tensor as 16-bit words."""
    assert t.device.type == "cpu" and t.element_size() == 2
    w = t.view(torch.int16)
    return w.data_ptr(), tuple(w.stride())


def _cache_strides(t: torch.Tensor, layout: int):
    """Strides for (page, token, kv head, d) of a pool in NHD or HND order."""
    s = t.stride()
    if layout == NHD:  # [NB, P, Hkv, D]
        return s[0], s[1], s[2], s[3]
    return s[0], s[2], s[1], s[3]  # HND: [NB, Hkv, P, D]


def _common_args(case):
    q = case.q.cpu()
    k = case.k_cache.cpu() if case.k_cache.device.type != "cpu" else case.k_cache
    v = case.v_cache.cpu() if case.v_cache.device.type != "cpu" else case.v_cache
    bt = case.block_table.cpu().to(torch.int32).contiguous()
    sl = case.seq_lens.cpu().to(torch.int32).contiguous()
    qp, (qs0, qs1, qs2) = _raw(q)
    kp, _ = _raw(k)
    vp, _ = _raw(v)
    sp, st, sh, sd = _cache_strides(k.view(torch.int16), case.layout)
    sp2, st2, sh2, sd2 = _cache_strides(v.view(torch.int16), case.layout)
    assert (sp, st, sh, sd) == (sp2, st2, sh2, sd2), "K and V must share strides"
    keep = (q, k, v, bt, sl)
    args = [qp, qs0, qs1, qs2, kp, vp, sp, st, sh, sd, bt.data_ptr(), bt.stride(0), bt.shape[1],
            sl.data_ptr(), int(sl.shape[0]), int(case.dtype == torch.bfloat16),
            case.num_q_heads, case.num_kv_heads, case.head_size, case.page_size,
            case.max_query_len, int(case.window), float(case.scale)]
    return args, keep


def attention(case, rows=None, nthreads: int | None = None, lib=None) -> np.ndarray:
    """Oracle outputs.  ``rows``: optional list of (token row t, q head hq)."""
    lib = lib or _load()
    args, keep = _common_args(case)
    nthreads = nthreads or default_threads()
    D = case.head_size
    qs = getattr(case, "query_start", None)
    if qs is not None:
        # variable query lengths: rows are the batch's tokens
        qsl = qs.cpu().to(torch.int32).contiguous()
        T = int(case.q.shape[0])
        extra = [qsl.data_ptr(), T]
        if rows is None:
            sel, nsel, shape = None, 0, (T, case.num_q_heads, D)
            n = T * case.num_q_heads
        else:
            sel_a = np.asarray([int(t) * case.num_q_heads + int(h) for t, h in rows], dtype=np.int64)
            sel, nsel, shape, n = sel_a.ctypes.data, len(sel_a), (len(sel_a), D), len(sel_a)
        out = np.empty((n, D), dtype=np.float64)
        rc = lib.pdo_attention_varlen(*args, *extra, sel, nsel, out.ctypes.data, nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle failed: {rc}")
        del keep, qsl
        return out.reshape(shape)
    if rows is None:
        n = case.q.shape[0] * case.num_q_heads
        out = np.empty((n, D), dtype=np.float64)
        rc = lib.pdo_attention(*args, None, 0, out.ctypes.data, nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle failed: {rc}")
        return out.reshape(case.q.shape[0], case.num_q_heads, D)
    sel = np.asarray([int(t) * case.num_q_heads + int(h) for t, h in rows], dtype=np.int64)
    out = np.empty((len(sel), D), dtype=np.float64)
    rc = lib.pdo_attention(*args, sel.ctypes.data, len(sel), out.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle failed: {rc}")
    del keep
    return out


def partial(case, key_lo: int, key_hi: int, nthreads: int | None = None, lib=None):
    """Unnormalised (acc [S*M, Hq, D], m [S*M, Hq], l [S*M, Hq]) over keys
    [key_lo, key_hi) intersected with each row's visible keys."""
    lib = lib or _load()
    args, keep = _common_args(case)
    nthreads = nthreads or default_threads()
    T, Hq, D = case.q.shape[0], case.num_q_heads, case.head_size
    acc = np.empty((T * Hq, D), dtype=np.float64)
    m = np.empty((T * Hq,), dtype=np.float64)
    l = np.empty((T * Hq,), dtype=np.float64)
    rc = lib.pdo_partial(*args, int(key_lo), int(key_hi), acc.ctypes.data, m.ctypes.data,
                         l.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle failed: {rc}")
    del keep
    return acc.reshape(T, Hq, D), m.reshape(T, Hq), l.reshape(T, Hq)


def merge(parts):
    """Combine unnormalised partials [(acc, m, l), ...] into outputs."""
    ms = np.stack([p[1] for p in parts])
    m_star = ms.max(axis=0)
    safe = np.where(np.isfinite(m_star), m_star, 0.0)
    total_l = np.zeros_like(m_star)
    total_acc = np.zeros_like(parts[0][0])
    for acc, m, l in parts:
        w = np.where(l > 0, np.exp(np.where(np.isfinite(m), m, 0.0) - safe), 0.0)
        total_l += l * w
        total_acc += acc * w[..., None]
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(total_l[..., None] > 0, total_acc / np.where(total_l > 0, total_l, 1.0)[..., None], 0.0)
    return out


def widen(word: int, is_bf16: bool) -> float:
    return _load().pdo_widen(word & 0xFFFF, int(is_bf16))
