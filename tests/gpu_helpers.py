"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and
compare with the fp64 oracle on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_split_kv_02_gb300 as pd

# max-abs error bounds on O(1)-scaled outputs, per input dtype
TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
# Bounds on each output row's max-abs error relative to that row's largest
# oracle value, which keep a check meaningful where the outputs themselves
# are small (long contexts of N(0,1) values average towards zero, where the
# max-abs bound alone is near the outputs' size).  Rounding the output to the
# input dtype costs at most half a unit in the last place, 2^-9 (bf16) /
# 2^-12 (fp16) of a value; rounding P to the input dtype before PV adds noise
# of that relative size divided by the square root of the keys that matter.
# The bound is four times the rounding: 2^-7 (bf16), 2^-10 (fp16).  A row
# whose oracle output is all zeros must come out all zeros.
REL_TOL = {torch.float16: 2.0 ** -10, torch.bfloat16: 2.0 ** -7}


def scratch_for(case, splits=256):
    return pd.Scratch(case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_size,
                      case.max_query_len, max_splits=splits)


def run(case_gpu, scratch=None, opts=None, out=None):
    out = pd.decode_case(case_gpu, out=out, scratch=scratch, opts=opts)
    torch.cuda.synchronize()
    return out


def max_err(gpu_out: torch.Tensor, ref: np.ndarray, rows=None):
    g = gpu_out.double().cpu().numpy()
    if rows is not None:
        g = np.stack([g[t, h] for t, h in rows])
    return float(np.max(np.abs(g - ref))) if ref.size else 0.0


def row_rel_err(gpu_out: torch.Tensor, ref: np.ndarray, rows=None):
    """Largest over output rows of (the row's max-abs error) / (the row's
    largest |oracle| value), and the number of all-zero oracle rows whose
    output is not all zeros."""
    g = gpu_out.double().cpu().numpy()
    if rows is not None:
        g = np.stack([g[t, h] for t, h in rows])
    D = ref.shape[-1]
    g, r = g.reshape(-1, D), ref.reshape(-1, D)
    err = np.max(np.abs(g - r), axis=1)
    scale = np.max(np.abs(r), axis=1)
    zero = scale == 0
    rel = np.where(zero, 0.0, err / np.where(zero, 1.0, scale))
    return (float(rel.max()) if rel.size else 0.0), int(np.count_nonzero(zero & (err > 0)))


def check(case_cpu, gpu_out, rows=None, tol=None, ref=None, rel_tol=None):
    """Assert the GPU output matches the oracle within the dtype's max-abs
    bound and, row by row, within the dtype's bound relative to the row's
    largest oracle value; returns (max abs error, error relative to the
    oracle's RMS)."""
    if ref is None:
        ref = oracle.attention(case_cpu, rows=rows)
    err = max_err(gpu_out, ref, rows)
    tol = TOL[case_cpu.dtype] if tol is None else tol
    rel_tol = REL_TOL[case_cpu.dtype] if rel_tol is None else rel_tol
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    assert np.all(np.isfinite(gpu_out.float().cpu().numpy())), "non-finite output"
    assert err <= tol, f"{case_cpu.name}: max abs err {err:.3g} > {tol:g} (oracle rms {rms:.3g})"
    rel, bad_zero = row_rel_err(gpu_out, ref, rows)
    assert bad_zero == 0, f"{case_cpu.name}: {bad_zero} rows should be all zeros"
    assert rel <= rel_tol, (
        f"{case_cpu.name}: a row's max-abs error is {rel:.3g} of its largest oracle value "
        f"(bound {rel_tol:g})")
    return err, (err / rms if rms > 0 else 0.0)


def sample_rows(case, n, seed=0):
    """n (token row, q head) pairs spread over the call, always including
    the first and last rows of every sequence (of every request, with
    variable query lengths) and the call's last row."""
    g = np.random.default_rng(seed)
    T, Hq = case.q.shape[0], case.num_q_heads
    n = min(n, T * Hq)  # a small call has fewer rows than asked for
    rows = {(0, 0), (T - 1, Hq - 1)}
    M = case.max_query_len
    qsl = getattr(case, "query_start_host", None)
    for s in range(case.num_seqs):
        first, last = (s * M, s * M + M - 1) if qsl is None else (qsl[s], qsl[s + 1] - 1)
        if last >= first:
            rows.add((last, int(g.integers(Hq))))
            rows.add((first, int(g.integers(Hq))))
    while len(rows) < n:
        rows.add((int(g.integers(T)), int(g.integers(Hq))))
    return sorted(rows)
