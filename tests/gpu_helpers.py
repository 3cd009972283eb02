"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and
compare with the fp64 oracle on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_split_kv_02_gb300 as pd

# max-abs error bounds on O(1)-scaled outputs, per input dtype
TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}


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


def check(case_cpu, gpu_out, rows=None, tol=None, ref=None):
    """Assert the GPU output matches the oracle within the dtype's bound;
    returns (max abs error, error relative to the oracle's RMS)."""
    if ref is None:
        ref = oracle.attention(case_cpu, rows=rows)
    err = max_err(gpu_out, ref, rows)
    tol = TOL[case_cpu.dtype] if tol is None else tol
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    assert np.all(np.isfinite(gpu_out.float().cpu().numpy())), "non-finite output"
    assert err <= tol, f"{case_cpu.name}: max abs err {err:.3g} > {tol:g} (oracle rms {rms:.3g})"
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
