"""Seeded synthetic inputs for paged decode attention.

This module only builds inputs: query rows, a paged K/V pool, a block table
and per-sequence lengths.  It holds none of the attention arithmetic, so the
CUDA path and the CPU oracle can both read the same tensors without sharing
any of the method.

Shapes follow the decode-attention API of the ROCm RDNA3.5 decode kernels
(vllm.v1.attention.ops.rocm_rdna_hip, ``KernelVariant`` fields and
``expected_kv_cache_strides``) and the decode metadata of the Octave backend
(vllm.v1.attention.backends.rocm_octave_attn, ``forward``):

* ``q`` / ``out``: ``[S*M, Hq, D]``; tokens of sequence ``s`` are rows
  ``s*M .. s*M+M-1`` (uniform decode, M query tokens per sequence).
* K/V pool, layout NHD: ``[NB, P, Hkv, D]``; layout HND: ``[NB, Hkv, P, D]``.
  ``packed=True`` stores K and V side by side in one row of ``2*D``
  (the packed-cache stride order of ``expected_kv_cache_strides``), so
  ``v_cache`` is the view ``k_cache + D`` with the same strides.
* ``block_table``: int32 ``[S, W]``, logical page -> physical page.
* ``seq_lens``: int32 ``[S]``, keys of each sequence *including* its M new
  query tokens.

Every value is drawn in fp32 from a ``torch.Generator`` seeded per stream
(q, k, v, page permutation, lengths) and rounded once (round to nearest even)
to fp16 or bf16.  Pool slots that hold no key of any sequence (the tail of a
partial last page, pages a sliding window never reaches, slack pages) are
filled with NaN so that any read of them shows up in the output.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

NHD = 0
HND = 1

_STREAM_Q, _STREAM_K, _STREAM_V, _STREAM_PERM, _STREAM_LEN = range(5)


def _gen(seed: int, stream: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + stream * 7919 + 17)
    return g


@dataclasses.dataclass
class DecodeCase:
    """One decode call's inputs (all tensors on ``device``)."""

    name: str
    dtype: torch.dtype
    head_size: int
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    max_query_len: int
    window: int
    scale: float
    layout: int
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    packed: bool = False
    # host copy of seq_lens (the inputs are made on the host; kept for sizing)
    seq_lens_host: Optional[list] = None
    # variable query lengths: [S + 1] int32, request s owns q rows
    # query_start[s] .. query_start[s+1] - 1 (None: uniform, s*M .. s*M+M-1)
    query_start: Optional[torch.Tensor] = None
    query_start_host: Optional[list] = None

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    def to(self, device) -> "DecodeCase":
        """Copy every tensor to ``device``; a packed pool stays one allocation."""
        if self.packed:
            pool = self.k_cache.as_strided(
                self._pool_shape(), self._pool_strides(), self.k_cache.storage_offset()
            )
            pool_d = pool.to(device)
            k = pool_d[..., : self.head_size]
            v = pool_d[..., self.head_size :]
        else:
            k = self.k_cache.to(device)
            v = self.v_cache.to(device)
        return dataclasses.replace(
            self,
            q=self.q.to(device),
            k_cache=k,
            v_cache=v,
            block_table=self.block_table.to(device),
            seq_lens=self.seq_lens.to(device),
            query_start=None if self.query_start is None else self.query_start.to(device),
        )

    def _pool_shape(self):
        s = list(self.k_cache.shape)
        s[-1] = 2 * self.head_size
        return tuple(s)

    def _pool_strides(self):
        return tuple(self.k_cache.stride())

    def kv_bytes_touched(self) -> int:
        """Bytes of K and V that the M rows of every sequence can see (union
        over rows): the algorithmic K+V read of one call."""
        e = self.q.element_size()
        total = 0
        lens = self.seq_lens_host or self.seq_lens.tolist()
        for s, L in enumerate(lens):
            L = max(int(L), 0)
            m = self.query_len(s)
            if m == 0:
                continue
            u = min(L, self.window + m - 1) if self.window else L
            total += u * self.num_kv_heads * 2 * self.head_size * e
        return total

    def query_len(self, s: int) -> int:
        """Query tokens of sequence s."""
        if self.query_start_host is None:
            return self.max_query_len
        return self.query_start_host[s + 1] - self.query_start_host[s]

    def pages_touched(self) -> int:
        lens = self.seq_lens_host or self.seq_lens.tolist()
        n = 0
        for L in lens:
            L = max(int(L), 0)
            lo = max(0, L - self.max_query_len + 1 - self.window) if self.window else 0
            if L > lo:
                n += (L - 1) // self.page_size - lo // self.page_size + 1
        return n

    def algorithmic_bytes(self) -> int:
        """K+V read, Q read and O write, block-table entries and seq_lens."""
        e = self.q.element_size()
        qo = 2 * self.q.shape[0] * self.num_q_heads * self.head_size * e
        return self.kv_bytes_touched() + qo + 4 * self.pages_touched() + 4 * self.num_seqs


def _rounded_normal(shape, std, mean, dtype, gen, device="cpu"):
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(dtype)


def make_case(
    name: str,
    *,
    seed: int,
    dtype: torch.dtype,
    head_size: int,
    num_q_heads: int,
    num_kv_heads: int,
    page_size: int,
    max_query_len: int,
    seq_lens: Sequence[int],
    layout: int = HND,
    window: int = 0,
    std: float = 1.0,
    v_mean: float = 0.0,
    scale: Optional[float] = None,
    pool_pages: Optional[int] = None,
    table_width: Optional[int] = None,
    window_pages_only: bool = False,
    packed: bool = False,
    poison: bool = True,
    device: str = "cpu",
    gen_device: str = "cpu",
) -> DecodeCase:
    """Build one call's inputs.

    ``pool_pages``: physical pages in the pool (default: exactly the pages
    used, plus one poison page when ``window_pages_only``).  Logical pages are
    mapped to a random permutation of the pool.  ``window_pages_only`` keeps
    only the pages a sliding window reaches in the block table; entries
    before the window's first page point at a NaN page, as in a block table
    that holds only the blocks the window reaches.  ``gen_device="cuda"``
    draws q, K and V with a seeded CUDA generator (fast for large pools;
    other values than the CPU streams of the same seed).
    """
    D, P = head_size, page_size
    S, M = len(seq_lens), max_query_len
    lens = [max(int(x), 0) for x in seq_lens]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    pages_needed = [(L + P - 1) // P for L in lens]
    W = table_width if table_width is not None else max(1, max(pages_needed))
    assert W >= max(pages_needed)
    first_page = []
    for L in lens:
        if window_pages_only and window and L > 0:
            lo = max(0, L - M + 1 - window)
            first_page.append(lo // P)
        else:
            first_page.append(0)
    used = [pn - fp for pn, fp in zip(pages_needed, first_page)]
    n_used = sum(used)
    extra_poison = 1 if window_pages_only else 0
    NB = pool_pages if pool_pages is not None else n_used + extra_poison
    assert NB >= n_used + extra_poison, (NB, n_used)

    g_perm = _gen(seed, _STREAM_PERM)
    perm = torch.randperm(NB, generator=g_perm)
    poison_page = int(perm[-1]) if extra_poison else None
    block_table = torch.zeros((S, W), dtype=torch.int32)
    cursor = 0
    for s in range(S):
        for j in range(W):
            if first_page[s] <= j < pages_needed[s]:
                block_table[s, j] = int(perm[cursor])
                cursor += 1
            elif j < first_page[s]:
                block_table[s, j] = poison_page
            else:
                # past the sequence end: a valid page index that is never read
                block_table[s, j] = int(perm[0]) if n_used else 0

    shape_pool = (NB, P, num_kv_heads, D) if layout == NHD else (NB, num_kv_heads, P, D)
    if packed:
        full = list(shape_pool)
        full[-1] = 2 * D
        pool = torch.full(full, float("nan") if poison else 0.0, dtype=dtype, device=device)
        k_cache, v_cache = pool[..., :D], pool[..., D:]
    else:
        fill = float("nan") if poison else 0.0
        k_cache = torch.full(shape_pool, fill, dtype=dtype, device=device)
        v_cache = torch.full(shape_pool, fill, dtype=dtype, device=device)

    g_q, g_k, g_v = (_gen(seed, st, gen_device) for st in (_STREAM_Q, _STREAM_K, _STREAM_V))
    q = _rounded_normal((S * M, num_q_heads, D), std, 0.0, dtype, g_q, gen_device)
    for s in range(S):
        L = lens[s]
        lo_pos = first_page[s] * P
        n = L - lo_pos
        if n <= 0:
            continue
        kvals = _rounded_normal((n, num_kv_heads, D), std, 0.0, dtype, g_k, gen_device)
        vvals = _rounded_normal((n, num_kv_heads, D), std, v_mean, dtype, g_v, gen_device)
        pos = torch.arange(lo_pos, L)
        phys = block_table[s, (pos // P)].long().to(device)
        tok = (pos % P).long().to(device)
        if layout == NHD:
            k_cache[phys, tok] = kvals.to(device)
            v_cache[phys, tok] = vvals.to(device)
        else:
            k_cache.permute(0, 2, 1, 3)[phys, tok] = kvals.to(device)
            v_cache.permute(0, 2, 1, 3)[phys, tok] = vvals.to(device)
    if window_pages_only and window and not poison:
        raise ValueError("window_pages_only needs poison=True")
    return DecodeCase(
        name=name,
        dtype=dtype,
        head_size=D,
        num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads,
        page_size=P,
        max_query_len=M,
        window=window,
        scale=float(scale),
        layout=layout,
        q=q.to(device),
        k_cache=k_cache,
        v_cache=v_cache,
        block_table=block_table.to(device),
        seq_lens=torch.tensor(lens, dtype=torch.int32, device=device),
        packed=packed,
        seq_lens_host=list(lens),
    )


def make_varlen_case(name: str, *, seed: int, q_lens: Sequence[int], pad_tokens: int = 0,
                     **kw) -> DecodeCase:
    """A batch with a query length per request (zero allowed; the decode
    call takes up to 8, a prefill call any) and ``pad_tokens`` rows past the
    last request, as in a captured batch padded to a fixed token count.  The
    pool and block table are those of ``make_case`` with ``max_query_len =
    max(q_lens)`` (at least 1); q holds sum(q_lens) + pad_tokens rows,
    request s at query_start[s]."""
    q_lens = [int(m) for m in q_lens]
    assert all(0 <= m for m in q_lens) and len(q_lens) == len(kw["seq_lens"])
    M = max(1, max(q_lens) if q_lens else 1)
    if kw.get("max_query_len") is None:
        kw["max_query_len"] = M
    assert kw["max_query_len"] >= M
    case = make_case(name, seed=seed, **kw)
    qsl = [0]
    for m in q_lens:
        qsl.append(qsl[-1] + m)
    T = qsl[-1] + int(pad_tokens)
    g_q = _gen(seed, _STREAM_Q, kw.get("gen_device", "cpu"))
    q = _rounded_normal((T, case.num_q_heads, case.head_size), kw.get("std", 1.0), 0.0,
                        case.dtype, g_q, kw.get("gen_device", "cpu"))
    dev = case.q.device
    return dataclasses.replace(case, q=q.to(dev),
                               query_start=torch.tensor(qsl, dtype=torch.int32, device=dev),
                               query_start_host=qsl)


# ---------------------------------------------------------------------------
# The five workloads.  Sizes follow the decode configurations the kernel is
# specified on; the pages' own harness (vLLM's attention_benchmarks, HND,
# batch 1) is not available, so these seeded shapes stand in for it.
# ---------------------------------------------------------------------------

def single_seq_nhd(seed: int = 0, device: str = "cpu") -> DecodeCase:
    """fp16, D=128, 8 q / 2 kv heads, M=1, one sequence of 300 keys (the last
    of 19 pages holds 12 keys), P=16, NHD, 19 random pages of a 64-page pool."""
    return make_case(
        "single_seq_nhd_fp16_d128_L300",
        seed=seed, dtype=torch.float16, head_size=128, num_q_heads=8,
        num_kv_heads=2, page_size=16, max_query_len=1, seq_lens=[300],
        layout=NHD, pool_pages=64, device=device,
    )


def spec_decode_hnd(M: int, L: int, seed: int = 0, device: str = "cpu",
                    gen_device: str = "cpu", v_mean: float = 0.0,
                    packed: bool = False) -> DecodeCase:
    """bf16, D=128, 32 q / 8 kv heads, P=16, HND, batch 1, M in 1..4.
    ``v_mean`` shifts the V values (outputs stay O(1) at long contexts);
    ``packed`` stores K and V side by side in one pool."""
    return make_case(
        f"spec_decode_hnd_bf16_d128_M{M}_L{L}" + (f"_vmean{v_mean:g}" if v_mean else "")
        + ("_packed" if packed else ""),
        seed=seed, dtype=torch.bfloat16, head_size=128, num_q_heads=32,
        num_kv_heads=8, page_size=16, max_query_len=M, seq_lens=[L],
        layout=HND, v_mean=v_mean, packed=packed, device=device, gen_device=gen_device,
    )


def sliding_window(dtype: torch.dtype, M: int, L: int, seed: int = 0,
                   device: str = "cpu", gen_device: str = "cpu",
                   v_mean: float = 0.0) -> DecodeCase:
    """D=256, 8 q / 1 kv head, window 512, P=32; the block table holds only
    the pages the window reaches (earlier entries point at a NaN page)."""
    tag = "fp16" if dtype == torch.float16 else "bf16"
    return make_case(
        f"sliding_window_{tag}_d256_w512_M{M}_L{L}" + (f"_vmean{v_mean:g}" if v_mean else ""),
        seed=seed, dtype=dtype, head_size=256, num_q_heads=8, num_kv_heads=1,
        page_size=32, max_query_len=M, seq_lens=[L], layout=HND, window=512,
        window_pages_only=True, v_mean=v_mean, device=device, gen_device=gen_device,
    )


def wide_head(M: int, L: int, seed: int = 0, device: str = "cpu",
              gen_device: str = "cpu", v_mean: float = 0.0,
              packed: bool = False) -> DecodeCase:
    """fp16, D=512, 8 q / 1 kv head, full causal, P=16, values N(0, 0.5)."""
    return make_case(
        f"wide_head_fp16_d512_M{M}_L{L}" + (f"_vmean{v_mean:g}" if v_mean else "")
        + ("_packed" if packed else ""),
        seed=seed, dtype=torch.float16, head_size=512, num_q_heads=8,
        num_kv_heads=1, page_size=16, max_query_len=M, seq_lens=[L],
        layout=HND, std=0.5, v_mean=v_mean, packed=packed, device=device,
        gen_device=gen_device,
    )


def batched_hybrid_pages(seed: int = 0, num_seqs: int = 64, max_len: int = 16384,
                         device: str = "cpu", gen_device: str = "cpu", v_mean: float = 0.0,
                         page_size: int = 1056) -> DecodeCase:
    """bf16, D=256, 16 q / 2 kv heads, P=1056, M=4, 64 sequences with lengths
    uniform in [1, max_len] and one empty (padded) slot; a shared pool with
    10 % slack pages, randomly permuted."""
    g = _gen(seed, _STREAM_LEN)
    lens = torch.randint(1, max_len + 1, (num_seqs,), generator=g).tolist()
    lens[num_seqs // 3] = 0
    P = page_size
    used = sum((L + P - 1) // P for L in lens)
    return make_case(
        f"batched_hybrid_bf16_d256_P{P}_S{num_seqs}" + (f"_vmean{v_mean:g}" if v_mean else ""),
        seed=seed, dtype=torch.bfloat16, head_size=256, num_q_heads=16,
        num_kv_heads=2, page_size=P, max_query_len=4, seq_lens=lens,
        layout=HND, pool_pages=used + max(1, used // 10), v_mean=v_mean,
        table_width=(max_len + P - 1) // P, device=device, gen_device=gen_device,
    )


def hybrid_page(P: int, M: int, L: int, seed: int = 0, device: str = "cpu",
                gen_device: str = "cpu", v_mean: float = 0.0, packed: bool = False,
                layout: int = HND) -> DecodeCase:
    """One sequence on the page sizes of hybrid attention / state-space
    models (528, 544, 784, 1056 tokens): bf16, D=256, 16 q / 2 kv heads."""
    return make_case(
        f"hybrid_page_bf16_d256_P{P}_M{M}_L{L}" + (f"_vmean{v_mean:g}" if v_mean else "")
        + ("_packed" if packed else ""),
        seed=seed, dtype=torch.bfloat16, head_size=256, num_q_heads=16, num_kv_heads=2,
        page_size=P, max_query_len=M, seq_lens=[L], layout=layout, v_mean=v_mean,
        packed=packed, device=device, gen_device=gen_device,
    )


SPEC_DECODE_CONTEXTS = (128, 1024, 4096, 16384, 32768)
SPEC_DECODE_M = (1, 2, 3, 4)


def varlen_spec_decode_batch(seed: int = 0, num_seqs: int = 32, min_len: int = 1024,
                             max_len: int = 16384, max_draft: int = 4, pad_tokens: int = 0,
                             uniform: bool = False, device: str = "cpu",
                             gen_device: str = "cpu", v_mean: float = 0.0) -> DecodeCase:
    """Speculative decoding over a batch: bf16, D=128, 32 q / 8 kv heads,
    P=16, HND; request s has 1..max_draft query tokens (seeded) and a context
    uniform in [min_len, max_len].  ``uniform=True`` gives the same requests
    padded to max_draft query rows each (the uniform call's layout)."""
    g = torch.Generator().manual_seed(seed * 7919 + 3)
    q_lens = torch.randint(1, max_draft + 1, (num_seqs,), generator=g).tolist()
    lens = torch.randint(min_len, max_len + 1, (num_seqs,), generator=g).tolist()
    kw = dict(seed=seed, dtype=torch.bfloat16, head_size=128, num_q_heads=32, num_kv_heads=8,
              page_size=16, seq_lens=lens, layout=HND, v_mean=v_mean, device=device,
              gen_device=gen_device)
    if uniform:
        return make_case("varlen_batch_padded", max_query_len=max_draft, **kw)
    return make_varlen_case("varlen_batch", q_lens=q_lens, pad_tokens=pad_tokens,
                            max_query_len=max_draft, **kw)


# ---------------------------------------------------------------------------
# Inputs of the rotary embedding + paged KV-cache write that runs ahead of
# decode: new tokens' q, k, v, their positions and cache slots, a cos / sin
# table, and the pools to write into.
# ---------------------------------------------------------------------------

def rope_cos_sin_table(max_pos: int, rot_dim: int, base: float = 10000.0) -> torch.Tensor:
    """fp32 [max_pos, rot_dim]: cos of position x frequency i in the first
    rot_dim/2 columns, sin in the rest, frequency i = base^(-2i/rot_dim)
    (the table a model's rotary embedding precomputes; computed in fp64 and
    rounded once)."""
    i = torch.arange(rot_dim // 2, dtype=torch.float64)
    inv_freq = base ** (-2.0 * i / rot_dim)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv_freq[None, :]
    return torch.cat([ang.cos(), ang.sin()], dim=1).to(torch.float32).contiguous()


@dataclasses.dataclass
class RopeCase:
    """One call's inputs of the rotary embedding + cache write."""

    name: str
    dtype: torch.dtype
    head_size: int
    rot_dim: int
    is_neox: bool
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    layout: int
    q: torch.Tensor            # [T, Hq, D]
    k: torch.Tensor            # [T, Hkv, D]
    v: torch.Tensor            # [T, Hkv, D]
    positions: torch.Tensor    # [T] int32
    slot_mapping: torch.Tensor  # [T] int32, -1 = padding token
    cos_sin: torch.Tensor      # [max_pos, rot_dim] fp32
    k_cache: torch.Tensor      # pool before the call
    v_cache: torch.Tensor
    packed: bool = False

    def to(self, device) -> "RopeCase":
        if self.packed:
            pool = self.k_cache.as_strided(
                tuple(list(self.k_cache.shape[:-1]) + [2 * self.head_size]),
                self.k_cache.stride(), self.k_cache.storage_offset()).to(device)
            k_cache, v_cache = pool[..., :self.head_size], pool[..., self.head_size:]
        else:
            k_cache, v_cache = self.k_cache.to(device), self.v_cache.to(device)
        return dataclasses.replace(
            self, q=self.q.to(device), k=self.k.to(device), v=self.v.to(device),
            positions=self.positions.to(device), slot_mapping=self.slot_mapping.to(device),
            cos_sin=self.cos_sin.to(device), k_cache=k_cache, v_cache=v_cache)

    def bytes_moved(self) -> int:
        """q read + q_out written + k, v read + k, v written for every token
        with a slot, + one table row per token (fp32)."""
        e = self.q.element_size()
        T = self.q.shape[0]
        live = int((self.slot_mapping >= 0).sum())
        D = self.head_size
        return (2 * T * self.num_q_heads * D * e + 2 * T * self.num_kv_heads * D * e
                + 2 * live * self.num_kv_heads * D * e + T * self.rot_dim * 4)


def make_rope_case(name: str, *, seed: int, dtype: torch.dtype, num_tokens: int,
                   num_q_heads: int, num_kv_heads: int, head_size: int, rot_dim: int,
                   page_size: int, num_pages: int, layout: int = HND, is_neox: bool = True,
                   max_pos: int = 4096, pad_tokens: int = 0, packed: bool = False,
                   device: str = "cpu", gen_device: str = "cpu") -> RopeCase:
    """T = num_tokens new tokens at random distinct positions and random
    distinct cache slots; the last ``pad_tokens`` of them are padding (slot
    -1).  The pools hold seeded values before the call, so an untouched slot
    can be checked bit for bit."""
    D, P = head_size, page_size
    T = num_tokens
    assert num_pages * P >= T and max_pos >= 1
    g = _gen(seed, _STREAM_PERM)
    slots = torch.randperm(num_pages * P, generator=g)[:T].to(torch.int32)
    if pad_tokens:
        slots[T - pad_tokens:] = -1
    positions = torch.randint(0, max_pos, (T,), generator=_gen(seed, _STREAM_LEN),
                              dtype=torch.int64).to(torch.int32)
    if T:
        positions[0] = 0                       # position 0 (no rotation) is always in
        positions[-1] = max_pos - 1            # and the table's last row
    g_q, g_k, g_v = (_gen(seed, st, gen_device) for st in (_STREAM_Q, _STREAM_K, _STREAM_V))
    q = _rounded_normal((T, num_q_heads, D), 1.0, 0.0, dtype, g_q, gen_device)
    k = _rounded_normal((T, num_kv_heads, D), 1.0, 0.0, dtype, g_k, gen_device)
    v = _rounded_normal((T, num_kv_heads, D), 1.0, 0.0, dtype, g_v, gen_device)
    shape_pool = (num_pages, P, num_kv_heads, D) if layout == NHD else (num_pages, num_kv_heads, P, D)
    g_pool = _gen(seed + 1, _STREAM_K, gen_device)
    if packed:
        full = list(shape_pool)
        full[-1] = 2 * D
        pool = _rounded_normal(tuple(full), 1.0, 0.0, dtype, g_pool, gen_device)
        k_cache, v_cache = pool[..., :D], pool[..., D:]
    else:
        k_cache = _rounded_normal(shape_pool, 1.0, 0.0, dtype, g_pool, gen_device)
        v_cache = _rounded_normal(shape_pool, 1.0, 0.0, dtype, g_pool, gen_device)
    case = RopeCase(name=name, dtype=dtype, head_size=D, rot_dim=rot_dim, is_neox=is_neox,
                    num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, page_size=P,
                    layout=layout, q=q, k=k, v=v, positions=positions, slot_mapping=slots,
                    cos_sin=rope_cos_sin_table(max_pos, rot_dim), k_cache=k_cache,
                    v_cache=v_cache, packed=packed)
    return case.to(device)


def make_prefill_case(name: str, *, seed: int, q_lens: Sequence[int], contexts: Sequence[int],
                      dtype: torch.dtype = torch.bfloat16, head_size: int = 128,
                      num_q_heads: int = 32, num_kv_heads: int = 8, page_size: int = 16,
                      layout: int = HND, window: int = 0, pad_tokens: int = 0,
                      v_mean: float = 0.0, std: float = 1.0, device: str = "cpu",
                      gen_device: str = "cpu") -> DecodeCase:
    """A prefill batch: request s has q_lens[s] new tokens after contexts[s]
    cached ones (seq_lens = context + q_len, the new tokens' keys included),
    rows as in ``make_varlen_case``; q, K and V drawn with standard
    deviation ``std``."""
    lens = [int(c) + int(m) for c, m in zip(contexts, q_lens)]
    return make_varlen_case(name, seed=seed, q_lens=q_lens, pad_tokens=pad_tokens, dtype=dtype,
                            head_size=head_size, num_q_heads=num_q_heads,
                            num_kv_heads=num_kv_heads, page_size=page_size, seq_lens=lens,
                            layout=layout, window=window, v_mean=v_mean, std=std,
                            device=device, gen_device=gen_device)


def prefill_flops(case) -> int:
    """Multiply-adds x 2 of QK^T and PV over the keys each query row sees."""
    qs, lens = case.query_start_host, case.seq_lens_host
    total = 0
    for s in range(case.num_seqs):
        q_len = qs[s + 1] - qs[s]
        ctx = max(lens[s], q_len) - q_len
        for i in range(q_len):
            n = ctx + i + 1
            lo = max(0, n - case.window) if case.window else 0
            total += n - lo
    return 4 * case.head_size * case.num_q_heads * total
