"""GB300 (sm_103a) paged split-KV decode attention.

Thin Python binding of ``libpaged_decode.so`` (C ABI in
``include/paged_decode.h``).  This module only marshals torch tensors into
the ABI's descriptors: every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing the calls
raise, and ``build()`` compiles it with nvcc.

Names follow the C ABI:

* ``paged_decode_attn(q, k_cache, v_cache, block_table, seq_lens, out,
  num_q_heads, num_kv_heads, head_size, page_size, max_query_len, window,
  scale, layout, scratch, stream)``
* ``paged_decode_scratch_bytes(...)`` / ``Scratch`` (``paged_decode_scratch_init``)
* ``paged_decode_plan(...)``, ``paged_decode_device_status(...)``
* ``paged_rope_cache_write(...)``: rotary embedding of the new tokens' q
  and k and the store of k and v into the paged cache, ahead of decode
* ``paged_prefill_plan(...)`` / ``paged_prefill_attn(...)``: attention for
  requests of any query length over a host-made work list
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

from . import _build

NHD = 0
HND = 1
PATH_AUTO, PATH_MMA, PATH_DOT = 0, 1, 2

PD_OK = 0
STATUS_NAMES = {
    0: "PD_OK", -1: "PD_EINVAL", -2: "PD_EDTYPE", -3: "PD_EHEAD", -4: "PD_EQLEN",
    -5: "PD_EALIGN", -6: "PD_ESCRATCH", -7: "PD_ECUDA", -8: "PD_ENODEV",
}
DEV_WAIT_TIMEOUT, DEV_BAD_PAGE, DEV_BAD_SEQLEN, DEV_BAD_QSTART = 0x1, 0x2, 0x4, 0x8
DEV_BAD_SCRATCH, DEV_BAD_POSITION, DEV_BAD_SLOT, DEV_BAD_WORK = 0x10, 0x20, 0x40, 0x80
COUNTERS_PER_PAIR = 16  # PD_COUNTERS_PER_PAIR

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "paged_decode.h")


class PagedDecodeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({_strerror(code)})")


class PdTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class PdScratch(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("bytes", ctypes.c_size_t),
                ("counter_slots", ctypes.c_int64)]


class PdOptions(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("segments", "row_groups", "key_groups", "stages", "cluster", "path",
                 "max_ctas_hint", "merge", "wait_limit_us", "early_reads", "mergers")]


class PdPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("path", "merge", "mergers", "rows", "row_groups", "rows_per_cta", "n_tiles", "key_groups", "stages",
                 "seg_blocks", "max_segments", "cluster", "max_parts", "grid_x", "grid_y",
                 "block_threads", "smem_bytes")] + [("scratch_needed", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class PdPrefillItem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("seq", "tile", "seg", "nseg", "split", "slot", "blocks", "reserved")]


class PdPrefillPlanInfo(ctypes.Structure):
    _fields_ = [("num_items", ctypes.c_int64), ("num_split_tiles", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("tile_rows", ctypes.c_int32),
                ("max_segments", ctypes.c_int32), ("target_ctas", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("total_blocks", ctypes.c_int64),
                ("load_blocks", ctypes.c_double)]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_ if n != "reserved"}


_lib = None


def library_path() -> str:
    return _build.LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libpaged_decode.so in-tree for sm_103a."""
    global _lib
    path = _build.build(force=force, verbose=verbose)
    return path


def lib():
    """The loaded C library; raises if it was never built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with paged_split_kv_02_gb300.build() "
                "(there is no fallback implementation)")
        L = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        T = ctypes.POINTER(PdTensor)
        L.paged_decode_scratch_bytes.argtypes = [i32] * 6
        L.paged_decode_scratch_bytes.restype = sz
        L.paged_decode_scratch_init.argtypes = [ctypes.POINTER(PdScratch), vp, sz, i32, i32, vp]
        L.paged_decode_scratch_init.restype = i32
        attn_args = [T, T, T, T, T, T, i32, i32, i32, i32, i32, i32, f32, i32,
                     ctypes.POINTER(PdScratch), vp]
        L.paged_decode_attn.argtypes = attn_args
        L.paged_decode_attn.restype = i32
        L.paged_decode_attn_opts.argtypes = attn_args + [ctypes.POINTER(PdOptions)]
        L.paged_decode_attn_opts.restype = i32
        L.paged_decode_attn_varlen.argtypes = [T] * 7 + attn_args[6:] + [ctypes.POINTER(PdOptions)]
        L.paged_decode_attn_varlen.restype = i32
        L.paged_decode_attn_static.argtypes = attn_args[:14] + [vp]
        L.paged_decode_attn_static.restype = i32
        L.paged_decode_plan.argtypes = [i32] * 9 + [ctypes.POINTER(PdScratch),
                                                    ctypes.POINTER(PdOptions),
                                                    ctypes.POINTER(PdPlan)]
        L.paged_decode_plan.restype = i32
        L.paged_decode_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i32, vp]
        L.paged_decode_device_status.restype = i32
        L.paged_decode_strerror.argtypes = [i32]
        L.paged_decode_strerror.restype = ctypes.c_char_p
        L.paged_decode_version.argtypes = []
        L.paged_decode_version.restype = i32
        L.paged_rope_cache_write.argtypes = [T] * 9 + [i32] * 7 + [vp]
        L.paged_rope_cache_write.restype = i32
        L.paged_prefill_plan.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp, i64,
                                         ctypes.POINTER(PdPrefillPlanInfo)]
        L.paged_prefill_plan.restype = i32
        L.paged_prefill_scratch_bytes.argtypes = [i32, i32, i32]
        L.paged_prefill_scratch_bytes.restype = sz
        L.paged_prefill_attn.argtypes = [T] * 7 + [ctypes.POINTER(PdPrefillPlanInfo), T] + \
            [i32] * 5 + [f32, i32, ctypes.POINTER(PdScratch), vp]
        L.paged_prefill_attn.restype = i32
        _lib = L
    return _lib


def declared_symbols() -> list:
    """Function names the public header declares."""
    text = open(HEADER).read()
    return re.findall(r"PD_API\s+[\w\s\*]*?\b(paged_\w+)\s*\(", text)


def _strerror(code: int) -> str:
    try:
        return lib().paged_decode_strerror(int(code)).decode()
    except Exception:  # pragma: no cover
        return "?"


_DTYPES = {torch.float16: 0, torch.bfloat16: 1, torch.int32: 2, torch.float32: 3}


def tensor_desc(t: torch.Tensor) -> PdTensor:
    """Descriptor of a tensor: pointer, dtype code, shape and element strides."""
    d = PdTensor()
    d.data = t.data_ptr()
    d.dtype = _DTYPES.get(t.dtype, 99)  # 99: a type the library does not take
    d.ndim = t.dim()
    for i in range(min(t.dim(), 4)):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def options(**kw) -> PdOptions:
    o = PdOptions()
    for k, v in kw.items():
        setattr(o, k, int(v))
    return o


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        if not torch.cuda.is_available():
            return None  # the call itself reports the missing device
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def paged_decode_scratch_bytes(max_num_seqs, num_q_heads, num_kv_heads, head_size,
                               max_query_len, max_splits=256) -> int:
    return int(lib().paged_decode_scratch_bytes(max_num_seqs, num_q_heads, num_kv_heads,
                                                head_size, max_query_len, max_splits))


class Scratch:
    """Caller-owned split-KV scratch in device memory (torch allocation)
    prepared by ``paged_decode_scratch_init``; create it outside graph
    capture and reuse it for every call of one stream."""

    def __init__(self, max_num_seqs, num_q_heads, num_kv_heads, head_size, max_query_len,
                 max_splits=256, device=None, stream=None, nbytes=None):
        if nbytes is None:
            nbytes = paged_decode_scratch_bytes(max_num_seqs, num_q_heads, num_kv_heads,
                                                head_size, max_query_len, max_splits)
            if nbytes == 0:
                raise PagedDecodeError(-1, "paged_decode_scratch_bytes")
        self.buffer = torch.empty(int(nbytes) + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buffer.data_ptr()) % 256
        self.view = self.buffer[off: off + int(nbytes)]
        self.desc = PdScratch()
        self._init_args = (int(max_num_seqs), int(num_kv_heads))
        self.reinit(stream)

    def reinit(self, stream=None):
        """``paged_decode_scratch_init`` again on the same buffer: zero the
        counters (needed after a call reported a wait timeout or a bad
        scratch)."""
        rc = lib().paged_decode_scratch_init(ctypes.byref(self.desc), self.view.data_ptr(),
                                             int(self.view.numel()), *self._init_args,
                                             _stream_handle(stream))
        if rc != PD_OK:
            raise PagedDecodeError(rc, "paged_decode_scratch_init")

    def counters(self) -> torch.Tensor:
        """The int32 counter area (every call leaves it zero)."""
        n = int(self.desc.counter_slots)
        return self.view[: 4 * n].view(torch.int32)


def paged_decode_attn(q, k_cache, v_cache, block_table, seq_lens, out, num_q_heads,
                      num_kv_heads, head_size, page_size, max_query_len, window, scale, layout,
                      scratch: Optional[Scratch] = None, stream=None,
                      opts: Optional[PdOptions] = None, check: bool = True) -> int:
    """Launch the decode kernel; raises PagedDecodeError on a non-zero status
    (returns the status when ``check`` is False)."""
    L = lib()
    descs = [tensor_desc(t) for t in (q, k_cache, v_cache, block_table, seq_lens, out)]
    sp = ctypes.byref(scratch.desc) if scratch is not None else None
    args = [ctypes.byref(d) for d in descs] + [
        int(num_q_heads), int(num_kv_heads), int(head_size), int(page_size), int(max_query_len),
        int(window), float(scale), int(layout), sp, _stream_handle(stream)]
    if opts is None:
        rc = L.paged_decode_attn(*args)
    else:
        rc = L.paged_decode_attn_opts(*args, ctypes.byref(opts))
    if check and rc != PD_OK:
        raise PagedDecodeError(rc, "paged_decode_attn")
    return rc


def paged_decode_attn_varlen(q, k_cache, v_cache, block_table, seq_lens, query_start, out,
                             num_q_heads, num_kv_heads, head_size, page_size, max_query_len,
                             window, scale, layout, scratch: Optional[Scratch] = None,
                             stream=None, opts: Optional[PdOptions] = None,
                             check: bool = True) -> int:
    """The decode call for a batch with a query length per request:
    ``query_start`` [S + 1] int32 gives each request's first row of q / out
    (see the C header); rows past the last request are written as zeros."""
    L = lib()
    descs = [tensor_desc(t) for t in (q, k_cache, v_cache, block_table, seq_lens, query_start,
                                      out)]
    sp = ctypes.byref(scratch.desc) if scratch is not None else None
    rc = L.paged_decode_attn_varlen(
        *[ctypes.byref(d) for d in descs], int(num_q_heads), int(num_kv_heads), int(head_size),
        int(page_size), int(max_query_len), int(window), float(scale), int(layout), sp,
        _stream_handle(stream), ctypes.byref(opts) if opts is not None else None)
    if check and rc != PD_OK:
        raise PagedDecodeError(rc, "paged_decode_attn_varlen")
    return rc


def paged_decode_attn_static(q, k_cache, v_cache, block_table, seq_lens, out, num_q_heads,
                             num_kv_heads, head_size, page_size, max_query_len, window, scale,
                             layout, stream=None, check: bool = True) -> int:
    """The decode call with the library's own fixed scratch array, for
    callers that cannot allocate device memory (see the C header).  Calls
    share that array, so do not overlap them on the GPU; make the first call
    on a device before any stream capture."""
    L = lib()
    descs = [tensor_desc(t) for t in (q, k_cache, v_cache, block_table, seq_lens, out)]
    rc = L.paged_decode_attn_static(*[ctypes.byref(d) for d in descs], int(num_q_heads),
                                    int(num_kv_heads), int(head_size), int(page_size),
                                    int(max_query_len), int(window), float(scale), int(layout),
                                    _stream_handle(stream))
    if check and rc != PD_OK:
        raise PagedDecodeError(rc, "paged_decode_attn_static")
    return rc


def paged_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_size, page_size, max_query_len,
                      window, block_table_width, num_sms, scratch: Optional[Scratch] = None,
                      opts: Optional[PdOptions] = None, scratch_desc: Optional[PdScratch] = None
                      ) -> dict:
    plan = PdPlan()
    sd = scratch.desc if scratch is not None else scratch_desc
    rc = lib().paged_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_size, page_size,
                                 max_query_len, window, block_table_width, num_sms,
                                 ctypes.byref(sd) if sd is not None else None,
                                 ctypes.byref(opts) if opts is not None else None,
                                 ctypes.byref(plan))
    if rc != PD_OK:
        raise PagedDecodeError(rc, "paged_decode_plan")
    return plan.as_dict()


def paged_rope_cache_write(q, k, v, positions, slot_mapping, cos_sin_cache, q_out, k_cache,
                           v_cache, num_q_heads, num_kv_heads, head_size, rot_dim, page_size,
                           layout, is_neox=True, stream=None, check: bool = True) -> int:
    """Rotary embedding of q and k and the store of k and v into the paged
    cache at ``slot_mapping`` (see the C header); ``q_out`` may be ``q``."""
    descs = [tensor_desc(t) for t in (q, k, v, positions, slot_mapping, cos_sin_cache, q_out,
                                      k_cache, v_cache)]
    rc = lib().paged_rope_cache_write(*[ctypes.byref(d) for d in descs], int(num_q_heads),
                                      int(num_kv_heads), int(head_size), int(rot_dim),
                                      int(page_size), int(layout), int(bool(is_neox)),
                                      _stream_handle(stream))
    if check and rc != PD_OK:
        raise PagedDecodeError(rc, "paged_rope_cache_write")
    return rc


def rope_case(case, q_out=None, stream=None):
    """Run the rotary embedding + cache write on a ``workloads.RopeCase``
    (tensors on the GPU); returns q_out (the caches are written in place)."""
    if q_out is None:
        q_out = torch.empty_like(case.q)
    paged_rope_cache_write(case.q, case.k, case.v, case.positions, case.slot_mapping,
                           case.cos_sin, q_out, case.k_cache, case.v_cache, case.num_q_heads,
                           case.num_kv_heads, case.head_size, case.rot_dim, case.page_size,
                           case.layout, case.is_neox, stream)
    return q_out


def paged_prefill_plan(query_start, seq_lens, num_q_heads, num_kv_heads, head_size, window,
                       num_sms=0):
    """The work list of a prefill launch for this head size, made on the host
    (see the C header): returns (items int32 [n, 8] as a CPU tensor,
    PdPrefillPlanInfo)."""
    qs = torch.as_tensor(query_start, dtype=torch.int32).contiguous()
    sl = torch.as_tensor(seq_lens, dtype=torch.int32).contiguous()
    S = int(sl.shape[0])
    if qs.shape[0] != S + 1:
        raise PagedDecodeError(-1, "paged_prefill_plan")
    info = PdPrefillPlanInfo()
    L = lib()
    rc = L.paged_prefill_plan(qs.data_ptr(), sl.data_ptr(), S, int(num_q_heads),
                              int(num_kv_heads), int(head_size), int(window), int(num_sms), None,
                              0, ctypes.byref(info))
    if rc != PD_OK:
        raise PagedDecodeError(rc, "paged_prefill_plan")
    items = torch.zeros((int(info.num_items), 8), dtype=torch.int32)
    rc = L.paged_prefill_plan(qs.data_ptr(), sl.data_ptr(), S, int(num_q_heads),
                              int(num_kv_heads), int(head_size), int(window), int(num_sms),
                              items.data_ptr() if items.numel() else None, int(info.num_items),
                              ctypes.byref(info))
    if rc != PD_OK:
        raise PagedDecodeError(rc, "paged_prefill_plan")
    return items, info


def paged_prefill_scratch_bytes(num_kv_heads, head_size, num_sms) -> int:
    return int(lib().paged_prefill_scratch_bytes(int(num_kv_heads), int(head_size), int(num_sms)))


def prefill_scratch(num_kv_heads, head_size, num_sms=None, device=None, stream=None) -> "Scratch":
    """A scratch buffer for every prefill plan made with ``num_sms``."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(device or 0).multi_processor_count
    nbytes = paged_prefill_scratch_bytes(num_kv_heads, head_size, num_sms)
    if nbytes == 0:
        raise PagedDecodeError(-1, "paged_prefill_scratch_bytes")
    return Scratch(num_sms, 1, 1, head_size, 1, nbytes=nbytes, device=device, stream=stream)


def paged_prefill_attn(q, k_cache, v_cache, block_table, seq_lens, query_start, work, info, out,
                       num_q_heads, num_kv_heads, head_size, page_size, window, scale, layout,
                       scratch: Optional["Scratch"] = None, stream=None, check: bool = True) -> int:
    """The prefill call over a work list (``work``: the plan's items on the
    device, ``info``: its PdPrefillPlanInfo)."""
    descs = [tensor_desc(t) for t in (q, k_cache, v_cache, block_table, seq_lens, query_start,
                                      work)]
    od = tensor_desc(out)
    sp = ctypes.byref(scratch.desc) if scratch is not None else None
    rc = lib().paged_prefill_attn(*[ctypes.byref(d) for d in descs], ctypes.byref(info),
                                  ctypes.byref(od), int(num_q_heads), int(num_kv_heads),
                                  int(head_size), int(page_size), int(window), float(scale),
                                  int(layout), sp, _stream_handle(stream))
    if check and rc != PD_OK:
        raise PagedDecodeError(rc, "paged_prefill_attn")
    return rc


def prefill_case(case, out=None, scratch=None, stream=None, num_sms=0, plan=None):
    """Plan (on the host, from the case's host lengths) and run a prefill
    call on a ``workloads.DecodeCase`` with ``query_start``; returns out."""
    if plan is None:
        plan = paged_prefill_plan(case.query_start_host, case.seq_lens_host, case.num_q_heads,
                                  case.num_kv_heads, case.head_size, case.window, num_sms)
    items, info = plan
    work = items.to(case.q.device)
    if out is None:
        out = torch.empty_like(case.q)
    paged_prefill_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens,
                       case.query_start, work, info, out, case.num_q_heads, case.num_kv_heads,
                       case.head_size, case.page_size, case.window, case.scale, case.layout,
                       scratch, stream)
    return out


def paged_decode_device_status(reset: bool = False, stream=None) -> int:
    v = ctypes.c_uint(0)
    rc = lib().paged_decode_device_status(ctypes.byref(v), int(bool(reset)), _stream_handle(stream))
    if rc != PD_OK:
        raise PagedDecodeError(rc, "paged_decode_device_status")
    return int(v.value)


def paged_decode_version() -> int:
    return int(lib().paged_decode_version())


def decode_case(case, out=None, scratch=None, stream=None, opts=None):
    """Run the kernel on a ``workloads.DecodeCase`` (tensors on the GPU)."""
    if out is None:
        out = torch.empty_like(case.q)
    if getattr(case, "query_start", None) is not None:
        paged_decode_attn_varlen(case.q, case.k_cache, case.v_cache, case.block_table,
                                 case.seq_lens, case.query_start, out, case.num_q_heads,
                                 case.num_kv_heads, case.head_size, case.page_size,
                                 case.max_query_len, case.window, case.scale, case.layout,
                                 scratch, stream, opts)
        return out
    paged_decode_attn(case.q, case.k_cache, case.v_cache, case.block_table, case.seq_lens, out,
                      case.num_q_heads, case.num_kv_heads, case.head_size, case.page_size,
                      case.max_query_len, case.window, case.scale, case.layout, scratch,
                      stream, opts)
    return out
