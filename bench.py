"""Benchmark of the paged decode-attention kernel on GB300.

Workload (the spec-decode sweep the headline metric is quoted on): bf16,
head size 128, 32 q / 8 kv heads, page size 16, HND cache, batch 1,
M in {1, 2, 3, 4} query tokens x contexts {128, 1k, 4k, 16k, 32k}.
One step = one decode call for each of those 20 cases.

Every input is seeded synthetic data made on the device.  Between two uses
of a replica at least the rest of the sweep (~850 MB, more than the 126 MB
L2) passes, so every call reads its K/V from HBM.  Per-case times come from
CUDA graphs that cycle through enough replicas of the case to exceed 2.2x
the L2 size.  Times are CUDA events on the launching stream around graph
replays; the clocks are sampled with nvidia-smi during the timed region.
Each call reads its block table, seq_lens and older pages while the
previous call finishes (early reads, programmatic dependent launch); the
same steps and cases are also timed with every call waiting first.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs the same workload on its own GPU (replicas
only: the path has no cross-GPU exchange); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KV-read GB/s and % of GB300 HBM peak; µs per decode attention call"
UNIT = "GB/s"
CONTEXTS = (128, 1024, 4096, 16384, 32768)
MS = (1, 2, 3, 4)
WORKLOAD = ("spec-decode sweep: bf16, head_size 128, 32 q / 8 kv heads, page_size 16, HND, "
            "batch 1, M in {1,2,3,4} x contexts {128, 1k, 4k, 16k, 32k}; one step = one call "
            "per case")


# DRAM bytes (read + write) over algorithmic bytes of the decode kernel, from
# one ncu capture of the spec-decode case M=4, 32768 keys.  It holds for the
# kernel sources the capture was taken on only: with any other sources
# `traffic` is null.
TRAFFIC_CAPTURE = {"sources": "fd94399eaeea17e1", "dram_over_algorithmic": 1.0229}
# the same for the variable-length batch (one capture of an 8-request batch)
VARLEN_TRAFFIC_CAPTURE = {"sources": "fd94399eaeea17e1", "dram_over_algorithmic": 1.0113}


def _kernel_sources_digest(csrc: str | None = None) -> str:
    """Digest of the CUDA sources with comments and blank lines removed, so
    that a comment edit keeps an ncu capture valid and a code edit does not."""
    import glob
    import hashlib
    import re

    h = hashlib.sha256()
    if csrc is None:
        csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "paged_split_kv_02_gb300",
                            "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                    glob.glob(os.path.join(csrc, "*.h"))):
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            text = fh.read()
        # drop /* */ and // comments outside string literals, then blank lines
        text = re.sub(r'"(?:\\.|[^"\\])*"|/\*.*?\*/|//[^\n]*',
                      lambda m: m.group(0) if m.group(0).startswith('"') else "", text, flags=re.S)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during a timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in self.samples if num(p[0]) is not None]
        mx = [num(p[1]) for p in self.samples if num(p[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for p in self.samples for n, v in zip(names, p[3:7]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


def build_sweep(device, l2_bytes, only=None, rep_factor=2.2, seed0=0):
    """Per case: replicas of the inputs, enough to exceed rep_factor x L2."""
    from paged_split_kv_02_gb300 import workloads as W

    cases = {}
    for M in MS:
        for L in CONTEXTS:
            if only and (M, L) not in only:
                continue
            probe = W.spec_decode_hnd(M, 16)
            kv = L * probe.num_kv_heads * 2 * probe.head_size * 2
            n_rep = max(2, math.ceil(rep_factor * l2_bytes / kv))
            reps = [W.spec_decode_hnd(M, L, seed=seed0 + 1000 * M + r, device=device,
                                      gen_device=device) for r in range(n_rep)]
            cases[(M, L)] = reps
    return cases


def run_ours(args, world, rank, local):
    import paged_split_kv_02_gb300 as pd

    pd.build()
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20))
    peak, peak_kind = _peaks()
    cases = build_sweep(device, l2, only=args.only)
    first = next(iter(cases.values()))[0]
    scratch = pd.Scratch(1, first.num_q_heads, first.num_kv_heads, first.head_size, max(MS),
                         max_splits=256, device=device)
    outs = {k: [torch.empty_like(r.q) for r in reps] for k, reps in cases.items()}
    stream = torch.cuda.Stream(device=device)
    keys = sorted(cases)

    # Every call of the sweep reads inputs written before the previous call
    # started, so it may read its block table, seq_lens and pages while that
    # call finishes (pd_options.early_reads); the same steps are also timed
    # with every call waiting for the previous one first.
    opts = pd.options(early_reads=1) if args.early_reads else None

    def n_reps(k):
        return len(cases[k])

    def call(k, r, st=None, o=opts):
        pd.decode_case(cases[k][r], out=outs[k][r], scratch=scratch, stream=st, opts=o)

    # warm the library (attributes, tensor maps) outside capture
    with torch.cuda.stream(stream):
        for k in keys:
            for r in range(len(cases[k])):
                call(k, r)
    torch.cuda.synchronize()

    # ---- step graphs: one call per case, replicas alternating ------------
    n_step_graphs = 2

    def step_graphs_for(o):
        gs = []
        for gi in range(n_step_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for k in keys:
                    call(k, gi % len(cases[k]), o=o)
            gs.append(g)
        torch.cuda.synchronize()
        return gs

    step_graphs = step_graphs_for(opts)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step_graphs[i % n_step_graphs].replay()
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream), torch.cuda.nvtx.range("bench_timed_steps"):
            ev0.record(stream)
            for i in range(args.steps):
                step_graphs[i % n_step_graphs].replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        _barrier(world)
        torch.cuda.synchronize()
    step_ms = ev0.elapsed_time(ev1) / args.steps
    step_ms = _max_over_ranks(step_ms, world)
    kv_step = sum(cases[k][0].kv_bytes_touched() for k in keys)
    alg_step = sum(cases[k][0].algorithmic_bytes() for k in keys)
    value = world * kv_step / (step_ms * 1e-3) / 1e9
    launches = args.steps * len(keys)

    # the same steps with every call waiting for the previous one first
    wait_first = None
    if opts is not None:
        del step_graphs
        graphs_w = step_graphs_for(None)
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                graphs_w[i % n_step_graphs].replay()
            ev0.record(stream)
            for i in range(args.steps):
                graphs_w[i % n_step_graphs].replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        ms_w = _max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
        wait_first = {"value": round(world * kv_step / (ms_w * 1e-3) / 1e9, 1),
                      "ms_per_step": round(ms_w, 5)}
        del graphs_w

    # ---- per case: graphs over the case's replicas -------------------------
    def case_us(k, o):
        g = torch.cuda.CUDAGraph()
        n = len(cases[k])
        with torch.cuda.graph(g, stream=stream):
            for r in range(n):
                call(k, r, o=o)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            reps = max(3, min(50, int(2000 / n)))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (reps * n)

    per_case, pct_w = [], []
    for k in keys:
        us = case_us(k, opts)
        c = cases[k][0]
        kv_gbs = c.kv_bytes_touched() / (us * 1e-6) / 1e9
        alg_gbs = c.algorithmic_bytes() / (us * 1e-6) / 1e9
        row = {"M": k[0], "context": k[1], "us": round(us, 3),
               "kv_gbs": round(kv_gbs, 1), "pct_hbm": round(100 * alg_gbs / peak, 2),
               "replicas": n_reps(k)}
        if opts is not None:
            us_w = case_us(k, None)
            row["us_wait_first"] = round(us_w, 3)
            if k[1] >= 4096:
                pct_w.append(100 * c.algorithmic_bytes() / (us_w * 1e-6) / 1e9 / peak)
        per_case.append(row)
    long_ctx = [c["pct_hbm"] for c in per_case if c["context"] >= 4096]
    if wait_first is not None and pct_w:
        wait_first["median_pct_hbm_4k_32k"] = round(statistics.median(pct_w), 2)
    traffic, traffic_basis = None, "no ncu capture of these kernel sources"
    if _kernel_sources_digest() == TRAFFIC_CAPTURE["sources"]:
        traffic = round(TRAFFIC_CAPTURE["dram_over_algorithmic"] * alg_step / len(keys))
        traffic_basis = ("bytes per launch, averaged over the step's calls: the DRAM/algorithmic "
                         "ratio of one ncu capture (M=4, 32768 keys) x the algorithmic bytes")

    # ---- the other decode configurations, timed the same way ----------------
    configs = None
    if not args.no_configs:
        configs = measure_other_configs(pd, device, l2, peak, stream, opts=opts)

    # ---- end to end through the C ABI with host buffers --------------------
    e2e = None
    if rank == 0 or world > 1:
        e2e = measure_e2e(pd, cases, outs, scratch, stream, keys, args)

    # ---- the oracle on the host (rank 0 only) -------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cases, keys)

    status = pd.paged_decode_device_status(reset=True)
    if rank != 0:
        return
    workload = WORKLOAD if not args.only else WORKLOAD + f"; restricted to (M, context) {sorted(args.only)}"
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/K/V, random page permutation)",
        "config": {
            "workload": workload,
            "l2": "inputs larger than L2: rotating replicas, >= 2.2x L2 per case",
            "timing": "CUDA graphs of the calls, CUDA events on the launching stream",
            "launch": ("early reads: a call reads its block table, seq_lens and older pages "
                       "while the previous call finishes (programmatic dependent launch); "
                       "wait_first: every call waits for the previous one")
                      if opts is not None else "every call waits for the previous one",
            "parallelism": f"replicas x{world}",
        },
        "gpu_launches": launches,
        "roofline": {
            "bound": "hbm",
            "achieved": round(alg_step / (step_ms * 1e-3) / 1e9, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(alg_step / (step_ms * 1e-3) / 1e9 / peak, 4),
            "traffic": traffic,
            "traffic_basis": traffic_basis,
            "peak_kind": peak_kind,
        },
        "median_pct_hbm_4k_32k": round(statistics.median(long_ctx), 2) if long_ctx else None,
        "wait_first": wait_first,
        "cases": per_case,
        "other_configs": configs,
        "clocks": clk.summary(),
        "e2e": e2e,
        "cpu_baseline": cpu,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def other_configs():
    """The other decode configurations, timed beside the sweep: (name, maker
    of replica r, L2-resident note)."""
    from paged_split_kv_02_gb300 import workloads as W

    out = [("single sequence: fp16 D=128 8/2, 300 keys, P=16, NHD",
            lambda r, dev: W.single_seq_nhd(seed=r).to(dev), True)]
    for M in (1, 4):
        out.append((f"sliding window 512: fp16 D=256 8/1, P=32, M={M}, 32768 keys",
                    lambda r, dev, M=M: W.sliding_window(torch.float16, M, 32768, seed=r,
                                                         device=dev, gen_device=dev), True))
    for L in (4096, 32768):
        for M in (1, 4, 8):
            out.append((f"wide head: fp16 D=512 8/1, P=16, M={M}, {L} keys",
                        lambda r, dev, M=M, L=L: W.wide_head(M, L, seed=r, device=dev,
                                                             gen_device=dev), False))
    out.append(("batched: bf16 D=256 16/2, P=1056, 64 sequences U[1,16384], M=4",
                lambda r, dev: W.batched_hybrid_pages(seed=r, device=dev, gen_device=dev), False))
    for P in (784, 1056):
        out.append((f"hybrid page: bf16 D=256 16/2, P={P}, M=4, 16384 keys",
                    lambda r, dev, P=P: W.hybrid_page(P, 4, 16384, seed=r, device=dev,
                                                      gen_device=dev), False))
    out.append(("packed K|V: bf16 D=128 32/8, P=16, HND, M=4, 32768 keys",
                lambda r, dev: W.spec_decode_hnd(4, 32768, seed=r, device=dev, gen_device=dev,
                                                 packed=True), False))
    return out


def run_configs(args, world, rank, local):
    """--workload configs: only the other decode configurations (those whose
    name contains --config-filter), one JSON line; for profiling runs."""
    import paged_split_kv_02_gb300 as pd

    pd.build()
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    l2 = int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 126 << 20))
    peak, peak_kind = _peaks()
    stream = torch.cuda.Stream(device=device)
    res = measure_other_configs(pd, device, l2, peak, stream, args.config_filter,
                                opts=pd.options(early_reads=1) if args.early_reads else None)
    status = pd.paged_decode_device_status(reset=True)
    if rank == 0:
        print(json.dumps({"metric": METRIC, "unit": "us per call", "n_gpus": world,
                          "configs": res, "peak": peak, "peak_kind": peak_kind,
                          "device_status": status}), flush=True)


def measure_other_configs(pd, device, l2, peak, stream, name_filter="", opts=None):
    """µs per call, K+V GB/s and % of the HBM peak of each configuration
    (CUDA graphs over replicas that exceed 2.2 x L2, as for the sweep; a
    windowed or 300-key call moves under 1 MB and is timed on 16 replicas
    that stay in L2: it is bound by latency either way)."""
    res = []
    for name, make, small in other_configs():
        if name_filter and name_filter not in name:
            continue
        first = make(0, device)
        kv = max(1, first.kv_bytes_touched())
        n = 16 if small else max(2, min(12, math.ceil(2.2 * l2 / kv)))
        reps = [first] + [make(r, device) for r in range(1, n)]
        sc = pd.Scratch(first.num_seqs, first.num_q_heads, first.num_kv_heads, first.head_size,
                        first.max_query_len, max_splits=256, device=device)
        outs = [torch.empty_like(c.q) for c in reps]
        calls = [(lambda c=c, o=o: pd.decode_case(c, out=o, scratch=sc, opts=opts))
                 for c, o in zip(reps, outs)]
        with torch.cuda.stream(stream):
            for c in calls:
                c()
        torch.cuda.synchronize()
        us = _time_graph(calls, stream, max(3, min(50, int(600 / n))))
        res.append({"config": name, "us": round(us, 3),
                    "kv_gbs": round(kv / (us * 1e-6) / 1e9, 1),
                    "pct_hbm": round(100 * first.algorithmic_bytes() / (us * 1e-6) / 1e9 / peak, 2),
                    "replicas": n, "l2_resident": small})
        del reps, outs, calls, sc
        torch.cuda.empty_cache()
    return res


def measure_e2e(pd, cases, outs, scratch, stream, keys, args):
    """The same sweep through the C ABI with pinned host buffers, driven the
    way a serving loop would: each step copies every case's q, block table
    and seq_lens host->device in one transfer (one pinned staging buffer),
    makes the C calls with descriptors built once, copies every output back
    in one transfer, and the host reads the step's outputs once that copy has
    landed.  Two sets of buffers alternate, so a step's host->device copy
    (its own stream) and the device->host copy of the step before (a third
    stream) overlap the calls, as a serving loop overlaps its next batch's
    transfers with the current one's compute; the host waits for a step's
    outputs two steps later, before it reuses that step's buffers."""
    import ctypes

    def layout_of(tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    ins = [t for k in keys for t in (cases[k][0].q, cases[k][0].block_table, cases[k][0].seq_lens)]
    in_offs, in_bytes = layout_of(ins)
    out_shapes = [cases[k][0].q for k in keys]
    out_offs, out_bytes = layout_of(out_shapes)
    dev = ins[0].device
    nb = 2  # buffer sets in flight
    host_in = [torch.empty(in_bytes, dtype=torch.uint8).pin_memory() for _ in range(nb)]
    dev_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(nb)]
    host_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(nb)]
    dev_out = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(nb)]

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    for b in range(nb):
        for t, off in zip(ins, in_offs):
            view(host_in[b], off, t).copy_(t.cpu())
    lib = pd.lib()
    early = pd.options(early_reads=1)
    calls = [[] for _ in range(nb)]
    for b in range(nb):
        for i, k in enumerate(keys):
            c = cases[k][0]
            q, bt, sl = (view(dev_in[b], in_offs[3 * i + j], t)
                         for j, t in enumerate((c.q, c.block_table, c.seq_lens)))
            o = view(dev_out[b], out_offs[i], c.q)
            descs = [pd.tensor_desc(t) for t in (q, c.k_cache, c.v_cache, bt, sl, o)]
            cargs = [ctypes.byref(d) for d in descs] + [
                c.num_q_heads, c.num_kv_heads, c.head_size, c.page_size, c.max_query_len,
                c.window, ctypes.c_float(c.scale), c.layout, ctypes.byref(scratch.desc),
                ctypes.c_void_p(stream.cuda_stream)]
            if args.early_reads:
                # (q, block table and seq_lens come from the step's one host
                # copy, complete before the step's first call: every call may
                # read early)
                cargs = cargs + [ctypes.byref(early)]
            calls[b].append((descs, cargs))
    h2d, d2h = in_bytes, out_bytes
    entry = lib.paged_decode_attn_opts if args.early_reads else lib.paged_decode_attn
    kv_step = sum(cases[k][0].kv_bytes_touched() for k in keys)
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(nb)]
    out_ready = [torch.cuda.Event() for _ in range(nb)]
    out_landed = [torch.cuda.Event() for _ in range(nb)]
    checksum = [0.0]

    def consume(b):
        out_landed[b].synchronize()
        checksum[0] += float(host_out[b][:2].view(torch.bfloat16)[0])  # the host reads it

    def issue(i):
        b = i % nb
        if i >= nb:
            consume(b)  # step i - nb's outputs; its buffers are free again
        with torch.cuda.stream(h2d_stream):
            dev_in[b].copy_(host_in[b], non_blocking=True)
            in_ready[b].record(h2d_stream)
        stream.wait_event(in_ready[b])
        for _, a in calls[b]:
            rc = entry(*a)
            if rc != 0:
                raise RuntimeError(f"paged_decode_attn: {rc}")
        out_ready[b].record(stream)
        d2h_stream.wait_event(out_ready[b])
        with torch.cuda.stream(d2h_stream):
            host_out[b].copy_(dev_out[b], non_blocking=True)
            out_landed[b].record(d2h_stream)

    def run(n):
        for i in range(n):
            issue(i)
        for i in range(max(0, n - nb), n):
            consume(i % nb)

    run(args.warmup)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(args.steps)
    dt = (time.perf_counter() - t0) / args.steps
    return {"value": round(kv_step / dt / 1e9, 1), "unit": UNIT, "ms_per_step": round(dt * 1e3, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "transfers": "one pinned host->device copy of every call's inputs and one "
                         "device->host copy of every output per step, read by the host; two "
                         "buffer sets alternate, so the copies of neighbouring steps overlap "
                         "the calls",
            "call": "paged_decode_attn_opts (early reads)" if args.early_reads
                    else "paged_decode_attn"}


def _oracle_sweep(host_cases, keys, nthreads):
    import oracle

    t0 = time.perf_counter()
    for k in keys:
        oracle.attention(host_cases[k], nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(cases, keys, min_seconds=10.0, max_sweeps=200):
    """The fp64 oracle on the host cores, repeating one call of every case
    until at least `min_seconds` have passed (a bounded sample)."""
    import oracle

    oracle.build()
    host = {k: cases[k][0].to("cpu") for k in keys}
    n = oracle.default_threads()
    dt, sweeps = 0.0, 0
    while dt < min_seconds and sweeps < max_sweeps:
        dt += _oracle_sweep(host, keys, n)
        sweeps += 1
    kv = sum(host[k].kv_bytes_touched() for k in keys)
    # and on one thread, over the cases up to 4k keys (a bounded sample)
    small = [k for k in keys if k[1] <= 4096] or list(keys)
    dt1 = _oracle_sweep(host, small, 1)
    kv1 = sum(host[k].kv_bytes_touched() for k in small)
    return {"value": round(sweeps * kv / dt / 1e9, 4), "unit": UNIT, "cores": n,
            "single_thread": {"value": round(kv1 / dt1 / 1e9, 4), "unit": UNIT,
                              "seconds": round(dt1, 2),
                              "sample": "one call of each sweep case up to 4096 keys"},
            "kind": "oracle",
            "sample": f"{sweeps} repetitions of one call of each of the {len(keys)} sweep "
                      "cases (all heads), fp64 C oracle",
            "seconds": round(dt, 2)}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step runs it on the host cores
    over one call of every sweep case (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from paged_split_kv_02_gb300 import workloads as W

    oracle.build()
    keys = [(M, L) for M in MS for L in CONTEXTS]
    host = {(M, L): W.spec_decode_hnd(M, L, seed=1000 * M) for (M, L) in keys}
    n = oracle.default_threads()
    kv = sum(host[k].kv_bytes_touched() for k in keys)
    for _ in range(args.warmup):
        _oracle_sweep(host, keys, n)
    t = 0.0
    for _ in range(args.steps):
        t += _oracle_sweep(host, keys, n)
    dt = t / args.steps
    value = kv / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/K/V, random page permutation)",
        "config": {"workload": WORKLOAD, "parallelism": "host threads"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": n, "kind": "oracle",
                         "sample": "one call of each of the 20 sweep cases per step"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


VARLEN_WORKLOAD = ("speculative-decode batch with a query length per request: bf16, head_size "
                   "128, 32 q / 8 kv heads, page_size 16, HND, 32 requests, draft lengths "
                   "U{1..4}, contexts U[1k, 16k] (one call = paged_decode_attn_varlen)")


def _time_graph(calls, stream, reps):
    """Mean µs per call of a CUDA graph of `calls`, replayed `reps` times."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    with torch.cuda.stream(stream):
        for _ in range(2):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * len(calls))


def run_varlen(args, world, rank, local):
    """--workload varlen: the variable-query-length call on a batch (replicas
    past 2.2 x L2), with the same requests padded to a uniform call timed
    beside it."""
    import paged_split_kv_02_gb300 as pd
    from paged_split_kv_02_gb300 import workloads as W

    pd.build()
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20))
    peak, peak_kind = _peaks()
    nreq = args.requests
    probe = W.varlen_spec_decode_batch(seed=0, num_seqs=nreq)
    n_rep = max(2, math.ceil(2.2 * l2 / probe.kv_bytes_touched()))
    var = [W.varlen_spec_decode_batch(seed=r, num_seqs=nreq, device=device, gen_device=device)
           for r in range(n_rep)]
    uni = [W.varlen_spec_decode_batch(seed=r, num_seqs=nreq, uniform=True, device=device,
                                      gen_device=device) for r in range(n_rep)]
    c0 = var[0]
    scratch = pd.Scratch(c0.num_seqs, c0.num_q_heads, c0.num_kv_heads, c0.head_size, 4,
                         max_splits=256, device=device)
    outs_v = [torch.empty_like(c.q) for c in var]
    outs_u = [torch.empty_like(c.q) for c in uni]
    stream = torch.cuda.Stream(device=device)
    calls_v = [(lambda c=c, o=o: pd.decode_case(c, out=o, scratch=scratch)) for c, o in zip(var, outs_v)]
    calls_u = [(lambda c=c, o=o: pd.decode_case(c, out=o, scratch=scratch)) for c, o in zip(uni, outs_u)]
    with torch.cuda.stream(stream):
        for c in calls_v + calls_u:
            c()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        _time_graph(calls_v, stream, 1)
    _barrier(world)
    with ClockSampler(local) as clk:
        us = _time_graph(calls_v, stream, args.steps)
    us = _max_over_ranks(us, world)
    us_u = _time_graph(calls_u, stream, args.steps)
    kv = sum(c.kv_bytes_touched() for c in var) / n_rep
    alg = sum(c.algorithmic_bytes() for c in var) / n_rep
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        host = var[0].to("cpu")
        rows = [(t, h) for t in range(0, host.q.shape[0], 8) for h in range(host.num_q_heads)]
        n = oracle.default_threads()
        t0 = time.perf_counter()
        oracle.attention(host, rows=rows, nthreads=n)
        dt = time.perf_counter() - t0
        frac = len(rows) / (host.q.shape[0] * host.num_q_heads)
        cpu = {"value": round(kv * frac / dt / 1e9, 4), "unit": UNIT, "cores": n,
               "kind": "oracle", "seconds": round(dt, 2),
               "sample": f"every 8th token row of one batch, all heads ({frac:.3f} of the "
                         "rows), fp64 C oracle; value scaled to the sampled rows"}
    status = pd.paged_decode_device_status(reset=True)
    if rank != 0:
        return
    traffic, traffic_basis = None, "no ncu capture of these kernel sources"
    if _kernel_sources_digest() == VARLEN_TRAFFIC_CAPTURE["sources"]:
        traffic = round(VARLEN_TRAFFIC_CAPTURE["dram_over_algorithmic"] * alg)
        traffic_basis = ("bytes per launch: the DRAM/algorithmic ratio of one ncu capture of "
                         "an 8-request batch of this workload x the algorithmic bytes")
    line = {
        "metric": METRIC, "value": round(world * kv / (us * 1e-6) / 1e9, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us * 1e-3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/K/V, random page permutation)",
        "config": {"workload": VARLEN_WORKLOAD.replace("32 requests", f"{nreq} requests"),
                   "l2": f"inputs larger than L2: {n_rep} rotating replicas",
                   "timing": "CUDA graph of the calls, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps * n_rep,
        "us_per_call": round(us, 3),
        "padded_uniform_us_per_call": round(us_u, 3),
        "roofline": {"bound": "hbm", "achieved": round(alg / (us * 1e-6) / 1e9, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(alg / (us * 1e-6) / 1e9 / peak, 4), "traffic": traffic,
                     "traffic_basis": traffic_basis, "peak_kind": peak_kind},
        "clocks": clk.summary(),
        "e2e": None,
        "cpu_baseline": cpu,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


ROPE_WORKLOAD = ("rotary embedding + paged KV-cache write ahead of decode: bf16, head_size 128, "
                 "32 q / 8 kv heads, all 128 dims rotated (NeoX pairing), page_size 16, HND; "
                 "16384 new tokens at random positions and distinct cache slots (one call)")


def run_rope(args, world, rank, local):
    """--workload rope: paged_rope_cache_write on a prefill-sized token
    batch (HBM-bound: ~0.4 GB per call), with a decode-sized batch (64
    sequences x 4 tokens, latency-bound) timed beside it."""
    import paged_split_kv_02_gb300 as pd
    from paged_split_kv_02_gb300 import workloads as W

    pd.build()
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    peak, peak_kind = _peaks()
    stream = torch.cuda.Stream(device=device)

    def make(T, pages, seed):
        return W.make_rope_case(f"rope_T{T}", seed=seed, dtype=torch.bfloat16, num_tokens=T,
                                num_q_heads=32, num_kv_heads=8, head_size=128, rot_dim=128,
                                page_size=16, num_pages=pages, layout=W.HND, max_pos=32768,
                                device=device, gen_device=device)

    big = [make(16384, 2048, r) for r in range(2)]  # two replicas of ~0.4 GB each
    small = [make(256, 64, 10 + r) for r in range(64)]
    outs_b = [torch.empty_like(c.q) for c in big]
    outs_s = [torch.empty_like(c.q) for c in small]
    calls_b = [(lambda c=c, o=o: pd.rope_case(c, q_out=o)) for c, o in zip(big, outs_b)]
    calls_s = [(lambda c=c, o=o: pd.rope_case(c, q_out=o)) for c, o in zip(small, outs_s)]
    with torch.cuda.stream(stream):
        for c in calls_b + calls_s:
            c()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        _time_graph(calls_b, stream, 1)
    _barrier(world)
    with ClockSampler(local) as clk:
        us = _time_graph(calls_b, stream, args.steps)
    us = _max_over_ranks(us, world)
    us_small = _time_graph(calls_s, stream, max(3, args.steps // 4))
    nbytes = big[0].bytes_moved()
    status = pd.paged_decode_device_status(reset=True)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        from oracle import rope_cache as R

        c = make(512, 64, 99).to("cpu")
        n = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            R.rope_cache_write(c.q, c.k, c.v, c.positions, c.slot_mapping, c.cos_sin,
                               c.k_cache, c.v_cache, c.layout, c.rot_dim, c.is_neox)
            n += 1
        dt = (time.perf_counter() - t0) / n
        cpu = {"value": round(c.bytes_moved() / dt / 1e9, 4), "unit": UNIT, "cores": 1,
               "kind": "oracle", "seconds": round(dt * n, 2),
               "sample": f"{n} calls on 512 tokens of the same shape (fp64 numpy oracle, "
                         "one thread)"}
    line = {
        "metric": "GB/s moved by the rotary embedding + KV-cache write, and us per call",
        "value": round(world * nbytes / (us * 1e-6) / 1e9, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us * 1e-3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, random positions and slots)",
        "config": {"workload": ROPE_WORKLOAD,
                   "l2": "inputs larger than L2: two replicas of ~0.4 GB alternate",
                   "timing": "CUDA graph of the calls, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps * len(calls_b),
        "us_per_call": round(us, 3),
        "decode_batch_us_per_call": round(us_small, 3),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4),
                     "traffic": None, "traffic_basis": "no ncu capture of this kernel",
                     "peak_kind": peak_kind},
        "clocks": clk.summary(),
        "e2e": None,
        "cpu_baseline": cpu,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


PREFILL_WORKLOAD = ("paged prefill: bf16, head_size 128, 32 q / 8 kv heads, page_size 16, HND; "
                    "4 requests x 2048 new tokens after 2048 cached ones (one call over the "
                    "host-made work list)")


def run_prefill(args, world, rank, local):
    """--workload prefill: paged_prefill_attn on a batch of long requests;
    the plan is made once on the host, its work list copied to the device."""
    import paged_split_kv_02_gb300 as pd
    from paged_split_kv_02_gb300 import workloads as W

    pd.build()
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        peak, peak_kind = float(peaks["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"
    stream = torch.cuda.Stream(device=device)
    reps = [W.make_prefill_case("prefill_bench", seed=r, q_lens=[2048] * 4, contexts=[2048] * 4,
                                device=device, gen_device=device) for r in range(2)]
    c0 = reps[0]
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    plan = pd.paged_prefill_plan(c0.query_start_host, c0.seq_lens_host, c0.num_q_heads,
                                 c0.num_kv_heads, c0.head_size, c0.window, sms)
    items, info = plan
    work = items.to(device)
    sc = pd.prefill_scratch(c0.num_kv_heads, c0.head_size, sms, device=device)
    outs = [torch.empty_like(c.q) for c in reps]

    def call(c, o):
        pd.paged_prefill_attn(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens,
                              c.query_start, work, info, o, c.num_q_heads, c.num_kv_heads,
                              c.head_size, c.page_size, c.window, c.scale, c.layout, sc)

    calls = [(lambda c=c, o=o: call(c, o)) for c, o in zip(reps, outs)]
    with torch.cuda.stream(stream):
        for c in calls:
            c()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        _time_graph(calls, stream, 1)
    _barrier(world)
    with ClockSampler(local) as clk:
        us = _time_graph(calls, stream, args.steps)
    us = _max_over_ranks(us, world)
    flops = W.prefill_flops(c0)
    status = pd.paged_decode_device_status(reset=True)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        host = c0.to("cpu")
        T = host.q.shape[0]
        rows = [(t, h) for t in range(0, T, 64) for h in range(host.num_q_heads)]
        n = oracle.default_threads()
        t0 = time.perf_counter()
        oracle.attention(host, rows=rows, nthreads=n)
        dt = time.perf_counter() - t0
        frac = len(rows) / (T * host.num_q_heads)
        cpu = {"value": round(flops * frac / dt / 1e12, 5), "unit": "TFLOP/s", "cores": n,
               "kind": "oracle", "seconds": round(dt, 2),
               "sample": f"every 64th token row of the batch, all heads ({frac:.4f} of the "
                         "rows), fp64 C oracle; value scaled to the sampled rows"}
    tflops = flops / (us * 1e-6) / 1e12
    line = {
        "metric": "TFLOP/s of a paged prefill call (QK^T and PV over the keys each row sees)",
        "value": round(world * tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us * 1e-3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/K/V, random page permutation)",
        "config": {"workload": PREFILL_WORKLOAD,
                   "l2": "two replicas alternate (prefill is bound by arithmetic)",
                   "timing": "CUDA graph of the calls, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}",
                   "plan": info.as_dict()},
        "gpu_launches": args.steps * len(calls),
        "us_per_call": round(us, 3),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "traffic": None,
                     "traffic_basis": "no ncu capture of this launch", "peak_kind": peak_kind,
                     "note": "products on tcgen05 (256-row tiles: two 128-row halves per "
                             "K/V stage, M = 128; S, P and O in tensor memory; four softmax "
                             "warps per half, one warp issuing S, one per half issuing PV), "
                             "against the measured cuBLAS bf16 peak"},
        "clocks": clk.summary(),
        "e2e": None,
        "cpu_baseline": cpu,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other decode configurations timed beside the sweep")
    ap.add_argument("--config-filter", default="",
                    help="--workload configs: only configurations whose name contains this")
    ap.add_argument("--workload", default="sweep",
                    choices=["sweep", "varlen", "rope", "prefill", "configs"],
                    help="sweep: the spec-decode sweep (default); varlen: a batch with a "
                         "query length per request; rope: the rotary embedding + KV-cache "
                         "write; prefill: paged prefill over a work list; configs: the other "
                         "decode configurations only")
    ap.add_argument("--requests", type=int, default=32,
                    help="requests of the varlen batch (fewer for profiling runs)")
    ap.add_argument("--cases", default="",
                    help="restrict the sweep, e.g. 4:32768,1:4096 (profiling runs only)")
    ap.add_argument("--early-reads", type=int, default=1, choices=[0, 1],
                    help="1 (default): decode calls read their block table, seq_lens and "
                         "older pages while the previous call finishes "
                         "(pd_options.early_reads); 0: every call waits for the previous one")
    args = ap.parse_args()
    args.only = None
    if args.cases:
        args.only = {tuple(int(x) for x in c.split(":")) for c in args.cases.split(",")}
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload == "varlen":
        run_varlen(args, world, rank, local)
    elif args.workload == "rope":
        run_rope(args, world, rank, local)
    elif args.workload == "prefill":
        run_prefill(args, world, rank, local)
    elif args.workload == "configs":
        run_configs(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
