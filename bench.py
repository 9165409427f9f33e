"""Benchmark: paged-decode KV bandwidth on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one paged_decode call over the workload's whole batch (window
restriction, page gather, logits, online softmax, P.V, Split-KV merge and
epilogue, all in one kernel launch).  Inputs are resident in HBM; the L2 is
flushed before every timed step (a 512 MiB write, then a 256 MiB read so that
no dirty line of the flush is written back inside the step; --l2-flush write
keeps only the write) and the KV stream is larger than the L2 anyway.  Each step is timed with CUDA events on the launching
stream, around a direct call (--graph replays one captured call instead, so
that host-side launch overhead cannot open gaps inside a step).  value =
algorithmic KV bytes of all ranks / max over ranks of the summed step time.
One JSON line is printed by rank 0.  The end-to-end figure (e2e) always goes
through the direct call.

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload per step, in the same metric.

Under torchrun (N > 1) each rank runs an independent replica of the workload
on its own GPU (the path has no exchange step): weak scaling.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s and % of GB300 HBM peak; µs/call at B=64 bf16 decode"
DEFAULT_WORKLOAD = "gqa_decode_b64"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth (the measured copy peak is the roofline)


# ------------------------------------------------------------- accounting
def visible_keys(case) -> np.ndarray:
    """Keys each request reads (page-aligned window start, as the kernel sees them)."""
    L = case.seq_lens.astype(np.int64)
    if case.window > 0 and not case.causal:
        start = np.maximum(0, (L - (case.window + case.sq - 1)) // case.page_size) * case.page_size
    elif case.window > 0:
        start = np.maximum(0, L - case.sq - case.window + 1)
    else:
        start = np.zeros_like(L)
    return np.maximum(L - start, 0)


def algorithmic_bytes(case) -> dict:
    """Bytes a perfect kernel must move: visible K and V rows, q, out, lse,
    the block-table entries of the visible pages and seq_lens."""
    elt = 1 if case.dtype == "fp8" else 2
    vis = visible_keys(case)
    kv = int(vis.sum()) * case.num_kv_heads * 2 * case.head_dim * elt
    B, sq, Hq, D = case.q.shape
    q = case.q.nbytes
    out = B * sq * Hq * D * 2
    lse = B * sq * Hq * 4
    table = int(np.ceil(vis / case.page_size).sum()) * 4
    return {"kv": kv, "total": kv + q + out + lse + table + B * 4}


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


# sources that build neither the paged-decode kernels nor their launch plan
NON_DECODE_SOURCES = ("segment.cu", "segment.cuh", "cache_write.cu", "static_ws.cu")
# sources of the tcgen05 query-block kernel only
TC05_SOURCES = ("decode_tc05.cu", "decode_tc05.cuh", "tc05.cuh")


def source_digest(tc05: bool = True) -> str:
    """sha256 over the paged-decode kernel sources and their launch plan (with
    tc05=False, leaving out the files only the tcgen05 kernel is built from):
    a traffic figure is valid only for the digest of the sources its kernel
    is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_15_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in NON_DECODE_SOURCES and \
                (tc05 or name not in TC05_SOURCES):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = ""):
    """dram bytes per launch from the committed ncu summary, if it matches the
    sources of the kernel the workload runs (`kernel`: the library's name)."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    d = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not t or not d or d.group(1) != source_digest(tc05="tcgen05" in kernel):
        return None
    return int(t.group(1))


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        if not inside and rows:
            inside = [min(rows, key=lambda r: abs(r[0] - t1))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------ device side
def pack(torch, tensors):
    """Copy device tensors into one allocation (views at 256-byte aligned
    offsets), so that an end-to-end step moves all of them with one copy.
    Returns (buffer, views)."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device="cuda")
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        v = buf[o:o + n].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class PagedRunner:
    """One paged_decode call over a PagedCase, inputs resident on the device."""
    kernel = "paged decode (one launch per step)"

    def __init__(self, case, args, torch, pkd):
        from workloads import to_torch
        self.case, self.pkd = case, pkd
        self.q = to_torch(case.q, case.dtype)
        self.cache = to_torch(case.kv_cache, case.dtype)
        self.bt = to_torch(case.block_table, "int32")
        self.lens = to_torch(case.seq_lens, "int32")
        self.out = torch.empty(case.q.shape, dtype=torch.bfloat16 if case.dtype != "fp16" else torch.float16,
                               device="cuda")
        self.lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
        self.max_kv_len = int(case.block_table.shape[1] * case.page_size)
        kv_code = {"bf16": pkd.BF16, "fp16": pkd.FP16, "fp8": pkd.FP8_E4M3}[case.dtype]
        self.chunk, self.path, self.grid, self.flat = effective_chunk(case, args), args.path, args.grid, args.flat
        self.balanced = args.balanced
        flags = paged_flags(case, args, pkd)
        self.ws = torch.empty(pkd.workspace_size(case.batch, case.sq, case.num_heads, case.num_kv_heads,
                                                 case.head_dim, case.page_size, self.max_kv_len, kv_code, case.window,
                                                 self.chunk, flags), dtype=torch.uint8, device="cuda")
        pkd.workspace_init(self.ws)
        # q, table and lengths in one allocation, out and lse in another: an
        # end-to-end step copies each pack once
        in_buf, (self.q, self.bt, self.lens) = pack(torch, [self.q, self.bt, self.lens])
        out_buf, (self.out, self.lse) = pack(torch, [self.out, self.lse])
        self.inputs = [in_buf]    # copied in every end-to-end step
        self.outputs = [out_buf]  # copied back every end-to-end step
        self.acct = algorithmic_bytes(case)
        self.flags, self.kv_code = flags, kv_code

    def host_same_kernel(self) -> bool:
        """Whether a call with host_io launches the kernel of the device call
        (the tcgen05 kernel does not take host memory: its shapes move to the
        chunked grid, and their end-to-end figure keeps the copy path)."""
        c, pkd = self.case, self.pkd
        shape = (c.batch, c.sq, c.num_heads, c.num_kv_heads, c.head_dim, c.page_size, self.max_kv_len, self.kv_code,
                 c.window, self.chunk)
        return pkd.kernel_name(*shape, flags=self.flags | pkd.FLAG_HOST_IO) == pkd.kernel_name(*shape, flags=self.flags)

    def prepare_host(self):
        """Pinned host q, table and lengths (and out, lse) for calls with
        host_io: the kernels read and write them in place over the host link.
        Returns (bytes read from the host, bytes written to it) per call."""
        torch, c = __import__("torch"), self.case
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
        self.hq, self.hbt, self.hlens = pin(self.q), pin(self.bt), pin(self.lens)
        self.hout = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        self.hlse = torch.empty(self.lse.shape, dtype=torch.float32, pin_memory=True)
        self.ws_host = torch.empty(self.pkd.workspace_size(
            c.batch, c.sq, c.num_heads, c.num_kv_heads, c.head_dim, c.page_size, self.max_kv_len, self.kv_code,
            c.window, self.chunk, self.flags | self.pkd.FLAG_HOST_IO), dtype=torch.uint8, device="cuda")
        self.pkd.workspace_init(self.ws_host)
        nbytes = lambda ts: sum(t.numel() * t.element_size() for t in ts)
        return nbytes([self.hq, self.hbt, self.hlens]), nbytes([self.hout, self.hlse])

    def call_host(self):
        c = self.case
        self.pkd.paged_decode(self.hq, self.cache, self.hbt, self.hlens, c.scale, c.window, out=self.hout,
                              lse=self.hlse, q_scale=c.q_scale, k_scale=c.k_scale, v_scale=c.v_scale,
                              max_kv_len=self.max_kv_len, workspace=self.ws_host, causal=c.causal,
                              chunk_tokens=self.chunk, force_fma=self.path == "fma", grid=self.grid, flat=self.flat,
                              balanced=self.balanced, host_io=True)

    def check_host(self):
        if self.pkd.workspace_check(self.ws_host) != self.pkd.OK:
            raise RuntimeError("device status word set: " + self.pkd.load_library().pkd_last_error().decode())

    def call(self):
        c = self.case
        self.pkd.paged_decode(self.q, self.cache, self.bt, self.lens, c.scale, c.window, out=self.out, lse=self.lse,
                              q_scale=c.q_scale, k_scale=c.k_scale, v_scale=c.v_scale, max_kv_len=self.max_kv_len,
                              workspace=self.ws, causal=c.causal, chunk_tokens=self.chunk,
                              force_fma=self.path == "fma", grid=self.grid, flat=self.flat,
                              balanced=self.balanced)

    def check(self):
        if self.pkd.workspace_check(self.ws) != self.pkd.OK:
            raise RuntimeError("device status word set: " + self.pkd.load_library().pkd_last_error().decode())


class SegmentRunner:
    """One segmented_attention call (attention per segment + combine)."""
    kernel = "DASH segmented attention with fused combine (one launch per step)"

    def __init__(self, case, args, torch, pkd):
        from workloads import to_torch
        self.case, self.pkd = case, pkd
        self.q = to_torch(case.q, case.dtype)
        self.k = to_torch(case.k, case.dtype)
        self.v = to_torch(case.v, case.dtype)
        self.used = to_torch(case.used, "int32")
        self.bias = to_torch(case.bias, "fp32")
        self.out = torch.empty_like(self.q)
        in_buf, (self.q, self.k, self.v, self.used, self.bias) = pack(
            torch, [self.q, self.k, self.v, self.used, self.bias])
        self.inputs = [in_buf]
        self.outputs = [self.out]
        self.acct = segment_bytes(case)

    def call(self):
        self.pkd.segmented_attention(self.q, self.k, self.v, self.used, self.bias, self.case.bs, self.case.local,
                                     out=self.out)

    def check(self):
        pass


class PagedSegmentRunner:
    """One segmented_attention_paged call: segments read through the block table."""
    kernel = "DASH segmented attention from the paged cache, fused combine (one launch per step)"

    def __init__(self, case, args, torch, pkd):
        from workloads import to_torch
        self.case, self.pkd = case, pkd
        self.q = to_torch(case.q, case.dtype)
        self.cache = to_torch(case.kv_cache, case.dtype)
        self.bt = to_torch(case.block_table, "int32")
        self.seg_start = to_torch(case.seg_start, "int32")
        self.used = to_torch(case.used, "int32")
        self.bias = to_torch(case.bias, "fp32")
        self.out = torch.empty_like(self.q)
        in_buf, (self.q, self.bt, self.seg_start, self.used, self.bias) = pack(
            torch, [self.q, self.bt, self.seg_start, self.used, self.bias])
        self.inputs = [in_buf]
        self.outputs = [self.out]
        Hkv, D = case.num_kv_heads, case.q.shape[2]
        kv = int(case.used.sum()) * Hkv * 2 * D * 2
        self.acct = {"kv": kv, "total": kv + case.q.nbytes * 2 + case.used.nbytes * 2 + case.bias.nbytes}

    def call(self):
        c = self.case
        self.pkd.segmented_attention_paged(self.q, self.cache, self.bt, self.seg_start, self.used, self.bias, c.bs,
                                           c.local, out=self.out)

    def check(self):
        pass


class CacheWriteRunner:
    """One cache_write call: new key/value rows quantised into their slots."""
    kernel = "KV-cache write (one launch per step)"

    def __init__(self, case, args, torch, pkd):
        from workloads import to_torch
        self.case, self.pkd = case, pkd
        self.key = to_torch(case.key, case.in_dtype)
        self.value = to_torch(case.value, case.in_dtype)
        self.slots = torch.from_numpy(case.slots).cuda()
        self.cache = to_torch(case.kv_cache, case.kv_dtype)
        in_buf, (self.key, self.value, self.slots) = pack(torch, [self.key, self.value, self.slots])
        self.inputs = [in_buf]
        self.outputs = []
        live = int((case.slots >= 0).sum())
        Hkv, D = case.key.shape[1], case.key.shape[2]
        out_elt = 1 if case.kv_dtype == "fp8" else 2
        kv = live * Hkv * 2 * D * (2 + out_elt)
        self.acct = {"kv": kv, "total": kv + case.slots.nbytes}

    def call(self):
        self.pkd.cache_write(self.key, self.value, self.slots, self.cache, k_scale=self.case.k_scale,
                             v_scale=self.case.v_scale)

    def check(self):
        pass


def segment_bytes(case) -> dict:
    """Algorithmic bytes of segmented attention: the used K and V rows of every
    segment for every kv head, plus q, out, used and bias."""
    elt = 2
    kv = int(np.clip(case.used, 0, None).sum()) * case.num_kv_heads * 2 * case.q.shape[2] * elt
    extra = case.q.nbytes * 2 + case.used.nbytes + case.bias.nbytes
    return {"kv": kv, "total": kv + extra}


def runner_kind(case):
    import workloads as wl
    return SegmentRunner if isinstance(case, wl.SegmentCase) else \
        CacheWriteRunner if isinstance(case, wl.CacheWriteCase) else \
        PagedSegmentRunner if isinstance(case, wl.PagedSegmentCase) else PagedRunner


def make_flush(torch, args):
    """Evict L2 before a step: write a buffer larger than L2; with write-read,
    then read half of it back so that L2 holds clean lines and no write-back
    of the flush is left to compete with the step."""
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    words = flush_buf.view(torch.int32)

    class _Flush:
        @staticmethod
        def zero_():
            flush_buf.zero_()
            if args.l2_flush == "write-read":
                words[:words.numel() // 2].amax()
    return _Flush()


# The other configurations, timed after the headline in the default run so
# that one measured line carries them all (each with its own roofline figure).
SECONDARY = ("query_block_sq8", "query_block_sq8_w4096", "fp8_long_b8", "dash_segments_n256", "dash_paged_n256",
             "kv_write_32k")


def run_secondary(args, peak_gbs) -> dict:
    """Time each SECONDARY workload like the headline (L2 flushed before every
    step, CUDA events on the launching stream, the workload's own Split-KV)."""
    import copy
    import torch
    import paged_kv_decode_15_gb300 as pkd
    import workloads as wl
    flush = make_flush(torch, args)
    stream = torch.cuda.current_stream()
    sub_args = copy.copy(args)
    sub_args.chunk, sub_args.path, sub_args.grid, sub_args.flat, sub_args.balanced = None, "auto", False, False, False
    res = {}
    for name in SECONDARY:
        case = wl.WORKLOADS[name]()
        runner = runner_kind(case)(case, sub_args, torch, pkd)
        for _ in range(5):
            flush.zero_()
            runner.call()
        torch.cuda.synchronize()
        runner.check()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.secondary_steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.secondary_steps)]
        for i in range(args.secondary_steps):
            flush.zero_()
            starts[i].record(stream)
            runner.call()
            ends[i].record(stream)
        torch.cuda.synchronize()
        runner.check()
        ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        avg = sum(ms) / len(ms) / 1e3
        entry = {"us_per_call": round(avg * 1e6, 2), "us_per_call_median": round(statistics.median(ms) * 1e3, 2),
                 "kv_gbs": round(runner.acct["kv"] / avg / 1e9, 1),
                 "roofline_frac": round(runner.acct["total"] / avg / 1e9 / peak_gbs, 4),
                 "algorithmic_bytes_per_launch": runner.acct["total"], "kernel": runner.kernel,
                 "steps": args.secondary_steps}
        if isinstance(runner, PagedRunner):
            entry["paged_kernel"] = paged_kernel_name(case, sub_args)
            entry["chunk_tokens"] = effective_chunk(case, sub_args)
        res[name] = entry
        del runner, case
        torch.cuda.empty_cache()
    return res


def run_gpu(args, rank, world, dist):
    import torch
    import paged_kv_decode_15_gb300 as pkd
    import workloads as wl
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    pkd.build()
    pkd.load_library()
    case = wl.WORKLOADS[args.workload]()
    runner = runner_kind(case)(case, args, torch, pkd)
    flush = make_flush(torch, args)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        flush.zero_()
        runner.call()
    torch.cuda.synchronize()
    runner.check()

    # With --graph the timed steps replay one captured call, so that the
    # host's launch overhead (the binding's argument checks, ctypes) cannot
    # open gaps between a step's events even when the host falls behind the
    # GPU; the kernel and its arguments are those of the direct call.
    step_call, launch_mode = runner.call, "direct"
    if args.graph:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(graph, stream=side):
                    runner.call()
            stream.wait_stream(side)
            torch.cuda.synchronize()
            step_call, launch_mode = graph.replay, "CUDA graph of one call, replayed every step"
        except RuntimeError as e:  # capture refused: time direct calls and say so
            launch_mode = f"direct (graph capture failed: {e})"
    args.launch_mode = launch_mode

    sampler = ClockSampler(torch.cuda.current_device())
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step_call()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist:
        dist.barrier()
    clocks = sampler.stop(t0, t1)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = float(sum(step_ms))

    # end to end through the public call: pinned host inputs in, results out
    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu()) for t in runner.inputs]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in runner.outputs]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def copy_step():
        for dev, host in zip(runner.inputs, host_in):
            dev.copy_(host, non_blocking=True)
        runner.call()
        for dev, host in zip(runner.outputs, host_out):
            host.copy_(dev, non_blocking=True)

    def timed(step):
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for _ in range(args.warmup):
            flush.zero_()
            step()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            es[i].record(stream)
            step()
            ee[i].record(stream)
        torch.cuda.synchronize()
        return float(sum(s.elapsed_time(e) for s, e in zip(es, ee)))

    e2e_copy_ms = None
    if hasattr(runner, "call_host") and runner.host_same_kernel():
        # the kernels read the step's inputs from pinned host memory and write its
        # results there (PKD_FLAG_HOST_IO); the copy-in / copy-out step is timed too
        e2e_copy_ms = timed(copy_step)
        runner.check()
        h2d, d2h = runner.prepare_host()
        e2e_ms = timed(runner.call_host)
        runner.check_host()
    else:
        e2e_ms = timed(copy_step)
        runner.check()
    args.e2e_copy_ms = e2e_copy_ms
    args.e2e_host_io = e2e_copy_ms is not None

    if dist:
        total_ms, e2e_ms, copy_ms = max_over_ranks([total_ms, e2e_ms, args.e2e_copy_ms or 0.0], dist, "cuda")
        args.e2e_copy_ms = copy_ms if args.e2e_copy_ms is not None else None
    return case, runner, step_ms, total_ms, e2e_ms, h2d, d2h, clocks


def max_over_ranks(values, dist, device):
    """Element-wise max of per-rank timings (the slowest replica sets the job time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(bytes_per_step_per_rank: int, world: int, steps: int, total_ms: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_per_step_per_rank * world * steps / (total_ms / 1e3) / 1e9


def cpu_baseline(case, budget_s: float = 12.0) -> dict:
    """Time the oracle, as it stands, on a bounded sample of the workload's requests."""
    import oracle
    threads = os.cpu_count() or 1
    order = np.random.default_rng(0).permutation(case.batch)
    n = 1
    t = _time_oracle(case, order[:1], threads)
    n = int(min(case.batch, max(1, budget_s / max(t, 1e-6))))
    if n > 1:
        t = _time_oracle(case, order[:n], threads)
    sub = _subcase(case, order[:n])
    gbs = algorithmic_bytes(sub)["kv"] / t / 1e9
    # the same oracle on one thread, on a sample sized for about 4 s
    n1 = int(min(n, max(1, 4.0 / max(t * threads / n, 1e-6))))
    t1 = _time_oracle(case, order[:n1], 1)
    gbs1 = algorithmic_bytes(_subcase(case, order[:n1]))["kv"] / t1 / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {case.batch} requests (all heads), fp64 C oracle with OpenMP over "
                      f"(request, head), {t:.2f} s",
            "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "sample": f"{n1} requests, {t1:.2f} s"}}


def _subcase(case, idx):
    import copy
    sub = copy.copy(case)
    sub.q = case.q[idx]
    sub.block_table = case.block_table[idx]
    sub.seq_lens = case.seq_lens[idx]
    return sub


def _time_oracle(case, idx, threads):
    import oracle
    sub = _subcase(case, idx)
    t = time.perf_counter()
    oracle.paged_decode(sub.q, sub.dtype, sub.kv_cache, sub.dtype, sub.block_table, sub.seq_lens,
                        threads=threads, **sub.oracle_kwargs())
    return time.perf_counter() - t


def run_reference(args, rank):
    """The oracle arm: each step is a bounded sample of the workload on the host cores."""
    import oracle
    import workloads as wl
    oracle.build()
    case = wl.WORKLOADS[args.workload]()
    threads = os.cpu_count() or 1
    order = np.random.default_rng(0).permutation(case.batch)
    t1 = _time_oracle(case, order[:1], threads)
    per_step_budget = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    n = int(min(case.batch, max(1, per_step_budget / max(t1, 1e-6))))
    sub = _subcase(case, order[:n])
    for _ in range(args.warmup):
        _time_oracle(case, order[:n], threads)
    total = 0.0
    for _ in range(args.steps):
        total += _time_oracle(case, order[:n], threads)
    kv = algorithmic_bytes(sub)["kv"]
    value = kv * args.steps / total / 1e9
    cfg = workload_config(case, args, gpu_kernel=False)
    sample = f"{n} of {case.batch} requests per step (all heads), fp64 C oracle, OpenMP over (request, head)"
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def workload_config(case, args, gpu_kernel=True) -> dict:
    """The workload's description; gpu_kernel=False (the oracle arm) leaves
    out the library's kernel label, so that arm never loads the library."""
    if hasattr(case, "slots"):
        return {"workload": case.name, "num_tokens": case.num_tokens, "num_kv_heads": case.key.shape[1],
                "head_dim": case.key.shape[2], "page_size": case.page_size, "in_dtype": case.in_dtype,
                "kv_dtype": case.kv_dtype, "l2": l2_note(args)}
    if hasattr(case, "seg_start"):
        return {"workload": case.name, "n": case.n, "num_heads": case.q.shape[1], "num_kv_heads": case.num_kv_heads,
                "head_dim": case.q.shape[2], "page_size": case.page_size, "topk": case.topk, "bs": case.bs,
                "local": case.local, "dtype": case.dtype, "used_keys": int(case.used.sum()),
                "l2": l2_note(args)}
    if not hasattr(case, "seq_lens"):
        return {"workload": case.name, "n": case.n, "num_heads": case.q.shape[1], "num_kv_heads": case.num_kv_heads,
                "head_dim": case.q.shape[2], "topk": case.topk, "bs": case.bs, "local": case.local,
                "dtype": case.dtype, "used_rows": int(case.used.sum()),
                "l2": l2_note(args)}
    cfg = {"workload": case.name, "batch": case.batch, "sq": case.sq, "num_heads": case.num_heads,
           "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim, "page_size": case.page_size,
           "kv_dtype": case.dtype, "window": case.window, "causal": case.causal,
           "scales": {"q": case.q_scale, "k": case.k_scale, "v": case.v_scale},
           "seq_lens": {"min": int(case.seq_lens.min()), "max": int(case.seq_lens.max()),
                        "total": int(case.seq_lens.sum())},
           "pool_pages": case.num_pages, "l2": l2_note(args) + "; KV stream larger than L2",
           "parallelism": f"replicas{args.gpus}" if args.gpus > 1 else "single",
           "chunk_tokens": effective_chunk(case, args)}
    if gpu_kernel:
        cfg["kernel_path"] = getattr(args, "path", "auto")
        cfg["kernel"] = paged_kernel_name(case, args)
    return cfg


def effective_chunk(case, args) -> int:
    """Split-KV chunk of a run: --chunk if given, else the one the workload's
    configuration fixes, else 0 (the library's plan)."""
    chunk = getattr(args, "chunk", None)
    return int(getattr(case, "chunk_tokens", 0)) if chunk is None else int(chunk)


def paged_flags(case, args, pkd) -> int:
    return (pkd.FLAG_CAUSAL if case.causal else 0) | (pkd.FLAG_FMA if args.path == "fma" else 0) | \
        (pkd.FLAG_GRID if args.grid else 0) | (pkd.FLAG_FLAT if args.flat else 0) | \
        (pkd.FLAG_BALANCED if args.balanced else 0)


def paged_kernel_name(case, args) -> str:
    """The library's own account of the kernel it launches for this workload."""
    import paged_kv_decode_15_gb300 as pkd
    try:
        kv_code = {"bf16": pkd.BF16, "fp16": pkd.FP16, "fp8": pkd.FP8_E4M3}[case.dtype]
        return pkd.kernel_name(case.batch, case.sq, case.num_heads, case.num_kv_heads, case.head_dim,
                               case.page_size, int(case.block_table.shape[1] * case.page_size), kv_code,
                               case.window, effective_chunk(case, args), paged_flags(case, args, pkd))
    except (OSError, RuntimeError) as e:  # library not built on this host
        return f"unknown ({e})"


def l2_note(args) -> str:
    if args.l2_flush == "write-read":
        return "L2 flushed before every timed step: 512 MiB write, then 256 MiB read (clean lines)"
    return "L2 flushed (512 MiB write) before every timed step"


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="pkd", choices=["pkd", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other configurations' timings (run by default with the default workload on 1 GPU)")
    ap.add_argument("--secondary-steps", type=int, default=100)
    ap.add_argument("--chunk", type=int, default=None,
                    help="Split-KV chunk in keys (0 = the library's plan; default: the workload's own, else 0)")
    ap.add_argument("--path", default="auto", choices=["auto", "fma"],
                    help="library default (tensor cores for 16-bit caches) or CUDA cores")
    ap.add_argument("--grid", action="store_true", help="force the chunked grid (one CTA per Split-KV chunk)")
    ap.add_argument("--flat", action="store_true", help="force the persistent flat partition")
    ap.add_argument("--balanced", action="store_true", help="force the persistent per-CTA partition")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one captured call instead of direct calls")
    ap.add_argument("--l2-flush", default="write-read", choices=["write", "write-read"],
                    help="how L2 is evicted before every timed step: a 512 MiB write (it leaves up to an L2 of "
                         "dirty lines whose write-back lands inside the timed step), or that write followed by a "
                         "256 MiB read that leaves L2 holding clean, unrelated lines")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank)), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group(backend="nccl")
        dist = tdist
    case, runner, step_ms, total_ms, e2e_ms, h2d, d2h, clocks = run_gpu(args, rank, world, dist)
    acct = runner.acct
    kind_is_paged = isinstance(runner, PagedRunner)
    if rank == 0:
        peaks = load_peaks()
        steps = args.steps
        gbs = job_throughput(acct["kv"], world, steps, total_ms)
        avg_ms = total_ms / steps
        achieved = acct["total"] / (avg_ms / 1e3) / 1e9
        traffic = profiled_traffic(case.name, paged_kernel_name(case, args) if kind_is_paged else "")
        line = {
            "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(avg_ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": getattr(case, "dtype", getattr(case, "kv_dtype", None)),
            "data": "synthetic", "config": workload_config(case, args),
            "us_per_call": round(avg_ms * 1e3, 2), "us_per_call_median": round(statistics.median(step_ms) * 1e3, 2),
            "pct_of_hbm_peak": round(100 * gbs / world / peaks["hbm_gbs"], 2),
            "pct_of_nominal_hbm": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": acct["total"], "peak_source": peaks["source"],
                         "kernel": runner.kernel},
            "e2e": {"value": round(job_throughput(acct["kv"], world, steps, e2e_ms), 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "us_per_call": round(e2e_ms / steps * 1e3, 2),
                    **({"copy_path_us_per_call": round(args.e2e_copy_ms / steps * 1e3, 2)}
                       if getattr(args, "e2e_copy_ms", None) is not None else {}),
                    "note": ("q, block_table, seq_lens read by the kernels from pinned host memory and out, lse "
                             "written there, in place over the host link (PKD_FLAG_HOST_IO), every step; the KV "
                             "cache is resident device state. copy_path_us_per_call: the same step with one packed "
                             "copy in and one out around a device-memory call")
                    if isinstance(runner, PagedRunner) and getattr(args, "e2e_host_io", False) else
                            ("q, block_table, seq_lens in from pinned host memory (one packed copy), out and lse "
                             "back (one packed copy), every step; the KV cache is resident device state")
                    if isinstance(runner, PagedRunner) else
                            ("key, value, slot_mapping in from pinned host memory; the cache is resident "
                             "device state") if isinstance(runner, CacheWriteRunner) else
                            ("q, block_table, seg_start, used, bias in, out back; the cache is resident device "
                             "state") if isinstance(runner, PagedSegmentRunner) else
                            "q, k, v, used, bias in from pinned host memory and out back, every step"},
            "gpu_launches": steps,
            "launch": getattr(args, "launch_mode", "direct"),
            "clocks": clocks,
        }
        if not args.no_secondary and world == 1 and args.workload == DEFAULT_WORKLOAD:
            del runner
            line["secondary"] = run_secondary(args, peaks["hbm_gbs"])
        if not args.no_cpu_baseline and kind_is_paged:
            line["cpu_baseline"] = cpu_baseline(case)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
