"""Benchmark: paged varlen GQA attention on GB300.

Default workload: long-context sliding-window decode (batch 8, kv_len 6700, window
4096, 32 q / 8 kv heads, head_dim 128, per-head sinks, bf16 KV), the shape the
pages quote decode tokens/s on.  One step is one ``ua_unified_attention`` call (the
split-KV partition kernel plus the merge kernel).  The cache holds several replicas
of the working set on disjoint physical blocks and step i reads replica i mod R, so
consecutive steps never hit L2 (R x algorithmic bytes > 3 x L2).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU fp64 oracle on
the host cores on the same workload instead (a deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import ctypes
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# --------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# The source files each kernel is built from (a recorded ncu traffic figure stays valid
# only while these are unchanged).
KERNEL_SOURCES = {
    "ua_attn_tile_kernel": ["ua_tile.cuh", "ua_tile_d*.cu", "ua_device.cuh", "ua_internal.h"],
    "ua_decode_kernel": ["ua_decode.cuh", "ua_decode_*.cu", "ua_tile.cuh", "ua_device.cuh",
                         "ua_internal.h"],
    "ua_prefill_tm_kernel": ["ua_prefill_tm.cuh", "ua_prefill.cuh", "ua_prefill_d64.cu",
                             "ua_prefill_d128.cu", "ua_device.cuh", "ua_internal.h"],
    "ua_prefill_wide_kernel": ["ua_prefill_wide.cuh", "ua_prefill.cuh", "ua_prefill_d256.cu",
                               "ua_device.cuh", "ua_internal.h"],
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "varlen_gqa_attention_paged_gb300", "csrc")
    files = sorted({f for pat in KERNEL_SOURCES[kernel] for f in glob.glob(os.path.join(csrc, pat))})
    for p in files:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode() + f.read())
    return h.hexdigest()[:16]


def kernel_name(plan, head_dim):
    """The attention kernel a plan launches."""
    if plan["kernel"] in (8, 16):
        return "ua_prefill_tm_kernel" if head_dim <= 128 else "ua_prefill_wide_kernel"
    if plan["kernel"] in (2, 32, 64):
        return "ua_decode_kernel"
    return "ua_attn_tile_kernel"


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d[f"{kernel}/{workload}"]
        if rec.get("source_hash") != kernel_source_hash(kernel):
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the GPU works (start before, stop after)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu=timestamp,{self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        t0, t1 = self.marks.get("timed_start"), self.marks.get("timed_end")
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(ts=ts, sm=float(parts[2]), sm_max=float(parts[3]),
                                 active=parts[5], hw=parts[6], hwt=parts[7], swt=parts[8],
                                 swpc=parts[9]))
            except ValueError:
                continue
        if not rows:
            return None
        window = "timed"
        sel = [r for r in rows if t0 is not None and t0 - 0.03 <= r["ts"] <= t1 + 0.03]
        if not sel:
            sel, window = rows, "whole run"
        reasons = set()
        for r in sel:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swpc", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in sel),
                "sm_max_mhz": max(r["sm_max"] for r in sel), "reasons": sorted(reasons),
                "samples": len(sel), "window": window}


def max_over_ranks(elapsed_ms, world, device):
    """The slowest rank's timed-region length (replicas: each rank runs its own copy)."""
    if world <= 1:
        return float(elapsed_ms)
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step, steps, elapsed_ms, world):
    """Whole-job tokens/s: every rank processes its own steps (weak scaling)."""
    return world * tokens_per_step * steps / (elapsed_ms * 1e-3)


# --------------------------------------------------------------------------- our arm

class Call:
    """Pre-marshalled arguments of ua_unified_attention for one input set on the GPU."""

    def __init__(self, inp, dev, backend="auto", replica=0):
        import varlen_gqa_attention_paged_gb300 as ua
        from varlen_gqa_attention_paged_gb300 import _lib
        self.ua, self.lib = ua, _lib.load()
        self.inp = inp
        self.d = {n: (None if getattr(inp, n) is None else getattr(inp, n).to(dev).contiguous())
                  for n in ("q", "k_cache", "v_cache", "cu_seqlens_q", "seq_lens_k",
                            "block_table", "alibi_slopes", "qq_bias", "sinks")}
        bt = self.d["block_table"]
        self.tables = [bt] if bt.dim() == 2 else [bt[r].contiguous() for r in range(bt.shape[0])]
        self.kv_scale = None
        if inp.spec.kv_dtype == torch.float8_e4m3fn:
            self.kv_scale = torch.tensor([inp.k_scale, inp.v_scale], dtype=torch.float32,
                                         device=dev)
        # per-token fp8 scales keep their strides (V's differ from K's)
        self.tok = [None if t is None else t.to(dev) for t in (inp.k_scale_tok, inp.v_scale_tok)]
        self.out = torch.empty_like(self.d["q"])
        self.backend = ua.BACKENDS[backend]
        self.plan = ua.plan(num_seqs=inp.num_seqs, total_q=inp.total_q,
                            max_seqlen_q=inp.max_seqlen_q, max_seqlen_k=inp.max_seqlen_k,
                            block_size=inp.spec.block_size, num_q_heads=inp.spec.num_q_heads,
                            num_kv_heads=inp.spec.num_kv_heads, head_dim=inp.spec.head_dim,
                            window_left=inp.window_left,
                            kv_dtype=ua._DTYPES[inp.spec.kv_dtype],
                            q_dtype=ua._DTYPES[inp.spec.q_dtype], backend=backend,
                            max_blocks_per_seq=self.tables[0].shape[-1],
                            num_blocks=self.d["k_cache"].shape[0],
                            per_token_scales=inp.k_scale_tok is not None)
        self.shape = ua._shape(self.d["q"], self.d["k_cache"], self.tables[0],
                               self.d["cu_seqlens_q"], inp.max_seqlen_q, inp.max_seqlen_k,
                               self.d["qq_bias"], ua._DTYPES[self.out.dtype], 0, None, None,
                               self.tok[0], self.tok[1])
        p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
        spec = inp.spec
        self.head = [p(self.d["q"]), p(self.d["k_cache"]), p(self.d["v_cache"]), p(self.out),
                     p(self.d["cu_seqlens_q"]), p(self.d["seq_lens_k"])]
        self.table_ptrs = [p(t) for t in self.tables]
        self.tail = [spec.block_size, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                     float(inp.scale), float(inp.softcap), int(inp.window_left),
                     p(self.d["alibi_slopes"]), p(self.d["qq_bias"]), p(self.d["sinks"]),
                     ua._DTYPES[spec.kv_dtype], p(self.kv_scale), self.backend]
        # the split path merges in a second kernel unless its partitions merge in-cluster
        self.launches_per_call = (2 if self.plan["path"] == ua.UA_PATH_SPLIT and
                                  self.plan["cluster_z"] <= 1 else 1)

    def __call__(self, stream, replica=0, events=None):
        if events is not None:
            self.shape.events = ctypes.cast(events, ctypes.c_void_p)
        else:
            self.shape.events = None
        rc = self.lib.ua_unified_attention(*self.head, self.table_ptrs[replica % len(self.tables)],
                                           *self.tail, ctypes.c_void_p(stream.cuda_stream),
                                           ctypes.byref(self.shape))
        if rc != 0:
            raise self.ua.UaError(rc, "ua_unified_attention")


def event_triplets(n):
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for trip in evs:  # torch creates the CUDA event lazily, on its first record
        for e in trip:
            e.record()
    torch.cuda.synchronize()
    arrs = [(ctypes.c_void_p * 3)(*[e.cuda_event for e in trip]) for trip in evs]
    return evs, arrs


def n_replicas(spec):
    """Cache replicas so that R x per-step KV bytes exceed 3 x L2 (bounded)."""
    esz = torch.empty((), dtype=spec.kv_dtype).element_size()
    keys = 0
    for a, kv in spec.seqs:
        lo = 0 if not spec.window else max(0, kv - a - (spec.window - 1))
        keys += kv - lo
    per_step = keys * spec.num_kv_heads * spec.head_dim * esz * 2
    return int(min(64, max(1, math.ceil(3 * L2_BYTES / max(per_step, 1)))))


def measure_workload(spec, dev, stream, steps, warmup, backend="auto"):
    """Device time per call (library events around each kernel, median over calls) and the
    average step of the same calls back to back (events around the whole loop only)."""
    reps = n_replicas(spec)
    inp = W.make(spec, replicas=reps)
    call = Call(inp, dev, backend=backend)
    evs, arrs = event_triplets(steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            call(stream, replica=i)
        torch.cuda.synchronize()
        for i in range(steps):
            call(stream, replica=i, events=arrs[i])
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(steps):
            call(stream, replica=i)
        e1.record(stream)
        torch.cuda.synchronize()
    attn = [evs[i][0].elapsed_time(evs[i][1]) for i in range(steps)]
    total = [evs[i][0].elapsed_time(evs[i][2]) for i in range(steps)]
    return inp, call, reps, attn, total, e0.elapsed_time(e1) / steps


def workload_record(inp, call, reps, attn_ms, total_ms, step_ms, hbm_peak, tc_peak):
    """us_per_call: one call alone (events around it); step_us: the same calls back to back.
    The kernel time behind the roofline fractions is the back-to-back step where a call is
    one kernel launch, else the attention kernel's own events."""
    spec = inp.spec
    med = statistics.median(total_ms)
    kbytes = W.kv_bytes_read(inp)
    flops = W.attention_flops(inp)
    kern_ms = step_ms if call.launches_per_call == 1 else statistics.median(attn_ms)
    rec = {"kernel": kernel_name(call.plan, spec.head_dim),
           "path": "split" if call.plan["path"] == 2 else "2d", "n_part": call.plan["n_part"],
           "kernel_block_m": call.plan["block_m"], "launches_per_call": call.launches_per_call,
           "us_per_call": round(med * 1e3, 2), "step_us": round(step_ms * 1e3, 2),
           "attn_kernel_us": round(kern_ms * 1e3, 2),
           "tokens_per_s": round(inp.total_q / (step_ms * 1e-3), 1),
           "kv_gbs": round(kbytes / (step_ms * 1e-3) / 1e9, 1),
           "hbm_frac": round(kbytes / (kern_ms * 1e-3) / 1e9 / hbm_peak, 4),
           "tflops": round(flops / (step_ms * 1e-3) / 1e12, 2),
           "tensor_frac": round(flops / (kern_ms * 1e-3) / 1e12 / tc_peak, 4),
           "l2": f"{reps} cache replicas rotated"}
    return rec


class Cudart:
    """The few CUDA runtime calls the end-to-end loop issues itself (through ctypes, so no
    framework dispatch sits between the steps)."""

    def __init__(self):
        self.lib = None
        for name in ("libcudart.so.13", "libcudart.so"):
            try:
                self.lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.lib is None:
            raise RuntimeError("libcudart not found")
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        self.lib.cudaMemcpyAsync.argtypes = [vp, vp, sz, ctypes.c_int, vp]
        self.lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
        self.lib.cudaEventRecord.argtypes = [vp, vp]
        self.lib.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
        self.lib.cudaEventDestroy.argtypes = [vp]

    def event(self):
        ev = ctypes.c_void_p()
        assert self.lib.cudaEventCreateWithFlags(ctypes.byref(ev), 2) == 0  # disable timing
        return ev

    def copy(self, dst, src, nbytes, kind, stream):
        assert self.lib.cudaMemcpyAsync(dst, src, nbytes, kind, stream) == 0

    def record(self, ev, stream):
        assert self.lib.cudaEventRecord(ev, stream) == 0

    def wait(self, stream, ev):
        assert self.lib.cudaStreamWaitEvent(stream, ev, 0) == 0


def e2e_pipelined(inp, call, dev, stream, reps, steps):
    """End-to-end steps through the public prepared call, with host buffers.

    A step's inputs (q, cu_seqlens_q, seq_lens_k and the block table of the step's cache
    replica) sit in one pinned host buffer and travel in one host-to-device copy; its
    output comes back in one device-to-host copy into pinned memory.  The input copies,
    the attention calls and the output copies run on three streams, with two device
    buffers used in turn, so step i's input copy and step i-1's output copy overlap step
    i-1's and step i's kernels (one copy stream would queue step i's input behind step
    i-1's output, which waits for step i-1's kernel); events order each buffer's reuse.
    Time: host wall clock from a synchronised start to a synchronised end.
    Returns (milliseconds, host-to-device bytes a step, device-to-host bytes a step)."""
    import varlen_gqa_attention_paged_gb300 as ua
    rt = Cudart()
    tables = [inp.block_table[r] for r in range(reps)] if inp.block_table.dim() == 3 \
        else [inp.block_table]
    pieces = [inp.q, inp.cu_seqlens_q, inp.seq_lens_k, tables[0]]
    sizes = [t.numel() * t.element_size() for t in pieces]
    offs = [0]
    for n in sizes[:-1]:
        offs.append(offs[-1] + (n + 15) // 16 * 16)
    total = offs[-1] + sizes[-1]
    stages = []
    for tb in tables:
        st = torch.empty(total, dtype=torch.uint8).pin_memory()
        for t, o, n in zip([inp.q, inp.cu_seqlens_q, inp.seq_lens_k, tb], offs, sizes):
            st[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        stages.append(st)
    in_stream, out_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ins, outs = ctypes.c_void_p(in_stream.cuda_stream), ctypes.c_void_p(out_stream.cuda_stream)
    ks = ctypes.c_void_p(stream.cuda_stream)
    bufs = []
    for _ in range(2):
        dstage = torch.empty(total, dtype=torch.uint8, device=dev)
        dq = dstage[offs[0]:offs[0] + sizes[0]].view(inp.q.dtype).view(inp.q.shape)
        dcu = dstage[offs[1]:offs[1] + sizes[1]].view(torch.int32)
        dsl = dstage[offs[2]:offs[2] + sizes[2]].view(torch.int32)
        dbt = dstage[offs[3]:offs[3] + sizes[3]].view(torch.int32).view(tables[0].shape)
        dout = torch.empty_like(call.out)
        hout = torch.empty(call.out.shape, dtype=call.out.dtype).pin_memory()
        prep = ua.prepare(dq, call.d["k_cache"], call.d["v_cache"], dcu, dsl, dbt,
                          max_seqlen_q=inp.max_seqlen_q, max_seqlen_k=inp.max_seqlen_k,
                          scale=inp.scale, softcap=inp.softcap, window_left=inp.window_left,
                          alibi_slopes=call.d["alibi_slopes"], qq_bias=call.d["qq_bias"],
                          sinks=call.d["sinks"], kv_scale=call.kv_scale,
                          k_scale_tok=call.tok[0], v_scale_tok=call.tok[1], out=dout,
                          stream=stream)
        bufs.append(dict(dstage=dstage, dout=dout, hout=hout, prep=prep,
                         ev_in=rt.event(), ev_k=rt.event(), ev_out=rt.event(),
                         pd=ctypes.c_void_p(dstage.data_ptr()),
                         po=ctypes.c_void_p(dout.data_ptr()), ph=ctypes.c_void_p(hout.data_ptr())))
    out_bytes = call.out.numel() * call.out.element_size()
    host_ptrs = [ctypes.c_void_p(st.data_ptr()) for st in stages]

    def step(i):
        b = bufs[i & 1]
        if i >= 2:
            rt.wait(ins, b["ev_k"])   # the kernel of step i-2 has read this buffer's inputs
        rt.copy(b["pd"], host_ptrs[i % len(stages)], total, 1, ins)   # host -> device
        rt.record(b["ev_in"], ins)
        rt.wait(ks, b["ev_in"])
        if i >= 2:
            rt.wait(ks, b["ev_out"])  # the copy-out of step i-2 has read this buffer's out
        b["prep"]()
        rt.record(b["ev_k"], ks)
        rt.wait(outs, b["ev_k"])
        rt.copy(b["ph"], b["po"], out_bytes, 2, outs)                  # device -> host
        rt.record(b["ev_out"], outs)

    for i in range(4):  # warm-up
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3
    for b in bufs:  # the last steps' outputs came back intact
        assert torch.isfinite(b["hout"].float()).all()
        for ev in (b["ev_in"], b["ev_k"], b["ev_out"]):
            rt.lib.cudaEventDestroy(ev)
    return ms, total, out_bytes


def run_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)
    hbm_peak, tc_burst, tc_sust, peak_kind = peaks()
    spec = W.WORKLOADS[args.workload]

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    reps = n_replicas(spec)
    inp = W.make(spec, replicas=reps)
    call = Call(inp, dev)
    evs, arrs = event_triplets(args.steps)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(stream, replica=i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark("timed_start")
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            call(stream, replica=i)
        end.record(stream)
    torch.cuda.synchronize()
    sampler.mark("timed_end")
    # Kernel-timing pass: the same K steps again, with the library's events recorded
    # around the attention kernel and the merge kernel of every step.  (Events between
    # the kernels stop them overlapping through programmatic dependent launch, so this
    # pass is kept out of the timed region above.)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            call(stream, replica=i, events=arrs[i])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    attn_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(args.steps)]
    merge_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(args.steps)]

    # end-to-end through the public API with host buffers: each step's inputs travel from
    # pinned host memory and its output comes back, all inside the timed region
    e2e_steps = max(200, min(args.steps, 1000))
    e2e_ms, h2d, d2h = e2e_pipelined(inp, call, dev, stream, reps, e2e_steps)
    clocks = sampler.stop() if rank == 0 else None

    extra = {}
    if rank == 0 and not args.skip_workloads:
        for name in args.workloads.split(","):
            if not name or name == args.workload:
                continue
            try:
                w_inp, w_call, w_reps, a_ms, t_ms, s_ms = measure_workload(
                    W.WORKLOADS[name], dev, stream, steps=args.workload_steps, warmup=3)
                extra[name] = workload_record(w_inp, w_call, w_reps, a_ms, t_ms, s_ms, hbm_peak,
                                              tc_burst)
                del w_inp, w_call
                torch.cuda.empty_cache()
            except Exception as exc:  # a workload that fails is reported, not hidden
                extra[name] = {"error": str(exc)[:200]}

    if rank != 0:
        return
    tokens_per_step = inp.total_q
    value = job_throughput(tokens_per_step, args.steps, elapsed_ms, world)
    # One kernel launch per step: its average duration is the timed region over K steps
    # (launch gaps included).  Two (partition + merge kernel): the partition kernel's own
    # events in the pass after the timed region.
    one_launch = call.launches_per_call == 1
    attn_us = elapsed_ms / args.steps * 1e3 if one_launch else statistics.mean(attn_ms) * 1e3
    kbytes = W.kv_bytes_read(inp)
    flops = W.attention_flops(inp)
    kname = kernel_name(call.plan, spec.head_dim)
    if kname in ("ua_attn_tile_kernel", "ua_decode_kernel"):  # bandwidth-bound: K/V bytes
        achieved = kbytes / (attn_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "algorithmic_bytes_per_launch": kbytes}
    else:  # dense contraction: algorithmic flops, dense bf16 peak (burst: the kernel is timed alone)
        achieved = flops / (attn_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tc_burst,
                "unit": "TFLOP/s", "frac": round(achieved / tc_burst, 4),
                "algorithmic_flops_per_launch": flops}
    cpu = cpu_baseline(inp, budget_s=args.cpu_seconds)
    line = {
        "metric": "decode tokens/s (kernel-level, whole job)",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16"}.get(spec.kv_dtype, "f16 (e4m3 KV)"),
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled block table)",
        "config": workload_config(spec, world),
        "plan": {"path": "split" if call.plan["path"] == 2 else "2d",
                 "n_part": call.plan["n_part"], "kernel_code": call.plan["kernel"]},
        "hbm_gbs": round(kbytes * args.steps / (elapsed_ms * 1e-3) / 1e9, 1),
        "roofline": {**roof,
                     "traffic": recorded_traffic(kname, spec.name), "peak_source": peak_kind,
                     "kernel": kname + (" (split-KV partition)" if call.plan["path"] == 2 else ""),
                     "kernel_us_mean": round(attn_us, 3),
                     "kernel_timing": (
                         "CUDA events around the K timed steps on the launching stream, one "
                         "kernel launch a step (split partitions merged in-cluster): timed "
                         "region / K, launch gaps included" if one_launch else
                         "CUDA events around the attention kernel, every step of a pass of "
                         "the same K steps right after the timed region"),
                     "merge_us_mean": None if one_launch else
                     round(statistics.mean(merge_ms) * 1e3, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * tokens_per_step * e2e_steps / (e2e_ms * 1e-3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "note": "public Python API per step (the prepared call of "
                        "varlen_gqa_attention_paged_gb300.prepare): one pinned H2D of q + "
                        "cu_seqlens_q + seq_lens_k + block table (staged together), the call, "
                        "D2H of out; input and output copies on two copy streams overlap "
                        "the neighbouring steps' kernels (two buffers, events); host wall "
                        "clock between synchronised ends; the KV cache stays resident"},
        "gpu_launches": call.launches_per_call * args.steps,
        "clocks": clocks,
        "workloads": extra,
    }
    print(json.dumps(line), flush=True)


def run_launches(args):
    """warmup + steps calls of the workload on cuda:0, nothing else (for ncu captures)."""
    spec = W.WORKLOADS[args.workload]
    inp = W.make(spec, replicas=n_replicas(spec))
    call = Call(inp, torch.device("cuda", 0), backend=args.backend)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            call(stream, replica=i)
    torch.cuda.synchronize()
    print(json.dumps({"launch_only": spec.name, "calls": args.warmup + args.steps,
                      "plan": call.plan}))


def sample_heads(total_heads, threads, budget_heads):
    """Heads of a CPU sample: a multiple of the thread count (or every head when there are
    fewer heads than threads), within the budget, at least one round."""
    if total_heads <= threads:
        return total_heads
    rounds = max(1, min(total_heads // threads, budget_heads // threads))
    return rounds * threads


def workload_config(spec, world):
    """The `config` of both arms' JSON line: the workload and its input rule."""
    reps = n_replicas(spec)
    return {"workload": spec.name, "desc": spec.desc, "batch": len(spec.seqs),
            "q_len": spec.seqs[0][0], "kv_len": spec.seqs[0][1], "window": spec.window,
            "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads,
            "head_dim": spec.head_dim, "block_size": spec.block_size,
            "l2": f"inputs larger than L2: {reps} cache replicas on disjoint blocks, "
                  f"step i reads replica i mod {reps}",
            "parallelism": f"replicas x{world}"}


def cpu_baseline(inp, budget_s=12.0, sample_seqs=None):
    """The oracle as it stands, on the host cores, over a bounded sample of the workload."""
    import oracle
    threads = os.cpu_count() or 1
    kw = inp.oracle_kwargs()
    total_heads = inp.spec.num_q_heads
    # one sample = every query token of the step for a slice of heads, sized to ~1 s; the
    # oracle runs one head per host thread, so the slice is a whole number of rounds of
    # `threads` heads (no thread idles in a last, partial round)
    t0 = time.time()
    oracle.attention(threads=threads, head_range=(0, 1), **kw)
    one = max(time.time() - t0, 1e-3)
    heads = sample_heads(total_heads, threads, int(1.0 / one) * threads)
    threads = min(threads, heads)
    done_tokens = 0.0
    t0 = time.time()
    reps = 0
    while True:
        oracle.attention(threads=threads, head_range=(0, heads), **kw)
        reps += 1
        done_tokens += inp.total_q * heads / total_heads
        if time.time() - t0 > budget_s or reps >= 1000:
            break
    el = time.time() - t0
    return {"value": round(done_tokens / el, 3), "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{reps} x (all {inp.total_q} query tokens, heads 0..{heads - 1} of "
                      f"{total_heads}) in {el:.1f} s; tokens scaled by heads/{total_heads}"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    spec = W.WORKLOADS[args.workload]
    inp = W.make(spec)
    threads = os.cpu_count() or 1
    kw = inp.oracle_kwargs()
    total_heads = spec.num_q_heads
    t0 = time.time()
    oracle.attention(threads=threads, head_range=(0, 1), **kw)
    one = max(time.time() - t0, 1e-3)
    # each step: all query tokens, a slice of heads sized so K+W steps take ~2 minutes,
    # a whole number of rounds of one head per thread
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    heads = sample_heads(total_heads, threads, int(per_step_budget / one) * threads)
    threads = min(threads, heads)
    for _ in range(args.warmup):
        oracle.attention(threads=threads, head_range=(0, heads), **kw)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.attention(threads=threads, head_range=(0, heads), **kw)
    el = time.time() - t0
    tokens = inp.total_q * heads / total_heads * args.steps
    value = tokens / el
    sample = (f"each step: all {inp.total_q} query tokens x heads 0..{heads - 1} of "
              f"{total_heads}; tokens scaled by heads/{total_heads}")
    line = {"impl": "reference", "metric": "decode tokens/s (kernel-level, whole job)",
            "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) q/k/v, shuffled block table)",
            "config": workload_config(spec, world),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="swdecode_bf16", choices=sorted(W.WORKLOADS))
    ap.add_argument("--workloads", default=",".join(W.WORKLOADS),
                    help="other workloads measured per call and reported under 'workloads'")
    ap.add_argument("--workload-steps", type=int, default=20)
    ap.add_argument("--skip-workloads", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--launch-only", action="store_true",
                    help="only run --warmup + --steps calls of --workload (a small, fixed "
                         "launch sequence for profilers); print nothing else")
    ap.add_argument("--backend", default="auto", choices=["auto", "2d", "split"])
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.launch_only:
        run_launches(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
