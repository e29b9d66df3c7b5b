"""Benchmark of libsar on one GB300 (or N replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-rows] [--rows-only REGEX] [--rows-out PATH]

Workload (a "step"): one sar_allreduce, rsag style, over 8 simulated ranks of
32M fp16 elements (64 MiB) each, values N(0,1) from seed 1 -- reduce every
rank chunk in binary32 in rank order, round once, write to all 8 outputs.
Bytes counted per step: N*S read + N*S written = 1 GiB (GB = 1e9 below).
The working set (1 GiB) is far larger than the 129 MB L2, so no flush is
needed between steps.

stdout: ONE short JSON line, the last line printed.  `value` is whole-job HBM
GB/s over all GPUs (each GPU runs the same workload on its own buffers:
replicas, weak scaling), `e2e` the same metric through the C ABI with the
inputs copied in from pinned host memory and all outputs copied back inside
the timed region (pipelined copies issued eagerly; the fastest of the other
ways is named beside it), `roofline` the dominant kernel's achieved bandwidth
against the measured copy peak, and `cpu_baseline` the CPU oracle timed on a
sample of the same workload.

stderr: one `row: {...}` line per other workload (eager and CUDA-graph
us/call and GB/s), one `oracle_per_config: [...]` line (the oracle on every
measured configuration) and one `e2e_detail: {...}` line; --rows-out writes
the same objects to a JSON file.

--impl reference times the CPU oracle itself on a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

GB = 1e9
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic of one launch of the dominant kernel (rsag fused, fp16, 8 ranks,
# 64 MiB per rank) from one ncu capture with the caches flushed before the
# launch (dram__bytes_read.sum 536,891,648 + dram__bytes_write.sum 485,169,664;
# the rest of the 536.9 MB of outputs is still dirty in L2 when the launch
# ends), valid while the kernel sources hash to `sources_sha`; otherwise
# `traffic` is reported as null.
TRAFFIC = {"sources_sha": "365562bd70618ef1", "bytes_per_launch": 1022055424}
KERNEL_SOURCES = ["allreduce_reduction_rank_gb300/csrc/rsag_kernels.cuh",
                  "allreduce_reduction_rank_gb300/csrc/rsag_fp16.cu",
                  "allreduce_reduction_rank_gb300/csrc/sar_device.cuh"]


def sources_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# Distributed plumbing (host-side only: barrier and max over ranks).
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# Clock sampling during the timed region.
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": inside[0][2],
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# The GPU arm.
# ---------------------------------------------------------------------------
NP_VIEW = {"bf16": np.int16, "fp16": np.int16, "fp32": np.float32, "e4m3fn": np.uint8, "e4m3b15": np.uint8}


def upload(torch, codes, dt, dev):
    return torch.from_numpy(np.ascontiguousarray(codes).view(NP_VIEW[dt])).to(dev)


def time_calls(torch, fn, calls: int, stream) -> float:
    """Average ms per call of `calls` back-to-back calls, CUDA events on `stream`."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(calls):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / calls


def time_graph(torch, fn, calls: int, stream) -> float:
    """Average ms per call with `calls` calls captured into one CUDA graph."""
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(calls):
            fn()
    with torch.cuda.stream(stream):        # replay() launches on the current stream
        graph.replay()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / calls


def rsag_row(torch, sar, wl, dev, stream, l2_bytes, algo=0, calls=20, warm=5, graph=True, ins=None, accum=None):
    ins = ins if ins is not None else wl.inputs()
    din = [upload(torch, x, wl.dtype, dev) for x in ins]
    dout = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    pi, po = [t.data_ptr() for t in din], [t.data_ptr() for t in dout]

    def call():
        if accum is None:
            sar.sar_allreduce(pi, po, count=wl.count, dtype=wl.dtype, algo=algo, stream=stream.cuda_stream)
        else:
            sar.sar_allreduce_accum(pi, po, accum, count=wl.count, dtype=wl.dtype, stream=stream.cuda_stream)

    with torch.cuda.stream(stream):
        for _ in range(warm):
            call()
        eager = time_calls(torch, call, calls, stream)
        g = time_graph(torch, call, calls, stream) if graph else None
    name = ["rsag", "rsag_two_phase", "ll_allpair"][algo] if accum is None else f"rsag, {accum} accumulation"
    row = {"workload": wl.name, "algo": name, "bytes": wl.algo_bytes,
           "eager_us": round(eager * 1e3, 3), "eager_GBps": round(wl.algo_bytes / (eager * 1e-3) / GB, 1),
           "l2_resident": wl.algo_bytes <= l2_bytes}
    if g is not None:
        row["graph_us"] = round(g * 1e3, 3)
        row["graph_GBps"] = round(wl.algo_bytes / (g * 1e-3) / GB, 1)
    if algo == 2:      # the LL rows' check: the outputs equal the rsag allreduce
        want = rsag_result(torch, sar, din, wl, stream)
        row["outputs_ok"] = all(torch.equal(o.view(torch.uint8), want.view(torch.uint8)) for o in dout)
    del din, dout
    if g is not None and algo == 0 and accum is None:
        row["copy_graph_us"] = round(copy_floor_ms(torch, wl.nranks * wl.bytes_per_rank, dev, calls, stream) * 1e3, 3)
    return row


def copy_floor_ms(torch, nbytes: int, dev, calls: int, stream) -> float:
    """Context for a row: a device-to-device copy of the call's N*S bytes (N*S
    read, N*S written, as the allreduce), timed the same way in a CUDA graph
    (torch's same-type contiguous copy_, a cudaMemcpyAsync)."""
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    with torch.cuda.stream(stream):
        dst.copy_(src)
    ms = time_graph(torch, lambda: dst.copy_(src), calls, stream)
    del src, dst
    return ms


def rsag_result(torch, sar, din, wl, stream):
    """The fused rsag allreduce of `din` (bit-exact against the oracle in the
    GPU tests): the value every LL row's outputs must equal."""
    outs = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    sar.sar_allreduce([t.data_ptr() for t in din], [t.data_ptr() for t in outs], count=wl.count, dtype=wl.dtype,
                      stream=stream.cuda_stream)
    stream.synchronize()
    return outs[0]


def ll_row(torch, sar, wl, dev, stream, calls):
    ins = wl.inputs()
    din = [upload(torch, x, wl.dtype, dev) for x in ins]
    dout = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    pk = [torch.zeros(sar.sar_ll_packet_bytes(wl.count, wl.dtype), dtype=torch.uint8, device=dev)
          for _ in range(wl.nranks)]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pi, po, pp = [t.data_ptr() for t in din], [t.data_ptr() for t in dout], [t.data_ptr() for t in pk]
    epoch = [0]

    def call():
        epoch[0] += 1
        sar.sar_allreduce_ll(pi, po, pp, epoch[0], st.data_ptr(), count=wl.count, dtype=wl.dtype,
                             stream=stream.cuda_stream)

    with torch.cuda.stream(stream):
        ms = time_calls(torch, call, calls, stream)
        # CUDA graph: `calls` calls with epochs calls+1 .. 2*calls captured once;
        # a replay re-packs every packet before it is polled, so replays are safe.
        g_ms = time_graph(torch, call, calls, stream)
    ok = sar.sar_read_device_status(st.data_ptr(), stream.cuda_stream) == sar.SAR_OK
    want = rsag_result(torch, sar, din, wl, stream)
    same = all(torch.equal(t, want) for t in dout)
    phys = 6 * wl.nranks * wl.bytes_per_rank
    return {"workload": wl.name, "calls": calls, "epochs": f"1..{calls}", "us_per_call": round(ms * 1e3, 3),
            "GBps": round(wl.algo_bytes / (ms * 1e-3) / GB, 2),
            "physical_GBps": round(phys / (ms * 1e-3) / GB, 2),
            "graph_us_per_call": round(g_ms * 1e3, 3), "graph_GBps": round(wl.algo_bytes / (g_ms * 1e-3) / GB, 2),
            "status_ok": ok, "outputs_ok": same}


def ll_double_row(torch, sar, wl, dev, calls):
    """LL on a double-buffered scratch shared by two streams that run at the
    same time: stream 0 uses odd epochs (the second half), stream 1 even
    epochs (the first half), `calls` calls each; the time is the whole span
    over both streams, reported per call (2 * calls calls)."""
    ins = wl.inputs()
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    din = [upload(torch, x, wl.dtype, dev) for x in ins]
    dout = [[torch.empty_like(din[0]) for _ in range(wl.nranks)] for _ in range(2)]
    nb = sar.ll_double_packet_bytes(wl.count, wl.dtype)
    pk = [torch.zeros(nb, dtype=torch.uint8, device=dev) for _ in range(wl.nranks)]
    st = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in range(2)]
    pi, pp = [t.data_ptr() for t in din], [t.data_ptr() for t in pk]
    po = [[t.data_ptr() for t in dout[s]] for s in range(2)]

    def run(first_epoch):
        for i in range(calls):
            for s in range(2):
                sar.sar_allreduce_ll_double(pi, po[s], pp, first_epoch + 2 * i + s, st[s].data_ptr(),
                                            count=wl.count, dtype=wl.dtype, stream=streams[s].cuda_stream)

    run(1)                                   # warm-up, epochs 1 .. 2 * calls
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(streams[0])
    streams[1].wait_event(start)
    run(2 * calls + 1)
    streams[0].wait_stream(streams[1])
    end.record(streams[0])
    end.synchronize()
    ms = start.elapsed_time(end) / (2 * calls)
    # The same calls captured in one CUDA graph (stream 1 forked from the
    # capturing stream and joined at the end): the GPU time, without the
    # host's issue rate.
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=streams[0]):
        streams[1].wait_stream(streams[0])
        run(4 * calls + 1)
        streams[0].wait_stream(streams[1])
    with torch.cuda.stream(streams[0]):       # replay() launches on the current stream
        graph.replay()
        torch.cuda.synchronize()
        start.record(streams[0])
        graph.replay()
        end.record(streams[0])
    end.synchronize()
    g_ms = start.elapsed_time(end) / (2 * calls)
    del graph
    ok = all(sar.sar_read_device_status(x.data_ptr(), streams[0].cuda_stream) == sar.SAR_OK for x in st)
    want = rsag_result(torch, sar, din, wl, streams[0])
    same = all(torch.equal(dout[s][j], want) for s in range(2) for j in range(wl.nranks))
    return {"workload": wl.name + "_double_two_streams", "calls": 2 * calls, "us_per_call": round(ms * 1e3, 3),
            "GBps": round(wl.algo_bytes / (ms * 1e-3) / GB, 2), "graph_us_per_call": round(g_ms * 1e3, 3),
            "graph_GBps": round(wl.algo_bytes / (g_ms * 1e-3) / GB, 2), "status_ok": ok, "outputs_ok": same}


def ll_fused_row(torch, sar, wl, dev, stream, calls):
    """LL in one cooperative launch: eager with host epochs 1..calls, and a
    CUDA graph of `calls` launches that take their epochs from the device
    epoch counter (so every replay continues the epoch sequence)."""
    ins = wl.inputs()
    din = [upload(torch, x, wl.dtype, dev) for x in ins]
    dout = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    pk = [torch.zeros(sar.sar_ll_packet_bytes(wl.count, wl.dtype), dtype=torch.uint8, device=dev)
          for _ in range(wl.nranks)]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ctrl = torch.zeros(1, dtype=torch.int64, device=dev)
    pi, po, pp = [t.data_ptr() for t in din], [t.data_ptr() for t in dout], [t.data_ptr() for t in pk]
    epoch = [0]

    def host_epoch_call():
        epoch[0] += 1
        sar.sar_allreduce_ll_fused(pi, po, pp, st.data_ptr(), epoch=epoch[0], count=wl.count, dtype=wl.dtype,
                                   stream=stream.cuda_stream)

    def device_epoch_call():
        sar.sar_allreduce_ll_fused(pi, po, pp, st.data_ptr(), epoch_ctrl=ctrl.data_ptr(), count=wl.count,
                                   dtype=wl.dtype, stream=stream.cuda_stream)

    with torch.cuda.stream(stream):
        ms = time_calls(torch, host_epoch_call, calls, stream)
        # continue the epoch sequence on the device after the host epochs
        sar.ll_set_device_epoch(ctrl, epoch[0])
        g_ms = time_graph(torch, device_epoch_call, calls, stream)
    ok = sar.sar_read_device_status(st.data_ptr(), stream.cuda_stream) == sar.SAR_OK
    want = rsag_result(torch, sar, din, wl, stream)
    same = all(torch.equal(t, want) for t in dout)
    return {"workload": wl.name + "_fused", "calls": calls, "us_per_call": round(ms * 1e3, 3),
            "GBps": round(wl.algo_bytes / (ms * 1e-3) / GB, 2),
            "graph_us_per_call": round(g_ms * 1e3, 3), "graph_GBps": round(wl.algo_bytes / (g_ms * 1e-3) / GB, 2),
            "epochs_on_device": sar.ll_device_epoch(ctrl), "status_ok": ok, "outputs_ok": same}


def ll_writeback_row(torch, sar, wl, dev, stream, calls, multi_dest):
    """LL with the write-back as a second packet round (one cooperative
    launch), eager with host epochs and as a CUDA graph with device epochs."""
    ins = wl.inputs()
    din = [upload(torch, x, wl.dtype, dev) for x in ins]
    dout = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    nbp = sar.sar_ll_packet_bytes(wl.count, wl.dtype)
    pk = [torch.zeros(nbp, dtype=torch.uint8, device=dev) for _ in range(wl.nranks)]
    res = torch.zeros(nbp, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ctrl = torch.zeros(1, dtype=torch.int64, device=dev)
    pi, po, pp = [t.data_ptr() for t in din], [t.data_ptr() for t in dout], [t.data_ptr() for t in pk]
    epoch = [0]

    def host_epoch_call():
        epoch[0] += 1
        sar.sar_allreduce_ll_writeback(pi, po, pp, res.data_ptr(), st.data_ptr(), multi_dest=multi_dest,
                                       epoch=epoch[0], count=wl.count, dtype=wl.dtype, stream=stream.cuda_stream)

    def device_epoch_call():
        sar.sar_allreduce_ll_writeback(pi, po, pp, res.data_ptr(), st.data_ptr(), multi_dest=multi_dest,
                                       epoch_ctrl=ctrl.data_ptr(), count=wl.count, dtype=wl.dtype,
                                       stream=stream.cuda_stream)

    with torch.cuda.stream(stream):
        ms = time_calls(torch, host_epoch_call, calls, stream)
        sar.ll_set_device_epoch(ctrl, epoch[0])
        g_ms = time_graph(torch, device_epoch_call, calls, stream)
    ok = sar.sar_read_device_status(st.data_ptr(), stream.cuda_stream) == sar.SAR_OK
    want = rsag_result(torch, sar, din, wl, stream)
    same = all(torch.equal(t, want) for t in dout)
    mode = "multi_dest" if multi_dest else "own_output"
    return {"workload": f"{wl.name}_writeback_{mode}", "calls": calls, "us_per_call": round(ms * 1e3, 3),
            "GBps": round(wl.algo_bytes / (ms * 1e-3) / GB, 2),
            "graph_us_per_call": round(g_ms * 1e3, 3), "graph_GBps": round(wl.algo_bytes / (g_ms * 1e-3) / GB, 2),
            "status_ok": ok, "outputs_ok": same}


def ll_cluster_row(torch, sar, wl, dev, stream, calls):
    """LL through the shared memory of thread-block clusters: eager and a
    CUDA graph of `calls` calls (no epoch or scratch, so the graph replays
    as it is)."""
    ins = wl.inputs()
    din = [upload(torch, x, wl.dtype, dev) for x in ins]
    dout = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pi, po = [t.data_ptr() for t in din], [t.data_ptr() for t in dout]

    def call():
        sar.sar_allreduce_ll_cluster(pi, po, st.data_ptr(), count=wl.count, dtype=wl.dtype, stream=stream.cuda_stream)

    with torch.cuda.stream(stream):
        ms = time_calls(torch, call, calls, stream)
        g_ms = time_graph(torch, call, calls, stream)
    ok = sar.sar_read_device_status(st.data_ptr(), stream.cuda_stream) == sar.SAR_OK
    want = rsag_result(torch, sar, din, wl, stream)
    same = all(torch.equal(t, want) for t in dout)
    return {"workload": wl.name + "_cluster", "calls": calls, "us_per_call": round(ms * 1e3, 3),
            "GBps": round(wl.algo_bytes / (ms * 1e-3) / GB, 2),
            "graph_us_per_call": round(g_ms * 1e3, 3), "graph_GBps": round(wl.algo_bytes / (g_ms * 1e-3) / GB, 2),
            "status_ok": ok, "outputs_ok": same}


def convert_row(torch, sar, dev, stream, count=1 << 26):
    x = torch.randn(count, dtype=torch.float32, device=dev, generator=torch.Generator(device=dev).manual_seed(0))
    y = torch.empty(count, dtype=torch.uint8, device=dev)
    z = torch.empty(count, dtype=torch.float32, device=dev)

    def down():
        sar.sar_fp8_convert(x.data_ptr(), y.data_ptr(), src_dtype="fp32", dst_dtype="e4m3fn", count=count,
                            stream=stream.cuda_stream)

    def up():
        sar.sar_fp8_convert(y.data_ptr(), z.data_ptr(), src_dtype="e4m3fn", dst_dtype="fp32", count=count,
                            stream=stream.cuda_stream)

    with torch.cuda.stream(stream):
        down(); up()
        t_down = time_calls(torch, down, 20, stream)
        t_up = time_calls(torch, up, 20, stream)
    b = count * 5
    return {"workload": f"fp8_convert_{count}", "fp32_to_e4m3fn_us": round(t_down * 1e3, 2),
            "fp32_to_e4m3fn_GBps": round(b / (t_down * 1e-3) / GB, 1),
            "e4m3fn_to_fp32_us": round(t_up * 1e3, 2), "e4m3fn_to_fp32_GBps": round(b / (t_up * 1e-3) / GB, 1)}


def cpu_baseline(ins, wl, budget_s: float = 10.0) -> dict:
    """The oracle as it stands, single-threaded, on a slice of the workload."""
    import oracle
    sample = 1 << 20
    part = [x[:sample] for x in ins]
    runs, t_total = [], 0.0
    while t_total < budget_s or len(runs) < 2:
        t = time.perf_counter()
        oracle.allreduce(part, wl.dtype)
        dt = time.perf_counter() - t
        runs.append(dt)
        t_total += dt
    med = statistics.median(runs)
    bytes_ = 2 * wl.nranks * sample * W.ESIZE[wl.dtype]
    return {"value": round(bytes_ / med / GB, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {sample} elements of each of the {wl.nranks} ranks, median of {len(runs)} runs "
                      f"({t_total:.1f} s)",
            "us_per_call_sample": round(med * 1e6, 1), "host_cpus": os.cpu_count(), "cpu_model": cpu_model(),
            "all_cores": cpu_all_cores(ins, wl)}


def host_threads() -> int:
    """The cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_all_cores(ins, wl, budget_s: float = 5.0, per_thread: int = 1 << 20) -> dict:
    """The same oracle call, unchanged, on disjoint element slices, one thread
    per host core (the C call runs without the GIL).  Context for the
    single-core figure, not a target: every element is still reduced on its
    own, so the slices change nothing but who computes them."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    threads = host_threads()
    total = min(wl.count, per_thread * threads)
    edges = [total * t // threads for t in range(threads + 1)]
    slices = [[x[edges[t]:edges[t + 1]] for x in ins] for t in range(threads) if edges[t + 1] > edges[t]]
    runs, t_total = [], 0.0
    with ThreadPoolExecutor(len(slices)) as ex:
        while t_total < budget_s or len(runs) < 2:
            t = time.perf_counter()
            list(ex.map(lambda part: oracle.allreduce(part, wl.dtype), slices))
            dt = time.perf_counter() - t
            runs.append(dt)
            t_total += dt
    med = statistics.median(runs)
    bytes_ = 2 * wl.nranks * total * W.ESIZE[wl.dtype]
    return {"value": round(bytes_ / med / GB, 4), "cores": len(slices),
            "sample": f"first {total} elements of each rank in {len(slices)} slices, median of {len(runs)} runs"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu-style), or the Arm part number."""
    parts = {"0xd4f": "Neoverse-V2", "0xd40": "Neoverse-V1", "0xd0c": "Neoverse-N1", "0xd49": "Neoverse-N2"}
    try:
        with open("/proc/cpuinfo") as fh:
            info = fh.read()
    except OSError:
        return "unknown"
    for ln in info.splitlines():
        if ln.lower().startswith("model name"):
            return ln.split(":", 1)[1].strip()
    for ln in info.splitlines():
        if ln.startswith("CPU part"):
            part = ln.split(":", 1)[1].strip().lower()
            return parts.get(part, f"Arm part {part}")
    return "unknown"


ORACLE_SAMPLE = 1 << 20


def oracle_per_config(reps: int = 3) -> list:
    """The oracle as it stands, single-threaded, on every measured
    configuration: median of `reps` runs per config, in us per call and GB/s
    under the same byte convention.  Configurations of at most ORACLE_SAMPLE
    elements per rank run whole; larger ones run on their first ORACLE_SAMPLE
    elements of every rank.  LL configurations time the oracle's pack and
    unpack-reduce together."""
    import oracle
    out = []
    for w in [W.C1] + W.C3 + [W.C4, W.C4_B15] + W.C5:
        n = min(w.count, ORACLE_SAMPLE)
        ins = W.sample_inputs(w.dist, w.seed, w.dtype, w.count, w.nranks, np.arange(n, dtype=np.uint64), w.sigma)
        runs = []
        for _ in range(reps):
            t = time.perf_counter()
            if w.algo == "ll":
                rc, _ = oracle.ll_unpack_reduce(oracle.ll_pack(ins, w.dtype, 1), n, w.dtype, 1)
                assert rc == oracle.OK
            else:
                oracle.allreduce(ins, w.dtype)
            runs.append(time.perf_counter() - t)
        med = statistics.median(runs)
        out.append({"workload": w.name, "elements_per_rank": n, "whole": n == w.count,
                    "us_per_call": round(med * 1e6, 1),
                    "GBps": round(2 * w.nranks * n * W.ESIZE[w.dtype] / med / GB, 4)})
    return out


def run_gpu(args, d: Dist) -> None:
    import torch
    import allreduce_reduction_rank_gb300 as sar

    torch.cuda.set_device(d.local)
    dev = torch.device("cuda", d.local)
    stream = torch.cuda.Stream(device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = getattr(props, "L2_cache_size", 0) or (129 << 20)
    peak, peak_kind = measured_peaks()
    wl = WORKLOADS[args.workload]

    ins = wl.inputs()
    din = [upload(torch, x, wl.dtype, dev) for x in ins]
    dout = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    pi, po = [t.data_ptr() for t in din], [t.data_ptr() for t in dout]

    def step():
        sar.sar_allreduce(pi, po, count=wl.count, dtype=wl.dtype, algo=sar.SAR_ALGO_RSAG,
                          stream=stream.cuda_stream)

    clocks = ClockSampler(d.local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        # keep the GPU busy for a moment so the clock samples see it under load
        t_settle = time.time()
        while time.time() - t_settle < args.settle_s:
            step()
            torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        d.barrier()
    clocks.stop()
    ms_total = d.max(start.elapsed_time(end))
    ms_step = ms_total / args.steps
    value = d.world * wl.algo_bytes * args.steps / (ms_total * 1e-3) / GB
    kernel_gbs = wl.algo_bytes / (ms_step * 1e-3) / GB      # one launch per step

    # CUDA graph of the same step
    with torch.cuda.stream(stream):
        g_ms = time_graph(torch, step, min(args.steps, 50), stream)

    # End to end through the C ABI with host buffers: every step copies all
    # inputs in from pinned host memory, runs the allreduce and copies all
    # outputs back.  Pipelined in chunks over three streams (H2D, compute,
    # D2H): chunk c's allreduce runs while chunk c+1 comes in and chunk c-1
    # goes out; the next step's H2D of a chunk waits for this step's compute
    # of it (the inputs are overwritten), and its compute waits for this
    # step's D2H of it (the outputs are overwritten).
    h_in = [torch.from_numpy(x.view(NP_VIEW[wl.dtype])).pin_memory() for x in ins]
    h_out = [torch.empty(wl.count, dtype=din[0].dtype).pin_memory() for _ in range(wl.nranks)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # Two chunks: each chunk costs 2 x N separate copies, and on GB300 (8 x 64
    # MiB fp16) 1, 2, 3, 4, 8, 16 and 32 chunks measured 3.44, 3.34, 3.38,
    # 3.45-3.58, 3.72, 4.12 and 4.18 ms per step against 3.23 ms for the
    # copies alone; consecutive steps overlap anyway (a chunk's next copy in
    # waits only for this step's kernel on it).
    nchunk = 2
    step_c = -(-wl.count // nchunk)
    step_c = -(-step_c // 4096) * 4096
    bounds = [(lo, min(wl.count, lo + step_c)) for lo in range(0, wl.count, step_c)]
    es = din[0].element_size()
    ev_in = [torch.cuda.Event() for _ in bounds]
    ev_c = [torch.cuda.Event() for _ in bounds]
    ev_out = [torch.cuda.Event() for _ in bounds]
    first = [True]

    def e2e_step():
        for c, (lo, hi) in enumerate(bounds):
            if not first[0]:
                s_in.wait_event(ev_c[c])
            with torch.cuda.stream(s_in):
                for h, t in zip(h_in, din):
                    t[lo:hi].copy_(h[lo:hi], non_blocking=True)
                ev_in[c].record(s_in)
            stream.wait_event(ev_in[c])
            if not first[0]:
                stream.wait_event(ev_out[c])
            sar.sar_allreduce([p + lo * es for p in pi], [p + lo * es for p in po], count=hi - lo, dtype=wl.dtype,
                              algo=sar.SAR_ALGO_RSAG, stream=stream.cuda_stream)
            ev_c[c].record(stream)
            s_out.wait_event(ev_c[c])
            with torch.cuda.stream(s_out):
                for h, t in zip(h_out, dout):
                    h[lo:hi].copy_(t[lo:hi], non_blocking=True)
                ev_out[c].record(s_out)
        first[0] = False

    e2e_steps = max(3, min(args.steps, 20))
    e2e_step()
    torch.cuda.synchronize()
    d.barrier()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # best of three trials: a host-side hiccup in one trial stalls the issue of
    # every later copy in it
    eager_ms = float("inf")
    for _ in range(3):
        torch.cuda.synchronize()
        t_start.record(s_in)
        for _ in range(e2e_steps):
            e2e_step()
        t_end.record(s_out)
        t_end.synchronize()
        eager_ms = min(eager_ms, d.max(t_start.elapsed_time(t_end)) / e2e_steps)
    e2e_ok = all(torch.equal(h_out[j], h_out[0]) for j in range(wl.nranks)) and \
        bool(torch.equal(h_out[0].to(dev), dout[0]))

    # The same pipelined steps captured in a CUDA graph (4 steps per graph, so
    # consecutive steps still overlap inside it): no host launch overhead.
    per_graph = 4
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        first[0] = True
        for _ in range(per_graph):
            e2e_step()
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
    for h in h_out:
        h.zero_()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    graph_ok = all(torch.equal(h_out[j].to(dev), dout[0]) for j in range(wl.nranks))
    replays = max(1, e2e_steps // per_graph)
    graph_ms = float("inf")
    for _ in range(3):                       # best of three trials
        with torch.cuda.stream(stream):      # replay() launches on the current stream
            torch.cuda.synchronize()
            t_start.record(stream)
            for _ in range(replays):
                graph.replay()
            t_end.record(stream)
        t_end.synchronize()
        graph_ms = min(graph_ms, d.max(t_start.elapsed_time(t_end)) / (replays * per_graph))
    del graph

    # Zero copy: the kernel reads the pinned host inputs and writes the pinned
    # host outputs itself over the CPU-GPU link (one launch per step).
    hi_p, ho_p = [h.data_ptr() for h in h_in], [h.data_ptr() for h in h_out]

    def zero_copy_step():
        sar.sar_allreduce(hi_p, ho_p, count=wl.count, dtype=wl.dtype, algo=sar.SAR_ALGO_RSAG,
                          stream=stream.cuda_stream)

    for h in h_out:
        h.zero_()
    with torch.cuda.stream(stream):
        zero_copy_step()
        torch.cuda.synchronize()
        zc_ok = all(torch.equal(h_out[j].to(dev), dout[0]) for j in range(wl.nranks))
        zc_ms = min(d.max(time_calls(torch, zero_copy_step, max(3, e2e_steps // 2), stream)) for _ in range(3))
    # Three ways through the C ABI from pinned host buffers: pipelined copies
    # issued eagerly or from a CUDA graph, or the kernel on the host buffers
    # themselves.  Each moves every input in and every output out per step.
    # The headline e2e is the plain way, pipelined copies issued eagerly; the
    # fastest of the three is reported beside it.
    variants = {"pipelined_eager": eager_ms, "pipelined_cuda_graph": graph_ms, "zero_copy_kernel": zc_ms}
    best_variant = min(variants, key=variants.get)
    e2e_ms = eager_ms
    e2e_ok = e2e_ok and graph_ok and zc_ok

    # The platform's ceiling for that traffic: the same pinned copies alone
    # (H2D of all inputs, D2H of all outputs) and both directions at once.
    def copy_ms(direction: str, reps: int = 5) -> float:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(s_in)
        s_out.wait_event(t0)
        for _ in range(reps):
            if direction in ("h2d", "both"):
                with torch.cuda.stream(s_in):
                    for h, t in zip(h_in, din):
                        t.copy_(h, non_blocking=True)
            if direction in ("d2h", "both"):
                with torch.cuda.stream(s_out):
                    for h, t in zip(h_out, dout):
                        h.copy_(t, non_blocking=True)
        s_in.wait_stream(s_out)
        t1.record(s_in)
        t1.synchronize()
        return t0.elapsed_time(t1) / reps

    io_bytes = wl.nranks * wl.bytes_per_rank
    # best of three trials: the host link is shared with the machine's other
    # GPUs, so a single trial can catch a transient slowdown
    h2d_ms = min(copy_ms("h2d") for _ in range(3))
    d2h_ms = min(copy_ms("d2h") for _ in range(3))
    both_ms = min(copy_ms("both") for _ in range(3))
    # A step moves io_bytes each way, so it cannot beat the copies alone by
    # more than noise.  Far faster means the e2e timing itself is wrong (a
    # replay timed on the wrong stream once read 4x too fast): stop.  A little
    # faster is noise on the shared link: keep the number and say so.
    if e2e_ms < 0.5 * both_ms:
        raise RuntimeError(f"e2e step {e2e_ms:.3f} ms beats its own copies ({both_ms:.3f} ms): timing error")
    timing_note = None
    if e2e_ms < 0.9 * both_ms:
        timing_note = (f"e2e step {e2e_ms:.3f} ms is faster than the best of three copy-only trials "
                       f"({both_ms:.3f} ms): the shared host link was slower during the copy trials")
    copy_limits = {"h2d_GBps": round(io_bytes / (h2d_ms * 1e-3) / GB, 1),
                   "d2h_GBps": round(io_bytes / (d2h_ms * 1e-3) / GB, 1),
                   "both_directions_GBps": round(2 * io_bytes / (both_ms * 1e-3) / GB, 1),
                   "both_directions_ms_per_step": round(both_ms, 3),
                   "e2e_vs_copies_alone": round(both_ms / e2e_ms, 3)}
    del h_in, h_out

    e2e = {"value": round(d.world * wl.algo_bytes / (e2e_ms * 1e-3) / GB, 2), "unit": "GB/s",
           "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes, "steps": e2e_steps,
           "ms_per_step": round(e2e_ms, 3), "outputs_identical": e2e_ok,
           "how": (f"pinned host -> {wl.nranks} inputs, sar_allreduce, {wl.nranks} outputs -> pinned host; "
                   f"{len(bounds)} chunks pipelined over 3 streams, eager, best of 3 trials"),
           "best_variant": best_variant,
           "best_value": round(d.world * wl.algo_bytes / (variants[best_variant] * 1e-3) / GB, 2),
           "vs_copies_alone": copy_limits["e2e_vs_copies_alone"]}
    e2e_detail = {"variants_ms_per_step": {k: round(v, 3) for k, v in variants.items()},
                  "copy_limits": copy_limits, "timing_note": timing_note, "zero_copy_outputs_ok": zc_ok,
                  "zero_copy": "sar_allreduce on the pinned host buffers themselves: the kernel's loads and "
                               "stores cross the CPU-GPU link, no copies",
                  "pipelined_cuda_graph": f"the eager pipeline captured {per_graph} steps per CUDA graph"}

    side = {"rows": [], "oracle_per_config": None, "e2e_detail": e2e_detail}
    if d.rank == 0:
        emit_side("e2e_detail", e2e_detail)
    if args.rows and d.rank == 0 and wl is W.C2:
        del din, dout
        torch.cuda.empty_cache()
        c4 = {}

        def c4_ins():
            if "ins" not in c4:
                c4["ins"] = W.C4.inputs()
            return c4["ins"]

        def any_count_row(w):      # any rank count: reuse the 8-rank inputs, draw the ranks past 8
            assert (w.dtype, w.count, w.dist, w.seed, w.sigma) == (wl.dtype, wl.count, wl.dist, wl.seed, wl.sigma)
            extra = [W.rank_input(w.dist, w.seed, w.dtype, w.count, r, w.sigma) for r in range(len(ins), w.nranks)]
            return rsag_row(torch, sar, w, dev, stream, l2_bytes, ins=(list(ins) + extra)[:w.nranks])

        # (row name, thunk): --rows-only selects rows by name
        plan = [(wl.name + "/two_phase", lambda: rsag_row(torch, sar, wl, dev, stream, l2_bytes, algo=1, ins=ins)),
                (W.C1.name, lambda: rsag_row(torch, sar, W.C1, dev, stream, l2_bytes))]
        plan += [(w.name, lambda w=w: rsag_row(torch, sar, w, dev, stream, l2_bytes)) for w in W.C3]
        plan += [(w.name, lambda w=w: any_count_row(w)) for w in W.C6]
        plan.append((W.C4.name, lambda: rsag_row(torch, sar, W.C4, dev, stream, l2_bytes, ins=c4_ins())))
        plan += [(f"{W.C4.name}/acc_{acc}",
                  lambda acc=acc: rsag_row(torch, sar, W.C4, dev, stream, l2_bytes, ins=c4_ins(), accum=acc))
                 for acc in ("e4m3fn", "fp16")]
        plan.append((W.C4_B15.name, lambda: rsag_row(torch, sar, W.C4_B15, dev, stream, l2_bytes)))
        plan += [(w.name, lambda w=w: ll_row(torch, sar, w, dev, stream, W.LL_CALLS)) for w in W.C5]
        plan += [(w.name + "_allpair",
                  lambda w=w: dict(rsag_row(torch, sar, w, dev, stream, l2_bytes, algo=2, calls=W.LL_CALLS),
                                   workload=w.name + "_allpair")) for w in W.C5]
        plan += [(w.name + "_double", lambda w=w: ll_double_row(torch, sar, w, dev, W.LL_CALLS)) for w in W.C5]
        plan += [(w.name + "_fused", lambda w=w: ll_fused_row(torch, sar, w, dev, stream, W.LL_CALLS)) for w in W.C5]
        plan += [(w.name + "_cluster", lambda w=w: ll_cluster_row(torch, sar, w, dev, stream, W.LL_CALLS))
                 for w in W.C5]
        plan += [(f"{w.name}_writeback_{'multi_dest' if m else 'own_output'}",
                  lambda w=w, m=m: ll_writeback_row(torch, sar, w, dev, stream, W.LL_CALLS, m))
                 for w in W.C5 for m in (True, False)]
        plan.append(("fp8_convert", lambda: convert_row(torch, sar, dev, stream)))
        pick = re.compile(args.rows_only) if args.rows_only else None
        for name, run in plan:
            if pick is None or pick.search(name):
                row = run()
                side["rows"].append(row)
                emit_side("row", row)

    cpu = cpu_baseline(ins, wl) if d.rank == 0 and d.world == 1 and args.cpu_baseline else None
    if cpu is not None and wl is W.C2 and args.rows:
        side["oracle_per_config"] = oracle_per_config()
        emit_side("oracle_per_config", side["oracle_per_config"])
    sha = sources_sha()
    traffic = TRAFFIC["bytes_per_launch"] if (TRAFFIC["sources_sha"] == sha and wl is W.C2) else None
    clk = clocks.summary(t0 - args.settle_s - 0.1, t1)
    if d.rank == 0:
        if args.rows_out:
            with open(args.rows_out, "w") as fh:
                json.dump(side, fh, indent=1)
        line = headline(wl, d.world, args, value, ms_step, g_ms, kernel_gbs, peak, peak_kind, traffic, sha, l2_bytes,
                        e2e, clk, cpu)
        sys.stderr.flush()
        print(json.dumps(line, separators=(",", ":")), flush=True)


METRIC = "simulated-allreduce HBM GB/s (% of GB300 peak) and us/call vs message size"
# The headline line stays well under this many characters: a log that keeps
# only the tail of the output must still hold all of it.
HEADLINE_MAX_CHARS = 2048


def emit_side(kind: str, obj) -> None:
    """One line of the side output (stderr): `kind: <json>`."""
    sys.stderr.write(f"{kind}: {json.dumps(obj)}\n")
    sys.stderr.flush()


def headline(wl, world, args, value, ms_step, g_ms, kernel_gbs, peak, peak_kind, traffic, sha, l2_bytes, e2e, clk,
             cpu) -> dict:
    """The one JSON line of our arm (the side output carries the rest)."""
    resident = wl.algo_bytes <= l2_bytes
    return {
        "metric": METRIC,
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "us_per_call": round(ms_step * 1e3, 2),
        "pct_of_peak": round(100 * kernel_gbs / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{wl.dtype} (fp32 accumulate)",
        "data": f"synthetic (seeded splitmix64, {wl.dist}, seed {wl.seed})",
        "config": {"workload": wl.name, "nranks": wl.nranks, "count_per_rank": wl.count,
                   "algo": "rsag (fused reduce + write-back)", "bytes_per_step": wl.algo_bytes,
                   "byte_convention": "N*S read + N*S written",
                   "l2": ("L2-resident: fraction of HBM peak not meaningful" if resident
                          else f"working set {wl.algo_bytes >> 20} MiB > L2 {l2_bytes >> 20} MiB, no flush needed"),
                   "parallelism": f"replicas x{world}"},
        "graph": {"us_per_call": round(g_ms * 1e3, 2), "GBps": round(wl.algo_bytes / (g_ms * 1e-3) / GB, 1)},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": round(kernel_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(kernel_gbs / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": traffic, "kernel": f"rsag_vec_kernel<{wl.dtype},{wl.nranks},fused>",
                     "kernel_sources_sha": sha},
        "clocks": clk,
        "cpu_baseline": cpu,
    }


def run_reference(args, d: Dist) -> None:
    """The CPU oracle as it stands, on a bounded sample of the same workload:
    the first `sample` elements of each rank, with `sample` chosen so that the
    whole --warmup + --steps run takes about a minute of CPU time."""
    if d.rank != 0:
        return
    import oracle
    wl = W.C2
    probe = 1 << 14
    ins = [W.rank_input(wl.dist, wl.seed, wl.dtype, probe, r, wl.sigma) for r in range(wl.nranks)]
    t = time.perf_counter()
    oracle.allreduce(ins, wl.dtype)
    per_elem = max(1e-9, (time.perf_counter() - t) / probe)
    budget_s = 60.0
    sample = int(budget_s / ((args.steps + args.warmup) * per_elem))
    sample = max(probe, min(1 << 20, sample)) // 256 * 256
    ins = [W.rank_input(wl.dist, wl.seed, wl.dtype, sample, r, wl.sigma) for r in range(wl.nranks)]
    for _ in range(args.warmup):
        oracle.allreduce(ins, wl.dtype)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.allreduce(ins, wl.dtype)
    el = time.perf_counter() - t
    bytes_ = 2 * wl.nranks * sample * W.ESIZE[wl.dtype]
    value = bytes_ * args.steps / el / GB
    what = f"first {sample} elements of each of the {wl.nranks} ranks of {wl.name} per step"
    # The GB/s of the sample is the arm's value: the same byte convention, on
    # the first `sample` elements of every rank instead of all of them.
    line = {"impl": "reference", "metric": METRIC,
            "value": round(value, 4), "unit": "GB/s", "n_gpus": d.world, "steps": args.steps,
            "same_config": False, "sample": what,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": wl.name, "nranks": wl.nranks, "count_per_rank": wl.count,
                       "algo": "rsag (oracle: plain rank-ordered sum)", "sample": what},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": what,
                             "cpu_model": cpu_model(), "host_cpus": os.cpu_count()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


WORKLOADS = {w.name: w for w in [W.C1, W.C2, W.C4, W.C4_STRESS, W.C4_B15] + W.C3 + W.C6}


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=W.C2.name,
                    help="rsag workload timed as the step (default: the 8x64MiB fp16 headline)")
    ap.add_argument("--settle-s", type=float, default=0.5,
                    help="seconds of untimed calls before the timed region (clock samples under load)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", dest="rows", action="store_false")
    ap.add_argument("--rows-only", default=None, metavar="REGEX",
                    help="run only the rows whose name matches (for example to profile one kernel)")
    ap.add_argument("--rows-out", default=None, metavar="PATH",
                    help="also write the rows, the oracle per configuration and the e2e detail to this JSON file")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    d = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, d)
        else:
            run_gpu(args, d)
    finally:
        d.close()


if __name__ == "__main__":
    main()
