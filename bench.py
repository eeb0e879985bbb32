#!/usr/bin/env python3
"""Benchmark of the single-GPU MoE expert-parallel permute / unpermute path.

One step = one pass of the whole path over one batch: the dispatch layout with
its expert offsets (one launch), the permute and the combine, all on one stream
with no host synchronisation in between. The metric is source tokens per second,
with the achieved HBM bandwidth (algorithmic bytes / time) against the measured
peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl epd|reference]
                    [--workload dsv3_fp8|prefill_bf16|skew_bf16|tiny|decode_fp8]

The default (dsv3_fp8) line also carries, outside its timed region, one record
per other workload ("configs": prefill, skew, tiny, and decode latency over graph
replays). --impl reference times the CPU oracle (plain single-threaded C) on a
bounded token sample of the same workload. With N > 1 (torchrun) every rank runs
an independent replica on its own GPU; the time is the maximum over ranks.
Prints one JSON line on rank 0.

    python bench.py --record-traffic launches.csv [--traffic-workload W --traffic-tokens T]

writes profiles/ncu_traffic.json from an ncu CSV of dram__bytes_read.sum and
dram__bytes_write.sum per launch (the command is in that file).
"""
from __future__ import annotations

import argparse
import ctypes
import csv
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "permute+unpermute tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
DOM_EVERY = 8  # timed-region steps between two event-bracketed launches of the dominant kernel
CSRC = os.path.join(ROOT, "unpermute_ep_dispatch_gb300", "csrc")
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "ncu_traffic.json")

# launch name -> (kernel-name pattern in ncu's launch list, source files of its device code)
KERNELS = {
    "ep_dispatch_layout_offsets": (r"layout_kernel", ["layout.cu"]),
    "ep_dispatch_layout": (r"layout_kernel", ["layout.cu"]),
    "ep_scan_offsets": (r"scan_kernel", ["scan.cu"]),
    "ep_permute": (r"permute_tma_kernel", ["permute.cu"]),
    "ep_unpermute": (r"unpermute_kernel", ["unpermute.cu"]),
}


# ----------------------------------------------------------------------------- distributed
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of a float over ranks (identity for one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    on = device if (device is not None and dist.get_backend() == "nccl") else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units every rank processed divided by the slowest rank's time."""
    return units_per_rank * world / seconds


# ----------------------------------------------------------------------------- bytes of the path
def algorithmic_bytes(case, P: int, M: int, T_rows=None) -> dict:
    """Minimum HBM bytes of each step: every row read once and written once per
    pick, plus the index, weight and count traffic. T_rows: tokens whose row is
    read by the permute (all of them unless a view leaves some without a pick)."""
    T, H, k, E, R = case.T, case.H, case.k, case.E, case.R
    fp8 = case.dtype == "fp8"
    b = 1 if fp8 else 2
    sc = case.x_scale.shape[1] * 4 if case.x_scale is not None else 0
    Tr = T if T_rows is None else T_rows
    layout = T * k * 8 + T * R + 3 * E * 4
    scan = 2 * E * 4 + 4
    permute = Tr * H * b + Tr * sc + P * H * b + P * sc + T * k * 8 + T * k * 4 + M * 4
    unpermute = P * H * 2 + T * H * 2 + T * k * 4 + T * k * 4
    return dict(ep_dispatch_layout=layout, ep_scan_offsets=scan, ep_permute=permute,
                ep_unpermute=unpermute, ep_dispatch_layout_offsets=layout + scan)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- measured traffic
def _function_bodies(text: str):
    """Text of every __global__ / __device__ function definition in a CUDA source
    (declaration through its matching closing brace), in file order."""
    out = []
    for m in re.finditer(r"^(?:template <[^\n]*>\n)?(?:__global__|__device__|__host__ __device__)"
                         r"[^;{]*\{", text, re.M):
        depth, i = 0, m.end() - 1
        while i < len(text):
            if text[i] == "{":
                depth += 1
            elif text[i] == "}":
                depth -= 1
                if depth == 0:
                    break
            i += 1
        out.append(text[m.start(): i + 1])
    return out


def _function_name(body: str) -> str:
    head = body.split("{", 1)[0]
    m = re.findall(r"(\w+)\s*\(", head)
    return m[-1] if m else ""


def device_code_hash(sources) -> str:
    """Hash of the device code a kernel is built from: the __global__ / __device__
    functions of its source files, and the shared header's device functions that
    they call (directly or through one another). Host-side edits (launch set-up,
    argument checks) and header functions the kernel does not use leave it
    unchanged; any edit of the kernel or of a function it calls changes it."""
    own = []
    for name in sources:
        with open(os.path.join(CSRC, name)) as f:
            own += _function_bodies(f.read())
    with open(os.path.join(CSRC, "epd_common.cuh")) as f:
        shared = [(_function_name(b), b) for b in _function_bodies(f.read())]
    used, todo = set(), list(own)
    while todo:
        text = todo.pop()
        for fn, b in shared:
            if fn not in used and re.search(r"\b" + re.escape(fn) + r"\s*[<(]", text):
                used.add(fn)
                todo += [b2 for fn2, b2 in shared if fn2 == fn]
    h = hashlib.sha256()
    for body in own:
        h.update(body.encode())
    for fn, body in shared:      # file order; overloads share a name
        if fn in used:
            h.update(body.encode())
    return h.hexdigest()[:16]


def profiled_traffic(launch: str, workload: str, units: int):
    """DRAM bytes per launch from the committed ncu record, scaled to `units`
    tokens, or None when there is no record or the kernel's device code changed
    since the counters were taken."""
    try:
        with open(TRAFFIC_JSON) as f:
            e = json.load(f)[launch]
    except Exception:
        return None
    if e.get("device_sha256_16") != device_code_hash(KERNELS[launch][1]):
        return None
    if e.get("workload") != workload:
        return None
    return float(e["dram_bytes_per_launch"]) * units / float(e["tokens"])


_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}


def record_traffic(csv_path: str, workload: str, tokens: int, command: str):
    """profiles/ncu_traffic.json from an ncu CSV (ncu --metrics
    dram__bytes_read.sum,dram__bytes_write.sum --csv): per launch name, the mean of
    read + write bytes over the captured launches of its kernel."""
    per_id = {}
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        mid = row.get("ID")
        if mid is None or row.get("Metric Name") not in ("dram__bytes_read.sum",
                                                         "dram__bytes_write.sum"):
            continue
        v = float(row["Metric Value"].replace(",", "")) * _UNITS.get(row["Metric Unit"], 1.0)
        d = per_id.setdefault(mid, {"kernel": row["Kernel Name"], "bytes": 0.0})
        d["bytes"] += v
    out = {}
    for launch, (pat, srcs) in KERNELS.items():
        got = [d["bytes"] for d in per_id.values() if re.search(pat, d["kernel"])]
        if not got:
            continue
        out[launch] = {"kernel": pat, "sources": srcs, "device_sha256_16": device_code_hash(srcs),
                       "workload": workload, "tokens": tokens, "launches": len(got),
                       "dram_bytes_per_launch": statistics.mean(got),
                       "from": "dram__bytes_read.sum + dram__bytes_write.sum, mean over launches",
                       "command": command}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    return out


# ----------------------------------------------------------------------------- clocks
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x2: "applications_clocks_setting", 0x1: "gpu_idle"}


def _nvml_handle(nv, uuid, index):
    h = ctypes.c_void_p()
    if uuid and nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0:
        return h
    if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0:
        return h
    return None


def _sampler_main(uuid, index, period, stop, conn):
    """Child process: reads SM clock, clock-event reasons and power through NVML
    (read only) every `period` seconds until `stop` is set, then sends the samples
    (monotonic time, MHz, reason bits, W) and the maximum SM clock."""
    samples, max_mhz = [], None
    try:
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() == 0:
            h = _nvml_handle(nv, uuid, index)
            if h is not None:
                mx = ctypes.c_uint()
                if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                    max_mhz = int(mx.value)
                get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                    nv.nvmlDeviceGetCurrentClocksThrottleReasons
                mhz, reasons, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
                conn.send(("ready", max_mhz))
                while not stop.is_set():
                    t = time.monotonic()
                    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                        r = reasons.value if get_reasons(h, ctypes.byref(reasons)) == 0 else 0
                        p = mw.value / 1000.0 if nv.nvmlDeviceGetPowerUsage(
                            h, ctypes.byref(mw)) == 0 else None
                        samples.append((t, int(mhz.value), int(r), p))
                    time.sleep(period)
    except OSError:
        pass
    conn.send(("done", max_mhz, samples))


class ClockSampler:
    """Samples SM clock, power and clock-event reasons through NVML (read only) in a
    child process, so that the samples keep coming while this process launches
    kernels; phases are marked here by time and the samples binned into them."""

    def __init__(self, cuda_index: int, period_s: float = 0.0002):
        self.period = period_s
        self.cuda_index = cuda_index
        self.max_mhz = None
        self.samples = []
        self.marks = []          # (time, phase or None)
        self.phase = None
        self.ok = False
        self._proc = None

    def start(self):
        import multiprocessing as mp
        import torch
        uuid = None
        try:
            u = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
            uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        index = self.cuda_index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            try:
                index = int(vis.split(",")[self.cuda_index])
            except ValueError:
                pass
        ctx = mp.get_context("spawn")
        self._stop = ctx.Event()
        self._conn, child = ctx.Pipe(duplex=False)
        self._proc = ctx.Process(target=_sampler_main,
                                 args=(uuid, index, self.period, self._stop, child), daemon=True)
        self._proc.start()
        if self._conn.poll(60):
            msg = self._conn.recv()
            if msg[0] == "ready":
                self.ok = True
                self.max_mhz = msg[1]
            else:
                self.max_mhz = msg[1]

    def set_phase(self, name):
        self.phase = name
        self.marks.append((time.monotonic(), name))

    def stop(self):
        self.set_phase(None)
        if self._proc is not None:
            self._stop.set()
            if self.ok and self._conn.poll(60):
                msg = self._conn.recv()
                self.samples = msg[2]
            self._proc.join(10)
            self._proc = None

    def _phase_at(self, t):
        ph = None
        for tm, name in self.marks:
            if tm > t:
                break
            ph = name
        return ph

    def summary(self, phase="timed"):
        sam = [s for s in self.samples if self._phase_at(s[0]) == phase]
        if not sam:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "source": "nvml" if self.ok else "unavailable"}
        mhz = [s[1] for s in sam]
        bits = 0
        for s in sam:
            bits |= s[2]
        reasons = sorted(n for b, n in _REASONS.items() if bits & b and n != "gpu_idle")
        powers = [s[3] for s in sam if s[3] is not None]
        return {"sm_mhz": statistics.median(mhz), "sm_min_mhz": min(mhz),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(mhz),
                "power_w_max": max(powers) if powers else None, "source": "nvml"}

    def phases(self):
        names = []
        for _, n in self.marks:
            if n is not None and n not in names:
                names.append(n)
        return {n: self.summary(n) for n in names}


# ----------------------------------------------------------------------------- CPU oracle timing
def time_oracle(name: str, tokens: int, min_seconds: float, max_reps: int = 1000, seed=None):
    """The CPU oracle on a `tokens`-token instance of the workload, repeated until
    min_seconds of work; returns (tokens per second, reps, seconds per rep)."""
    import oracle
    from unpermute_ep_dispatch_gb300 import workloads
    case = workloads.make_case(name, T=tokens, seed=seed)
    args = _oracle_args(case)
    oracle.build()
    oracle.run_path(*args[0], **args[1])          # warm (page in, build)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.run_path(*args[0], **args[1])
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return tokens * reps / el, reps, el / reps


def _oracle_args(case):
    import numpy as np
    import torch

    def u8rows(t):
        t = t.contiguous()
        return t.view(torch.uint8).numpy().reshape(t.shape[0], -1)
    eo = None
    if case.expert_out is not None:
        eo = case.expert_out.contiguous().view(torch.int16).numpy().view(np.uint16)
    xs = None if case.x_scale is None else case.x_scale.numpy()
    return ((u8rows(case.x), xs, case.topk_idx.numpy(), case.topk_weights.numpy(), case.E,
             case.R, case.N), dict(expert_out=eo))


# ----------------------------------------------------------------------------- one workload on the device
class DevicePath:
    """Device-resident inputs and outputs of one workload (allocated once; a step
    allocates nothing) and the launches of one step, in order."""

    def __init__(self, case, dev, stream, align=1, scales="f32", scale_layout="row",
                 view_rank=None, fused=True):
        import torch
        import unpermute_ep_dispatch_gb300 as epd
        self.case, self.dev, self.stream = case, dev, stream
        T, H, k, E, R, N = case.T, case.H, case.k, case.E, case.R, case.N
        self.A = A = max(1, int(align))
        self.M = M = case.capacity if A == 1 else epd.aligned_capacity(T, k, E, A)
        self.fused = fused
        self.topk = case.topk_idx.to(dev)
        self.w = case.topk_weights.to(dev)
        self.x = case.x.to(dev)
        self.xs = None if case.x_scale is None else case.x_scale.to(dev)
        eo = None if case.expert_out is None else case.expert_out.to(dev)
        if eo is not None and M > eo.shape[0]:
            # an aligned layout's expert outputs span every padded row: repeat the seeded rows
            eo = torch.cat([eo, eo[: M - eo.shape[0]]])
        self.eo = eo
        self.ws = epd.new_workspace(T, k, E, R, N, dev)
        self.status = epd.new_status(dev)
        self.per_e = torch.empty(E, dtype=torch.int32, device=dev)
        self.per_r = torch.empty(R, dtype=torch.int32, device=dev)
        self.per_n = torch.empty(N, dtype=torch.int32, device=dev)
        self.itr = torch.empty(T, R, dtype=torch.bool, device=dev)
        self.start = torch.empty(E, dtype=torch.int32, device=dev)
        self.total = torch.empty(1, dtype=torch.int32, device=dev)
        self.out = torch.empty(M, H, dtype=self.x.dtype, device=dev)
        col = scale_layout == "col"
        self.col = col
        # ep_permute_ex adds its column-major scale pass for > 16 words per row over a
        # view of at least a quarter of the experts
        self.scale_pass = (col and self.xs is not None and self.xs.shape[1] > 16
                           and (view_rank is None or 4 * (E // R) >= E))
        self.use_ex = col or scales != "f32" or view_rank is not None
        self.v_begin, self.v_end = 0, E
        if view_rank is not None:
            self.v_begin, self.v_end = view_rank * (E // R), (view_rank + 1) * (E // R)
        if self.xs is None:
            self.out_scale = None
        else:
            C = self.xs.shape[1]
            self.out_scale = torch.empty((C, M) if col else (M, C), dtype=self.xs.dtype,
                                         device=dev)
        self.m_idx = torch.empty(M, dtype=torch.int32, device=dev)
        self.out_idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.io0 = dict(topk=self.topk, w=self.w, x=self.x, xs=self.xs, eo=self.eo, y=self.y)
        self.names = (["ep_dispatch_layout_offsets", "ep_permute", "ep_unpermute"] if fused else
                      ["ep_dispatch_layout", "ep_scan_offsets", "ep_permute", "ep_unpermute"])

    def launches(self, io=None):
        """The step's launches as (name, call) pairs; `io` selects the input / output
        buffers (double-buffered end to end)."""
        import unpermute_ep_dispatch_gb300 as epd
        c, s, A = self.case, self.stream, self.A
        E, R, N = c.E, c.R, c.N
        io = self.io0 if io is None else io
        topk, w, x, xs, eo, y = io["topk"], io["w"], io["x"], io["xs"], io["eo"], io["y"]
        out = []
        if self.fused:
            out.append(("ep_dispatch_layout_offsets", lambda: epd.ep_dispatch_layout_offsets(
                topk, E, R, N, self.ws, self.status, alignment=A, tokens_per_expert=self.per_e,
                tokens_per_rank=self.per_r, tokens_per_rdma_rank=self.per_n,
                is_token_in_rank=self.itr, expert_start_loc=self.start, total_rows=self.total,
                stream=s)))
        else:
            out.append(("ep_dispatch_layout", lambda: epd.ep_dispatch_layout(
                topk, E, R, N, self.ws, self.status, tokens_per_expert=self.per_e,
                tokens_per_rank=self.per_r, tokens_per_rdma_rank=self.per_n,
                is_token_in_rank=self.itr, stream=s)))
            out.append(("ep_scan_offsets", (lambda: epd.ep_scan_offsets(
                self.per_e, self.status, expert_start_loc=self.start, total_rows=self.total,
                stream=s)) if A == 1 else (lambda: epd.ep_scan_offsets_aligned(
                    self.per_e, A, self.status, expert_start_loc=self.start,
                    total_rows=self.total, stream=s))))
        if not self.use_ex:
            out.append(("ep_permute", lambda: epd.ep_permute(
                x, xs, topk, E, self.start, self.ws, self.status, capacity_rows=self.M,
                out=self.out, out_scale=self.out_scale, m_indices=self.m_idx,
                output_index=self.out_idx, stream=s)))
        else:
            out.append(("ep_permute", lambda: epd.ep_permute_ex(
                x, xs, topk, E, self.start, self.ws, self.status, capacity_rows=self.M,
                expert_begin=self.v_begin, expert_end=self.v_end, scale_col_major=self.col,
                scale_ld=self.M if self.col else None, out=self.out, out_scale=self.out_scale,
                m_indices=self.m_idx, output_index=self.out_idx, stream=s)))
        out.append(("ep_unpermute", lambda: epd.ep_unpermute(
            self.out if eo is None else eo, self.out_idx, w, self.status, y=y, stream=s)))
        return out

    def step(self, ev=None, around=None, io=None):
        """One pass of the path; with `ev`, events bracket the launches whose index
        is in `around` (all of them when around is None)."""
        for j, (_, call) in enumerate(self.launches(io)):
            timed = ev is not None and (around is None or j in around)
            if timed:
                ev[2 * j].record(self.stream)
            call()
            if timed:
                ev[2 * j + 1].record(self.stream)

    def valid_pairs(self):
        return int((self.out_idx >= 0).sum().item())

    def bytes(self):
        P = self.valid_pairs()
        T_rows = int((self.out_idx >= 0).any(dim=1).sum().item())
        return algorithmic_bytes(self.case, P, self.M, T_rows)


def _events(n, k=8):
    import torch
    return [[torch.cuda.Event(enable_timing=True) for _ in range(k)] for _ in range(n)]


def chained_launch_us(path, n=16, replays=4):
    """Each launch of the step on its own: n copies captured in one CUDA graph and
    replayed, back to back with their programmatic overlap (as the step runs them);
    mean device time per launch (µs)."""
    import torch
    out = {}
    for name, call in path.launches():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=path.stream):
            for _ in range(n):
                call()
        with torch.cuda.stream(path.stream):
            g.replay()
        torch.cuda.synchronize(path.dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(path.stream):
            a.record(path.stream)
            for _ in range(replays):
                g.replay()
            b.record(path.stream)
        torch.cuda.synchronize(path.dev)
        out[name] = a.elapsed_time(b) * 1e3 / (n * replays)
        del g
    return out


def sets_record(name, dev, stream, sets=4, steps=20, peak=None):
    """The headline step cycling `sets` distinct input and output sets (routing, rows,
    expert outputs, permuted buffer, y): no input is reused within `sets` steps, so
    nothing a step reads can still sit in L2 from the step that last used it."""
    import torch
    import unpermute_ep_dispatch_gb300 as epd
    from unpermute_ep_dispatch_gb300 import workloads
    paths = [DevicePath(workloads.make_case(name, seed=700 + i), dev, stream)
             for i in range(sets)]
    for p in paths:
        p.step()
    filler = torch.empty(1 << 28, dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        filler.fill_(0.0)     # the device stays busy while the first steps are enqueued
    a.record(stream)
    for i in range(steps):
        paths[i % sets].step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    for p in paths:
        epd.check_status(p.status, f"{name} steps over {sets} input sets")
    ms = a.elapsed_time(b) / steps
    byt = paths[0].bytes()
    pb = byt["ep_dispatch_layout_offsets"] + byt["ep_permute"] + byt["ep_unpermute"]
    gbs = pb / (ms * 1e-3) / 1e9
    rec = {"input_sets": sets, "steps": steps, "ms_per_step": round(ms, 5),
           "tokens_per_s": paths[0].case.T / (ms * 1e-3), "path_bytes": pb,
           "path_gbs": round(gbs, 1), "frac": round(gbs / peak, 4) if peak else None,
           "note": f"distinct routing, rows, expert outputs and output buffers cycled every "
                   f"step ({sets} sets)"}
    del paths, filler
    torch.cuda.empty_cache()
    return rec


def config_record(name, dev, stream, steps=20, peak=None):
    """A few timed steps of another workload (outside the headline's timed region):
    ms per step, tokens/s, path GB/s and fraction of the HBM peak."""
    import torch
    import unpermute_ep_dispatch_gb300 as epd
    from unpermute_ep_dispatch_gb300 import workloads
    case = workloads.make_case(name)
    path = DevicePath(case, dev, stream)
    for _ in range(3):
        path.step()
    filler = torch.empty(1 << 28, dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        filler.fill_(0.0)     # the device stays busy while the first steps are enqueued
    a.record(stream)
    for _ in range(steps):
        path.step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    epd.check_status(path.status, f"{name} steps")
    ms = a.elapsed_time(b) / steps
    # the same step captured once in a CUDA graph and replayed: the device time per
    # step without the host's launch cost (which bounds a step that fits in L2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        path.step()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms_graph = a.elapsed_time(b) / steps
    del g, filler
    byt = path.bytes()
    pb = byt["ep_dispatch_layout_offsets"] + byt["ep_permute"] + byt["ep_unpermute"]
    gbs = pb / (ms * 1e-3) / 1e9
    chained = chained_launch_us(path)
    rec = {"tokens": case.T, "hidden": case.H, "top_k": case.k, "experts": case.E,
           "simulated_ranks": case.R, "simulated_rdma_nodes": case.N,
           "rows": "fp8_e4m3 + f32 scale per 128 columns" if case.dtype == "fp8" else "bf16",
           "valid_pairs": path.valid_pairs(), "steps": steps, "ms_per_step": round(ms, 5),
           "ms_per_step_graph": round(ms_graph, 5),
           "tokens_per_s": case.T / (ms * 1e-3), "path_bytes": pb, "path_gbs": round(gbs, 1),
           "frac": round(gbs / peak, 4) if peak else None,
           "launch_us_chained": {k: round(v, 2) for k, v in chained.items()},
           "l2": "no flush" + (f": {pb / 1e6:.0f} MB per step > 129 MB L2" if pb > L2_BYTES
                               else ": the step fits in L2 (latency, not bandwidth)")}
    if name == "skew_bf16":
        cnt = path.per_e.cpu()
        rec["max_expert_share"] = round(float(cnt.max()) / float(cnt.sum()), 4)
        rec["empty_experts"] = int((cnt == 0).sum())
    del path
    torch.cuda.empty_cache()
    return rec


def link_rates(dev, nbytes=1 << 30):
    """Pinned host <-> device copy rates (GB/s) on this machine: each direction alone and
    both at once (two streams), best of three."""
    import torch
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2 = torch.empty(nbytes // 8, dtype=torch.uint8, device=dev)
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(nbytes // 8, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def once(fn):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        fn()
        torch.cuda.synchronize(dev)
        return time.perf_counter() - t0

    def both():
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
    h2d = max(nbytes / once(lambda: d.copy_(h, non_blocking=True)) for _ in range(3)) / 1e9
    d2h = max(nbytes / once(lambda: h.copy_(d, non_blocking=True)) for _ in range(3)) / 1e9
    t_both = min(once(both) for _ in range(3))
    return {"h2d_gbs": round(h2d, 1), "d2h_gbs": round(d2h, 1),
            "h2d_with_d2h_gbs": round(nbytes / t_both / 1e9, 1),
            "d2h_ratio_in_both": 0.125, "bytes": nbytes}


def numa_note(dev):
    """Which host NUMA nodes this process may use and the GPU's node (sysfs)."""
    import glob
    nodes = sorted(os.path.basename(n) for n in glob.glob("/sys/devices/system/node/node*"))
    gpu_node = None
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            gpu_node = int(f.read().strip())
    except Exception:
        pass
    return {"host_nodes": nodes, "gpu_numa_node": gpu_node,
            "cpus_allowed": len(os.sched_getaffinity(0))}


# ----------------------------------------------------------------------------- decode latency
def decode_latency(dev, pool=16, replays=128, mode="dispatch", G=1, warmup=3,
                   clocks=None, steps_timed=None, phase_timed=None, phase_lat=None):
    """Many small independent steps (decode_fp8, T=128): each step's chain is
    captured once in a CUDA graph per input set and replayed, so the per-step time
    carries no host launch cost; `pool` distinct device-resident input sets (seeds
    1000 + i) are cycled. mode: "dispatch" (ep_dispatch: one kernel for a decode
    batch, then ep_unpermute), "fused" (layout with offsets, permute, combine),
    "separate" (layout, offsets, permute, combine), "lowlatency" (ep_dispatch_lowlatency
    fixed rectangles, then the combine over them), "lowlatency_separate".
    Returns (per-step latencies in µs, total ms of the timed replays, bytes, extra)."""
    import torch
    import unpermute_ep_dispatch_gb300 as epd
    from unpermute_ep_dispatch_gb300 import workloads
    ll = mode.startswith("lowlatency")
    cases = [workloads.make_case("decode_fp8", seed=1000 + i, dtype="bf16" if ll else None)
             for i in range(pool)]
    c0 = cases[0]
    T, H, k, E, R, N = c0.T, c0.H, c0.k, c0.E, c0.R, c0.N
    M = T * k
    rows = T  # low-latency rectangles: the worst case, every token on one expert
    stream = torch.cuda.Stream(dev)
    ws = epd.new_workspace(T, k, E, R, N, dev)
    status = epd.new_status(dev)
    o = dict(per_e=torch.empty(E, dtype=torch.int32, device=dev),
             per_r=torch.empty(R, dtype=torch.int32, device=dev),
             per_n=torch.empty(N, dtype=torch.int32, device=dev),
             itr=torch.empty(T, R, dtype=torch.bool, device=dev),
             start=torch.empty(E, dtype=torch.int32, device=dev),
             total=torch.empty(1, dtype=torch.int32, device=dev),
             out=torch.empty(M, H, dtype=c0.x.dtype, device=dev),
             out_scale=torch.empty(M, H // 128, dtype=torch.float32, device=dev),
             m_idx=torch.empty(M, dtype=torch.int32, device=dev),
             out_idx=torch.empty(T, k, dtype=torch.int32, device=dev),
             y=torch.empty(T, H, dtype=torch.bfloat16, device=dev))
    rect = None
    if ll:
        gen = torch.Generator(device=dev)
        gen.manual_seed(99)
        o["q"] = torch.empty(E, rows, H, dtype=torch.float8_e4m3fn, device=dev)
        o["qs"] = torch.empty(E, H // 128, rows, dtype=torch.float32, device=dev)
        o["recv"] = torch.empty(E, dtype=torch.int32, device=dev)
        o["src"] = torch.empty(E, rows, dtype=torch.int32, device=dev)
        # one rectangle buffer reused by every step, as a serving loop does (470 MB of
        # bf16 at decode_fp8: larger than L2 by itself)
        rect = torch.randn(E * rows, H, generator=gen, device=dev).to(torch.bfloat16)
    inputs = [dict(topk=c.topk_idx.to(dev), w=c.topk_weights.to(dev), x=c.x.to(dev),
                   xs=None if c.x_scale is None else c.x_scale.to(dev),
                   eo=rect if ll else c.expert_out.to(dev)) for c in cases]

    def chain(inp):
        if mode == "lowlatency_separate":
            epd.ep_dispatch_layout(inp["topk"], E, R, N, ws, status, tokens_per_expert=o["per_e"],
                                   tokens_per_rank=o["per_r"], tokens_per_rdma_rank=o["per_n"],
                                   is_token_in_rank=o["itr"], stream=stream)
            epd.ep_permute_lowlatency(inp["x"], inp["topk"], E, rows, ws, status, out_q=o["q"],
                                      out_scale=o["qs"], recv_count=o["recv"],
                                      output_index=o["out_idx"], src_token=o["src"],
                                      stream=stream)
        elif mode == "lowlatency":
            epd.ep_dispatch_lowlatency(inp["x"], inp["topk"], E, R, N, rows, ws, status,
                                       out_q=o["q"], out_scale=o["qs"], recv_count=o["recv"],
                                       output_index=o["out_idx"], src_token=o["src"],
                                       stream=stream)
        elif mode == "dispatch":
            epd.ep_dispatch(inp["x"], inp["xs"], inp["topk"], E, R, N, ws, status,
                            capacity_rows=M, tokens_per_expert=o["per_e"],
                            tokens_per_rank=o["per_r"], tokens_per_rdma_rank=o["per_n"],
                            is_token_in_rank=o["itr"], expert_start_loc=o["start"],
                            total_rows=o["total"], out=o["out"], out_scale=o["out_scale"],
                            m_indices=o["m_idx"], output_index=o["out_idx"], stream=stream)
        else:
            if mode == "separate":
                epd.ep_dispatch_layout(inp["topk"], E, R, N, ws, status,
                                       tokens_per_expert=o["per_e"], tokens_per_rank=o["per_r"],
                                       tokens_per_rdma_rank=o["per_n"],
                                       is_token_in_rank=o["itr"], stream=stream)
                epd.ep_scan_offsets(o["per_e"], status, expert_start_loc=o["start"],
                                    total_rows=o["total"], stream=stream)
            else:
                epd.ep_dispatch_layout_offsets(inp["topk"], E, R, N, ws, status,
                                               tokens_per_expert=o["per_e"],
                                               tokens_per_rank=o["per_r"],
                                               tokens_per_rdma_rank=o["per_n"],
                                               is_token_in_rank=o["itr"],
                                               expert_start_loc=o["start"],
                                               total_rows=o["total"], stream=stream)
            epd.ep_permute(inp["x"], inp["xs"], inp["topk"], E, o["start"], ws, status,
                           capacity_rows=M, out=o["out"], out_scale=o["out_scale"],
                           m_indices=o["m_idx"], output_index=o["out_idx"], stream=stream)
        epd.ep_unpermute(inp["eo"], o["out_idx"], inp["w"], status, y=o["y"], stream=stream)

    for inp in inputs:                       # attributes set, caches warm
        chain(inp)
    torch.cuda.synchronize(dev)
    graphs = []
    for gi in range(len(inputs)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(G):
                chain(inputs[(gi * G + j) % len(inputs)])
        graphs.append(g)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize(dev)
    epd.check_status(status, "decode warm-up")
    n_rep = replays if steps_timed is None else steps_timed // G
    outer = clocks.phase if clocks is not None else None
    if clocks is not None and phase_timed is not None:
        clocks.set_phase(phase_timed)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for i in range(n_rep):
            graphs[i % len(graphs)].replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    total_ms = a.elapsed_time(b)
    # per-step latency: every replay bracketed by events (divided by its G steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(replays)]
    if clocks is not None:
        clocks.set_phase(phase_lat if phase_lat is not None else outer)
    with torch.cuda.stream(stream):
        for i in range(replays):
            ev[i][0].record(stream)
            graphs[i % len(graphs)].replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if clocks is not None:
        clocks.set_phase(outer)
    epd.check_status(status, "decode steps")
    lat = sorted(e0.elapsed_time(e1) * 1e3 / G for e0, e1 in ev)
    P = int((o["out_idx"] >= 0).sum().item())
    bytes_k = algorithmic_bytes(c0, P, M)
    if ll:  # no offset scan; the permute reads bf16 rows and writes e4m3 rows + scales
        bytes_k.pop("ep_scan_offsets")
        bytes_k["ep_permute"] = (T * H * 2 + P * H + P * (H // 128) * 4 + T * k * 16 + E * 4
                                 + P * 4)
    path_bytes = (bytes_k["ep_dispatch_layout"] + bytes_k.get("ep_scan_offsets", 0)
                  + bytes_k["ep_permute"] + bytes_k["ep_unpermute"])
    del graphs
    return lat, total_ms, n_rep * G, path_bytes, dict(T=T, H=H, k=k, E=E, R=R, N=N, P=P,
                                                      rows=rows if ll else None)


def latency_stats(lat):
    return {"mean": round(statistics.mean(lat), 3), "p50": round(lat[len(lat) // 2], 3),
            "p99": round(lat[min(len(lat) - 1, int(0.99 * len(lat)))], 3),
            "min": round(lat[0], 3), "replays": len(lat)}


DECODE_PATH = {
    "dispatch": "ep_dispatch (layout, offsets, permute: one kernel) -> combine",
    "fused": "layout with offsets -> permute -> combine",
    "separate": "layout -> offsets -> permute -> combine",
    "lowlatency": "ep_dispatch_lowlatency (fixed rectangles, bf16->e4m3 cast: one kernel) "
                  "-> combine",
    "lowlatency_separate": "layout -> fixed-rectangle permute with bf16->e4m3 cast -> combine",
}


# ----------------------------------------------------------------------------- the GPU arm
def run_epd(args, rank, world, local):
    import torch
    import unpermute_ep_dispatch_gb300 as epd
    from unpermute_ep_dispatch_gb300 import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist(world, "nccl")
    epd.load_library()
    name = args.workload
    case = workloads.make_case(name, T=args.tokens, scales=args.scales)
    T, H, k, E, R, N = case.T, case.H, case.k, case.E, case.R, case.N
    stream = torch.cuda.Stream(dev)
    fused = not args.separate_offsets  # steps 1 and 2 in one launch
    path = DevicePath(case, dev, stream, align=args.align, scales=args.scales,
                      scale_layout=args.scale_layout, view_rank=args.view_rank, fused=fused)
    M, A = path.M, path.A
    torch.cuda.synchronize(dev)
    peak, peak_src = load_peaks()
    clocks = ClockSampler(local, args.clock_period_ms * 1e-3)
    clocks.start()

    for _ in range(args.warmup):
        path.step()
    torch.cuda.synchronize(dev)
    epd.check_status(path.status, "warm-up")
    names = path.names
    bytes_k = path.bytes()
    # the dominant kernel by algorithmic bytes carries events inside the timed region;
    # events around every kernel would break the launch overlap between them
    dom = max(names, key=lambda n: bytes_k[n])
    dom_j = names.index(dom)

    evs = _events(args.steps)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    filler = torch.empty(1 << 28, dtype=torch.float32, device=dev)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    # ~150 us of device work queued ahead of the region's start event, so the device
    # is still busy while this thread enqueues the first steps: the region then times
    # the K steps, not the host's first launches (its time on the device is excluded)
    with torch.cuda.stream(stream):
        filler.fill_(0.0)
    clocks.set_phase("timed")
    t_start.record(stream)
    for i in range(args.steps):
        # events around the dominant kernel on every DOM_EVERY-th step: events block the
        # launch overlap between kernels, so bracketing every step would slow the step
        path.step(evs[i], around=(dom_j,) if i % DOM_EVERY == 0 else ())
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks.set_phase(None)
    barrier(world, dev)
    del filler
    epd.check_status(path.status, "timed steps")
    ms_local = t_start.elapsed_time(t_end)
    ms = reduce_max(ms_local, world, dev)
    dom_ms = statistics.mean(evs[i][2 * dom_j].elapsed_time(evs[i][2 * dom_j + 1])
                             for i in range(0, args.steps, DOM_EVERY))

    # per-kernel breakdown outside the timed region: a pass with events around every
    # launch, and each launch on its own, chained in a CUDA graph
    clocks.set_phase("kernels")
    n_prof = max(3, min(args.steps, 50))
    evp = _events(n_prof)
    torch.cuda.synchronize(dev)
    for i in range(n_prof):
        path.step(evp[i])
    torch.cuda.synchronize(dev)
    per_kernel_ms = {n: statistics.mean(e[2 * j].elapsed_time(e[2 * j + 1]) for e in evp)
                     for j, n in enumerate(names)}
    chained = chained_launch_us(path)
    clocks.set_phase(None)
    evented_dom_ms = per_kernel_ms[dom]
    per_kernel_ms[dom] = dom_ms

    # ---- end to end through the public API: host inputs in, host result out, every step
    e2e = None
    if not args.no_e2e:
        clocks.set_phase("e2e")
        e2e = run_e2e(path, args, world, dev)
        clocks.set_phase(None)
        epd.check_status(path.status, "e2e steps")

    # ---- roofline of the dominant kernel and of the whole path
    achieved = bytes_k[dom] / (per_kernel_ms[dom] * 1e-3) / 1e9
    ms_per_step = ms / args.steps
    P = path.valid_pairs()
    path_bytes = sum(bytes_k[n] for n in names)
    path_gbs = path_bytes / (ms_per_step * 1e-3) / 1e9
    kernels = {}
    for n in names:
        us = per_kernel_ms[n] * 1e3
        rec = {"us": round(us, 2), "us_evented": round(
            evented_dom_ms * 1e3 if n == dom else us, 2), "us_chained": round(chained[n], 2),
            "bytes": bytes_k[n], "gbs": round(bytes_k[n] / (us * 1e-6) / 1e9, 1),
            "frac": round(bytes_k[n] / (us * 1e-6) / 1e9 / peak, 4)}
        tr = profiled_traffic(n, name, T) if A == 1 and not path.use_ex else None
        rec["traffic"] = tr
        rec["traffic_over_algorithmic"] = None if tr is None else round(tr / bytes_k[n], 4)
        kernels[n] = rec
    dom_traffic = kernels[dom]["traffic"]

    result = {
        "metric": METRIC,
        "value": whole_job_rate(T * args.steps, world, ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded routing, rows and expert outputs; no dataset)",
        "config": {"workload": name, "tokens": T, "hidden": H, "top_k": k, "experts": E,
                   "simulated_ranks": R, "simulated_rdma_nodes": N,
                   "rows": "fp8_e4m3 + f32 scale per 128 columns" if case.dtype == "fp8"
                   else "bf16",
                   "expert_out": "bf16 identity (permuted rows)" if path.eo is None
                   else "bf16 seeded",
                   "capacity_rows": M, "valid_pairs": P, "expert_alignment": A,
                   "scales": args.scales if case.dtype == "fp8" else None,
                   "scale_layout": args.scale_layout if case.dtype == "fp8" else None,
                   "experts_in_view": [path.v_begin, path.v_end],
                   "launches": "layout+offsets fused, permute, combine" if fused else
                               "layout, offsets, permute, combine",
                   "l2": f"no flush: {path_bytes / 1e6:.0f} MB moved per step > 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "hbm": {"path_gbs": round(path_gbs, 1), "path_bytes": path_bytes,
                "frac": round(path_gbs / peak, 4), "peak_gbs": peak, "peak_source": peak_src},
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": dom_traffic, "algorithmic_bytes": bytes_k[dom],
                     "traffic_over_algorithmic": kernels[dom]["traffic_over_algorithmic"],
                     "peak_source": peak_src},
        "kernels": kernels,
        "kernels_note": f"us: {dom} timed inside the timed region (events on every "
                        f"{DOM_EVERY}th step), the others from a separate {n_prof}-step pass "
                        "with events around every launch (us_evented; events break the "
                        "programmatic overlap between launches); us_chained: 16 copies of the "
                        "launch alone in one CUDA graph, per launch; traffic: ncu DRAM "
                        "read + write per launch (profiles/ncu_traffic.json), null when the "
                        "kernel's device code changed since",
        # column-major scales add the scale pass after the row copy (inside ep_permute_ex)
        # every rank's kernels in the timed region (the job's total, like value)
        "gpu_launches": (len(names) + (1 if path.scale_pass else 0)) * args.steps * world,
        "e2e": e2e,
    }
    if name == "dsv3_fp8" and not args.no_configs and args.tokens is None and A == 1 \
            and not path.use_ex and fused:
        del path
        torch.cuda.empty_cache()
        clocks.set_phase("configs")
        configs = {}
        configs["dsv3_fp8_4_sets"] = sets_record("dsv3_fp8", dev, stream, sets=4, steps=20,
                                                 peak=peak)
        for other, st in (("prefill_bf16", 20), ("skew_bf16", 10), ("tiny", 50)):
            configs[other] = config_record(other, dev, stream, steps=st, peak=peak)
        lat, tot_ms, n_steps, pb, info = decode_latency(dev, pool=16, replays=128,
                                                        mode="dispatch", clocks=clocks)
        clocks.set_phase(None)
        configs["decode_fp8"] = {
            "tokens": info["T"], "hidden": info["H"], "top_k": info["k"],
            "experts": info["E"], "simulated_ranks": info["R"],
            "simulated_rdma_nodes": info["N"], "path": DECODE_PATH["dispatch"],
            "latency_us": latency_stats(lat),
            "tokens_per_s": info["T"] * n_steps / (tot_ms * 1e-3),
            "ms_per_step": round(tot_ms / n_steps, 5), "path_bytes": pb,
            "input_sets": 16, "launch": "one CUDA graph per input set, replayed",
            "l2": "no flush: 16 input sets cycled (~250 MB), each step's inputs read from "
                  "HBM once the pool exceeds the 129 MB L2"}
        result["configs"] = configs
    clocks.stop()
    result["clocks"] = clocks.summary("timed")
    result["clocks_phases"] = clocks.phases()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, reps, sec = time_oracle(name, args.cpu_tokens, args.cpu_seconds)
        result["cpu_baseline"] = {
            "value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{name} routing at T={args.cpu_tokens} tokens (same H, k, E, R, N), "
                      f"{reps} full-path reps in {reps * sec:.1f} s, single-threaded C"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(path, args, world, dev):
    """The step end to end through the binding: every step copies its inputs host ->
    device from pinned memory and reads y back. Pipelined over two buffer sets:
    step i+1's inputs go host -> device on a copy stream while step i computes, and
    step i's result comes back on a third stream."""
    import torch
    case = path.case
    T, H = case.T, case.H
    pin = lambda t: None if t is None else t.contiguous().pin_memory()  # noqa: E731
    h_topk, h_w, h_x, h_xs, h_eo = (pin(case.topk_idx), pin(case.topk_weights), pin(case.x),
                                    pin(case.x_scale),
                                    None if path.eo is None else pin(path.eo.cpu()))
    h_y = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_topk, h_w, h_x, h_xs, h_eo)
              if t is not None)
    d2h = h_y.numel() * h_y.element_size()

    def clone(t):
        return None if t is None else torch.empty_like(t)
    io0 = path.io0
    ios = [io0, dict(topk=clone(io0["topk"]), w=clone(io0["w"]), x=clone(io0["x"]),
                     xs=clone(io0["xs"]), eo=clone(io0["eo"]), y=clone(io0["y"]))]
    h_ys = [h_y, torch.empty_like(h_y).pin_memory()]
    stream = path.stream
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n, start_ev=None, end_ev=None):
        if start_ev is not None:
            start_ev.record(stream)
            cin.wait_event(start_ev)
            cout.wait_event(start_ev)
        for i in range(n):
            bi = i % 2
            io = ios[bi]
            if i >= 2:
                cin.wait_event(free[bi])    # step i-2 consumed these inputs, y read back
            with torch.cuda.stream(cin):
                io["topk"].copy_(h_topk, non_blocking=True)
                io["w"].copy_(h_w, non_blocking=True)
                io["x"].copy_(h_x, non_blocking=True)
                if io["xs"] is not None:
                    io["xs"].copy_(h_xs, non_blocking=True)
                if io["eo"] is not None:
                    io["eo"].copy_(h_eo, non_blocking=True)
                ready[bi].record(cin)
            stream.wait_event(ready[bi])
            path.step(io=io)
            done[bi].record(stream)
            cout.wait_event(done[bi])
            with torch.cuda.stream(cout):
                h_ys[bi].copy_(io["y"], non_blocking=True)
                free[bi].record(cout)
        if end_ev is not None:
            stream.wait_stream(cout)
            stream.wait_stream(cin)
            end_ev.record(stream)

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 50))
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    e2e_run(e2e_steps, a, b)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(a.elapsed_time(b), world, dev) / e2e_steps
    links = link_rates(dev)
    # the floor: the host link moves h2d and d2h bytes at the rates measured with both
    # directions busy; the kernels run under the copies
    floor_ms = max(h2d / (links["h2d_with_d2h_gbs"] * 1e9),
                   d2h / (links["d2h_gbs"] * 1e9)) * 1e3
    return {"value": whole_job_rate(T, world, e2e_ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
            "ms_per_step": e2e_ms, "floor_ms_per_step": round(floor_ms, 4),
            "over_floor": round(e2e_ms / floor_ms, 4), "link": links, "numa": numa_note(dev),
            "note": "copies of step i+1 / read-back of step i overlap step i's kernels; the "
                    "floor is the step's host->device bytes at the copy rate measured in this "
                    "run with a device->host copy running beside it"}


# ----------------------------------------------------------------------------- decode: graph-captured steps
def run_decode(args, rank, world, local):
    """The decode workload as the headline: many small independent steps (T=128),
    graph-captured, per-step latency and throughput."""
    import torch
    import unpermute_ep_dispatch_gb300 as epd

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist(world, "nccl")
    epd.load_library()
    mode = ("lowlatency_separate" if args.lowlatency and args.separate_offsets else
            "lowlatency" if args.lowlatency else "dispatch" if args.dispatch else
            "separate" if args.separate_offsets else "fused")
    G = max(1, int(args.steps_per_graph))  # consecutive steps (input sets) per graph
    if args.steps % G:
        raise SystemExit(f"--steps {args.steps} is not a multiple of --steps-per-graph {G}")
    clocks = ClockSampler(local, args.clock_period_ms * 1e-3)
    clocks.start()
    barrier(world, dev)
    lat, tot_ms, n_steps, path_bytes, info = decode_latency(
        dev, pool=args.decode_pool, replays=max(64, args.steps // G), mode=mode, G=G,
        warmup=args.warmup, clocks=clocks, steps_timed=args.steps, phase_timed="timed",
        phase_lat="latency")
    clocks.stop()
    barrier(world, dev)
    ms = reduce_max(tot_ms, world, dev)
    T, H, k, E, R, N = info["T"], info["H"], info["k"], info["E"], info["R"], info["N"]
    peak, peak_src = load_peaks()
    ms_per_step = ms / n_steps
    ll = mode.startswith("lowlatency")
    result = {
        "metric": METRIC,
        "value": whole_job_rate(T * n_steps, world, ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": n_steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded routing, rows and expert outputs; no dataset)",
        "config": {"workload": "decode_fp8" + ("_lowlatency" if ll else ""), "tokens": T,
                   "hidden": H, "top_k": k, "experts": E, "path": DECODE_PATH[mode],
                   "rows_per_expert": info["rows"], "simulated_ranks": R,
                   "simulated_rdma_nodes": N,
                   "rows": "fp8_e4m3 + f32 scale per 128 columns", "expert_out": "bf16 seeded",
                   "input_sets": args.decode_pool,
                   "launch": (f"CUDA graphs of {G} consecutive steps (input sets), replayed"
                              if G > 1 else "one CUDA graph per input set, replayed"),
                   "l2": f"no flush: {args.decode_pool} input sets cycled, each step's inputs "
                         "read from HBM once the pool exceeds the 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "latency_us": dict(latency_stats(lat), note="per step: events around each replay" +
                           (f", divided by its {G} steps" if G > 1 else "")),
        "hbm": {"path_gbs": round(path_bytes / (ms_per_step * 1e-3) / 1e9, 1),
                "path_bytes": path_bytes, "peak_gbs": peak, "peak_source": peak_src},
        "roofline": {"kernel": "whole step", "bound": "hbm",
                     "achieved": round(path_bytes / (ms_per_step * 1e-3) / 1e9, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(path_bytes / (ms_per_step * 1e-3) / 1e9 / peak, 4),
                     "traffic": None, "algorithmic_bytes": path_bytes,
                     "note": "latency-bound at this size: the step's bytes over its time"},
        "gpu_launches": {"lowlatency_separate": 3, "lowlatency": 2, "dispatch": 2,
                         "separate": 4, "fused": 3}[mode] * n_steps * world,
        "clocks": clocks.summary("timed"),
        "clocks_phases": clocks.phases(),
        "e2e": None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not ll:
        v, reps, sec = time_oracle("decode_fp8", T, args.cpu_seconds, seed=1000)
        result["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                  "sample": f"decode_fp8 step of T={T}, {reps} reps in "
                                            f"{reps * sec:.1f} s, single-threaded C"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- the reference arm
def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: rank 0 only; other ranks exit at once."""
    if rank != 0:
        return
    import oracle
    from unpermute_ep_dispatch_gb300 import workloads
    name = args.workload
    cfg = workloads.CONFIGS[name]
    T_s = args.cpu_tokens
    case = workloads.make_case(name, T=T_s)
    a, kw = _oracle_args(case)
    oracle.build()
    for _ in range(args.warmup):
        oracle.run_path(*a, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_path(*a, **kw)
    el = time.perf_counter() - t0
    v = T_s * args.steps / el
    result = {
        "impl": "reference",
        "metric": METRIC,
        "value": v,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded routing, rows and expert outputs; no dataset)",
        "config": {"workload": name, "tokens": args.tokens or cfg["T"], "hidden": cfg["H"],
                   "top_k": cfg["k"], "experts": cfg["E"], "simulated_ranks": cfg["R"],
                   "simulated_rdma_nodes": cfg["N"], "parallelism": "CPU, 1 thread"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{name} routing at T={T_s} tokens per step (same H, k, E, "
                                   f"R, N), single-threaded C oracle"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["epd", "reference"], default="epd")
    ap.add_argument("--workload", default="dsv3_fp8")
    ap.add_argument("--tokens", type=int, default=None, help="override T (smaller instances)")
    ap.add_argument("--cpu-tokens", type=int, default=1024)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' records on the dsv3_fp8 line")
    ap.add_argument("--align", type=int, default=1,
                    help="pad every expert's rows to a multiple of this (grouped-GEMM layout)")
    ap.add_argument("--scales", choices=["f32", "ue8m0"], default="f32",
                    help="fp8 scale words: fp32 per 128 columns, or UE8M0 exponents packed by 4")
    ap.add_argument("--scale-layout", choices=["row", "col"], default="row",
                    help="permuted scales row-major [M, C] or column-major [C, M]")
    ap.add_argument("--view-rank", type=int, default=None,
                    help="permute only this simulated rank's experts (local rows and ids)")
    ap.add_argument("--separate-offsets", action="store_true",
                    help="run ep_dispatch_layout and ep_scan_offsets as two launches (with "
                         "--lowlatency: the layout, then ep_permute_lowlatency)")
    ap.add_argument("--steps-per-graph", type=int, default=1,
                    help="decode: consecutive steps (input sets) captured in one CUDA graph")
    ap.add_argument("--dispatch", action="store_true",
                    help="decode: ep_dispatch (layout, offsets and permute in one call: one "
                         "kernel for a decode batch) then ep_unpermute")
    ap.add_argument("--lowlatency", action="store_true",
                    help="decode: fixed-rectangle layout with the fused bf16->fp8 cast")
    ap.add_argument("--decode-pool", type=int, default=16,
                    help="distinct input sets cycled by the decode workload")
    ap.add_argument("--clock-period-ms", type=float, default=1.0,
                    help="NVML clock sampling period (a child process samples)")
    ap.add_argument("--record-traffic", default=None, metavar="CSV",
                    help="write profiles/ncu_traffic.json from an ncu CSV and exit")
    ap.add_argument("--traffic-workload", default="dsv3_fp8")
    ap.add_argument("--traffic-tokens", type=int, default=8192)
    ap.add_argument("--traffic-command", default="")
    args = ap.parse_args(argv)
    if args.record_traffic:
        out = record_traffic(args.record_traffic, args.traffic_workload, args.traffic_tokens,
                             args.traffic_command)
        print(json.dumps(out, indent=1))
        return
    if args.warmup < 3 and args.impl == "epd":
        print("note: at least 3 warm-up steps are used", file=sys.stderr)
        args.warmup = 3
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        if args.workload == "decode_fp8":
            run_decode(args, rank, world, local)
        else:
            run_epd(args, rank, world, local)


if __name__ == "__main__":
    main()
