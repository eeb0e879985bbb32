#!/usr/bin/env python3
"""Benchmark of the single-GPU MoE expert-parallel permute / unpermute path.

One step = one pass of the whole path over one batch: ep_dispatch_layout ->
ep_scan_offsets -> ep_permute -> ep_unpermute, all on one stream with no host
synchronisation in between. The metric is source tokens per second, with the
achieved HBM bandwidth (algorithmic bytes / time) against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl epd|reference]
                    [--workload dsv3_fp8|prefill_bf16|skew_bf16|tiny|decode_fp8]

--impl reference times the CPU oracle (plain single-threaded C) on a bounded
token sample of the same workload. With N > 1 (torchrun) every rank runs an
independent replica on its own GPU; the time is the maximum over ranks.
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
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
                ep_unpermute=unpermute)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(name: str) -> str:
    p = os.path.join(ROOT, "unpermute_ep_dispatch_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel: str, source: str, workload: str, units: int):
    """DRAM bytes per launch from the committed ncu summary, scaled to `units`
    tokens, or None when the kernel changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[kernel]
    except Exception:
        return None
    if e.get("source_sha256_16") != kernel_source_hash(source) or e.get("workload") != workload:
        return None
    return float(e["dram_bytes_per_launch"]) * units / float(e["tokens"])


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock, power and clock-event reasons through NVML (read only)
    in a background thread while the timed region runs."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if not self._handle(cuda_index):
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            self.ok = False

    def _handle(self, cuda_index):
        import torch
        try:
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
            u = ("GPU-" + uuid) if not uuid.startswith("GPU-") else uuid
            if self.nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h)) == 0:
                return True
        except Exception:
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = cuda_index
        if vis:
            try:
                idx = int(vis.split(",")[cuda_index])
            except ValueError:
                idx = cuda_index
        return self.nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h)) == 0

    def _run(self):
        mhz = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        mw = ctypes.c_uint()
        get_reasons = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                r = reasons.value if get_reasons(self.h, ctypes.byref(reasons)) == 0 else 0
                p = mw.value / 1000.0 if self.nv.nvmlDeviceGetPowerUsage(
                    self.h, ctypes.byref(mw)) == 0 else None
                self.samples.append((int(mhz.value), int(r), p))
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "source": "nvml" if self.ok else "unavailable"}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[1]
        reasons = sorted(n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle")
        powers = [s[2] for s in self.samples if s[2] is not None]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(mhz),
                "power_w_max": max(powers) if powers else None, "source": "nvml"}


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
    A = max(1, int(args.align))
    M = case.capacity if A == 1 else epd.aligned_capacity(T, k, E, A)
    stream = torch.cuda.Stream(dev)

    # device-resident inputs and outputs (allocated once; the step allocates nothing)
    topk = case.topk_idx.to(dev)
    w = case.topk_weights.to(dev)
    x = case.x.to(dev)
    xs = None if case.x_scale is None else case.x_scale.to(dev)
    eo = None if case.expert_out is None else case.expert_out.to(dev)
    if eo is not None and M > eo.shape[0]:
        # an aligned layout's expert outputs span every padded row: repeat the seeded rows
        eo = torch.cat([eo, eo[: M - eo.shape[0]]])
    ws = epd.new_workspace(T, k, E, R, N, dev)
    status = epd.new_status(dev)
    per_e = torch.empty(E, dtype=torch.int32, device=dev)
    per_r = torch.empty(R, dtype=torch.int32, device=dev)
    per_n = torch.empty(N, dtype=torch.int32, device=dev)
    itr = torch.empty(T, R, dtype=torch.bool, device=dev)
    start = torch.empty(E, dtype=torch.int32, device=dev)
    total = torch.empty(1, dtype=torch.int32, device=dev)
    out = torch.empty(M, H, dtype=x.dtype, device=dev)
    col = args.scale_layout == "col"
    # ep_permute_ex adds its column-major scale pass for > 16 words per row over a
    # view of at least a quarter of the experts
    scale_pass = (col and xs is not None and xs.shape[1] > 16
                  and (args.view_rank is None or 4 * (E // R) >= E))
    use_ex = col or args.scales != "f32" or args.view_rank is not None
    v_begin, v_end = 0, E
    if args.view_rank is not None:
        v_begin, v_end = args.view_rank * (E // R), (args.view_rank + 1) * (E // R)
    if xs is None:
        out_scale = None
    else:
        C = xs.shape[1]
        out_scale = torch.empty((C, M) if col else (M, C), dtype=xs.dtype, device=dev)
    m_idx = torch.empty(M, dtype=torch.int32, device=dev)
    out_idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize(dev)

    io0 = dict(topk=topk, w=w, x=x, xs=xs, eo=eo, y=y)
    fused = not args.separate_offsets  # steps 1 and 2 in one launch

    def step(ev=None, around=(0, 1, 2, 3), io=None):
        """One pass of the path; with `ev`, events bracket the kernels in `around`.
        `io` selects the input / output buffers (double-buffered end to end)."""
        io = io0 if io is None else io
        topk, w, x, xs, eo, y = io["topk"], io["w"], io["x"], io["xs"], io["eo"], io["y"]
        if fused:
            first = (lambda: epd.ep_dispatch_layout_offsets(
                topk, E, R, N, ws, status, alignment=A, tokens_per_expert=per_e,
                tokens_per_rank=per_r, tokens_per_rdma_rank=per_n, is_token_in_rank=itr,
                expert_start_loc=start, total_rows=total, stream=stream), lambda: None)
        else:
            first = (
                lambda: epd.ep_dispatch_layout(topk, E, R, N, ws, status, tokens_per_expert=per_e,
                                               tokens_per_rank=per_r, tokens_per_rdma_rank=per_n,
                                               is_token_in_rank=itr, stream=stream),
                (lambda: epd.ep_scan_offsets(per_e, status, expert_start_loc=start,
                                             total_rows=total, stream=stream)) if A == 1 else
                (lambda: epd.ep_scan_offsets_aligned(per_e, A, status, expert_start_loc=start,
                                                     total_rows=total, stream=stream)))
        calls = (
            first[0],
            first[1],
            (lambda: epd.ep_permute(x, xs, topk, E, start, ws, status, capacity_rows=M, out=out,
                                    out_scale=out_scale, m_indices=m_idx, output_index=out_idx,
                                    stream=stream)) if not use_ex else
            (lambda: epd.ep_permute_ex(x, xs, topk, E, start, ws, status, capacity_rows=M,
                                       expert_begin=v_begin, expert_end=v_end,
                                       scale_col_major=col, scale_ld=M if col else None,
                                       out=out, out_scale=out_scale, m_indices=m_idx,
                                       output_index=out_idx, stream=stream)),
            lambda: epd.ep_unpermute(out if eo is None else eo, out_idx, w, status, y=y,
                                     stream=stream),
        )
        for j, call in enumerate(calls):
            timed = ev is not None and j in around
            if timed:
                ev[2 * j].record(stream)
            call()
            if timed:
                ev[2 * j + 1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    epd.check_status(status, "warm-up")
    P = int((out_idx >= 0).sum().item())  # valid pairs

    names = ["ep_dispatch_layout", "ep_scan_offsets", "ep_permute", "ep_unpermute"]
    # the dominant kernel by algorithmic bytes carries events inside the timed region;
    # events around every kernel would break the launch overlap between them
    bytes_k = algorithmic_bytes(case, P, M)
    dom = max(names, key=lambda n: bytes_k[n])
    dom_j = names.index(dom)

    def new_events(n):
        return [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n)]

    evs = new_events(args.steps)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start.record(stream)
    for i in range(args.steps):
        # events around the dominant kernel on every DOM_EVERY-th step: events block the
        # launch overlap between kernels, so bracketing every step would slow the step
        step(evs[i], around=(dom_j,) if i % DOM_EVERY == 0 else ())
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    clocks.stop()
    epd.check_status(status, "timed steps")
    ms_local = t_start.elapsed_time(t_end)
    ms = reduce_max(ms_local, world, dev)
    dom_ms = statistics.mean(evs[i][2 * dom_j].elapsed_time(evs[i][2 * dom_j + 1])
                             for i in range(0, args.steps, DOM_EVERY))

    # per-kernel breakdown: a separate pass with events around every kernel
    n_prof = max(3, min(args.steps, 50))
    evp = new_events(n_prof)
    torch.cuda.synchronize(dev)
    for i in range(n_prof):
        step(evp[i])
    torch.cuda.synchronize(dev)
    per_kernel_ms = {n: statistics.mean(e[2 * j].elapsed_time(e[2 * j + 1]) for e in evp)
                     for j, n in enumerate(names)}
    per_kernel_ms[dom] = dom_ms

    # ---- end to end through the public API: host inputs in, host result out, every step
    e2e = None
    if not args.no_e2e:
        pin = lambda t: None if t is None else t.contiguous().pin_memory()  # noqa: E731
        h_topk, h_w, h_x, h_xs, h_eo = (pin(case.topk_idx), pin(case.topk_weights),
                                        pin(case.x), pin(case.x_scale),
                                        None if eo is None else pin(eo.cpu()))
        h_y = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (h_topk, h_w, h_x, h_xs, h_eo)
                  if t is not None)
        d2h = h_y.numel() * h_y.element_size()

        # Pipelined over two buffer sets: step i+1's inputs go host -> device on a copy
        # stream while step i computes, and step i's result comes back on a third
        # stream; every step still moves its own inputs in and its result out.
        def clone(t):
            return None if t is None else torch.empty_like(t)
        ios = [io0, dict(topk=clone(topk), w=clone(w), x=clone(x), xs=clone(xs), eo=clone(eo),
                         y=clone(y))]
        h_ys = [h_y, torch.empty_like(h_y).pin_memory()]
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
                step(io=io)
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
        e2e = {"value": whole_job_rate(T, world, e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": e2e_ms,
               "note": "copies of step i+1 / read-back of step i overlap step i's kernels"}
        epd.check_status(status, "e2e steps")

    if fused:  # one launch computes steps 1 and 2
        per_kernel_ms["ep_dispatch_layout_offsets"] = per_kernel_ms.pop("ep_dispatch_layout")
        per_kernel_ms.pop("ep_scan_offsets")
        names = ["ep_dispatch_layout_offsets", "ep_permute", "ep_unpermute"]
    # ---- roofline of the dominant kernel and of the whole path
    peak, peak_src = load_peaks()
    dom_src = {"ep_unpermute": "unpermute.cu", "ep_permute": "permute.cu",
               "ep_dispatch_layout": "layout.cu", "ep_scan_offsets": "scan.cu",
               "ep_dispatch_layout_offsets": "layout.cu"}[dom]
    achieved = bytes_k[dom] / (per_kernel_ms[dom] * 1e-3) / 1e9
    ms_per_step = ms / args.steps
    P = int((out_idx >= 0).sum().item())        # valid pairs (total is the padded row count)
    T_rows = int((out_idx >= 0).any(dim=1).sum().item())
    bytes_k = algorithmic_bytes(case, P, M, T_rows)
    if fused:
        bytes_k["ep_dispatch_layout_offsets"] = (bytes_k.pop("ep_dispatch_layout")
                                                 + bytes_k.pop("ep_scan_offsets"))
    path_bytes = sum(bytes_k.values())
    path_gbs = path_bytes / (ms_per_step * 1e-3) / 1e9
    kernels = {n: {"us": round(per_kernel_ms[n] * 1e3, 2), "bytes": bytes_k[n],
                   "gbs": round(bytes_k[n] / (per_kernel_ms[n] * 1e-3) / 1e9, 1),
                   "frac": round(bytes_k[n] / (per_kernel_ms[n] * 1e-3) / 1e9 / peak, 4)}
               for n in names}

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
                   "expert_out": "bf16 identity (permuted rows)" if eo is None else "bf16 seeded",
                   "capacity_rows": M, "valid_pairs": P, "expert_alignment": A,
                   "scales": args.scales if case.dtype == "fp8" else None,
                   "scale_layout": args.scale_layout if case.dtype == "fp8" else None,
                   "experts_in_view": [v_begin, v_end],
                   "launches": "layout+offsets fused, permute, combine" if fused else
                               "layout, offsets, permute, combine",
                   "l2": f"no flush: {path_bytes / 1e6:.0f} MB moved per step > 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "hbm": {"path_gbs": round(path_gbs, 1), "path_bytes": path_bytes,
                "frac": round(path_gbs / peak, 4), "peak_gbs": peak, "peak_source": peak_src},
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(dom, dom_src, name, T),
                     "algorithmic_bytes": bytes_k[dom], "peak_source": peak_src},
        "kernels": kernels,
        "kernels_note": f"{dom} timed inside the timed region (events on every {DOM_EVERY}th "
                        f"step); the others from a separate "
                        f"{n_prof}-step pass with events around every kernel",
        # column-major scales add the scale pass after the row copy (inside ep_permute_ex)
        # every rank's kernels in the timed region (the job's total, like value)
        "gpu_launches": ((3 if fused else 4) + (1 if scale_pass else 0)) * args.steps * world,
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
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


# ----------------------------------------------------------------------------- decode: graph-captured steps
def run_decode(args, rank, world, local):
    """Many small independent steps (T=128): each step's layout -> offsets ->
    permute -> combine chain is captured once in a CUDA graph per input set and
    replayed, so the per-step latency carries no host launch cost. A pool of
    distinct device-resident input sets (seeds 1000 + i) is cycled."""
    import torch
    import unpermute_ep_dispatch_gb300 as epd
    from unpermute_ep_dispatch_gb300 import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    init_dist(world, "nccl")
    epd.load_library()
    ll = bool(args.lowlatency)
    pool = [workloads.make_case("decode_fp8", seed=1000 + i, dtype="bf16" if ll else None)
            for i in range(args.decode_pool)]
    c0 = pool[0]
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
    if ll:
        gen = torch.Generator(device=dev)
        gen.manual_seed(99)
        o["q"] = torch.empty(E, rows, H, dtype=torch.float8_e4m3fn, device=dev)
        o["qs"] = torch.empty(E, H // 128, rows, dtype=torch.float32, device=dev)
        o["recv"] = torch.empty(E, dtype=torch.int32, device=dev)
        o["src"] = torch.empty(E, rows, dtype=torch.int32, device=dev)
    # The fixed rectangles are one buffer, allocated once and reused by every step, as
    # a serving loop does (470 MB of bf16 at decode_fp8: larger than L2 by itself).
    # The exact layout's expert outputs are per input set (15 MB each; the pool keeps
    # the inputs larger than L2).
    rect = (torch.randn(E * rows, H, generator=gen, device=dev).to(torch.bfloat16)
            if ll else None)
    inputs = [dict(topk=c.topk_idx.to(dev), w=c.topk_weights.to(dev), x=c.x.to(dev),
                   xs=None if c.x_scale is None else c.x_scale.to(dev),
                   eo=rect if ll else c.expert_out.to(dev)) for c in pool]

    def chain_ll(inp, ev=None):
        if args.separate_offsets:  # the layout as its own launch, then the rectangle permute
            epd.ep_dispatch_layout(inp["topk"], E, R, N, ws, status,
                                   tokens_per_expert=o["per_e"], tokens_per_rank=o["per_r"],
                                   tokens_per_rdma_rank=o["per_n"], is_token_in_rank=o["itr"],
                                   stream=stream)
            epd.ep_permute_lowlatency(inp["x"], inp["topk"], E, rows, ws, status, out_q=o["q"],
                                      out_scale=o["qs"], recv_count=o["recv"],
                                      output_index=o["out_idx"], src_token=o["src"],
                                      stream=stream)
        else:  # one call: one kernel for a decode batch
            epd.ep_dispatch_lowlatency(inp["x"], inp["topk"], E, R, N, rows, ws, status,
                                       out_q=o["q"], out_scale=o["qs"], recv_count=o["recv"],
                                       output_index=o["out_idx"], src_token=o["src"],
                                       stream=stream)
        if ev is not None:
            ev[0].record(stream)
        epd.ep_unpermute(inp["eo"], o["out_idx"], inp["w"], status, y=o["y"], stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def chain(inp, ev=None):
        if ll:
            return chain_ll(inp, ev)
        if args.dispatch:
            epd.ep_dispatch(inp["x"], inp["xs"], inp["topk"], E, R, N, ws, status,
                            capacity_rows=M, tokens_per_expert=o["per_e"],
                            tokens_per_rank=o["per_r"], tokens_per_rdma_rank=o["per_n"],
                            is_token_in_rank=o["itr"], expert_start_loc=o["start"],
                            total_rows=o["total"], out=o["out"], out_scale=o["out_scale"],
                            m_indices=o["m_idx"], output_index=o["out_idx"], stream=stream)
            if ev is not None:
                ev[0].record(stream)
            epd.ep_unpermute(inp["eo"], o["out_idx"], inp["w"], status, y=o["y"], stream=stream)
            if ev is not None:
                ev[1].record(stream)
            return
        if args.separate_offsets:
            epd.ep_dispatch_layout(inp["topk"], E, R, N, ws, status,
                                   tokens_per_expert=o["per_e"], tokens_per_rank=o["per_r"],
                                   tokens_per_rdma_rank=o["per_n"], is_token_in_rank=o["itr"],
                                   stream=stream)
            epd.ep_scan_offsets(o["per_e"], status, expert_start_loc=o["start"],
                                total_rows=o["total"], stream=stream)
        else:
            epd.ep_dispatch_layout_offsets(inp["topk"], E, R, N, ws, status,
                                           tokens_per_expert=o["per_e"],
                                           tokens_per_rank=o["per_r"],
                                           tokens_per_rdma_rank=o["per_n"],
                                           is_token_in_rank=o["itr"],
                                           expert_start_loc=o["start"], total_rows=o["total"],
                                           stream=stream)
        epd.ep_permute(inp["x"], inp["xs"], inp["topk"], E, o["start"], ws, status,
                       capacity_rows=M, out=o["out"], out_scale=o["out_scale"],
                       m_indices=o["m_idx"], output_index=o["out_idx"], stream=stream)
        if ev is not None:
            ev[0].record(stream)
        epd.ep_unpermute(inp["eo"], o["out_idx"], inp["w"], status, y=o["y"], stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for inp in inputs:                       # load the library, set attributes, warm
        chain(inp)
    torch.cuda.synchronize(dev)
    G = max(1, int(args.steps_per_graph))  # consecutive steps (input sets) per graph
    if args.steps % G:
        raise SystemExit(f"--steps {args.steps} is not a multiple of --steps-per-graph {G}")
    graphs = []
    for gi in range(len(inputs)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(G):
                chain(inputs[(gi * G + j) % len(inputs)])
        graphs.append(g)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize(dev)
    epd.check_status(status, "decode warm-up")

    steps = args.steps
    replays = steps // G
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(replays)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    clocks.start()
    with torch.cuda.stream(stream):
        a.record(stream)
        for i in range(replays):
            graphs[i % len(graphs)].replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    # per-step latency: every replay bracketed by events (divided by its G steps)
    with torch.cuda.stream(stream):
        for i in range(replays):
            ev[i][0].record(stream)
            graphs[i % len(graphs)].replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    clocks.stop()
    epd.check_status(status, "decode steps")
    ms = reduce_max(a.elapsed_time(b), world, dev)
    lat = sorted(e0.elapsed_time(e1) * 1e3 / G for e0, e1 in ev)

    # dominant kernel (largest bytes) timed with events on its stream, outside graphs
    P = int((o["out_idx"] >= 0).sum().item())
    bytes_k = algorithmic_bytes(c0, P, M)
    names = ["ep_dispatch_layout", "ep_scan_offsets", "ep_permute", "ep_unpermute"]
    if ll:  # no offset scan; the permute reads bf16 rows and writes e4m3 rows + scales
        bytes_k.pop("ep_scan_offsets")
        names.remove("ep_scan_offsets")
        bytes_k["ep_permute"] = (T * H * 2 + P * H + P * (H // 128) * 4 + T * k * 16 + E * 4
                                 + P * 4)
    dom = max(names, key=lambda n: bytes_k[n])
    evd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(min(steps, 100))]
    for i, e in enumerate(evd):
        chain(inputs[i % len(inputs)], ev=e)
    torch.cuda.synchronize(dev)
    dom_us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evd) * 1e3
    peak, peak_src = load_peaks()
    path_bytes = sum(bytes_k.values())
    ms_per_step = ms / steps
    result = {
        "metric": METRIC,
        "value": whole_job_rate(T * steps, world, ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded routing, rows and expert outputs; no dataset)",
        "config": {"workload": "decode_fp8" + ("_lowlatency" if ll else ""), "tokens": T,
                   "hidden": H, "top_k": k, "experts": E,
                   "path": ("layout -> fixed-rectangle permute with bf16->e4m3 cast -> combine"
                            if ll and args.separate_offsets else
                            "ep_dispatch_lowlatency (fixed rectangles, bf16->e4m3 cast: one "
                            "kernel) -> combine" if ll else
                            "ep_dispatch (layout, offsets, permute: one kernel) -> combine"
                            if args.dispatch else "layout -> offsets -> permute -> combine"),
                   "rows_per_expert": rows if ll else None,
                   "simulated_ranks": R, "simulated_rdma_nodes": N,
                   "rows": "fp8_e4m3 + f32 scale per 128 columns", "expert_out": "bf16 seeded",
                   "input_sets": len(pool),
                   "launch": (f"CUDA graphs of {G} consecutive steps (input sets), replayed"
                              if G > 1 else "one CUDA graph per input set, replayed"),
                   "l2": f"no flush: {len(pool)} input sets cycled, each step's inputs "
                         "read from HBM once the pool exceeds the 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "latency_us": {"mean": statistics.mean(lat), "p50": lat[len(lat) // 2],
                       "p99": lat[min(len(lat) - 1, int(0.99 * len(lat)))],
                       "note": "per step: events around each replay" +
                               (f", divided by its {G} steps" if G > 1 else "")},
        "hbm": {"path_gbs": round(path_bytes / (ms_per_step * 1e-3) / 1e9, 1),
                "path_bytes": path_bytes, "peak_gbs": peak, "peak_source": peak_src},
        "roofline": {"kernel": dom, "bound": "hbm",
                     "achieved": round(bytes_k[dom] / (dom_us * 1e-6) / 1e9, 1), "peak": peak,
                     "unit": "GB/s",
                     "frac": round(bytes_k[dom] / (dom_us * 1e-6) / 1e9 / peak, 4),
                     "traffic": None, "algorithmic_bytes": bytes_k[dom],
                     "note": "latency-bound at this size; timed outside the graphs"},
        "gpu_launches": ((3 if args.separate_offsets else 2) if ll else
                         2 if args.dispatch else
                         3 if not args.separate_offsets else 4) * steps * world,
        "clocks": clocks.summary(),
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
    args = ap.parse_args(argv)
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
