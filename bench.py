"""Benchmark of the owner-local optimizer step on GB300.

One step = the whole hot path over one owner's table: the Muon step on every
2D matrix (momentum, Frobenius normalisation, five quintic Newton-Schulz
iterations, shape-scaled update with weight decay), AdamW on the packed
non-matrix tail, and RMNP on the same matrices (its own momentum and weight
copies). Default workload: the Llama-style 8B matrix set (224 matrices,
6.98 G elements; AdamW tail 1.05 G elements: the RMSNorm vectors, the
embedding and the LM head), synthetic seeded inputs resident in HBM. The
working set (~200 GB) is far larger than L2, so no flush is needed. After the
headline the GPT-2 Large matrix set (144 matrices) is timed the same way and
reported under `secondary` (device-resident inputs only).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an
independent replica of the workload on its own GPU (the step has no exchange);
the time is the max over ranks and the value is the sum of all ranks' work.
`--impl reference` times the CPU oracle on the host cores instead (rank 0).
"""
from __future__ import annotations

import argparse
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

METRIC = "owner Muon step ms & NS TFLOP/s vs bf16 peak; RMNP/AdamW HBM GB/s"
DEFAULT_CONFIG = "llama8b"
SECONDARY_CONFIG = "gpt2l"
UNIT = "TFLOP/s"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one step's 15
# Newton-Schulz launches, per workload, from an ncu capture of the named
# capture workload scaled by `scale` (the capture workload holds 1/scale of
# the table's matrices). Valid only for the kernel source and tile schedule it
# was measured on (hash of ns_gemm.cu, its device helpers, plan.cpp, abi.cu and
# mo_internal.h); the profiles directory holds the capture summaries with their
# commands.
NS_TRAFFIC = {
    "llama8b": {"source_sha256_16": "4e806d95c73f9fef", "bytes_per_ns_segment": 469.903e9,
                "how": "ncu dram__bytes_read.sum + dram__bytes_write.sum (one pass) over the 15 NS launches of the "
                       "fourth step on the full table (tiles from the per-launch counter; 470-495 GB over captures)"},
    "gpt2l": {"source_sha256_16": "4e806d95c73f9fef", "bytes_per_ns_segment": 34.910e9,
              "how": "ncu dram__bytes_read.sum + dram__bytes_write.sum (one pass) over the 15 NS launches of the "
                     "fourth step on the full table (static tile assignment; the last launch from the counter)"},
}
# A timed region at least this long is "a kernel timed inside a long step":
# its roofline uses the sustained bf16 peak, a shorter one the burst peak.
SUSTAINED_REGION_S = 1.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def choose_peak(peaks, region_s: float):
    """(peak TFLOP/s, name): the sustained bf16 peak for a timed region of at
    least SUSTAINED_REGION_S seconds, the burst peak for a shorter one."""
    if region_s >= SUSTAINED_REGION_S:
        return peaks["bf16_tflops_sustained"], "bf16_tflops_sustained"
    return peaks["bf16_tflops"], "bf16_tflops (burst)"


def source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    # the kernel and its device helpers, the tile lists, and the per-launch
    # choice of tile schedule
    for name in ("ns_gemm.cu", "ptx.cuh", "device_common.cuh", "plan.cpp", "abi.cu", "mo_internal.h"):
        with open(os.path.join(ROOT, "matrix_optimizers_zero_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ns_traffic(workload: str):
    """(bytes, note): the profiled DRAM traffic of one step's NS launches for
    this workload, or (None, why) when there is no capture for it or the
    kernel or its tile schedule differs from the one profiled."""
    rec = NS_TRAFFIC.get(workload)
    if rec is None:
        return None, "no capture for this workload"
    if rec["source_sha256_16"] != source_hash():
        return None, "kernel source changed since the capture"
    return rec["bytes_per_ns_segment"], rec["how"]


# ---------------------------------------------------------------- multi-rank helpers

def max_over_ranks(x: float, device=None) -> float:
    """The maximum of x over all ranks of the default process group (x itself
    when there is none). NCCL groups reduce on `device`, others on the CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    on = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def min_over_ranks(x: float, device=None) -> float:
    """The minimum of x over all ranks (x itself without a process group)."""
    return -max_over_ranks(-float(x), device)


def whole_job_tflops(world: int, flops_per_rank: float, ms_max: float) -> float:
    """Aggregate throughput of `world` independent replicas that each did
    flops_per_rank of work, timed by the slowest rank."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if self.t0 is not None and self.t1 is not None and self.t0 - 0.06 <= ts <= self.t1 + 0.06]
        use = inside if inside else [r for _, r in rows]
        sm = [float(r[1]) for r in use if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in use for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_max": max((float(r[3]) for r in use if r[3].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------------- CPU oracle timing

def distinct_shapes_by_cost(wl):
    """Index of the first matrix of each distinct shape, cheapest NS first."""
    from matrix_optimizers_zero_gb300 import workloads
    seen, picks = set(), []
    for i, s in enumerate(wl.matrices):
        if (s.rows, s.cols) not in seen:
            seen.add((s.rows, s.cols))
            picks.append(i)
    return sorted(picks, key=lambda i: (workloads.ns_alg_flops(wl.matrices[i].rows, wl.matrices[i].cols,
                                                               wl.ns_steps), i))


def oracle_matrix_seconds(wl, i):
    """Seconds the oracle's whole-matrix Muon step takes on matrix i (seeded
    host inputs, momentum from an earlier step), and that step's NS flops."""
    import oracle
    from matrix_optimizers_zero_gb300 import workloads
    W, G, V = workloads.host_matrix(wl, i, v_std=1e-3)
    W, G, V = (t.float().double().numpy() for t in (W, G, V))
    t0 = time.perf_counter()
    oracle.muon_matrix_step(W, G, V, lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_steps=wl.ns_steps)
    s = wl.matrices[i]
    return time.perf_counter() - t0, workloads.ns_alg_flops(s.rows, s.cols, wl.ns_steps)


def cpu_oracle_sample(wl, max_seconds=25.0, min_seconds=10.0):
    """Times the CPU oracle (as it stands) on a bounded sample of the
    workload: whole-matrix Muon steps on one matrix per distinct shape,
    cheapest first, skipping a shape whose predicted time would overrun
    max_seconds, and cycling again while less than min_seconds were spent.
    The full table's oracle step time is extrapolated from the measured rate.
    Returns a dict (TFLOP/s, seconds, description, cores, extrapolated step
    seconds)."""
    from matrix_optimizers_zero_gb300 import workloads
    cores = len(os.sched_getaffinity(0))
    picks = distinct_shapes_by_cost(wl)
    flops = 0
    t_total = 0.0
    done = []
    for rnd in range(8):
        ran = False
        for i in picks:
            s = wl.matrices[i]
            f = workloads.ns_alg_flops(s.rows, s.cols, wl.ns_steps)
            if done and t_total + f / (flops / t_total) > max_seconds:
                continue
            secs, f = oracle_matrix_seconds(wl, i)
            t_total += secs
            flops += f
            done.append(f"{s.rows}x{s.cols}")
            ran = True
        if t_total >= min_seconds or not ran:
            break
    rate = flops / t_total
    full = workloads.workload_alg_flops(wl) / rate
    desc = (f"oracle muon_matrix_step (fp64 numpy, bf16 emulation) on {len(done)} matrices "
            f"[{', '.join(done)}] of the {wl.name} table; the whole table's NS flops at this rate "
            f"(extrapolated) take {full:.0f} s per step")
    return {"value": rate / 1e12, "seconds": t_total, "sample": desc, "cores": cores,
            "extrapolated_step_s": full}


def host_mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


# ---------------------------------------------------------------- our arm

class Owner:
    """One owner's state on the device: the Muon table (W, G, V), an RMNP copy
    (its own W and V, the same G) and the AdamW tail, each in one flat
    buffer with per-tensor views, plus the library tables and workspace."""

    def __init__(self, mo, wl, dev, seed):
        import torch
        self.mo, self.wl, self.dev = mo, wl, dev
        self.shapes = [(s.rows, s.cols) for s in wl.matrices]
        self.offs, tot = [], 0
        for r, c in self.shapes:
            self.offs.append(tot)
            tot += ((r * c + 63) // 64) * 64
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        self.Wf = torch.randn(tot, generator=gen, device=dev).mul_(wl.w_std)
        self.Gf = torch.randn(tot, generator=gen, device=dev).mul_(wl.g_std).to(torch.bfloat16)
        self.Vf = torch.randn(tot, generator=gen, device=dev).mul_(1e-3)
        self.Wr = self.Wf.clone()
        self.Vr = self.Vf.clone()
        self.W_l, self.G_l, self.V_l = self.views(self.Wf), self.views(self.Gf), self.views(self.Vf)
        self.Wr_l, self.Vr_l = self.views(self.Wr), self.views(self.Vr)
        self.muon_tbl = mo.MuonTable(list(zip(self.W_l, self.G_l, self.V_l)))
        self.rmnp_tbl = mo.MuonTable(list(zip(self.Wr_l, self.G_l, self.Vr_l)))
        self.tail_sizes = [t for t in wl.tail if t > 0]
        self.toffs, ttot = [], 0
        for t in self.tail_sizes:
            self.toffs.append(ttot)
            ttot += ((t + 63) // 64) * 64
        self.Pf = torch.randn(max(ttot, 1), generator=gen, device=dev).mul_(wl.tail_p_std)
        self.Tg = torch.randn(max(ttot, 1), generator=gen, device=dev).mul_(wl.tail_g_std)
        self.Tm = torch.zeros(max(ttot, 1), device=dev)
        self.Tv = torch.zeros(max(ttot, 1), device=dev)
        self.tail_tbl = self.tail_table(self.Tg)
        self.mp = mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_steps=wl.ns_steps)
        self.rp = mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu)
        self.ws = mo.muon_workspace(self.muon_tbl, self.mp, device=dev)
        self.adam_step = 0

    def views(self, flat):
        return [flat[o:o + r * c].view(r, c) for o, (r, c) in zip(self.offs, self.shapes)]

    def tail_table(self, g_flat):
        return self.mo.TailTable([(self.Pf[o:o + t], g_flat[o:o + t], self.Tm[o:o + t], self.Tv[o:o + t])
                                  for o, t in zip(self.toffs, self.tail_sizes)])

    def launches_per_step(self):
        """Kernel launches of one step: the prologue (a norm and a cast
        launch), 3 GEMM launches per iteration (plus one Gram reduction per iteration when a matrix has
        more than 32768 columns on its long side), AdamW one per 256 segments,
        RMNP one per 512 entries separately for rows shorter / not shorter
        than 8192 elements."""
        wl = self.wl
        n_long = sum(1 for _, c in self.shapes if c >= 8192)
        reduce = 1 if any(max(r, c) > 32768 for r, c in self.shapes) else 0
        return ((2 + (3 + reduce) * wl.ns_steps) + math.ceil(len(self.tail_sizes) / 256)
                + math.ceil((len(self.shapes) - n_long) / 512) + math.ceil(n_long / 512))

    def step(self, stream, ev=None, tabs=None, between=None):
        """One optimizer step on `stream`: Muon, AdamW on the tail, RMNP.
        ev: six events (Muon start, NS start, NS end, Muon end, AdamW end,
        RMNP end); tabs: (muon, rmnp, tail) tables to use (default: the
        resident ones); between: called after the Muon call, before AdamW and
        RMNP."""
        import ctypes
        import torch
        mo, wl = self.mo, self.wl
        lib = mo.load_library()
        nvtx = torch.cuda.nvtx      # names each library call on the host timeline; no device work
        m_tbl, r_tbl, t_tbl = tabs if tabs is not None else (self.muon_tbl, self.rmnp_tbl, self.tail_tbl)
        sptr = stream.cuda_stream
        ws_ptr, ws_bytes = self.ws.data_ptr(), self.ws.numel()
        nvtx.range_push("muon_owner_step")
        if ev is None:
            st = lib.muon_owner_step(m_tbl.ptr, m_tbl.n, ctypes.byref(self.mp), ws_ptr, ws_bytes, sptr)
        else:
            ev[0].record(stream)
            st = lib.muon_owner_step_timed(m_tbl.ptr, m_tbl.n, ctypes.byref(self.mp), ws_ptr, ws_bytes, sptr,
                                           ev[1].cuda_event, ev[2].cuda_event)
        nvtx.range_pop()
        if st != 0:
            raise mo.MoError(st, "muon_owner_step")
        if ev is not None:
            ev[3].record(stream)
        if between is not None:
            between()
        self.adam_step += 1
        ap = mo.AdamWParams(lr=wl.adam_lr, wd=wl.adam_wd, beta1=wl.beta1, beta2=wl.beta2, eps=wl.adam_eps,
                            step=self.adam_step)
        nvtx.range_push("adamw_tail_step")
        st = lib.adamw_tail_step(t_tbl.ptr, t_tbl.n, ctypes.byref(ap), sptr)
        nvtx.range_pop()
        if st != 0:
            raise mo.MoError(st, "adamw_tail_step")
        if ev is not None:
            ev[4].record(stream)
        nvtx.range_push("rmnp_step")
        st = lib.rmnp_step(r_tbl.ptr, r_tbl.n, ctypes.byref(self.rp), sptr)
        nvtx.range_pop()
        if st != 0:
            raise mo.MoError(st, "rmnp_step")
        if ev is not None:
            ev[5].record(stream)


def timed_steps(owner, stream, dev, steps, barrier, clocks=None):
    """Times `steps` whole steps with CUDA events on `stream` (barrier and
    synchronize on both sides). Returns the total and per-part means/minima
    in ms."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for e in evs:
        for x in e:
            x.record(stream)          # torch creates events lazily: force the handles to exist
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    if clocks is not None:
        clocks.mark("begin")
    t_start.record(stream)
    for k in range(steps):
        owner.step(stream, evs[k])
    t_end.record(stream)
    barrier()
    if clocks is not None:
        clocks.mark("end")
    total_ms = t_start.elapsed_time(t_end)
    return {
        "total_ms": total_ms,
        "ms_step": total_ms / steps,
        "pro_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
        "ns_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in evs),
        "muon_ms": statistics.mean(e[0].elapsed_time(e[3]) for e in evs),
        "adam_ms": statistics.mean(e[3].elapsed_time(e[4]) for e in evs),
        "rmnp_ms": statistics.mean(e[4].elapsed_time(e[5]) for e in evs),
        "step_min_ms": min(e[0].elapsed_time(e[5]) for e in evs),
        "ns_min_ms": min(e[1].elapsed_time(e[2]) for e in evs),
    }


def breakdown(wl, t, peaks, steps):
    """Per-part figures of a timed run: ms, TFLOP/s and GB/s at the
    algorithmic work counts, and the NS fraction of the bf16 peak chosen by
    the length of the timed region."""
    from matrix_optimizers_zero_gb300 import workloads
    shapes = [(s.rows, s.cols) for s in wl.matrices]
    ns_flops = workloads.workload_alg_flops(wl)
    ns_dense = sum(workloads.ns_dense_flops(r, c, wl.ns_steps) for r, c in shapes)
    n_el = wl.n_elements
    ns_tflops = ns_flops / (t["ns_ms"] * 1e-3) / 1e12
    rmnp_gbs = n_el * workloads.RMNP_BYTES_PER_EL / (t["rmnp_ms"] * 1e-3) / 1e9
    adam_gbs = wl.tail_elements * workloads.ADAMW_BYTES_PER_EL / (t["adam_ms"] * 1e-3) / 1e9
    pro_gbs = n_el * workloads.PROLOGUE_BYTES_PER_EL / (t["pro_ms"] * 1e-3) / 1e9
    region_s = t["total_ms"] * 1e-3
    peak, peak_name = choose_peak(peaks, region_s)
    return {
        "muon_step_ms": round(t["muon_ms"], 4),
        "prologue_ms": round(t["pro_ms"], 4),
        "prologue_gbs": round(pro_gbs, 1),
        "prologue_frac_hbm": round(pro_gbs / peaks["hbm_gbs"], 4),
        "prologue_bytes_per_el": workloads.PROLOGUE_BYTES_PER_EL,
        "ns_ms": round(t["ns_ms"], 4),
        "ns_tflops_alg": round(ns_tflops, 2),
        "ns_tflops_dense_equiv": round(ns_dense / (t["ns_ms"] * 1e-3) / 1e12, 2),
        "ns_frac_of_peak": round(ns_tflops / peak, 4),
        "ns_frac_of_burst_peak": round(ns_tflops / peaks["bf16_tflops"], 4),
        "ns_frac_of_sustained_peak": round(ns_tflops / peaks["bf16_tflops_sustained"], 4),
        "peak_used": peak_name,
        "timed_region_s": round(region_s, 3),
        "adamw_ms": round(t["adam_ms"], 4),
        "adamw_gbs": round(adam_gbs, 1),
        "adamw_frac_hbm": round(adam_gbs / peaks["hbm_gbs"], 4),
        "adamw_elements": wl.tail_elements,
        "rmnp_ms": round(t["rmnp_ms"], 4),
        "rmnp_gbs": round(rmnp_gbs, 1),
        "rmnp_frac_hbm": round(rmnp_gbs / peaks["hbm_gbs"], 4),
        "means_over_steps": steps,
        "step_min_ms": round(t["step_min_ms"], 4),
        "ns_min_ms": round(t["ns_min_ms"], 4),
        "ns_tflops_alg_best": round(ns_flops / (t["ns_min_ms"] * 1e-3) / 1e12, 2),
    }


def run_ours(args, rank, world, local_rank):
    import torch
    import matrix_optimizers_zero_gb300 as mo
    from matrix_optimizers_zero_gb300 import build as mo_build, workloads

    mo_build.build()
    mo.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    wl = workloads.get_workload(args.config)
    out = headline(args, mo, workloads, wl, dev, stream, peaks, rank, world, local_rank, barrier)
    time_secondary = args.secondary and args.config != SECONDARY_CONFIG
    if time_secondary or args.extras:
        torch.cuda.empty_cache()
        wl2 = workloads.get_workload(SECONDARY_CONFIG if time_secondary else args.extras_config)
        owner2 = Owner(mo, wl2, dev, 4321 + rank)
        for _ in range(args.warmup):
            owner2.step(stream)
        torch.cuda.synchronize(dev)
        if time_secondary:
            t2 = timed_steps(owner2, stream, dev, args.secondary_steps, barrier)
            if mo.mo_last_device_error() != 0:
                raise RuntimeError("device-side timeout in the secondary workload")
            sec = breakdown(wl2, t2, peaks, args.secondary_steps)
            sec["ms_per_step"] = round(t2["ms_step"], 4)
            sec["workload"] = (f"{wl2.name}: {len(wl2.matrices)} matrices, {wl2.n_elements} elements, "
                               f"tail {wl2.tail_elements}")
            sec["value_tflops_alg_per_step"] = round(
                workloads.workload_alg_flops(wl2) / (t2["ms_step"] * 1e-3) / 1e12, 2)
            sec["note"] = ("the pages' own matrix set (GPT-2 Large); the AdamW tail here is L2- and "
                           "latency-bound and not graded")
            traffic, how = ns_traffic(wl2.name)
            sec["ns_traffic_bytes"] = traffic
            sec["ns_traffic_note"] = how
            if out is not None:
                out["secondary"] = {wl2.name: sec}
        if args.extras and wl2.name != args.extras_config:
            del owner2
            torch.cuda.empty_cache()
            wl2 = workloads.get_workload(args.extras_config)
            owner2 = Owner(mo, wl2, dev, 4321 + rank)
        if args.extras:
            ex = measure_extras(args, mo, workloads, wl2, owner2.shapes, owner2.W_l, owner2.G_l, owner2.V_l,
                                owner2.Wr_l, owner2.Vr_l, dev, stream, peaks)
            if out is not None:
                out["extras"] = {"workload": wl2.name, **ex}
        del owner2
    if out is not None and not args.no_cpu_baseline:
        cb = cpu_oracle_sample(wl, max_seconds=args.cpu_seconds, min_seconds=10.0)
        out["cpu_baseline"] = {"value": round(cb["value"], 6), "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
                               "sample": cb["sample"], "seconds": round(cb["seconds"], 2),
                               "extrapolated_step_s": round(cb["extrapolated_step_s"], 1)}
    return out


def headline(args, mo, workloads, wl, dev, stream, peaks, rank, world, local_rank, barrier):
    """The headline line for workload `wl`: the device-resident timed run,
    then the end-to-end run through the C ABI with host buffers."""
    import torch
    owner = Owner(mo, wl, dev, 1234 + rank)
    shapes = owner.shapes

    # ---- warmup
    for _ in range(args.warmup):
        owner.step(stream)
    torch.cuda.synchronize(dev)
    if mo.mo_last_device_error() != 0:
        raise RuntimeError("device-side timeout during warmup")

    # ---- timed region (kernel-level: inputs resident in HBM)
    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()
    time.sleep(0.3)
    t = timed_steps(owner, stream, dev, args.steps, barrier, clocks)
    clk = clocks.stop()
    ms_max = max_over_ranks(t["ms_step"], dev)
    ns_flops = workloads.workload_alg_flops(wl)
    value = whole_job_tflops(world, ns_flops, ms_max)
    bd = breakdown(wl, t, peaks, args.steps)

    e2e = end_to_end(args, mo, owner, dev, stream, barrier, world, ns_flops)
    if mo.mo_last_device_error() != 0:
        raise RuntimeError("device-side timeout during the timed region")

    if rank != 0:
        return None

    ns_tflops = bd["ns_tflops_alg"]
    peak, peak_name = choose_peak(peaks, t["total_ms"] * 1e-3)
    traffic, traffic_note = ns_traffic(wl.name)
    n_el = wl.n_elements
    out = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{wl.name}: {len(shapes)} matrices, {n_el} elements, tail {wl.tail_elements}",
            "ns_steps": wl.ns_steps,
            "step": "muon_owner_step + adamw_tail_step + rmnp_step",
            "value_definition": "algorithmic Newton-Schulz flops 5(3m^2n+m^3) per matrix / whole-step time",
            "l2": "inputs larger than L2 (no flush)",
            "parallelism": f"replicas x{world}",
            "state": "fp32 W/V, bf16 G; NS operands bf16 with fp32 accumulation",
        },
        "breakdown": bd,
        "roofline": {
            "bound": "tensor",
            "kernel": "ns_gemm_pair_kernel (the 15 Gram, A.A and B.X launches of one step)",
            "achieved": round(ns_tflops, 2),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(ns_tflops / peak, 4),
            "traffic": traffic,
            "traffic_unit": "DRAM bytes per step's 15 NS launches",
            "traffic_note": traffic_note,
            "peak_source": f"{peak_name} ({peaks['source']}); timed region {t['total_ms'] * 1e-3:.2f} s",
            "frac_of_burst_peak": bd["ns_frac_of_burst_peak"],
            "frac_of_sustained_peak": bd["ns_frac_of_sustained_peak"],
        },
        "e2e": e2e,
        "gpu_launches": int(owner.launches_per_step() * args.steps),
        "clocks": clk,
    }
    return out


def end_to_end(args, mo, owner, dev, stream, barrier, world, ns_flops):
    """The same step through the C ABI with host buffers. Every step uploads
    its gradients (Muon/RMNP G and the tail's g) from pinned host memory and
    reads all updated weights back (Muon W, RMNP W, tail p). Uploads, compute
    and read-backs run on three streams. The gradients are double-buffered on
    the device, so step k+1's upload overlaps step k. The weights are updated
    in place, so each step snapshots them into device staging buffers right
    after its Muon (W) and RMNP/AdamW (RMNP W, tail p) calls; the read-back
    copies from the snapshots while the next step computes (a snapshot waits
    only until the previous step's read-back of that buffer is done). The
    snapshots are elementwise kernels (x * 1.0, bit-identical), not
    device-to-device memcpys: those would queue on the copy engines behind
    the read-backs and stall the compute stream."""
    import torch
    if args.no_e2e:
        return None
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    need = owner.Gf.numel() * 2 + owner.Tg.numel() * 4 + (owner.Wf.numel() + owner.Wr.numel() + owner.Pf.numel()) * 4
    # the ranks of one host share its memory; every rank takes the same
    # decision (the leg has barriers)
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = host_mem_available_bytes()
    fits = avail is None or need <= 0.7 * avail / local_world
    if not (min_over_ranks(1.0 if fits else 0.0, dev) > 0.0):
        share = (avail or 0) / local_world
        return {"value": None, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "unavailable": f"pinned host buffers need {need / 1e9:.1f} GB per rank, a rank's share of the host's "
                               f"available memory is {share / 1e9:.1f} GB"}
    t_pin = time.perf_counter()
    hG = torch.empty(owner.Gf.numel(), dtype=torch.bfloat16, pin_memory=True)
    hTg = torch.empty(owner.Tg.numel(), dtype=torch.float32, pin_memory=True)
    hW = torch.empty(owner.Wf.numel(), dtype=torch.float32, pin_memory=True)
    hWr = torch.empty(owner.Wr.numel(), dtype=torch.float32, pin_memory=True)
    hP = torch.empty(owner.Pf.numel(), dtype=torch.float32, pin_memory=True)
    pin_s = time.perf_counter() - t_pin
    h2d = hG.numel() * 2 + hTg.numel() * 4
    d2h = hW.numel() * 4 + hWr.numel() * 4 + hP.numel() * 4
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    hG.copy_(owner.Gf)
    hTg.copy_(owner.Tg)
    Gf, Tg = owner.Gf, owner.Tg
    Gf2, Tg2 = torch.empty_like(Gf), torch.empty_like(Tg)
    try:
        sW, sWr, sP = torch.empty_like(owner.Wf), torch.empty_like(owner.Wr), torch.empty_like(owner.Pf)
        staged = True
    except torch.cuda.OutOfMemoryError:
        # no room for the snapshots: read back from the live weights, each
        # step waiting until the previous read-back of them is done
        sW, sWr, sP = owner.Wf, owner.Wr, owner.Pf
        staged = False
    mo_ = owner.mo
    bufs = [(Gf, Tg, (owner.muon_tbl, owner.rmnp_tbl, owner.tail_tbl)),
            (Gf2, Tg2, (mo_.MuonTable(list(zip(owner.W_l, owner.views(Gf2), owner.V_l))),
                        mo_.MuonTable(list(zip(owner.Wr_l, owner.views(Gf2), owner.Vr_l))),
                        owner.tail_table(Tg2)))]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_free = [torch.cuda.Event(), torch.cuda.Event()]
    ev_w, ev_wout, ev_r, ev_rout = (torch.cuda.Event() for _ in range(4))
    owner.step(stream, tabs=bufs[1][2])     # plan the second tables outside the timed region
    torch.cuda.synchronize(dev)
    barrier()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(e2e_steps):
        b = k % 2
        Gd, Tgd, tabs = bufs[b]
        if k >= 2:
            s_in.wait_event(ev_free[b])   # step k-2 no longer reads buffer b
        with torch.cuda.stream(s_in):
            Gd.copy_(hG, non_blocking=True)
            Tgd.copy_(hTg, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])

        if k >= 1 and not staged:
            stream.wait_event(ev_wout)        # W is read back from the live buffer

        def after_muon():
            if staged:
                if k >= 1:
                    stream.wait_event(ev_wout)    # the previous snapshot of W has been read back
                torch.mul(owner.Wf, 1.0, out=sW)
            ev_w.record(stream)
            if k >= 1 and not staged:
                stream.wait_event(ev_rout)

        owner.step(stream, tabs=tabs, between=after_muon)
        ev_free[b].record(stream)
        if staged:
            if k >= 1:
                stream.wait_event(ev_rout)
            torch.mul(owner.Wr, 1.0, out=sWr)
            torch.mul(owner.Pf, 1.0, out=sP)
        ev_r.record(stream)
        s_out.wait_event(ev_w)
        with torch.cuda.stream(s_out):
            hW.copy_(sW, non_blocking=True)
        ev_wout.record(s_out)
        s_out.wait_event(ev_r)
        with torch.cuda.stream(s_out):
            hWr.copy_(sWr, non_blocking=True)
            hP.copy_(sP, non_blocking=True)
        ev_rout.record(s_out)
    stream.wait_event(ev_rout)
    e1.record(stream)
    barrier()
    e2e_ms_max = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    e2e_value = whole_job_tflops(world, ns_flops, e2e_ms_max)
    # the host link as this run sees it: one plain pinned copy each way, so a
    # link-bound e2e figure can be read against what the link delivered
    l0, l1, l2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    with torch.cuda.stream(s_out):
        l0.record(s_out)
        hW.copy_(owner.Wf, non_blocking=True)
        l1.record(s_out)
        Gf.copy_(hG, non_blocking=True)
        l2.record(s_out)
    l2.synchronize()
    link = {"d2h_gbs": round(hW.numel() * 4 / (l0.elapsed_time(l1) * 1e-3) / 1e9, 1),
            "h2d_gbs": round(hG.numel() * 2 / (l1.elapsed_time(l2) * 1e-3) / 1e9, 1)}
    return {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms_max, 3), "steps": e2e_steps,
            "link_measured": link, "pinned_alloc_s": round(pin_s, 1),
            "copies": "pinned host buffers; uploads, compute and read-backs on three streams, "
                      "gradients double-buffered on the device, "
                      + ("updated weights snapshotted on the device (an elementwise copy kernel inside the "
                         "step) and read back from the snapshots" if staged else
                         "updated weights read back from the live buffers (no device memory for snapshots)")}


# ---------------------------------------------------------------- next-row kernels (--extras)

def measure_extras(args, mo, workloads, wl, shapes, W_l, G_l, V_l, Wr_l, Vr_l, dev, stream, peaks):
    """Times the kernels beyond the benchmarked step on the same table (not
    part of the headline step): the Muon variants, column-cut RMNP, HTRMNP,
    the planned Muon step replayed from a CUDA graph, and the host-side owner
    planner. CUDA events on `stream`, 2 warm-up + 5 timed
    calls each."""
    import time
    import torch

    def timed(fn, reps=5, warm=2):
        for _ in range(warm):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    out = {}
    mats = list(zip(W_l, G_l, V_l))
    table = mo.MuonTable(mats)
    n_el = sum(r * c for r, c in shapes)

    def muon_variant(name, params, flops):
        ws = mo.muon_workspace(table, params, device=dev)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for e in evs:
            e.record(stream)
        ns = []

        def call():
            mo.muon_owner_step_timed(table, params, ws, evs[0], evs[1], stream=stream)

        total = timed(call)
        for _ in range(3):
            call()
            torch.cuda.synchronize(dev)
            ns.append(evs[0].elapsed_time(evs[1]))
        ns_ms = min(ns)
        out[name] = {"muon_step_ms": round(total, 4), "ns_ms": round(ns_ms, 4),
                     "ns_tflops_alg": round(flops / (ns_ms * 1e-3) / 1e12, 2),
                     "ns_frac_of_sustained_peak": round(flops / (ns_ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"], 4)}

    mn = [(min(r, c), max(r, c)) for r, c in shapes]
    muon_variant("muon_appendix_form", mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_form="appendix"),
                 sum(5 * 5 * m * m * n for m, n in mn))
    out["muon_appendix_form"]["flops_note"] = "5 iterations x (m^2 n Gram + 2 m^2 n A.X + 2 m^2 n A.B)"
    muon_variant("muon_convergence_settings",
                 mo.MuonParams(lr=1e-3, wd=1e-2, mu=0.5, ns_steps=2, lr_adjust="match_rms_adamw", nesterov=True),
                 sum(2 * (3 * m * m * n + m ** 3) for m, n in mn))

    # HTRMNP on the RMNP copy of the table, 18 bytes per element like RMNP
    rtable = mo.MuonTable(list(zip(Wr_l, G_l, Vr_l)))
    ms = timed(lambda: mo.htrmnp_step(rtable, mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu), stream=stream))
    gbs = n_el * workloads.RMNP_BYTES_PER_EL / (ms * 1e-3) / 1e9
    out["htrmnp"] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}

    # column-cut RMNP: every matrix cut into 4 column shards (own buffers)
    shards, groups, scales = [], [], []
    for g_id, (r, c) in enumerate(shapes):
        edges = [c * k // 4 for k in range(5)]
        for a, b in zip(edges[:-1], edges[1:]):
            if b > a:
                shards.append((torch.empty(r, b - a, device=dev).normal_(0, wl.w_std),
                               torch.empty(r, b - a, device=dev).normal_(0, wl.g_std).to(torch.bfloat16),
                               torch.zeros(r, b - a, device=dev)))
                groups.append(g_id)
                scales.append(max(1.0, r / c) ** 0.5)
    chunks = []
    k = 0
    while k < len(shards):                       # at most 512 shards per call, whole groups
        j = min(len(shards), k + 512)
        while j < len(shards) and j > k and groups[j] == groups[j - 1]:
            j -= 1
        chunks.append((k, j))
        k = j
    cp = mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, eps=1e-7)

    def colcut():
        for a, b in chunks:
            mo.rmnp_colcut_step(shards[a:b], groups[a:b], scales[a:b], cp, stream=stream)

    ms = timed(colcut)
    gbs = n_el * 22 / (ms * 1e-3) / 1e9
    out["rmnp_colcut_4_shards"] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                                   "bytes_per_el": 22}

    # the planned Muon step replayed from a CUDA graph against per-call
    # steps, on the whole table and on its first four matrices (one layer),
    # where launch and host overhead weigh most
    def graph_vs_eager(name, sub):
        t = mo.MuonTable(sub)
        p = mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu)
        ws_e = mo.muon_workspace(t, p, device=dev)
        eager = timed(lambda: mo.muon_owner_step(t, p, ws_e, stream=stream))
        plan = mo.MuonPlan(t, p, stream=stream)
        plan.step(stream=stream)                 # first launches outside the capture
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            plan.step()

        def replay():
            with torch.cuda.stream(stream):
                graph.replay()

        replayed = timed(replay)
        plan.close()
        out[name] = {"matrices": len(sub), "per_call_ms": round(eager, 4), "graph_replay_ms": round(replayed, 4)}

    graph_vs_eager("muon_graph_replay_table", mats)
    graph_vs_eager("muon_graph_replay_one_layer", mats[:4])

    # owner planner (host only): GPT-2 Large-style roles over 8 ranks
    roles = workloads.owner_roles(wl, 4 if len(shapes) % 4 == 0 else 1)
    t0 = time.perf_counter()
    for _ in range(20):
        mo.mo_plan_owners(roles, 8)
    out["owner_planner_8_ranks_us"] = round((time.perf_counter() - t0) / 20 * 1e6, 1)
    return out


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank):
    """The CPU oracle as it stands, on the host cores: each step is one
    whole-matrix Muon step of the oracle on a matrix of the workload, cycling
    through the distinct shapes whose oracle step costs at most three times
    the cheapest one (a bounded sample: the 8B table's largest matrices take
    the oracle about half a minute each)."""
    if rank != 0:
        return None
    from matrix_optimizers_zero_gb300 import workloads
    wl = workloads.get_workload(args.config)
    by_cost = distinct_shapes_by_cost(wl)

    def cost(i):
        return workloads.ns_alg_flops(wl.matrices[i].rows, wl.matrices[i].cols, wl.ns_steps)

    picks = [i for i in by_cost if cost(i) <= 3 * cost(by_cost[0])]
    cores = len(os.sched_getaffinity(0))
    for k in range(args.warmup):
        oracle_matrix_seconds(wl, picks[k % len(picks)])
    times, flops = [], 0
    for k in range(args.steps):
        secs, f = oracle_matrix_seconds(wl, picks[k % len(picks)])
        times.append(secs)
        flops += f
    total = sum(times)
    value = flops / total / 1e12
    shapes = ", ".join(f"{wl.matrices[i].rows}x{wl.matrices[i].cols}" for i in picks)
    desc = (f"each step: the oracle's whole-matrix Muon step (fp64 numpy, bf16 emulation) on one matrix of "
            f"the {wl.name} table, cycling through the shapes [{shapes}]")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {len(wl.matrices)} matrices, {wl.n_elements} elements, "
                               f"tail {wl.tail_elements}",
                   "sample": "bounded sample per step (see cpu_baseline)", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--cpu-seconds", type=float, default=25.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end loop (profiling runs)")
    ap.add_argument("--e2e-steps", type=int, default=10, help="end-to-end steps (at most --steps)")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false",
                    help=f"skip the second workload ({SECONDARY_CONFIG}) timed after the headline")
    ap.add_argument("--secondary-steps", type=int, default=20)
    ap.add_argument("--extras", action="store_true",
                    help="also time the next-row kernels (Muon variants, column-cut RMNP, HTRMNP, graph "
                         "replay, planner) on the --extras-config table")
    ap.add_argument("--extras-config", default=SECONDARY_CONFIG)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        out = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
