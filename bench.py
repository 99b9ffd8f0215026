"""Benchmark of the owner-local optimizer step on GB300.

One step = the whole hot path over one owner's table: the Muon step on every
2D matrix (momentum, Frobenius normalisation, five quintic Newton-Schulz
iterations, shape-scaled update with weight decay), AdamW on the packed
non-matrix tail, and RMNP on the same matrices (its own momentum and weight
copies). Default workload: the GPT-2 Large matrix set (144 matrices, 707.8 M
elements; tail 601,600 elements), synthetic seeded inputs resident in HBM.
The working set (~17 GB) is far larger than L2, so no flush is needed.

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

# DRAM bytes of one step's 15 Newton-Schulz launches on the GPT-2 Large table,
# from ncu (dram__bytes_read.sum + dram__bytes_write.sum, one pass) over the 15
# NS launches of one step on the full table
# (profiles/ns_gemm_pair_gpt2l_tensor_active.md).
# Valid only for the kernel source and tile schedule it was measured on.
NS_TRAFFIC = {"source_sha256_16": "27380c248ef7ee14", "workload": "gpt2l", "bytes_per_ns_segment": 36.92e9}
UNIT = "TFLOP/s"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def ns_traffic(workload: str):
    """The profiled DRAM traffic of the NS launches, or None when the kernel
    or its tile schedule differs from the one profiled (or for another
    workload)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("ns_gemm.cu", "plan.cpp"):
        with open(os.path.join(ROOT, "matrix_optimizers_zero_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != NS_TRAFFIC["source_sha256_16"] or workload != NS_TRAFFIC["workload"]:
        return None
    return NS_TRAFFIC["bytes_per_ns_segment"]


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

def cpu_oracle_sample(wl, max_seconds=20.0, indices=None, min_seconds=0.0):
    """Times the CPU oracle (as it stands) on a bounded sample of the
    workload: whole-matrix Muon steps on one matrix per distinct shape, in
    table order (repeated until min_seconds of work), stopping once
    max_seconds is spent. Returns (TFLOP/s, seconds, description, cores)."""
    import numpy as np
    import oracle
    from matrix_optimizers_zero_gb300 import workloads
    cores = len(os.sched_getaffinity(0))
    seen, picks = set(), []
    for i, s in enumerate(wl.matrices):
        if (s.rows, s.cols) not in seen:
            seen.add((s.rows, s.cols))
            picks.append(i)
    if indices is not None:
        picks = indices
    flops = 0
    t_total = 0.0
    done = []
    order = list(picks) * (8 if min_seconds > 0 else 1)
    for k, i in enumerate(order):
        if k >= len(picks) and t_total >= min_seconds:
            break
        W, G, V = workloads.host_matrix(wl, i, v_std=1e-3)
        W, G, V = (t.float().double().numpy() for t in (W, G, V))
        t0 = time.perf_counter()
        oracle.muon_matrix_step(W, G, V, lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_steps=wl.ns_steps)
        t_total += time.perf_counter() - t0
        s = wl.matrices[i]
        flops += workloads.ns_alg_flops(s.rows, s.cols, wl.ns_steps)
        done.append(f"{s.rows}x{s.cols}")
        if t_total > max_seconds:
            break
    desc = f"oracle muon_matrix_step (fp64 numpy, bf16 emulation) on {len(done)} matrices [{', '.join(done)}]"
    return flops / t_total / 1e12, t_total, desc, cores


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import matrix_optimizers_zero_gb300 as mo
    from matrix_optimizers_zero_gb300 import build as mo_build, workloads

    mo_build.build()
    mo.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = workloads.get_workload(args.config)
    peaks = load_peaks()

    # ---- state: flat device buffers with per-matrix views (one copy each for e2e)
    shapes = [(s.rows, s.cols) for s in wl.matrices]
    offs, tot = [], 0
    for r, c in shapes:
        offs.append(tot)
        tot += ((r * c + 63) // 64) * 64
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    Wf = torch.randn(tot, generator=gen, device=dev).mul_(wl.w_std)
    Gf = torch.randn(tot, generator=gen, device=dev).mul_(wl.g_std).to(torch.bfloat16)
    Vf = torch.randn(tot, generator=gen, device=dev).mul_(1e-3)
    Wr = Wf.clone()
    Vr = Vf.clone()

    def views(flat):
        return [flat[o:o + r * c].view(r, c) for o, (r, c) in zip(offs, shapes)]

    W_l, G_l, V_l, Wr_l, Vr_l = views(Wf), views(Gf), views(Vf), views(Wr), views(Vr)
    muon_tbl = mo.MuonTable(list(zip(W_l, G_l, V_l)))
    rmnp_tbl = mo.MuonTable(list(zip(Wr_l, G_l, Vr_l)))
    tail_sizes = [t for t in wl.tail if t > 0]
    toffs, ttot = [], 0
    for t in tail_sizes:
        toffs.append(ttot)
        ttot += ((t + 63) // 64) * 64
    Pf = torch.randn(max(ttot, 1), generator=gen, device=dev).mul_(wl.tail_p_std)
    Tg = torch.randn(max(ttot, 1), generator=gen, device=dev).mul_(wl.tail_g_std)
    Tm = torch.zeros(max(ttot, 1), device=dev)
    Tv = torch.zeros(max(ttot, 1), device=dev)
    segs = [(Pf[o:o + t], Tg[o:o + t], Tm[o:o + t], Tv[o:o + t]) for o, t in zip(toffs, tail_sizes)]
    tail_tbl = mo.TailTable(segs)

    mp = mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_steps=wl.ns_steps)
    rp = mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu)
    ws = mo.muon_workspace(muon_tbl, mp, device=dev)
    stream = torch.cuda.current_stream(dev)
    lib = mo.load_library()
    import ctypes
    ws_ptr, ws_bytes = ws.data_ptr(), ws.numel()
    sptr = stream.cuda_stream
    adam_step = [0]
    # NVTX ranges name each library call on the host timeline (ncu --nvtx
    # can filter on them); they add no device work
    nvtx = torch.cuda.nvtx

    def step(ev=None, tabs=None, between=None):
        """One optimizer step on `stream`: Muon, AdamW on the tail, RMNP.
        tabs: (muon, rmnp, tail) tables to use (default: the resident ones);
        between: called after the Muon call, before AdamW and RMNP."""
        m_tbl, r_tbl, t_tbl = tabs if tabs is not None else (muon_tbl, rmnp_tbl, tail_tbl)
        nvtx.range_push("muon_owner_step")
        if ev is None:
            st = lib.muon_owner_step(m_tbl.ptr, m_tbl.n, ctypes.byref(mp), ws_ptr, ws_bytes, sptr)
        else:
            ev[0].record(stream)
            st = lib.muon_owner_step_timed(muon_tbl.ptr, muon_tbl.n, ctypes.byref(mp), ws_ptr, ws_bytes, sptr,
                                           ev[1].cuda_event, ev[2].cuda_event)
        nvtx.range_pop()
        if st != 0:
            raise mo.MoError(st, "muon_owner_step")
        if ev is not None:
            ev[3].record(stream)
        if between is not None:
            between()
        adam_step[0] += 1
        ap = mo.AdamWParams(lr=wl.adam_lr, wd=wl.adam_wd, beta1=wl.beta1, beta2=wl.beta2, eps=wl.adam_eps,
                            step=adam_step[0])
        nvtx.range_push("adamw_tail_step")
        st = lib.adamw_tail_step(t_tbl.ptr, t_tbl.n, ctypes.byref(ap), sptr)
        nvtx.range_pop()
        if st != 0:
            raise mo.MoError(st, "adamw_tail_step")
        if ev is not None:
            ev[4].record(stream)
        nvtx.range_push("rmnp_step")
        st = lib.rmnp_step(r_tbl.ptr, r_tbl.n, ctypes.byref(rp), sptr)
        nvtx.range_pop()
        if st != 0:
            raise mo.MoError(st, "rmnp_step")
        if ev is not None:
            ev[5].record(stream)

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- warmup
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if mo.mo_last_device_error() != 0:
        raise RuntimeError("device-side timeout during warmup")

    # ---- timed region (kernel-level: inputs resident in HBM)
    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for e in evs:
        for x in e:
            x.record(stream)          # torch creates events lazily: force the handles to exist
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    clocks.mark("begin")
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    barrier()
    clocks.mark("end")
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    ms_step = total_ms / args.steps
    pro_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ns_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    muon_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in evs)
    adam_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)
    rmnp_ms = statistics.mean(e[4].elapsed_time(e[5]) for e in evs)
    # per-step minima (each step's events from its Muon start to its RMNP end)
    step_min_ms = min(e[0].elapsed_time(e[5]) for e in evs)
    ns_min_ms = min(e[1].elapsed_time(e[2]) for e in evs)

    ns_flops = workloads.workload_alg_flops(wl)
    ns_dense = sum(workloads.ns_dense_flops(r, c, wl.ns_steps) for r, c in shapes)
    n_el = wl.n_elements
    ns_tflops = ns_flops / (ns_ms * 1e-3) / 1e12
    rmnp_gbs = n_el * workloads.RMNP_BYTES_PER_EL / (rmnp_ms * 1e-3) / 1e9
    adam_gbs = wl.tail_elements * workloads.ADAMW_BYTES_PER_EL / (adam_ms * 1e-3) / 1e9
    pro_gbs = n_el * 16 / (pro_ms * 1e-3) / 1e9

    ms_max = max_over_ranks(ms_step, dev)
    value = whole_job_tflops(world, ns_flops, ms_max)

    # ---- end to end through the C ABI with host buffers. Every step uploads
    # its gradients (Muon/RMNP G and the tail's g) from pinned host memory and
    # reads all updated weights back (Muon W, RMNP W, tail p). Uploads, compute
    # and read-backs run on three streams: the gradients are double-buffered on
    # the device so step k+1's upload overlaps step k; a step's Muon call waits
    # until the previous step's Muon weights have been read back, its AdamW
    # and RMNP calls until the previous RMNP weights and tail have been.
    e2e_steps = 0 if args.no_e2e else max(1, min(args.steps, 10))
    pin = e2e_steps > 0
    hG = torch.empty(Gf.numel() if pin else 1, dtype=torch.bfloat16, pin_memory=pin)
    hTg = torch.empty(Tg.numel() if pin else 1, dtype=torch.float32, pin_memory=pin)
    hW = torch.empty(Wf.numel() if pin else 1, dtype=torch.float32, pin_memory=pin)
    hWr = torch.empty(Wr.numel() if pin else 1, dtype=torch.float32, pin_memory=pin)
    hP = torch.empty(Pf.numel() if pin else 1, dtype=torch.float32, pin_memory=pin)
    h2d = hG.numel() * 2 + hTg.numel() * 4
    d2h = hW.numel() * 4 + hWr.numel() * 4 + hP.numel() * 4
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if pin:
        hG.copy_(Gf)
        hTg.copy_(Tg)
        Gf2, Tg2 = torch.empty_like(Gf), torch.empty_like(Tg)
        G2_l = views(Gf2)
        segs2 = [(Pf[o:o + t], Tg2[o:o + t], Tm[o:o + t], Tv[o:o + t]) for o, t in zip(toffs, tail_sizes)]
        bufs = [(Gf, Tg, (muon_tbl, rmnp_tbl, tail_tbl)),
                (Gf2, Tg2, (mo.MuonTable(list(zip(W_l, G2_l, V_l))), mo.MuonTable(list(zip(Wr_l, G2_l, Vr_l))),
                            mo.TailTable(segs2)))]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_free = [torch.cuda.Event(), torch.cuda.Event()]
        ev_w, ev_wout, ev_r, ev_rout = (torch.cuda.Event() for _ in range(4))
        step(tabs=bufs[1][2])               # plan the second tables outside the timed region
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
            if k >= 1:
                stream.wait_event(ev_wout)

            def after_muon():
                ev_w.record(stream)
                if k >= 1:
                    stream.wait_event(ev_rout)

            step(tabs=tabs, between=after_muon)
            ev_r.record(stream)
            ev_free[b].record(stream)
            s_out.wait_event(ev_w)
            with torch.cuda.stream(s_out):
                hW.copy_(Wf, non_blocking=True)
            ev_wout.record(s_out)
            s_out.wait_event(ev_r)
            with torch.cuda.stream(s_out):
                hWr.copy_(Wr, non_blocking=True)
                hP.copy_(Pf, non_blocking=True)
            ev_rout.record(s_out)
        stream.wait_event(ev_rout)
        e1.record(stream)
    else:
        e0.record(stream)
        e1.record(stream)
    barrier()
    e2e_ms_max = max_over_ranks(e0.elapsed_time(e1) / max(e2e_steps, 1), dev)
    e2e_value = whole_job_tflops(world, ns_flops, e2e_ms_max)
    # the host link as this run sees it: one plain pinned copy each way, so a
    # link-bound e2e figure can be read against what the link delivered
    link = None
    if pin:
        l0, l1, l2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        with torch.cuda.stream(s_out):
            l0.record(s_out)
            hW.copy_(Wf, non_blocking=True)
            l1.record(s_out)
            Gf.copy_(hG, non_blocking=True)
            l2.record(s_out)
        l2.synchronize()
        link = {"d2h_gbs": round(hW.numel() * 4 / (l0.elapsed_time(l1) * 1e-3) / 1e9, 1),
                "h2d_gbs": round(hG.numel() * 2 / (l1.elapsed_time(l2) * 1e-3) / 1e9, 1)}
    if mo.mo_last_device_error() != 0:
        raise RuntimeError("device-side timeout during the timed region")

    extras = measure_extras(args, mo, workloads, wl, shapes, W_l, G_l, V_l, Wr_l, Vr_l, dev, stream, peaks) \
        if args.extras else None

    if rank != 0:
        return None

    # prologue + 3 GEMM launches per iteration; AdamW: one per 256 segments;
    # RMNP: one per 512 entries, separately for rows shorter / not shorter
    # than 8192 elements (warp-per-row and CTA-per-row kernels)
    n_long = sum(1 for _, c in shapes if c >= 8192)
    launches_per_step = ((1 + 3 * wl.ns_steps) + math.ceil(len(tail_sizes) / 256)
                         + math.ceil((len(shapes) - n_long) / 512) + math.ceil(n_long / 512))
    peak = peaks["bf16_tflops_sustained"]
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
        "breakdown": {
            "muon_step_ms": round(muon_ms, 4),
            "prologue_ms": round(pro_ms, 4),
            "prologue_gbs": round(pro_gbs, 1),
            "ns_ms": round(ns_ms, 4),
            "ns_tflops_alg": round(ns_tflops, 2),
            "ns_tflops_dense_equiv": round(ns_dense / (ns_ms * 1e-3) / 1e12, 2),
            "adamw_ms": round(adam_ms, 4),
            "adamw_gbs": round(adam_gbs, 1),
            "rmnp_ms": round(rmnp_ms, 4),
            "rmnp_gbs": round(rmnp_gbs, 1),
            "rmnp_frac_hbm": round(rmnp_gbs / peaks["hbm_gbs"], 4),
            "means_over_steps": args.steps,
            "step_min_ms": round(step_min_ms, 4),
            "ns_min_ms": round(ns_min_ms, 4),
            "ns_tflops_alg_best": round(ns_flops / (ns_min_ms * 1e-3) / 1e12, 2),
        },
        "roofline": {
            "bound": "tensor",
            "kernel": "ns_gemm_pair_kernel (the 15 Gram, A.A and B.X launches of one step)",
            "achieved": round(ns_tflops, 2),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(ns_tflops / peak, 4),
            "traffic": ns_traffic(wl.name),
            "traffic_unit": "DRAM bytes per step's 15 NS launches (ncu, full table, single-pass metrics)",
            "peak_source": f"bf16_tflops_sustained ({peaks['source']})",
        },
        "e2e": ({"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                 "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms_max, 3), "steps": e2e_steps,
                 "link_measured": link,
                 "copies": "pinned host buffers; uploads, compute and read-backs on three streams, "
                           "gradients double-buffered on the device"}
                if e2e_steps else None),
        "gpu_launches": int(launches_per_step * args.steps),
        **({"extras": extras} if extras is not None else {}),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        v, secs, desc, cores = cpu_oracle_sample(wl, max_seconds=args.cpu_seconds, min_seconds=10.0)
        out["cpu_baseline"] = {"value": round(v, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": desc, "seconds": round(secs, 2)}
    return out


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
    if rank != 0:
        return None
    from matrix_optimizers_zero_gb300 import workloads
    wl = workloads.get_workload(args.config)
    seen, picks = set(), []
    for i, s in enumerate(wl.matrices):
        if (s.rows, s.cols) not in seen:
            seen.add((s.rows, s.cols))
            picks.append(i)
    cores = len(os.sched_getaffinity(0))
    for k in range(args.warmup):
        cpu_oracle_sample(wl, max_seconds=0.0, indices=[picks[k % len(picks)]])
    times, flops = [], 0
    for k in range(args.steps):
        i = picks[k % len(picks)]
        v, secs, _, _ = cpu_oracle_sample(wl, max_seconds=0.0, indices=[i])
        s = wl.matrices[i]
        times.append(secs)
        flops += workloads.ns_alg_flops(s.rows, s.cols, wl.ns_steps)
    total = sum(times)
    value = flops / total / 1e12
    desc = (f"each step: the oracle's whole-matrix Muon step on one matrix of the {wl.name} table, cycling "
            f"through its {len(picks)} distinct shapes")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name} (bounded sample per step)", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="gpt2l")
    ap.add_argument("--cpu-seconds", type=float, default=25.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end loop (profiling runs)")
    ap.add_argument("--extras", action="store_true",
                    help="also time the next-row kernels (Muon variants, column-cut RMNP, HTRMNP, planner)")
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
