"""GB300 (sm_103a) owner-local optimizer step: Muon on whole 2D matrices,
AdamW on the packed tail, RMNP row normalisation.

This module is a thin ctypes binding over the C ABI in include/mo.h: it only
marshals torch tensors into the C tables and raises on error statuses. Every
step of the computation runs in the library's CUDA kernels; there is no
Python or CPU fallback, and importing the binding fails loudly when the
library has not been built (python -m matrix_optimizers_zero_gb300.build).

Typical use on one owner (tensors on the current CUDA device; W and V fp32,
G bf16, all of shape [rows, cols], contiguous):

    import matrix_optimizers_zero_gb300 as mo
    mats = [(W, G, V) for ...]                    # the owner's 2D matrices
    p = mo.MuonParams(lr=0.02, wd=0.01, mu=0.95)  # ns_form / lr_adjust / nesterov for the variants
    ws = mo.muon_workspace(mats, p)               # reuse it across steps
    mo.muon_owner_step(mats, p, ws)               # momentum, Newton-Schulz, weight update
    mo.adamw_tail_step(segments, mo.AdamWParams(step=t))
    mo.rmnp_step(mats_rmnp, mo.RmnpParams())
    assert mo.mo_last_device_error() == 0         # synchronises; bounded device waits

Plans (tile schedules, tensor maps) are cached per (table, workspace), so a
training loop that passes the same tensors every step plans once.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, List, Optional, Sequence, Tuple

from .build import LIB_PATH

__all__ = [
    "MoError", "MuonParams", "RmnpParams", "AdamWParams", "load_library",
    "mo_muon_workspace_bytes", "muon_workspace", "muon_owner_step", "muon_owner_step_timed",
    "rmnp_step", "rmnp_step_scaled", "htrmnp_step", "adamw_tail_step", "mo_last_device_error",
    "mo_status_string", "mo_selftest_bounded_wait", "mo_muon_tile_schedule", "MuonTable",
    "TailTable", "RmnpTable", "muon_owner_step_noalloc", "mo_static_scratch_bytes", "mo_plan_owners",
    "rmnp_colcut_step", "muon_owner_step_coverage",
]

MO_OK = 0
PHASE_GRAM, PHASE_POLY, PHASE_UPDATE = 0, 1, 2


class MoMatrix(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("G", ctypes.c_void_p), ("V", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


NS_FORMS = {"gram": 0, "appendix": 1}                  # mo_ns_form
LR_ADJUST = {"original": 0, "match_rms_adamw": 1}      # mo_lr_adjust


class MuonParams(ctypes.Structure):
    """mo_muon_params. ns_form and lr_adjust take the names of NS_FORMS and
    LR_ADJUST (or their integer codes)."""
    _fields_ = [("lr", ctypes.c_float), ("wd", ctypes.c_float), ("mu", ctypes.c_float),
                ("a", ctypes.c_float), ("b", ctypes.c_float), ("c", ctypes.c_float),
                ("eps", ctypes.c_float), ("ns_steps", ctypes.c_int32), ("ns_form", ctypes.c_int32),
                ("lr_adjust", ctypes.c_int32), ("nesterov", ctypes.c_int32)]

    def __init__(self, lr=0.02, wd=0.01, mu=0.95, a=3.4445, b=-4.7750, c=2.0315, eps=1e-7, ns_steps=5,
                 ns_form="gram", lr_adjust="original", nesterov=False):
        form = NS_FORMS[ns_form] if isinstance(ns_form, str) else int(ns_form)
        adj = LR_ADJUST[lr_adjust] if isinstance(lr_adjust, str) else int(lr_adjust)
        super().__init__(lr, wd, mu, a, b, c, eps, ns_steps, form, adj, int(nesterov))


class RmnpParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("wd", ctypes.c_float), ("mu", ctypes.c_float),
                ("eps", ctypes.c_float)]

    def __init__(self, lr=0.02, wd=0.01, mu=0.95, eps=1e-12):
        super().__init__(lr, wd, mu, eps)


class MoTailSeg(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("v", ctypes.c_void_p), ("numel", ctypes.c_int64)]


class AdamWParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("wd", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float), ("step", ctypes.c_int64)]

    def __init__(self, lr=1e-3, wd=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, step=1):
        super().__init__(lr, wd, beta1, beta2, eps, step)


class MoRole(ctypes.Structure):
    _fields_ = [("numel", ctypes.c_int64), ("block", ctypes.c_int32), ("is_tail", ctypes.c_int32)]


PLAN_ROLE_GREEDY, PLAN_SCOPE_GREEDY, PLAN_COST_AWARE = 0, 1, 2


class MoTile(ctypes.Structure):
    _fields_ = [("mat", ctypes.c_uint32), ("tm", ctypes.c_uint16), ("tn", ctypes.c_uint16)]


class MoError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = mo_status_string(status)
        if status == -7:
            msg += f" (cudaError {load_library().mo_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{status}]")


_lib = None


def load_library() -> ctypes.CDLL:
    """Loads the in-tree libmo.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m matrix_optimizers_zero_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "mo_muon_workspace_bytes": (SZ, [P, I32, P]),
        "muon_owner_step": (ctypes.c_int, [P, I32, P, P, SZ, P]),
        "muon_owner_step_timed": (ctypes.c_int, [P, I32, P, P, SZ, P, P, P]),
        "adamw_tail_step": (ctypes.c_int, [P, I32, P, P]),
        "rmnp_step": (ctypes.c_int, [P, I32, P, P]),
        "rmnp_step_scaled": (ctypes.c_int, [P, P, I32, P, P]),
        "htrmnp_step": (ctypes.c_int, [P, I32, P, ctypes.c_float, P]),
        "mo_last_device_error": (ctypes.c_int, [P]),
        "mo_last_cuda_error": (ctypes.c_int, []),
        "mo_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "mo_abi_version": (ctypes.c_int, []),
        "mo_muon_tile_schedule": (ctypes.c_int, [P, I32, I32, P, I64, P]),
        "muon_owner_step_coverage": (ctypes.c_int, [P, I32, P, P, SZ, P, I64, I32, P, P]),
        "mo_selftest_bounded_wait": (ctypes.c_int, [I64, P]),
        "muon_owner_step_noalloc": (ctypes.c_int, [P, I32, P, P]),
        "mo_plan_owners": (ctypes.c_int, [P, I32, I32, I32, I64, P, P, P]),
        "mo_rmnp_colcut_workspace_bytes": (SZ, [P, I32]),
        "rmnp_colcut_step": (ctypes.c_int, [P, P, P, I32, P, P, SZ, P]),
        "mo_static_scratch_bytes": (SZ, []),
        "adamw_tail_step_dev": (ctypes.c_int, [P, I32, P, P, P, P]),
        "rmnp_step_dev": (ctypes.c_int, [P, I32, P, ctypes.c_float, P, P]),
        "mo_muon_plan_create": (ctypes.c_int, [P, I32, P, P, SZ, P, P]),
        "mo_muon_plan_step": (ctypes.c_int, [P, P]),
        "mo_muon_plan_lr_ptr": (P, [P]),
        "mo_muon_plan_destroy": (ctypes.c_int, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != MO_OK:
        raise MoError(status, where)


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def mo_status_string(status: int) -> str:
    return load_library().mo_status_string(int(status)).decode()


# ---------------------------------------------------------------- tables

class MuonTable:
    """ctypes shape table for a list of (W fp32, G bf16, V fp32) CUDA tensors.
    Build it once and reuse it across steps to keep host overhead out of the
    step."""

    def __init__(self, mats: Sequence[Tuple["object", "object", "object"]]):
        import torch
        self.n = len(mats)
        self.arr = (MoMatrix * max(1, self.n))()
        for i, (W, G, V) in enumerate(mats):
            if W.dtype != torch.float32 or V.dtype != torch.float32 or G.dtype != torch.bfloat16:
                raise TypeError("expected W fp32, G bf16, V fp32")
            if W.dim() != 2 or W.shape != G.shape or W.shape != V.shape:
                raise ValueError("W, G, V must be 2D with equal shapes")
            if not (W.is_contiguous() and G.is_contiguous() and V.is_contiguous()):
                raise ValueError("W, G, V must be contiguous")
            self.arr[i] = MoMatrix(W.data_ptr(), G.data_ptr(), V.data_ptr(), W.shape[0], W.shape[1])
        self.keep = list(mats)

    @property
    def ptr(self):
        return ctypes.cast(self.arr, ctypes.c_void_p) if self.n else None


RmnpTable = MuonTable


class TailTable:
    """ctypes table of AdamW tail segments (p, g, m, v) fp32 CUDA tensors."""

    def __init__(self, segs: Sequence[Tuple["object", "object", "object", "object"]]):
        import torch
        self.n = len(segs)
        self.arr = (MoTailSeg * max(1, self.n))()
        for i, (p, g, m, v) in enumerate(segs):
            for t in (p, g, m, v):
                if t.dtype != torch.float32 or not t.is_contiguous():
                    raise TypeError("tail tensors must be contiguous fp32")
                if t.numel() != p.numel():
                    raise ValueError("p, g, m, v must have equal sizes")
            self.arr[i] = MoTailSeg(p.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr(), p.numel())
        self.keep = list(segs)

    @property
    def ptr(self):
        return ctypes.cast(self.arr, ctypes.c_void_p) if self.n else None


def _as_table(mats, cls=MuonTable):
    return mats if isinstance(mats, cls) else cls(mats)


# ---------------------------------------------------------------- Muon

def mo_muon_workspace_bytes(mats, params: Optional[MuonParams] = None) -> int:
    t = _as_table(mats)
    params = params or MuonParams()
    return int(load_library().mo_muon_workspace_bytes(t.ptr, t.n, ctypes.byref(params)))


def muon_workspace(mats, params: Optional[MuonParams] = None, device=None):
    """A torch uint8 device tensor large enough for muon_owner_step."""
    import torch
    t = _as_table(mats)
    nbytes = mo_muon_workspace_bytes(t, params)
    if device is None:
        device = t.keep[0][0].device if t.n else torch.device("cuda")
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def muon_owner_step(mats, params: Optional[MuonParams] = None, workspace=None, stream=None) -> None:
    t = _as_table(mats)
    params = params or MuonParams()
    if workspace is None:
        raise ValueError("muon_owner_step needs a workspace (see muon_workspace())")
    st = load_library().muon_owner_step(t.ptr, t.n, ctypes.byref(params), workspace.data_ptr(),
                                        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(st, "muon_owner_step")


def muon_owner_step_timed(mats, params, workspace, ev_begin, ev_end, stream=None) -> None:
    t = _as_table(mats)
    st = load_library().muon_owner_step_timed(
        t.ptr, t.n, ctypes.byref(params), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream), ev_begin.cuda_event if ev_begin is not None else None,
        ev_end.cuda_event if ev_end is not None else None)
    _check(st, "muon_owner_step_timed")


def muon_owner_step_noalloc(mats, params: Optional[MuonParams] = None, stream=None) -> None:
    """muon_owner_step without a caller workspace, for callers that cannot
    allocate device memory: the library's fixed scratch array is used instead
    (tables up to mo_static_scratch_bytes() of workspace). Calls that overlap
    on the GPU share that array and race."""
    t = _as_table(mats)
    params = params or MuonParams()
    _check(load_library().muon_owner_step_noalloc(t.ptr, t.n, ctypes.byref(params), _stream_ptr(stream)),
           "muon_owner_step_noalloc")


def mo_static_scratch_bytes() -> int:
    return int(load_library().mo_static_scratch_bytes())


class MuonPlan:
    """A Muon step planned once (mo_muon_plan_create): step() enqueues device
    work only, so it can be captured in a CUDA graph and replayed. The
    workspace belongs to the plan while it exists. `lr` is a one-element fp32
    device tensor viewing the learning rate every step reads; write it (for
    example with lr.fill_()) to follow a schedule between steps or replays."""

    def __init__(self, mats, params: Optional[MuonParams] = None, workspace=None, stream=None):
        import torch
        self.table = _as_table(mats)
        self.params = params or MuonParams()
        self.workspace = workspace if workspace is not None else muon_workspace(self.table, self.params)
        lib = load_library()
        handle = ctypes.c_void_p()
        st = lib.mo_muon_plan_create(self.table.ptr, self.table.n, ctypes.byref(self.params),
                                     self.workspace.data_ptr(),
                                     self.workspace.numel() * self.workspace.element_size(),
                                     _stream_ptr(stream), ctypes.byref(handle))
        _check(st, "mo_muon_plan_create")
        self._handle = handle
        lr_off = lib.mo_muon_plan_lr_ptr(handle) - self.workspace.data_ptr()
        self.lr = self.workspace[lr_off:lr_off + 4].view(torch.float32)

    def step(self, stream=None) -> None:
        _check(load_library().mo_muon_plan_step(self._handle, _stream_ptr(stream)), "mo_muon_plan_step")

    def close(self) -> None:
        if self._handle is not None and _lib is not None:
            _lib.mo_muon_plan_destroy(self._handle)
        self._handle = None

    def __del__(self):
        self.close()


# ---------------------------------------------------------------- RMNP / AdamW

def rmnp_step(mats, params: Optional[RmnpParams] = None, stream=None) -> None:
    t = _as_table(mats)
    params = params or RmnpParams()
    _check(load_library().rmnp_step(t.ptr, t.n, ctypes.byref(params), _stream_ptr(stream)), "rmnp_step")


HTRMNP_POWER = 0.125


def htrmnp_step(mats, params: Optional[RmnpParams] = None, power: float = HTRMNP_POWER, stream=None) -> None:
    """RMNP with the row direction scaled by ||V_i||^power (see include/mo.h)."""
    t = _as_table(mats)
    params = params or RmnpParams()
    _check(load_library().htrmnp_step(t.ptr, t.n, ctypes.byref(params), float(power), _stream_ptr(stream)),
           "htrmnp_step")


def rmnp_step_dev(mats, params, lr, power: float = 0.0, stream=None) -> None:
    """rmnp_step (power 0) or htrmnp_step with lr read from the one-element
    fp32 CUDA tensor `lr` when the kernels run (capturable in a CUDA graph)."""
    import torch
    t = _as_table(mats)
    if lr.dtype != torch.float32 or lr.numel() != 1 or not lr.is_cuda:
        raise TypeError("lr must be a one-element fp32 CUDA tensor")
    _check(load_library().rmnp_step_dev(t.ptr, t.n, ctypes.byref(params), float(power), lr.data_ptr(),
                                        _stream_ptr(stream)), "rmnp_step_dev")


def rmnp_step_scaled(mats, scales: Sequence[float], params: Optional[RmnpParams] = None, stream=None) -> None:
    t = _as_table(mats)
    params = params or RmnpParams()
    arr = (ctypes.c_float * max(1, len(scales)))(*[float(s) for s in scales])
    _check(load_library().rmnp_step_scaled(t.ptr, ctypes.cast(arr, ctypes.c_void_p), t.n,
                                           ctypes.byref(params), _stream_ptr(stream)), "rmnp_step_scaled")


def rmnp_colcut_step(shards, groups: Sequence[int], scales: Sequence[float], params: Optional[RmnpParams] = None,
                     workspace=None, stream=None) -> None:
    """Column-cut RMNP over column shards (W, G, V) of logical matrices;
    shards with equal group ids belong to one matrix. `workspace` is a device
    tensor of at least mo_rmnp_colcut_workspace_bytes bytes (allocated with
    torch when None)."""
    import torch
    t = _as_table(shards)
    params = params or RmnpParams(eps=1e-7)
    lib = load_library()
    nbytes = int(lib.mo_rmnp_colcut_workspace_bytes(t.ptr, t.n))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=t.keep[0][0].device)
    g = (ctypes.c_int32 * max(1, t.n))(*[int(x) for x in groups])
    sc = (ctypes.c_float * max(1, t.n))(*[float(x) for x in scales])
    _check(lib.rmnp_colcut_step(t.ptr, ctypes.cast(g, ctypes.c_void_p), ctypes.cast(sc, ctypes.c_void_p), t.n,
                                ctypes.byref(params), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "rmnp_colcut_step")


def adamw_tail_step(segs, params: Optional[AdamWParams] = None, stream=None) -> None:
    t = segs if isinstance(segs, TailTable) else TailTable(segs)
    params = params or AdamWParams()
    _check(load_library().adamw_tail_step(t.ptr, t.n, ctypes.byref(params), _stream_ptr(stream)),
           "adamw_tail_step")


def adamw_tail_step_dev(segs, params, step, lr=None, stream=None) -> None:
    """adamw_tail_step with t read from the one-element int64 CUDA tensor
    `step` (after the increment) and, if given, lr from the one-element fp32
    CUDA tensor `lr`, when the kernel runs (capturable in a CUDA graph)."""
    import torch
    t = segs if isinstance(segs, TailTable) else TailTable(segs)
    if step.dtype != torch.int64 or step.numel() != 1 or not step.is_cuda:
        raise TypeError("step must be a one-element int64 CUDA tensor")
    if lr is not None and (lr.dtype != torch.float32 or lr.numel() != 1 or not lr.is_cuda):
        raise TypeError("lr must be a one-element fp32 CUDA tensor")
    _check(load_library().adamw_tail_step_dev(t.ptr, t.n, ctypes.byref(params), step.data_ptr(),
                                              lr.data_ptr() if lr is not None else None, _stream_ptr(stream)),
           "adamw_tail_step_dev")


# ---------------------------------------------------------------- diagnostics

def mo_last_device_error(stream=None) -> int:
    return int(load_library().mo_last_device_error(_stream_ptr(stream)))


def mo_selftest_bounded_wait(timeout_ns: int, stream=None) -> None:
    _check(load_library().mo_selftest_bounded_wait(int(timeout_ns), _stream_ptr(stream)), "selftest")


def fake_table(shapes: Sequence[Tuple[int, int]]):
    """A MoMatrix array with distinct, aligned, non-overlapping fake addresses
    (never dereferenced) for the host-only planning entry points."""
    arr = (MoMatrix * max(1, len(shapes)))()
    addr = 1 << 20
    for i, (r, c) in enumerate(shapes):
        sz = ((r * c * 4 + 4095) // 4096) * 4096
        w, g, v = addr, addr + sz, addr + 2 * sz
        addr += 3 * sz
        arr[i] = MoMatrix(w, g, v, r, c)
    return arr


NS_SCHEDULES = {"auto": 0, "static": 1, "counter": 2}  # mo_ns_schedule


def muon_owner_step_coverage(mats, params, workspace, stream=None, schedule="auto"):
    """muon_owner_step that also returns the per-tile execution counters
    (a uint32 device tensor: two per tile of every GEMM launch; all ones when
    each tile ran exactly once on each CTA of its pair), under the tile
    schedule named by `schedule` (NS_SCHEDULES). For tests."""
    import torch
    t = _as_table(mats)
    lib = load_library()
    sched = NS_SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)
    needed = ctypes.c_int64(0)
    _check(lib.muon_owner_step_coverage(t.ptr, t.n, ctypes.byref(params), None, 0, None, 0, sched,
                                        ctypes.byref(needed), None), "muon_owner_step_coverage")
    cov = torch.zeros(max(1, needed.value), dtype=torch.int32, device=workspace.device)
    st = lib.muon_owner_step_coverage(t.ptr, t.n, ctypes.byref(params), workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(), cov.data_ptr(), needed.value,
                                      sched, ctypes.byref(needed), _stream_ptr(stream))
    _check(st, "muon_owner_step_coverage")
    return cov[:needed.value]


def mo_muon_tile_schedule(shapes: Sequence[Tuple[int, int]], phase: int) -> List[Tuple[int, int, int]]:
    lib = load_library()
    arr = fake_table(shapes)
    count = ctypes.c_int64(0)
    st = lib.mo_muon_tile_schedule(ctypes.cast(arr, ctypes.c_void_p), len(shapes), phase, None, 0,
                                   ctypes.byref(count))
    if st not in (MO_OK, -2):
        _check(st, "mo_muon_tile_schedule")
    out = (MoTile * max(1, count.value))()
    _check(lib.mo_muon_tile_schedule(ctypes.cast(arr, ctypes.c_void_p), len(shapes), phase,
                                     ctypes.cast(out, ctypes.c_void_p), count.value, ctypes.byref(count)),
           "mo_muon_tile_schedule")
    return [(t.mat, t.tm, t.tn) for t in out[:count.value]]


# ---------------------------------------------------------------- owner planning

def mo_plan_owners(roles: Sequence[Tuple[int, int, int]], world: int, strategy: int = PLAN_COST_AWARE,
                   block_cap: int = 0):
    """Owner assignment of roles (numel, block, is_tail) over `world` ranks.
    Returns (owners, loads, chosen_strategy)."""
    n = len(roles)
    arr = (MoRole * max(1, n))(*[MoRole(int(a), int(b), int(c)) for a, b, c in roles])
    owners = (ctypes.c_int32 * max(1, n))()
    loads = (ctypes.c_int64 * max(1, world))()
    chosen = ctypes.c_int32(-1)
    _check(load_library().mo_plan_owners(ctypes.cast(arr, ctypes.c_void_p), n, int(world), int(strategy),
                                         int(block_cap), ctypes.cast(owners, ctypes.c_void_p),
                                         ctypes.cast(loads, ctypes.c_void_p), ctypes.byref(chosen)),
           "mo_plan_owners")
    return list(owners[:n]), list(loads[:world]), int(chosen.value)
