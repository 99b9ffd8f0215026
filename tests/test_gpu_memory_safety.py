"""Memory safety and isolation on the GPU, without a sanitizer.

* Canary guard regions: every W, G, V tensor and the Muon workspace is carved
  out of one allocation with 4 KB of a fixed byte pattern before and after it
  (the workspace gets exactly the bytes mo_muon_workspace_bytes asks for), and
  after several steps on ragged shapes (partial tiles in both directions,
  tall, wide, tiny) every guard byte must be unchanged.
* NaN isolation: matrices, rows (RMNP) and elements (AdamW) are independent,
  so a NaN planted in one gradient must leave every other matrix, row or
  element bit-identical to a run without it."""
import ctypes

import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 4096
PATTERN = 0xA5
RAGGED = [(130, 257), (257, 130), (1, 64), (64, 1), (300, 300), (7, 1000), (1000, 7), (255, 513)]


class Arena:
    """One device allocation holding 256-byte-aligned views separated by
    guard regions filled with PATTERN."""

    def __init__(self, sizes):
        self.offsets = []
        off = GUARD
        for nbytes in sizes:
            self.offsets.append(off)
            off += -(-nbytes // 256) * 256 + GUARD
        self.buf = torch.full((off,), PATTERN, dtype=torch.uint8, device=DEV)
        self.sizes = list(sizes)

    def view(self, k, dtype, shape=None):
        nbytes = self.sizes[k]
        t = self.buf[self.offsets[k]:self.offsets[k] + nbytes].view(dtype)
        return t.view(shape) if shape is not None else t

    def guards_intact(self):
        mask = torch.ones_like(self.buf, dtype=torch.bool)
        for off, nbytes in zip(self.offsets, self.sizes):
            mask[off:off + nbytes] = False
        return bool((self.buf[mask] == PATTERN).all().item())


def _muon_arena(shapes, params):
    wl = workloads.custom_workload(shapes, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    sizes = []
    for R, C in shapes:
        sizes += [R * C * 4, R * C * 2, R * C * 4]
    table = mo.fake_table(shapes)                      # the size query reads shapes only
    ws_bytes = mo.load_library().mo_muon_workspace_bytes(ctypes.cast(table, ctypes.c_void_p), len(shapes),
                                                          ctypes.byref(params))
    sizes.append(ws_bytes)
    arena = Arena(sizes)
    mats = []
    for i, ((R, C), (W, G, V)) in enumerate(zip(shapes, host)):
        w = arena.view(3 * i, torch.float32, (R, C))
        g = arena.view(3 * i + 1, torch.bfloat16, (R, C))
        v = arena.view(3 * i + 2, torch.float32, (R, C))
        w.copy_(W.to(DEV))
        g.copy_(G.to(DEV))
        v.copy_(V.to(DEV))
        mats.append((w, g, v))
    return arena, mats, arena.view(len(sizes) - 1, torch.uint8)


@pytest.mark.parametrize("form", ["gram", "appendix"])
def test_muon_guard_regions_untouched(form):
    p = mo.MuonParams(ns_form=form, nesterov=(form == "appendix"))
    arena, mats, ws = _muon_arena(RAGGED, p)
    assert ws.numel() == mo.mo_muon_workspace_bytes(mats, p)
    for _ in range(3):
        mo.muon_owner_step(mats, p, ws)
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    assert arena.guards_intact()
    for W, _, V in mats:
        assert torch.isfinite(W).all() and torch.isfinite(V).all()


def test_planned_step_guard_regions_untouched():
    p = mo.MuonParams()
    arena, mats, ws = _muon_arena(RAGGED, p)
    plan = mo.MuonPlan(mats, p, workspace=ws)
    for _ in range(2):
        plan.step()
    torch.cuda.synchronize()
    assert arena.guards_intact()
    plan.close()


def test_rmnp_and_adamw_guard_regions_untouched():
    shapes = [(130, 257), (1, 9), (9, 1), (16, 9000), (33, 4096)]
    wl = workloads.custom_workload(shapes, g_std=1e-3, tail=[1, 3, 4097, 10_001])
    sizes = []
    for R, C in shapes:
        sizes += [R * C * 4, R * C * 2, R * C * 4]
    for n in wl.tail:
        sizes += [n * 4] * 4
    arena = Arena(sizes)
    mats = []
    for i, (R, C) in enumerate(shapes):
        W, G, V = workloads.host_matrix(wl, i, v_std=1e-3)
        views = [arena.view(3 * i, torch.float32, (R, C)), arena.view(3 * i + 1, torch.bfloat16, (R, C)),
                 arena.view(3 * i + 2, torch.float32, (R, C))]
        for dst, src in zip(views, (W, G, V)):
            dst.copy_(src.to(DEV))
        mats.append(tuple(views))
    segs = []
    base = 3 * len(shapes)
    for j, n in enumerate(wl.tail):
        host = workloads.host_tail(wl, j, state_std=1e-3)
        views = [arena.view(base + 4 * j + k, torch.float32) for k in range(4)]
        for dst, src in zip(views, host):
            dst.copy_(src.to(DEV))
        segs.append(tuple(views))
    for t in range(1, 3):
        mo.rmnp_step(mats, mo.RmnpParams())
        mo.htrmnp_step(mats, mo.RmnpParams())
        mo.adamw_tail_step(segs, mo.AdamWParams(step=t))
    torch.cuda.synchronize()
    assert arena.guards_intact()


def test_nan_stays_in_its_matrix():
    shapes = [(256, 640), (640, 256), (130, 257)]
    wl = workloads.custom_workload(shapes, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    p = mo.MuonParams()
    clean = [tuple(t.to(DEV) for t in m) for m in host]
    dirty = [tuple(t.to(DEV) for t in m) for m in host]
    dirty[1][1][17, 3] = float("nan")
    for mats in (clean, dirty):
        mo.muon_owner_step(mats, p, mo.muon_workspace(mats, p, device=DEV))
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    for k in (0, 2):
        assert torch.equal(clean[k][0], dirty[k][0]) and torch.equal(clean[k][2], dirty[k][2])
    # the whole matrix is normalised by its (NaN) norm, so all of it is NaN
    assert torch.isnan(dirty[1][0]).all()


def test_nan_stays_in_its_row_and_element():
    shapes = [(64, 300), (16, 9000)]
    wl = workloads.custom_workload(shapes, g_std=1e-3, tail=[5000])
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    clean = [tuple(t.to(DEV) for t in m) for m in host]
    dirty = [tuple(t.to(DEV) for t in m) for m in host]
    dirty[0][1][5, 11] = float("nan")
    dirty[1][1][3, 8191] = float("nan")
    for mats in (clean, dirty):
        mo.rmnp_step(mats, mo.RmnpParams())
    tail_host = workloads.host_tail(wl, 0, state_std=1e-3)
    tc = [tuple(t.to(DEV) for t in tail_host)]
    td = [tuple(t.to(DEV) for t in tail_host)]
    td[0][1][1234] = float("nan")
    mo.adamw_tail_step(tc, mo.AdamWParams())
    mo.adamw_tail_step(td, mo.AdamWParams())
    torch.cuda.synchronize()
    for (Wc, _, Vc), (Wd, _, Vd), row in zip(clean, dirty, (5, 3)):
        keep = torch.ones(Wc.shape[0], dtype=torch.bool, device=DEV)
        keep[row] = False
        assert torch.equal(Wc[keep], Wd[keep]) and torch.equal(Vc[keep], Vd[keep])
        assert torch.isnan(Wd[row]).all()
    keep = torch.ones(5000, dtype=torch.bool, device=DEV)
    keep[1234] = False
    for a, b in zip(tc[0], td[0]):
        assert torch.equal(a[keep], b[keep])
    assert torch.isnan(td[0][0][1234])
