"""Host-side tests of the C ABI (no GPU): the library loads and exports every
function include/mo.h declares; validation rejects bad arguments before any
CUDA call; the tile schedules are bit-exact against a plain Python restatement
of their rules and cover every output element exactly once."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import build as mo_build
from matrix_optimizers_zero_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mo_build.build()
    return mo.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "mo.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert "muon_owner_step" in names and "adamw_tail_step" in names and "rmnp_step" in names
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert lib.mo_abi_version() == 4


def test_status_strings(lib):
    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8, -9]:
        s = mo.mo_status_string(code)
        assert s and s != "unknown status"
    assert mo.mo_status_string(12345) == "unknown status"


# ---------------------------------------------------------------- schedules

BM = 256   # output tile height of the CTA-pair kernel
GRAM_SLICE = 32768   # Gram reductions longer than this are split into slices of this length


def py_schedule(shapes, phase):
    keys = []
    for i, (R, C) in enumerate(shapes):
        m, n = min(R, C), max(R, C)
        tiles_m = -(-m // BM)
        if phase == mo.PHASE_UPDATE:
            # m x n products: column-block by column-block within a matrix
            for tm in range(tiles_m):
                for tn in range(-(-n // 256)):
                    keys.append((-m, i, tn, tm))
        elif phase == mo.PHASE_POLY or n <= GRAM_SLICE:
            k = n if phase == mo.PHASE_GRAM else m
            for tm in range(tiles_m):
                for tn in range(-(-m // 256)):
                    if (tn + 1) * 256 > tm * BM:
                        keys.append((-k, i, tm, tn, i))
    if phase == mo.PHASE_GRAM:
        # longer Grams: one entry per GRAM_SLICE columns, numbered after the
        # table's matrices in (matrix, slice) order, reported as the matrix
        entry = len(shapes)
        for i, (R, C) in enumerate(shapes):
            m, n = min(R, C), max(R, C)
            if n <= GRAM_SLICE:
                continue
            for k0 in range(0, n, GRAM_SLICE):
                k = min(GRAM_SLICE, n - k0)
                for tm in range(-(-m // BM)):
                    for tn in range(-(-m // 256)):
                        if (tn + 1) * 256 > tm * BM:
                            keys.append((-k, entry, tm, tn, i))
                entry += 1
    keys.sort()
    if phase == mo.PHASE_UPDATE:
        return [(i, tm, tn) for _, i, tn, tm in keys]
    return [(i, tm, tn) for _, _, tm, tn, i in keys]


def gram_slices(n):
    return max(1, -(-n // GRAM_SLICE)) if n > GRAM_SLICE else 1


TABLES = {
    "gpt2l": [(s.rows, s.cols) for s in workloads.get_workload("gpt2l").matrices],
    "share32b": [(s.rows, s.cols) for s in workloads.get_workload("share32b").matrices],
    "ragged": [(130, 257), (257, 130), (1, 9), (9, 1), (128, 256), (300, 300), (1000, 70)],
    "long": [(3, 100_000), (70_000, 300), (130, 257), (600, 32_768), (32_769, 5), (1, 1 << 22)],
}


@pytest.mark.parametrize("table", sorted(TABLES))
@pytest.mark.parametrize("phase", [0, 1, 2])
def test_schedule_bit_exact(lib, table, phase):
    shapes = TABLES[table]
    assert mo.mo_muon_tile_schedule(shapes, phase) == py_schedule(shapes, phase)


@pytest.mark.parametrize("shape", [(130, 257), (257, 130), (300, 300), (700, 1500), (1, 5), (300, 70_000)])
def test_schedule_covers_outputs_exactly_once(lib, shape):
    """Once per Gram slice for the Gram (whose slices each cover the whole
    output), once otherwise."""
    m, n = min(shape), max(shape)
    for phase in (0, 1):
        cover = np.zeros((m, m), dtype=np.int32)
        for _, tm, tn in mo.mo_muon_tile_schedule([shape], phase):
            r0, c0 = tm * BM, tn * 256
            # the epilogue's store rule: direct for col >= row, mirror for col > row
            for r in range(r0, min(r0 + BM, m)):
                for c in range(c0, min(c0 + 256, m)):
                    if c >= r:
                        cover[r, c] += 1
                    if c > r:
                        cover[c, r] += 1
        assert np.all(cover == (gram_slices(n) if phase == 0 else 1)), phase
    cover = np.zeros((m, n), dtype=np.int32)
    for _, tm, tn in mo.mo_muon_tile_schedule([shape], 2):
        cover[tm * BM:tm * BM + BM, tn * 256:tn * 256 + 256] += 1
    assert np.all(cover == 1)


def test_workspace_bytes(lib):
    shapes = [(130, 257), (257, 130)]
    arr = mo.fake_table(shapes)
    p = mo.MuonParams()
    nb = lib.mo_muon_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), 2, ctypes.byref(p))
    # lower bound: two bf16 iterates and A, B per matrix with 64-element padded rows
    lower = sum(2 * min(s) * (-(-max(s) // 64) * 64) * 2 + 2 * min(s) * (-(-min(s) // 64) * 64) * 2 for s in shapes)
    assert nb >= lower and nb < lower + 64 * 1024
    bad = mo.MuonParams(ns_steps=0)
    assert lib.mo_muon_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), 2, ctypes.byref(bad)) == 0
    g = [(s.rows, s.cols) for s in workloads.get_workload("gpt2l").matrices]
    big = mo.fake_table(g)
    nb2 = lib.mo_muon_workspace_bytes(ctypes.cast(big, ctypes.c_void_p), len(g), ctypes.byref(p))
    buffers = sum(2 * min(r, c) * max(r, c) * 2 + 2 * min(r, c) ** 2 * 2 for r, c in g)
    assert buffers <= nb2 < buffers * 1.01
    # the appendix form keeps B = A X (m x n) instead of the m x m polynomial
    pa = mo.MuonParams(ns_form="appendix")
    nb3 = lib.mo_muon_workspace_bytes(ctypes.cast(big, ctypes.c_void_p), len(g), ctypes.byref(pa))
    buffers3 = sum(3 * min(r, c) * max(r, c) * 2 + min(r, c) ** 2 * 2 for r, c in g)
    assert buffers3 <= nb3 < buffers3 * 1.01
    assert lib.mo_muon_workspace_bytes(ctypes.cast(big, ctypes.c_void_p), len(g),
                                       ctypes.byref(mo.MuonParams(nesterov=True, lr_adjust="match_rms_adamw"))) == nb2


def test_workspace_bytes_with_gram_slices(lib):
    """A matrix with n > 32768 adds one fp32 m x m partial (rows padded to 64
    elements) per Gram slice; shorter ones add nothing."""
    p = mo.MuonParams()

    def ws(shapes):
        arr = mo.fake_table(shapes)
        return lib.mo_muon_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), len(shapes), ctypes.byref(p))

    for (R, C), slices in (((300, 70_000), 3), ((40_000, 130), 2), ((1, 1 << 20), 32)):
        m = min(R, C)
        lda = -(-m // 64) * 64
        part = -(-(m * lda * 4) // 1024) * 1024
        base = ws([(R, C), (130, 257)])
        # the same matrix just under the threshold has no slices
        short = ws([(min(R, C), 32_768) if R < C else (32_768, min(R, C)), (130, 257)])
        x_extra = 2 * m * (-(-max(R, C) // 64) * 64 - 32_768) * 2
        assert base - short >= slices * part + x_extra - 4096
        assert base - short <= slices * part + x_extra + 64 * 1024


# ---------------------------------------------------------------- validation (no GPU needed)

def _muon(lib, arr, n, params, ws=1 << 30, ws_bytes=1 << 40):
    return lib.muon_owner_step(ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None, n,
                               ctypes.byref(params), ws, ws_bytes, None)


def test_muon_validation_codes(lib):
    p = mo.MuonParams()
    ok = mo.fake_table([(16, 32)])
    assert _muon(lib, None, 1, p) == -1                        # null table
    assert _muon(lib, ok, -1, p) == -2
    assert _muon(lib, None, 0, p) == 0                          # empty table is a no-op
    zero = mo.fake_table([(16, 32)])
    zero[0].rows = 0
    assert _muon(lib, zero, 1, p) == -2
    mis = mo.fake_table([(16, 32)])
    mis[0].W += 4
    assert _muon(lib, mis, 1, p) == -3
    nulls = mo.fake_table([(16, 32)])
    nulls[0].V = None
    assert _muon(lib, nulls, 1, p) == -1
    over = mo.fake_table([(16, 32)])
    over[0].V = over[0].W + 16
    assert _muon(lib, over, 1, p) == -6
    alias = mo.fake_table([(16, 32)])
    alias[0].G = alias[0].W
    assert _muon(lib, alias, 1, p) == -6
    two = mo.fake_table([(16, 32), (16, 32)])
    two[1].W = two[0].V
    assert _muon(lib, two, 2, p) == -6
    for bad in (mo.MuonParams(lr=float("nan")), mo.MuonParams(ns_steps=0), mo.MuonParams(ns_steps=101),
                mo.MuonParams(eps=-1.0), mo.MuonParams(a=float("inf")), mo.MuonParams(ns_form=2),
                mo.MuonParams(ns_form=-1), mo.MuonParams(lr_adjust=2), mo.MuonParams(nesterov=2)):
        assert _muon(lib, ok, 1, bad) == -4
    assert _muon(lib, ok, 1, p, ws=0) == -1
    assert _muon(lib, ok, 1, p, ws=(1 << 30) + 16) == -3
    assert _muon(lib, ok, 1, p, ws_bytes=1024) == -5
    big = mo.fake_table([(70000, 70000)])
    assert _muon(lib, big, 1, p) == -2                          # m above the supported maximum


def test_muon_plan_validation_codes(lib):
    """mo_muon_plan_create rejects bad arguments before any CUDA call; the
    other plan entry points accept NULL plans."""
    p = mo.MuonParams()
    ok = mo.fake_table([(16, 32)])
    out = ctypes.c_void_p()

    def create(arr, n, params=p, ws=1 << 30, ws_bytes=1 << 40, out_ptr=ctypes.byref(out)):
        return lib.mo_muon_plan_create(ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None, n,
                                       ctypes.byref(params), ws, ws_bytes, None, out_ptr)

    assert create(ok, 1, out_ptr=None) == -1
    assert create(None, 1) == -1
    assert create(None, 0) == -2                     # a plan needs at least one matrix
    assert create(ok, 1, params=mo.MuonParams(ns_steps=0)) == -4
    assert create(ok, 1, ws=0) == -1
    assert create(ok, 1, ws=(1 << 30) + 16) == -3
    assert create(ok, 1, ws_bytes=1024) == -5
    mis = mo.fake_table([(16, 32)])
    mis[0].W += 4
    assert create(mis, 1) == -3
    assert out.value is None                         # never set on failure
    assert lib.mo_muon_plan_step(None, None) == -1
    assert lib.mo_muon_plan_lr_ptr(None) is None
    assert lib.mo_muon_plan_destroy(None) == 0


def test_adamw_and_rmnp_validation_codes(lib):
    seg = (mo.MoTailSeg * 1)()
    seg[0] = mo.MoTailSeg(1 << 20, 2 << 20, 3 << 20, 4 << 20, 1000)
    sp = ctypes.cast(seg, ctypes.c_void_p)
    assert lib.adamw_tail_step(sp, 1, ctypes.byref(mo.AdamWParams(step=0)), None) == -4
    assert lib.adamw_tail_step(sp, 1, ctypes.byref(mo.AdamWParams(beta1=1.0)), None) == -4
    assert lib.adamw_tail_step(sp, 1, ctypes.byref(mo.AdamWParams(eps=float("nan"))), None) == -4
    assert lib.adamw_tail_step(None, 1, ctypes.byref(mo.AdamWParams()), None) == -1
    assert lib.adamw_tail_step(None, 0, ctypes.byref(mo.AdamWParams()), None) == 0
    seg[0].m = seg[0].p + 8 * 16
    assert lib.adamw_tail_step(sp, 1, ctypes.byref(mo.AdamWParams()), None) == -6
    seg[0].m = (3 << 20) + 4
    assert lib.adamw_tail_step(sp, 1, ctypes.byref(mo.AdamWParams()), None) == -3
    seg[0].m = 3 << 20
    seg[0].g = seg[0].v
    assert lib.adamw_tail_step(sp, 1, ctypes.byref(mo.AdamWParams()), None) == -6

    t = mo.fake_table([(16, 32)])
    tp = ctypes.cast(t, ctypes.c_void_p)
    assert lib.rmnp_step(tp, 1, ctypes.byref(mo.RmnpParams(eps=-1.0)), None) == -4
    assert lib.rmnp_step(None, 0, ctypes.byref(mo.RmnpParams()), None) == 0
    assert lib.rmnp_step_scaled(tp, None, 1, ctypes.byref(mo.RmnpParams()), None) == -1
    sc = (ctypes.c_float * 1)(float("nan"))
    assert lib.rmnp_step_scaled(tp, ctypes.cast(sc, ctypes.c_void_p), 1, ctypes.byref(mo.RmnpParams()), None) == -4
    for bad_power in (-0.1, 1.5, float("nan"), float("inf")):
        assert lib.htrmnp_step(tp, 1, ctypes.byref(mo.RmnpParams()), ctypes.c_float(bad_power), None) == -4
    assert lib.htrmnp_step(None, 0, ctypes.byref(mo.RmnpParams()), ctypes.c_float(0.125), None) == 0
    assert lib.htrmnp_step(tp, 1, ctypes.byref(mo.RmnpParams(eps=-1.0)), ctypes.c_float(0.125), None) == -4


def test_device_hyperparameter_validation_codes(lib):
    """adamw_tail_step_dev / rmnp_step_dev: null or misaligned device
    pointers are rejected before any CUDA call; the by-value fields they
    replace are not validated."""
    seg = (mo.MoTailSeg * 1)()
    seg[0] = mo.MoTailSeg(1 << 20, 2 << 20, 3 << 20, 4 << 20, 1000)
    sp = ctypes.cast(seg, ctypes.c_void_p)
    step_ptr, lr_ptr = 5 << 20, 6 << 20
    assert lib.adamw_tail_step_dev(sp, 1, ctypes.byref(mo.AdamWParams()), None, None, None) == -1
    assert lib.adamw_tail_step_dev(sp, 1, ctypes.byref(mo.AdamWParams()), step_ptr + 4, None, None) == -3
    assert lib.adamw_tail_step_dev(sp, 1, ctypes.byref(mo.AdamWParams()), step_ptr, lr_ptr + 2, None) == -3
    assert lib.adamw_tail_step_dev(sp, 1, None, step_ptr, None, None) == -1
    assert lib.adamw_tail_step_dev(sp, 1, ctypes.byref(mo.AdamWParams(beta1=1.0)), step_ptr, None, None) == -4
    assert lib.adamw_tail_step_dev(None, 0, ctypes.byref(mo.AdamWParams(step=0)), step_ptr, None, None) == 0
    t = mo.fake_table([(16, 32)])
    tp = ctypes.cast(t, ctypes.c_void_p)
    assert lib.rmnp_step_dev(tp, 1, ctypes.byref(mo.RmnpParams()), ctypes.c_float(0.0), None, None) == -1
    assert lib.rmnp_step_dev(tp, 1, ctypes.byref(mo.RmnpParams()), ctypes.c_float(0.0), lr_ptr + 1, None) == -3
    assert lib.rmnp_step_dev(tp, 1, ctypes.byref(mo.RmnpParams(eps=-1.0)), ctypes.c_float(0.0), lr_ptr, None) == -4
    assert lib.rmnp_step_dev(tp, 1, ctypes.byref(mo.RmnpParams()), ctypes.c_float(2.0), lr_ptr, None) == -4
    assert lib.rmnp_step_dev(None, 0, ctypes.byref(mo.RmnpParams(lr=float("nan"))), ctypes.c_float(0.0),
                             lr_ptr, None) == 0


def test_tile_coverage_size_query(lib):
    """muon_owner_step_coverage with no buffer only reports how many counters
    a step needs: two per tile of every GEMM launch (Gram, A.A or A.X, B.X per
    iteration), the tile counts being those of the host schedule."""
    for shapes, form, steps in (([(130, 257), (300, 200), (1, 70_000)], "gram", 5),
                                ([(1280, 5120)] * 3 + [(64, 1)], "appendix", 2)):
        p = mo.MuonParams(ns_form=form, ns_steps=steps)
        arr = mo.fake_table(shapes)
        need = ctypes.c_int64(-1)
        for sched in (0, 1, 2):
            st = lib.muon_owner_step_coverage(ctypes.cast(arr, ctypes.c_void_p), len(shapes), ctypes.byref(p), None,
                                              0, None, 0, sched, ctypes.byref(need), None)
            assert st == 0
            mid = 1 if form == "gram" else 2
            per_iter = sum(len(mo.mo_muon_tile_schedule(shapes, ph)) for ph in (0, mid, 2))
            assert need.value == 2 * steps * per_iter
    # a null count pointer is rejected before anything else, then an unknown schedule
    arr = mo.fake_table([(16, 32)])
    assert lib.muon_owner_step_coverage(ctypes.cast(arr, ctypes.c_void_p), 1, ctypes.byref(mo.MuonParams()), None, 0,
                                        None, 0, 0, None, None) == -1
    need = ctypes.c_int64(-1)
    for bad in (-1, 3):
        assert lib.muon_owner_step_coverage(ctypes.cast(arr, ctypes.c_void_p), 1, ctypes.byref(mo.MuonParams()),
                                            None, 0, None, 0, bad, ctypes.byref(need), None) == -4
