"""muon_owner_step_noalloc: the Muon step for callers that cannot allocate
device memory (for example when a framework's allocator owns the device, or
in contexts where cudaMalloc is not allowed). It uses the library's fixed
scratch array instead of a caller workspace; these tests call it through the
C ABI and check it against muon_owner_step with a caller workspace, on two
calls in a row: within the parity tolerances of the other GPU tests, and
bit-identical (the same kernels run on the same inputs)."""
import ctypes

import numpy as np
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import build as mo_build
from matrix_optimizers_zero_gb300 import workloads
from gpu_util import FP32_MAX_REL_TOL, NS_REL_FROB_TOL, extract_update, f64, max_rel, rel_frob, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    mo_build.build()
    return mo.load_library()


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    shapes = [(130, 257), (300, 200), (128, 256), (64, 1000)]
    wl = workloads.custom_workload(shapes, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    ref = to_device(host, DEV)       # stepped by muon_owner_step with a caller workspace
    got = to_device(host, DEV)       # stepped by muon_owner_step_noalloc
    p = mo.MuonParams()
    t_ref, t_got = mo.MuonTable(ref), mo.MuonTable(got)
    assert mo.mo_muon_workspace_bytes(t_got, p) <= lib.mo_static_scratch_bytes()
    ws = mo.muon_workspace(t_ref, p, device=DEV)
    stream = torch.cuda.current_stream(DEV).cuda_stream
    for call in range(2):
        w0 = [f64(W) for W, _, _ in got]
        st = lib.muon_owner_step(t_ref.ptr, t_ref.n, ctypes.byref(p), ws.data_ptr(), ws.numel(), stream)
        assert st == 0, mo.mo_status_string(st)
        st = lib.muon_owner_step_noalloc(t_got.ptr, t_got.n, ctypes.byref(p), stream)
        assert st == 0, mo.mo_status_string(st)
        torch.cuda.synchronize(DEV)
        assert mo.mo_last_device_error() == 0
        for (Wr, _, Vr), (Wg, _, Vg), w, (R, C) in zip(ref, got, w0, shapes):
            # within the parity tolerances of the other GPU tests ...
            o_ref = extract_update(w, f64(Wr), p.lr, p.wd, R, C)
            o_got = extract_update(w, f64(Wg), p.lr, p.wd, R, C)
            assert rel_frob(o_got, o_ref) <= NS_REL_FROB_TOL, (call, R, C)
            assert max_rel(f64(Vg), f64(Vr)) <= FP32_MAX_REL_TOL, (call, R, C)
            # ... and bit-identical: the same kernels and schedule on the same inputs
            assert torch.equal(Wg, Wr), (call, R, C)
            assert torch.equal(Vg, Vr), (call, R, C)


def test_noalloc_rejects_tables_beyond_the_scratch(lib):
    W = torch.zeros(4096, 4096, device=DEV)
    G = torch.ones(4096, 4096, device=DEV, dtype=torch.bfloat16)
    V = torch.zeros(4096, 4096, device=DEV)
    t = mo.MuonTable([(W, G, V)])
    p = mo.MuonParams()
    assert mo.mo_muon_workspace_bytes(t, p) > lib.mo_static_scratch_bytes()
    st = lib.muon_owner_step_noalloc(t.ptr, t.n, ctypes.byref(p), torch.cuda.current_stream(DEV).cuda_stream)
    assert st == -10 and "scratch" in mo.mo_status_string(st)
    torch.cuda.synchronize(DEV)
    assert float(V.abs().max()) == 0.0 and float(W.abs().max()) == 0.0
