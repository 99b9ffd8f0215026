"""Device-side tile coverage: every Newton-Schulz GEMM launch of a step
executes each output tile of its schedule exactly once on each CTA of the
pair that computes it, under both tile schedules: static (pair c runs tiles
c, c + pairs, ...) and from a per-launch device counter (reset for every
step). The counting entry point (muon_owner_step_coverage) runs the same
launches as muon_owner_step, and a tile's arithmetic does not depend on which
pair runs it or when, so its weights and momentum must come out bit-identical
to a plain step's (which uses the static schedule on these tables)."""
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads
from gpu_util import to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

RAGGED = [(130, 257), (257, 130), (1, 64), (640, 128), (300, 300), (1, 40_000), (7, 1000)]


def host_table(shapes, config_id):
    wl = workloads.custom_workload(shapes, g_std=1e-3, config_id=config_id)
    return [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]


def check_coverage(host, params, schedule):
    counted = to_device(host, DEV)
    plain = to_device(host, DEV)
    ws = mo.muon_workspace(counted, params, device=DEV)
    cov = mo.muon_owner_step_coverage(counted, params, ws, schedule=schedule)
    ws2 = mo.muon_workspace(plain, params, device=DEV)
    mo.muon_owner_step(plain, params, ws2)
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    assert cov.numel() > 0
    bad = torch.nonzero(cov != 1).flatten()
    assert bad.numel() == 0, f"tile counters not 1 at {bad[:10].tolist()} (values {cov[bad[:10]].tolist()})"
    for (Wc, _, Vc), (Wp, _, Vp) in zip(counted, plain):
        assert torch.equal(Wc, Wp) and torch.equal(Vc, Vp)


@pytest.mark.parametrize("schedule", ["static", "counter"])
@pytest.mark.parametrize("form", ["gram", "appendix"])
def test_every_tile_once_ragged_table(form, schedule):
    check_coverage(host_table(RAGGED, 97), mo.MuonParams(ns_form=form), schedule)


@pytest.mark.parametrize("schedule", ["static", "counter"])
def test_every_tile_once_gpt2l_four_layers(schedule):
    wl = workloads.get_workload("gpt2l_4layers")
    mats = workloads.device_matrices(wl, DEV, v_std=1e-3)
    host = [(W.cpu(), G.cpu(), V.cpu()) for W, G, V in mats]
    del mats
    check_coverage(host, mo.MuonParams(ns_steps=2), schedule)


def test_every_tile_once_on_consecutive_steps():
    """Two steps on one workspace under the counter schedule: each step starts
    its launches' tile counters from zero, so the second step runs every tile
    again."""
    host = host_table(RAGGED, 98)
    params = mo.MuonParams()
    counted = to_device(host, DEV)
    plain = to_device(host, DEV)
    ws = mo.muon_workspace(counted, params, device=DEV)
    ws2 = mo.muon_workspace(plain, params, device=DEV)
    for _ in range(2):
        cov = mo.muon_owner_step_coverage(counted, params, ws, schedule="counter")
        mo.muon_owner_step(plain, params, ws2)
        torch.cuda.synchronize()
        assert mo.mo_last_device_error() == 0
        assert bool((cov == 1).all())
    for (Wc, _, Vc), (Wp, _, Vp) in zip(counted, plain):
        assert torch.equal(Wc, Wp) and torch.equal(Vc, Vp)
