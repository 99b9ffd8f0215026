"""The planned Muon step (mo_muon_plan_*): bit-identical to muon_owner_step,
capturable in a CUDA graph, with the learning rate read from device memory.
The plan path runs the same kernels on the same inputs, so the bar is exact
equality of W and V with the per-call entry point (which the other GPU tests
hold to the oracle); one case is also checked against the oracle directly."""
import numpy as np
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads
import oracle
from gpu_util import FP32_MAX_REL_TOL, NS_REL_FROB_TOL, extract_update, f64, max_rel, rel_frob, to_device
from test_gpu_muon import oracle_options

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SHAPES = [(384, 640), (640, 384), (130, 257), (1, 64), (300, 300)]


def _host(seed_shapes=SHAPES):
    wl = workloads.custom_workload(seed_shapes, g_std=1e-3)
    return [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(seed_shapes))]


def _grads(host, steps, seed):
    gen = torch.Generator().manual_seed(seed)
    return [[(torch.randn(W.shape, generator=gen) * 1e-3).to(torch.bfloat16) for W, _, _ in host]
            for _ in range(steps)]


def _assert_same(a, b):
    for (Wa, _, Va), (Wb, _, Vb) in zip(a, b):
        assert torch.equal(Wa, Wb) and torch.equal(Va, Vb)


@pytest.mark.parametrize("form", ["gram", "appendix"])
def test_plan_steps_match_owner_step_bit_exactly(form):
    host = _host()
    p = mo.MuonParams(ns_form=form, nesterov=(form == "appendix"))
    ref, got = to_device(host, DEV), to_device(host, DEV)
    ws_ref = mo.muon_workspace(ref, p, device=DEV)
    plan = mo.MuonPlan(got, p)
    for gs in _grads(host, 3, seed=5):
        for (_, G, _), g in zip(ref, gs):
            G.copy_(g.to(DEV))
        for (_, G, _), g in zip(got, gs):
            G.copy_(g.to(DEV))
        mo.muon_owner_step(ref, p, ws_ref)
        plan.step()
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    _assert_same(ref, got)
    plan.close()


def test_plan_against_oracle():
    host = _host()
    p = mo.MuonParams()
    dev = to_device(host, DEV)
    plan = mo.MuonPlan(dev, p)
    plan.step()
    torch.cuda.synchronize()
    for (Wh, Gh, Vh), (Wd, _, Vd) in zip(host, dev):
        R, C = Wh.shape
        _, Vn, O = oracle.muon_matrix_step(f64(Wh), f64(Gh), f64(Vh), **oracle_options(p))
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        assert rel_frob(extract_update(f64(Wh), f64(Wd), p.lr, p.wd, R, C), O) <= NS_REL_FROB_TOL


def test_plan_graph_replay_with_lr_schedule():
    """One eager plan step, then a CUDA graph of one plan step captured and
    replayed three times with new gradients copied into the table's G tensors
    and a new learning rate written to the plan's device lr before each
    replay; the per-call entry point with the same gradients and learning
    rates gives bit-identical W and V."""
    host = _host()
    p = mo.MuonParams()
    lrs = [0.02, 0.015, 0.01, 0.005]
    grads = _grads(host, len(lrs), seed=9)
    ref, got = to_device(host, DEV), to_device(host, DEV)
    ws_ref = mo.muon_workspace(ref, p, device=DEV)
    for lr, gs in zip(lrs, grads):
        for (_, G, _), g in zip(ref, gs):
            G.copy_(g.to(DEV))
        mo.muon_owner_step(ref, mo.MuonParams(lr=lr), ws_ref)

    plan = mo.MuonPlan(got, p)
    for (_, G, _), g in zip(got, grads[0]):
        G.copy_(g.to(DEV))
    plan.lr.fill_(lrs[0])
    plan.step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.step()
    for lr, gs in zip(lrs[1:], grads[1:]):
        for (_, G, _), g in zip(got, gs):
            G.copy_(g.to(DEV))
        plan.lr.fill_(lr)
        graph.replay()
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    _assert_same(ref, got)
    plan.close()


def test_plan_workspace_header_survives_other_work():
    """The header is uploaded once; steps after unrelated device work and a
    second plan on another workspace still match the per-call entry point."""
    host = _host([(256, 512), (512, 256)])
    p = mo.MuonParams()
    ref, got, other = to_device(host, DEV), to_device(host, DEV), to_device(host, DEV)
    ws_ref = mo.muon_workspace(ref, p, device=DEV)
    plan = mo.MuonPlan(got, p)
    plan2 = mo.MuonPlan(other, mo.MuonParams(ns_steps=2))
    for _ in range(2):
        mo.muon_owner_step(ref, p, ws_ref)
        plan2.step()
        torch.randn(1 << 20, device=DEV).sum()
        plan.step()
    torch.cuda.synchronize()
    _assert_same(ref, got)
