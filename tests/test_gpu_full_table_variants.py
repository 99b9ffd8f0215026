"""The variant configurations that the benchmark's extras time, checked in
the same launch configuration: all 144 GPT-2 Large matrices in one call,
with one matrix of each shape (and two others) compared against the oracle.

* the appendix iteration form (bar 2e-2, derived for five iterations of
  that form: see test_gpu_muon_variants);
* "MatrixFSDP" section 5.1's convergence settings (2 iterations, mu 0.5,
  Nesterov momentum, match_rms_adamw; bar 1e-3 for two iterations);
* the planned step (bit-identical to the per-call step on the full table);
* HTRMNP (the reading of its formula; fp32 bar 1e-5 on sampled rows)."""
import numpy as np
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads
import oracle
from gpu_util import FP32_MAX_REL_TOL, extract_update, f64, max_rel, rel_frob
from test_gpu_muon import oracle_options, update_scale

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SAMPLE = [0, 1, 2, 3, 77, 142]


def _full_table_check(p, tol):
    wl = workloads.get_workload("gpt2l")
    dev = workloads.device_matrices(wl, DEV, v_std=1e-3)
    snap = {i: tuple(f64(t) for t in dev[i]) for i in SAMPLE}
    mo.muon_owner_step(dev, p, mo.muon_workspace(dev, p, device=DEV))
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    for i in SAMPLE:
        W0, G0, V0 = snap[i]
        R, C = W0.shape
        _, Vn, O = oracle.muon_matrix_step(W0, G0, V0, **oracle_options(p))
        assert max_rel(f64(dev[i][2]), Vn) <= FP32_MAX_REL_TOL
        err = rel_frob(extract_update(W0, f64(dev[i][0]), p.lr, p.wd, R, C, update_scale(p, R, C)), O)
        assert err <= tol, (i, err)


def test_appendix_form_full_table():
    wl = workloads.get_workload("gpt2l")
    _full_table_check(mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_form="appendix"), 2e-2)


def test_convergence_settings_full_table():
    _full_table_check(mo.MuonParams(lr=1e-3, wd=1e-2, mu=0.5, ns_steps=2, lr_adjust="match_rms_adamw",
                                    nesterov=True), 1e-3)


def test_planned_step_full_table_bit_identical():
    wl = workloads.get_workload("gpt2l")
    p = mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu)
    ref = workloads.device_matrices(wl, DEV, v_std=1e-3)
    got = workloads.device_matrices(wl, DEV, v_std=1e-3)
    mo.muon_owner_step(ref, p, mo.muon_workspace(ref, p, device=DEV))
    plan = mo.MuonPlan(got, p)
    plan.step()
    torch.cuda.synchronize()
    for (Wa, _, Va), (Wb, _, Vb) in zip(ref, got):
        assert torch.equal(Wa, Wb) and torch.equal(Va, Vb)
    plan.close()


def test_htrmnp_full_table_sampled_rows():
    """The benchmark's HTRMNP extra on the full table: 64 sampled rows of one
    matrix per shape against the oracle's reading (rows are independent, so
    each sampled row is an exact check)."""
    wl = workloads.get_workload("gpt2l")
    dev = workloads.device_matrices(wl, DEV, v_std=1e-3)
    rng = np.random.default_rng(3)
    picks = {}
    for i in (0, 1, 2, 3):
        R = dev[i][0].shape[0]
        rows = torch.from_numpy(rng.choice(R, 64, replace=False)).to(DEV)
        picks[i] = (rows, tuple(f64(t[rows]) for t in dev[i]))
    p = mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu)
    mo.htrmnp_step(dev, p)
    torch.cuda.synchronize()
    for i, (rows, (W0, G0, V0)) in picks.items():
        R, C = dev[i][0].shape
        # the sampled rows with the whole matrix's shape scale
        Vn = oracle.momentum(V0, G0, p.mu)
        Wn = oracle.decoupled_update(W0, oracle.htrmnp_direction(Vn), p.lr, p.wd, oracle.shape_scale(R, C))
        assert max_rel(f64(dev[i][2][rows]), Vn) <= FP32_MAX_REL_TOL
        assert max_rel(f64(dev[i][0][rows]), Wn) <= FP32_MAX_REL_TOL


def test_colcut_rmnp_full_table_equals_unsharded():
    """Every matrix cut into 4 column shards (own buffers; at most 512 shards,
    whole matrices, per call, as the benchmark's extras run it): each
    reassembled matrix equals the unsharded RMNP step (with the column-cut
    form's clamp, 1e-7) within fp32 reassociation."""
    wl = workloads.get_workload("gpt2l")
    dev = workloads.device_matrices(wl, DEV, v_std=1e-3)
    p = mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, eps=1e-7)
    shards, groups, scales, cuts = [], [], [], []
    for g_id, (W, G, V) in enumerate(dev):
        R, C = W.shape
        edges = [C * k // 4 for k in range(5)]
        cuts.append(edges)
        for a, b in zip(edges[:-1], edges[1:]):
            shards.append((W[:, a:b].contiguous(), G[:, a:b].contiguous(), V[:, a:b].contiguous()))
            groups.append(g_id)
            scales.append(oracle.shape_scale(R, C))
    k = 0
    while k < len(shards):
        j = min(len(shards), k + 512)
        while j < len(shards) and groups[j] == groups[j - 1]:
            j -= 1
        mo.rmnp_colcut_step(shards[k:j], groups[k:j], scales[k:j], p)
        k = j
    mo.rmnp_step(dev, p)
    torch.cuda.synchronize()
    for g_id in SAMPLE:
        W, _, V = dev[g_id]
        mine = [s for s, g in zip(shards, groups) if g == g_id]
        Wc = torch.cat([s[0] for s in mine], dim=1)
        Vc = torch.cat([s[2] for s in mine], dim=1)
        assert max_rel(f64(Vc), f64(V)) <= FP32_MAX_REL_TOL
        assert max_rel(f64(Wc), f64(W)) <= FP32_MAX_REL_TOL
