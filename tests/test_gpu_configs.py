"""Parity at the full sizes of the larger configurations: every matrix of the
table goes through one grouped launch (as in the benchmark), and a sample of
matrices (one per distinct shape where the oracle finishes in seconds) is
checked against the CPU oracle. AdamW and RMNP are elementwise/row-wise, so
their full-size outputs are checked on sampled elements and rows.

Configurations: the Llama-style 8B table (224 matrices, 1.05 G-element AdamW
tail), the structured-spectrum batch (Haar singular vectors, log-uniform
spectra; rows with an exactly diagonal Gram matrix) and the 32B-scale owner
share (heterogeneous shapes up to 27648 x 5120)."""
import math

import numpy as np
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads
import oracle
from gpu_util import FP32_MAX_REL_TOL, NS_REL_FROB_TOL, extract_update, f64, max_rel, rel_frob

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def first_of_each_shape(wl, skip=()):
    seen, out = set(), []
    for i, s in enumerate(wl.matrices):
        if (s.rows, s.cols) not in seen and (s.rows, s.cols) not in skip:
            seen.add((s.rows, s.cols))
            out.append(i)
    return out


def muon_full_table_sampled(wl, dev_mats, sample):
    p = mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_steps=wl.ns_steps)
    snap = {i: tuple(f64(t) for t in dev_mats[i]) for i in sample}
    t = mo.MuonTable(dev_mats)
    ws = mo.muon_workspace(t, p, device=DEV)
    mo.muon_owner_step(t, p, ws)
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    del ws
    errs = {}
    for i in sample:
        W0, G0, V0 = snap[i]
        R, C = W0.shape
        _, Vn, O = oracle.muon_matrix_step(W0, G0, V0, lr=p.lr, wd=p.wd, mu=p.mu, ns_steps=p.ns_steps)
        assert max_rel(f64(dev_mats[i][2]), Vn) <= FP32_MAX_REL_TOL
        errs[i] = rel_frob(extract_update(W0, f64(dev_mats[i][0]), p.lr, p.wd, R, C), O)
        assert errs[i] <= NS_REL_FROB_TOL, (i, R, C, errs[i])
    return errs


def test_llama8b_muon_full_table():
    wl = workloads.get_workload("llama8b")
    mats = workloads.device_matrices(wl, DEV, v_std=1e-3)
    # one of each shape: 4096^2, 1024x4096, 14336x4096, 4096x14336
    muon_full_table_sampled(wl, mats, first_of_each_shape(wl))


def test_llama8b_rmnp_full_table_sampled_rows():
    wl = workloads.get_workload("llama8b")
    mats = workloads.device_matrices(wl, DEV, v_std=1e-3)
    rng = np.random.default_rng(0)
    picks = [(i, int(r)) for i in first_of_each_shape(wl) for r in rng.integers(0, wl.matrices[i].rows, 4)]
    snap = {(i, r): tuple(f64(t[r:r + 1]) for t in mats[i]) for i, r in picks}
    p = mo.RmnpParams(lr=wl.lr, wd=wl.wd, mu=wl.mu)
    mo.rmnp_step(mats, p)
    torch.cuda.synchronize()
    for (i, r), (W0, G0, V0) in snap.items():
        s = wl.matrices[i]
        Vn = oracle.momentum(V0, G0, p.mu)
        Wn = oracle.decoupled_update(W0, oracle.rmnp_direction(Vn), p.lr, p.wd, oracle.shape_scale(s.rows, s.cols))
        assert max_rel(f64(mats[i][0][r:r + 1]), Wn) <= FP32_MAX_REL_TOL
        assert max_rel(f64(mats[i][2][r:r + 1]), Vn) <= FP32_MAX_REL_TOL


def test_llama8b_adamw_tail_sampled():
    """The 1.05 G-element tail (norm vectors, embedding, LM head), checked on
    a random sample of elements of every segment."""
    wl = workloads.get_workload("llama8b")
    segs = workloads.device_tail(wl, DEV)
    rng = np.random.default_rng(1)
    idx = [torch.from_numpy(rng.integers(0, n, size=min(n, 20000))).to(DEV) for n in wl.tail]
    before = [tuple(f64(t[ix]) for t in seg) for seg, ix in zip(segs, idx)]
    p = mo.AdamWParams(lr=wl.adam_lr, wd=wl.adam_wd, beta1=wl.beta1, beta2=wl.beta2, eps=wl.adam_eps, step=1)
    mo.adamw_tail_step(segs, p)
    torch.cuda.synchronize()
    for seg, ix, (p0, g0, m0, v0) in zip(segs, idx, before):
        pr, mr, vr = oracle.adamw_step(p0, g0, m0, v0, lr=p.lr, wd=p.wd, beta1=p.beta1, beta2=p.beta2,
                                       eps=p.eps, step=1)
        assert max_rel(f64(seg[0][ix]), pr) <= FP32_MAX_REL_TOL
        assert max_rel(f64(seg[2][ix]), mr) <= FP32_MAX_REL_TOL
        assert max_rel(f64(seg[3][ix]), vr) <= FP32_MAX_REL_TOL


def test_spectrum_batch():
    """Structured spectra: Haar U, V and log-uniform singular values in
    [1e-4, 1]; plus rows that are exactly orthogonal (diagonal Gram matrix).
    The whole 56-matrix batch runs in one call; one matrix of each kind is
    checked against the oracle."""
    wl = workloads.get_workload("spectrum")
    sample = first_of_each_shape(wl)
    mats = []
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    for i, s in enumerate(wl.matrices):
        if i in sample:
            W, G, V = workloads.host_matrix(wl, i)
            mats.append((W.to(DEV), G.to(DEV), V.to(DEV)))
        else:
            # the unsampled matrices only need realistic content for the launch
            W = torch.randn(s.rows, s.cols, generator=gen, device=DEV).mul_(wl.w_std)
            G = torch.randn(s.rows, s.cols, generator=gen, device=DEV).mul_(0.01).to(torch.bfloat16)
            mats.append((W, G, torch.zeros_like(W)))
    muon_full_table_sampled(wl, mats, sample)


def test_share32b_grouped_launch():
    """28 heterogeneous matrices in one grouped launch; the two shapes the
    oracle finishes quickly (1024 x 5120 and 5120^2) plus one 27648 x 5120
    matrix are checked."""
    wl = workloads.get_workload("share32b")
    mats = workloads.device_matrices(wl, DEV, v_std=1e-3)
    sample = [1, 0, 4]
    muon_full_table_sampled(wl, mats, sample)
