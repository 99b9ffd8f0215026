"""Parity at the full sizes of the larger configurations for the row-wise
and elementwise kernels: RMNP on the whole Llama-style 8B table (sampled rows
checked against the oracle), AdamW on its 1.05 G-element tail (sampled
elements), and RMNP on the structured-spectrum batch's orthogonal-row
matrices against the exact polar factor. (The Muon step on whole tables is
covered by the full-table tests.)"""
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


def test_spectrum_orthorows_rmnp_matches_polar_factor():
    """The structured-spectrum batch's orthogonal-row matrices G = diag(z^2) Q
    have a diagonal Gram matrix, so their exact polar factor
    (G G^T)^{-1/2} G is Q itself, which is the RMNP direction ("Optimizers In
    A Sharded World", section 1: with an exactly diagonal Gram matrix RMNP and
    Muon give the same direction). The GPU's RMNP direction of the bf16 input
    is compared row by row with Q computed in fp64 on the host. Bound: the
    cast (fp64 -> fp32 -> bf16, nearest-even) moves each element by at most
    2^-9 + 2^-24 of itself, so each row by at most that fraction of its norm,
    and normalising a row at most doubles a relative perturbation: every row
    lies within 2 (2^-9 + 2^-24) of Q's row, plus 1e-5 for the fp32 row sums.
    The direction is also checked against the oracle's RMNP of the same bf16
    input (1e-5)."""
    wl = workloads.get_workload("spectrum")
    bound = 2.0 * (2.0 ** -9 + 2.0 ** -24) + 1e-5
    worst = 0.0
    for i, s in enumerate(wl.matrices):
        if s.kind != "orthorows":
            continue
        d, Q = workloads.spectral_factors(wl, i)
        gram = Q @ Q.T
        assert np.abs(gram - np.eye(s.rows)).max() < 1e-12          # orthonormal rows: the exact polar factor is Q
        G = torch.from_numpy(np.ascontiguousarray(d[:, None] * Q, dtype=np.float32)).to(torch.bfloat16)
        W = torch.zeros(s.rows, s.cols, device=DEV)
        V = torch.zeros(s.rows, s.cols, device=DEV)
        Gd = G.to(DEV)
        mo.rmnp_step([(W, Gd, V)], mo.RmnpParams(lr=1.0, wd=0.0, mu=0.95))
        torch.cuda.synchronize()
        D = -f64(W) / oracle.shape_scale(s.rows, s.cols)
        row_err = np.linalg.norm(D - Q, axis=1).max()
        assert row_err <= bound, (i, row_err, bound)
        worst = max(worst, row_err)
        assert max_rel(D, oracle.rmnp_direction(f64(G))) <= FP32_MAX_REL_TOL
    assert worst > 0.0      # the cast does perturb the rows: the comparison is not vacuous
