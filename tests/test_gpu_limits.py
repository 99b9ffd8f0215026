"""The largest supported sizes, against the oracle.

* Muon at the largest supported short side (65536 x 65536): a sign-pattern
  gradient that keeps every stored value exact, checked element for element
  against the oracle's scalar recursion (see the test).

* Muon and RMNP on matrices at the longest supported dimension (2^22 columns
  or rows; 16384 tile columns of 256) with one to three rows, ragged in both
  directions: full comparison, since such matrices are cheap for the oracle.
  Their Grams (and any longer than 32768 columns) are summed from slice
  partials; without the slicing the 1 x 2^22 update was 7.8% off.
* AdamW on one segment of 2^31 + 4097 elements (34 GB of fp32 state): every
  element index above 2^31 goes through 64-bit address arithmetic; checked on
  sampled elements (the oracle is elementwise, so each sample is exact),
  including the last ones and those around 2^31."""
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
LONG = 1 << 22


def test_muon_longest_dimension():
    shapes = [(1, LONG), (LONG, 1), (3, LONG - 5), (LONG - 5, 3)]
    wl = workloads.custom_workload(shapes, w_std=0.0, g_std=1e-3)   # W = 0: the update is exposed exactly
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    p = mo.MuonParams()
    dev = to_device(host, DEV)
    mo.muon_owner_step(dev, p, mo.muon_workspace(dev, p, device=DEV))
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    for (Wh, Gh, Vh), (Wd, _, Vd) in zip(host, dev):
        R, C = Wh.shape
        _, Vn, O = oracle.muon_matrix_step(f64(Wh), f64(Gh), f64(Vh), **oracle_options(p))
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        assert rel_frob(extract_update(f64(Wh), f64(Wd), p.lr, p.wd, R, C), O) <= NS_REL_FROB_TOL, (R, C)


@pytest.mark.parametrize("form", ["gram", "appendix"])
def test_gram_split_into_slices(form):
    """Grams longer than 32768 columns are summed from fp32 slice partials: a
    matrix just over the threshold (a 1000-column last slice), one of three
    slices, and a short matrix beside them in the same launches."""
    shapes = [(33_768, 512), (256, 70_000), (300, 700)]
    wl = workloads.custom_workload(shapes, w_std=0.0, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    p = mo.MuonParams(ns_form=form)
    dev, again = to_device(host, DEV), to_device(host, DEV)
    for mats in (dev, again):
        mo.muon_owner_step(mats, p, mo.muon_workspace(mats, p, device=DEV))
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    for (Wa, _, Va), (Wb, _, Vb) in zip(dev, again):   # partials are summed in a fixed order
        assert torch.equal(Wa, Wb) and torch.equal(Va, Vb)
    tol = 2e-2 if form == "appendix" else NS_REL_FROB_TOL
    for (Wh, Gh, Vh), (Wd, _, Vd) in zip(host, dev):
        R, C = Wh.shape
        _, Vn, O = oracle.muon_matrix_step(f64(Wh), f64(Gh), f64(Vh), **oracle_options(p))
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        assert rel_frob(extract_update(f64(Wh), f64(Wd), p.lr, p.wd, R, C), O) <= tol, (R, C)


def test_rmnp_longest_rows():
    """W = 0, lr = 1, wd = 0 exposes -s D directly (one CTA per row here)."""
    shapes = [(2, LONG), (1, LONG - 3)]
    wl = workloads.custom_workload(shapes, w_std=0.0, g_std=1.0)
    host = [workloads.host_matrix(wl, i, v_std=0.5) for i in range(len(shapes))]
    dev = to_device(host, DEV)
    mo.rmnp_step(dev, mo.RmnpParams(lr=1.0, wd=0.0, mu=0.9))
    torch.cuda.synchronize()
    for (Wh, Gh, Vh), (Wd, _, Vd) in zip(host, dev):
        _, Vn, D = oracle.rmnp_matrix_step(f64(Wh), f64(Gh), f64(Vh), lr=1.0, wd=0.0, mu=0.9)
        assert max_rel(-f64(Wd) / oracle.shape_scale(*Wh.shape), D) <= FP32_MAX_REL_TOL
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL


def test_adamw_segment_beyond_2_31_elements():
    n = (1 << 31) + 4097
    gen = torch.Generator(device=DEV).manual_seed(123)
    pt = torch.randn(n, generator=gen, device=DEV).mul_(0.02)
    g = torch.randn(n, generator=gen, device=DEV).mul_(1e-3)
    m = torch.randn(n, generator=gen, device=DEV).mul_(1e-3)
    v = m * m + torch.rand(n, generator=gen, device=DEV).mul_(1e-6)
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.integers(0, n, 4000), np.arange(n - 64, n),
                                    np.arange((1 << 31) - 64, (1 << 31) + 64), np.arange(64)]))
    it = torch.from_numpy(idx).to(DEV)
    before = [f64(t[it]) for t in (pt, g, m, v)]
    params = mo.AdamWParams(step=3)
    mo.adamw_tail_step([(pt, g, m, v)], params)
    torch.cuda.synchronize()
    ref = oracle.adamw_step(*before, lr=params.lr, wd=params.wd, beta1=params.beta1, beta2=params.beta2,
                            eps=params.eps, step=3)
    for got, want in zip((pt, m, v), ref):
        assert max_rel(f64(got[it]), want) <= FP32_MAX_REL_TOL
    del pt, g, m, v
    torch.cuda.empty_cache()


def test_muon_largest_square_sign_matrix():
    """m = n = 65536, the largest supported short side: the Gram is split
    into two slices, and A.A and B.X reduce over 65536 unsplit. The gradient
    is an outer product of random +-1 vectors times 2^-10, so every value the
    iteration stores is an exact power-of-two multiple of the same sign
    pattern: X_k = x_k s t^T / sqrt(m n), A_k = x_k^2 s s^T / m, and every
    fp32 sum of the products is exact. The iteration is then a scalar
    recursion whose bf16 roundings depend only on mantissas, so the oracle
    on a 64 x 64 matrix of the same kind gives the value the 65536 x 65536
    result must have. Checks: the momentum equals G exactly; every element of
    the update is the same value up to its sign s_i t_j (bit for bit: any
    tile computed wrongly, twice or not at all would break this); and that
    value matches the oracle's within the Newton-Schulz tolerance."""
    m = 65536
    gen = torch.Generator(device=DEV)
    gen.manual_seed(11)
    s = torch.randint(0, 2, (m,), generator=gen, device=DEV).float().mul_(2).sub_(1)
    t = torch.randint(0, 2, (m,), generator=gen, device=DEV).float().mul_(2).sub_(1)
    G = torch.empty(m, m, device=DEV, dtype=torch.bfloat16)
    for r0 in range(0, m, 4096):
        G[r0:r0 + 4096] = (s[r0:r0 + 4096, None] * t[None, :] * 2.0 ** -10).to(torch.bfloat16)
    W = torch.zeros(m, m, device=DEV)
    V = torch.zeros(m, m, device=DEV)
    p = mo.MuonParams(lr=1.0, wd=0.0)
    ws = mo.muon_workspace([(W, G, V)], p, device=DEV)
    mo.muon_owner_step([(W, G, V)], p, ws)
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    del ws
    # the oracle's value of x_5 on a small matrix of the same structure
    rs = np.random.default_rng(0)
    ss, tt = rs.choice([-1.0, 1.0], 64), rs.choice([-1.0, 1.0], 64)
    _, _, O = oracle.muon_matrix_step(np.zeros((64, 64)), np.outer(ss, tt) * 2.0 ** -10, np.zeros((64, 64)),
                                      **oracle_options(p))
    x5 = float((O * np.outer(ss, tt)).ravel()[0] * 64)
    lo, hi = float("inf"), -float("inf")
    for r0 in range(0, m, 4096):
        rows = slice(r0, r0 + 4096)
        assert torch.equal(V[rows], G[rows].float())
        d = W[rows] * s[rows, None] * t[None, :] * (-float(m))   # exact: powers of two and signs
        lo, hi = min(lo, float(d.min())), max(hi, float(d.max()))
    assert lo == hi, (lo, hi)
    assert abs(lo - x5) <= NS_REL_FROB_TOL * abs(x5), (lo, x5)
