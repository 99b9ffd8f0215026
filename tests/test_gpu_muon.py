"""GPU parity of muon_owner_step (called through the C ABI) against the CPU
oracle on the same seeded inputs: the Newton-Schulz direction within a
relative Frobenius error of 1e-2, the fp32 momentum within 1e-5 max relative
error. Covers the smoke matrix, ragged and degenerate shapes (tiles with
partial rows and columns, m = 1, tall and wide, square), heterogeneous tables
in one grouped launch, 1/2/5 iterations, custom coefficients, zero gradients,
determinism and multi-step state. (Whole tables in the benchmark's launch
configuration are covered by the full-table tests.)"""
import math

import numpy as np
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads
import oracle
from gpu_util import (FP32_MAX_REL_TOL, NS_REL_FROB_TOL, extract_update, f64, max_rel, rel_frob,
                      to_device)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run_muon(dev_mats, params):
    ws = mo.muon_workspace(dev_mats, params, device=DEV)
    mo.muon_owner_step(dev_mats, params, ws)
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0


FORM_NAMES = {v: k for k, v in mo.NS_FORMS.items()}
ADJUST_NAMES = {v: k for k, v in mo.LR_ADJUST.items()}


def oracle_options(params):
    """The oracle's keyword arguments for a MuonParams."""
    return dict(lr=params.lr, wd=params.wd, mu=params.mu, coeffs=(params.a, params.b, params.c),
                eps=params.eps, ns_steps=params.ns_steps, ns_form=FORM_NAMES[params.ns_form],
                lr_adjust=ADJUST_NAMES[params.lr_adjust], nesterov=bool(params.nesterov))


def update_scale(params, R, C):
    return oracle.match_rms_adamw_scale(R, C) if params.lr_adjust == 1 else oracle.shape_scale(R, C)


def check_table(host_mats, params, tol=NS_REL_FROB_TOL, direct=False):
    """Runs one step on the GPU and compares every matrix with the oracle."""
    dev = to_device(host_mats, DEV)
    W0 = [f64(W) for W, _, _ in host_mats]
    run_muon(dev, params)
    worst = 0.0
    for (Wh, Gh, Vh), (Wd, Gd, Vd), w0 in zip(host_mats, dev, W0):
        R, C = Wh.shape
        Wn, Vn, O = oracle.muon_matrix_step(w0, f64(Gh), f64(Vh), **oracle_options(params))
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        O_gpu = extract_update(w0, f64(Wd), params.lr, params.wd, R, C, update_scale(params, R, C))
        err = rel_frob(O_gpu, O)
        worst = max(worst, err)
        assert err <= tol, (R, C, err)
    return worst


def test_smoke_config():
    wl = workloads.get_workload("smoke")
    host = [workloads.host_matrix(wl, 0)]
    err = check_table(host, mo.MuonParams(lr=0.02, wd=0.01, mu=0.95, ns_steps=5))
    assert err < 5e-3


def test_direct_output_with_zero_weight():
    """W = 0, lr = 1, wd = 0: W_new = -s O exactly exposes the iteration output."""
    wl = workloads.custom_workload([(128, 256), (256, 128)], w_std=0.0, g_std=1.0)
    host = [workloads.host_matrix(wl, i) for i in range(2)]
    check_table(host, mo.MuonParams(lr=1.0, wd=0.0))


@pytest.mark.parametrize("shape", [(130, 257), (257, 130), (300, 300), (1, 64), (64, 1), (1, 1), (7, 1000),
                                   (129, 129), (255, 513), (640, 128)])
def test_ragged_and_degenerate_shapes(shape):
    wl = workloads.custom_workload([shape], g_std=1e-3)
    check_table([workloads.host_matrix(wl, 0)], mo.MuonParams())


def test_heterogeneous_table_one_launch():
    shapes = [(130, 257), (512, 384), (384, 512), (1000, 200), (200, 1000), (256, 256), (3, 700)]
    wl = workloads.custom_workload(shapes, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=5e-3) for i in range(len(shapes))]
    check_table(host, mo.MuonParams())


@pytest.mark.parametrize("steps", [1, 2, 5])
def test_iteration_counts_and_momentum(steps):
    """The convergence settings of MatrixFSDP section 5.1 (2 iterations,
    momentum 0.5) and the default 5 iterations."""
    wl = workloads.custom_workload([(384, 640), (640, 384)], g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(2)]
    check_table(host, mo.MuonParams(mu=0.5 if steps == 2 else 0.95, ns_steps=steps, lr=1e-3, wd=1e-2))


def test_custom_coefficients():
    wl = workloads.custom_workload([(256, 512)], g_std=1e-3)
    check_table([workloads.host_matrix(wl, 0)], mo.MuonParams(a=2.0, b=-1.5, c=0.5, ns_steps=6))


def test_zero_gradient_is_pure_decay():
    W = torch.randn(200, 300, device=DEV)
    G = torch.zeros(200, 300, device=DEV, dtype=torch.bfloat16)
    V = torch.zeros(200, 300, device=DEV)
    W0 = W.clone()
    p = mo.MuonParams()
    run_muon([(W, G, V)], p)
    assert torch.equal(V, torch.zeros_like(V))
    decay = torch.tensor(float(np.float32(1.0 - float(p.lr) * float(p.wd))), dtype=torch.float32)
    assert torch.equal(W, W0 * decay)


def test_deterministic_and_resume():
    """Two identical runs are bit-identical; three steps in one go equal
    step, copy out state, restore, two more steps."""
    wl = workloads.custom_workload([(300, 700), (700, 300), (256, 256)], g_std=1e-3)
    host = [workloads.host_matrix(wl, i) for i in range(3)]
    p = mo.MuonParams()
    a = to_device(host, DEV)
    b = to_device(host, DEV)
    run_muon(a, p)
    run_muon(b, p)
    for x, y in zip(a, b):
        assert torch.equal(x[0], y[0]) and torch.equal(x[2], y[2])
    # continue `a` two more steps; `c` restores a's state after one step
    c = [(W.clone(), G.clone(), V.clone()) for W, G, V in a]
    for _ in range(2):
        run_muon(a, p)
    for _ in range(2):
        run_muon(c, p)
    for x, y in zip(a, c):
        assert torch.equal(x[0], y[0]) and torch.equal(x[2], y[2])


def test_multi_step_matches_oracle():
    """Three steps with fresh gradients: momentum stays within 1e-5; the
    accumulated weight change within the Newton-Schulz tolerance."""
    wl = workloads.custom_workload([(256, 384), (384, 256)], g_std=1e-3)
    host = [workloads.host_matrix(wl, i) for i in range(2)]
    dev = to_device(host, DEV)
    p = mo.MuonParams()
    w_init = [f64(W) for W, _, _ in host]
    ref = [(f64(W), f64(V)) for W, _, V in host]
    for step in range(3):
        gs = [torch.randn(W.shape, generator=torch.Generator().manual_seed(100 + step)).mul_(1e-3).to(torch.bfloat16)
              for W, _, _ in host]
        dev = [(W, g.to(DEV), V) for (W, _, V), g in zip(dev, gs)]
        run_muon(dev, p)
        ref = [oracle.muon_matrix_step(W, f64(g), V, lr=p.lr, wd=p.wd, mu=p.mu)[:2] for (W, V), g in zip(ref, gs)]
    for (Wd, _, Vd), (Wr, Vr), w0 in zip(dev, ref, w_init):
        assert max_rel(f64(Vd), Vr) <= FP32_MAX_REL_TOL
        assert rel_frob(f64(Wd) - w0, Wr - w0) <= NS_REL_FROB_TOL


def test_bounded_wait_reports_timeout():
    mo.mo_selftest_bounded_wait(20_000_000)    # 20 ms
    assert mo.mo_last_device_error() == -8
    assert mo.mo_last_device_error() == 0      # cleared after reading
    # the context is still usable
    x = torch.ones(4, device=DEV)
    assert float((x * 2).sum()) == 8.0


def test_plan_cache_alternating_tables_on_one_workspace():
    """Plans are cached per (device, table, workspace address); alternating
    two different tables on the same workspace must stay correct on every
    call (each call re-uploads its own header)."""
    wl1 = workloads.custom_workload([(130, 257), (64, 640)], g_std=1e-3)
    wl2 = workloads.custom_workload([(257, 130), (300, 300), (512, 128)], g_std=1e-3, config_id=98)
    t1 = to_device([workloads.host_matrix(wl1, i) for i in range(2)], DEV)
    t2 = to_device([workloads.host_matrix(wl2, i) for i in range(3)], DEV)
    p = mo.MuonParams()
    nbytes = max(mo.mo_muon_workspace_bytes(t1, p), mo.mo_muon_workspace_bytes(t2, p))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    for tbl in (t1, t2, t1, t2, t1):
        snap = [tuple(f64(x) for x in m) for m in tbl]
        mo.muon_owner_step(tbl, p, ws)
        torch.cuda.synchronize()
        assert mo.mo_last_device_error() == 0
        for (W0, G0, V0), (Wd, _, Vd) in zip(snap, tbl):
            R, C = W0.shape
            _, Vn, O = oracle.muon_matrix_step(W0, G0, V0, lr=p.lr, wd=p.wd, mu=p.mu)
            assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
            assert rel_frob(extract_update(W0, f64(Wd), p.lr, p.wd, R, C), O) <= NS_REL_FROB_TOL


def test_many_small_matrices_in_one_table():
    """600 matrices of random small shapes (several per tile and per work
    item, tall and wide, some below the tile size in both directions) in one
    grouped launch sequence.

    Over a random population the bf16 rounding noise of five iterations
    itself reaches the 1e-2 bar for a few matrices: a NumPy restatement with
    fp32 accumulation and the same rounding points differs from the oracle by
    1.03e-2 on the 52 x 63 matrix of this set (and the GPU by the same
    amount). So each matrix is held to 1e-2 or, where larger, 1.25 times that
    fp32-accumulation noise on its own input; the table-wide error is held to
    1e-2."""
    from gpu_util import fp32_accumulation_noise
    rng = np.random.default_rng(77)
    shapes = [(int(rng.integers(1, 200)), int(rng.integers(1, 200))) for _ in range(600)]
    wl = workloads.custom_workload(shapes, g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(shapes))]
    p = mo.MuonParams()
    dev = to_device(host, DEV)
    W0 = [f64(W) for W, _, _ in host]
    run_muon(dev, p)
    num = den = 0.0
    over = 0
    for (Wh, Gh, Vh), (Wd, _, Vd), w0 in zip(host, dev, W0):
        R, C = Wh.shape
        _, Vn, O = oracle.muon_matrix_step(w0, f64(Gh), f64(Vh), **oracle_options(p))
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        O_gpu = extract_update(w0, f64(Wd), p.lr, p.wd, R, C)
        err = rel_frob(O_gpu, O)
        num += float(np.sum((O_gpu - O) ** 2))
        den += float(np.sum(O ** 2))
        if err > NS_REL_FROB_TOL:
            over += 1
            X0 = oracle.frobenius_normalize(Vn, p.eps)
            noise = fp32_accumulation_noise(X0, O, (p.a, p.b, p.c), p.ns_steps)
            assert err <= 1.25 * noise, (R, C, err, noise)
    assert math.sqrt(num / den) <= NS_REL_FROB_TOL
    assert over <= 6


def test_ten_iterations():
    """Twice the specified iteration count (even, so the ping-pong buffers end
    where they started). The bf16 rounding noise of the method grows with the
    iterations: a NumPy fp32-accumulation restatement is 1.8e-2 from the
    oracle here, so the bar is 1.5 times that noise on each input (1e-2 at
    least)."""
    from gpu_util import fp32_accumulation_noise
    wl = workloads.custom_workload([(192, 320), (320, 192)], g_std=1e-3)
    host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(2)]
    p = mo.MuonParams(ns_steps=10)
    dev = to_device(host, DEV)
    W0 = [f64(W) for W, _, _ in host]
    run_muon(dev, p)
    for (Wh, Gh, Vh), (Wd, _, Vd), w0 in zip(host, dev, W0):
        R, C = Wh.shape
        _, Vn, O = oracle.muon_matrix_step(w0, f64(Gh), f64(Vh), **oracle_options(p))
        assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
        err = rel_frob(extract_update(w0, f64(Wd), p.lr, p.wd, R, C), O)
        noise = fp32_accumulation_noise(oracle.frobenius_normalize(Vn, p.eps), O, (p.a, p.b, p.c), p.ns_steps)
        assert err <= max(NS_REL_FROB_TOL, 1.5 * noise), (R, C, err, noise)


def test_two_host_threads_two_streams():
    """Two host threads each run Muon steps on their own table, workspace and
    stream at the same time (the plan cache is shared and locked); both match
    the oracle."""
    import threading
    tables = []
    for seed_shapes in ([(256, 640), (640, 256)], [(384, 384), (130, 700)]):
        wl = workloads.custom_workload(seed_shapes, g_std=1e-3)
        host = [workloads.host_matrix(wl, i, v_std=1e-3) for i in range(len(seed_shapes))]
        tables.append(host)
    p = mo.MuonParams()
    devs = [to_device(h, DEV) for h in tables]
    W0 = [[f64(W) for W, _, _ in h] for h in tables]
    errors = []

    def work(k):
        try:
            torch.cuda.set_device(DEV)
            s = torch.cuda.Stream(DEV)
            ws = mo.muon_workspace(devs[k], p, device=DEV)
            with torch.cuda.stream(s):
                mo.muon_owner_step(devs[k], p, ws, stream=s)
            s.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert mo.mo_last_device_error() == 0
    for host, dev, w0s in zip(tables, devs, W0):
        for (Wh, Gh, Vh), (Wd, _, Vd), w0 in zip(host, dev, w0s):
            R, C = Wh.shape
            _, Vn, O = oracle.muon_matrix_step(w0, f64(Gh), f64(Vh), **oracle_options(p))
            assert max_rel(f64(Vd), Vn) <= FP32_MAX_REL_TOL
            assert rel_frob(extract_update(w0, f64(Wd), p.lr, p.wd, R, C), O) <= NS_REL_FROB_TOL
