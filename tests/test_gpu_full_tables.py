"""Whole tables in the benchmark's launch configuration: every matrix of a
configuration goes through one grouped muon_owner_step call, and the result
is checked two ways.

  * Every matrix, bit for bit, against the same matrix stepped alone through
    muon_owner_step. The kernels are deterministic and a matrix's arithmetic
    does not depend on the rest of the table (its norm partials, tiles and
    epilogues only touch its own data), so any difference is a scheduling or
    addressing fault of the grouped launch.
  * A sample against the CPU oracle (direction: relative Frobenius error
    <= 1e-2; momentum: max relative error <= 1e-5): the first matrix of each
    distinct shape plus two more drawn at random per shape, one more for the
    shapes whose oracle step exceeds 5 TFLOP (27648 x 5120 and 5120 x 27648,
    minutes of CPU time each). The oracle runs in spawned worker processes
    while the GPU comparisons go on.

Tables: GPT-2 Large (144 matrices), the Llama-style 8B set (224), the
32B-scale owner share (28 matrices up to 27648 x 5120) and the
structured-spectrum batch (56 matrices, each generated with its stated
structure: Haar singular vectors with log-uniform spectra, or orthogonal rows
with N(1, 0.3)^2 scales)."""
import numpy as np
import pytest
import torch

import matrix_optimizers_zero_gb300 as mo
from matrix_optimizers_zero_gb300 import workloads
import oracle
from gpu_util import FP32_MAX_REL_TOL, NS_REL_FROB_TOL, OraclePool

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# oracle steps above this many algorithmic flops get one random extra per shape
BIG_ORACLE_FLOPS = 5e12


@pytest.fixture(scope="module")
def pool():
    p = OraclePool(4)
    yield p
    p.close()


def oracle_sample(wl):
    """Matrix indices checked against the oracle: the first of each distinct
    shape, then two (one for the biggest shapes) drawn from the others."""
    rng = np.random.default_rng(1000 + wl.config_id)
    by_shape = {}
    for i, s in enumerate(wl.matrices):
        by_shape.setdefault((s.rows, s.cols), []).append(i)
    picks = []
    for (r, c), idx in by_shape.items():
        picks.append(idx[0])
        extra = 2 if workloads.ns_alg_flops(r, c, wl.ns_steps) <= BIG_ORACLE_FLOPS else 1
        rest = idx[1:]
        if rest:
            picks.extend(int(x) for x in rng.choice(rest, size=min(extra, len(rest)), replace=False))
    return picks


def host32(t):
    return t.detach().float().cpu().numpy()


def full_table_check(wl, mats, pool):
    p = mo.MuonParams(lr=wl.lr, wd=wl.wd, mu=wl.mu, ns_steps=wl.ns_steps)
    sample = oracle_sample(wl)
    W_init = [W.clone() for W, _, _ in mats]
    V_init = [V.clone() for _, _, V in mats]
    inputs = {i: (host32(mats[i][0]), host32(mats[i][1]), host32(mats[i][2])) for i in sample}

    table = mo.MuonTable(mats)
    ws = mo.muon_workspace(table, p, device=DEV)
    mo.muon_owner_step(table, p, ws)
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    del ws, table

    opts = dict(lr=p.lr, wd=p.wd, mu=p.mu, coeffs=(p.a, p.b, p.c), eps=p.eps, ns_steps=p.ns_steps)
    jobs = {}
    for i in sample:
        s = wl.matrices[i]
        jobs[i] = pool.muon_errors(*inputs[i], host32(mats[i][0]), host32(mats[i][2]), opts,
                                   oracle.shape_scale(s.rows, s.cols))
    del inputs

    # every matrix alone, in place on its saved inputs
    single_bytes = max(mo.mo_muon_workspace_bytes([(W_init[i], G, V_init[i])], p) for i, (_, G, _) in enumerate(mats))
    ws1 = torch.empty(single_bytes, dtype=torch.uint8, device=DEV)
    for i, (_, G, _) in enumerate(mats):
        mo.muon_owner_step([(W_init[i], G, V_init[i])], p, ws1)
    torch.cuda.synchronize()
    assert mo.mo_last_device_error() == 0
    differ = [i for i, (W, _, V) in enumerate(mats)
              if not (torch.equal(W_init[i], W) and torch.equal(V_init[i], V))]
    assert not differ, f"matrices whose grouped result differs from their single-matrix step: {differ[:20]}"

    errs = {}
    for i, job in jobs.items():
        v_err, o_err = job.result(timeout=1800)
        s = wl.matrices[i]
        assert v_err <= FP32_MAX_REL_TOL, (i, s.rows, s.cols, v_err)
        assert o_err <= NS_REL_FROB_TOL, (i, s.rows, s.cols, o_err)
        errs[i] = o_err
    return errs


def test_gpt2l_full_table(pool):
    wl = workloads.get_workload("gpt2l")
    full_table_check(wl, workloads.device_matrices(wl, DEV, v_std=1e-3), pool)


def test_llama8b_full_table(pool):
    wl = workloads.get_workload("llama8b")
    full_table_check(wl, workloads.device_matrices(wl, DEV, v_std=1e-3), pool)


def test_share32b_full_table(pool):
    wl = workloads.get_workload("share32b")
    full_table_check(wl, workloads.device_matrices(wl, DEV, v_std=1e-3), pool)


def test_spectrum_full_table(pool):
    wl = workloads.get_workload("spectrum")
    full_table_check(wl, workloads.device_structured_matrices(wl, DEV), pool)


def test_oracle_sample_covers_every_shape():
    for name in ("gpt2l", "llama8b", "share32b", "spectrum"):
        wl = workloads.get_workload(name)
        picks = oracle_sample(wl)
        assert len(set(picks)) == len(picks)
        shapes = {(wl.matrices[i].rows, wl.matrices[i].cols) for i in picks}
        assert shapes == {(s.rows, s.cols) for s in wl.matrices}
