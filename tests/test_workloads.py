"""The synthetic shape tables reproduce the figures the pages print about them
("Optimizers In A Sharded World", sections 3-5) and the configuration sizes."""
import math
import os

import numpy as np
import pytest

from matrix_optimizers_zero_gb300 import workloads as wl_mod

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_printed_values.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = (t.strip() for t in line.split("=", 1))
            out[k] = float(v)
    return out


def test_gpt2l_table_matches_printed_figures():
    g = golden()
    wl = wl_mod.get_workload("gpt2l")
    assert len(wl.matrices) == g["gpt2l_matrix_count"]
    assert round(wl.n_elements / 1e6) == g["gpt2l_params_millions_rounded"]
    assert wl.n_elements == 707_788_800
    sum_m = sum(s.rows for s in wl.matrices)
    assert abs(sum_m / 1e3 - g["gpt2l_colcut_vector_thousands"]) <= g["gpt2l_colcut_vector_tolerance"]
    gather_mib = sum(7 / 8 * s.rows * s.cols * 2 for s in wl.matrices) / 2 ** 20
    assert round(gather_mib) == g["muon_gather_mib_per_gpu"]
    assert 5120 * 1280 * 2 / 2 ** 20 == g["cfc_bf16_mib"]
    assert round(5120 * 4 / 1024) == g["colcut_partial_vector_kb"]
    assert wl.tail_elements == 601_600


def test_other_tables():
    w8 = wl_mod.get_workload("llama8b")
    assert len(w8.matrices) == 224 and w8.n_elements == 6_979_321_856
    assert w8.tail_elements == 1_050_939_392
    ws = wl_mod.get_workload("spectrum")
    assert len(ws.matrices) == 56 and ws.n_elements == 838_860_800
    w32 = wl_mod.get_workload("share32b")
    assert len(w32.matrices) == 28 and w32.n_elements == 1_950_351_360 and w32.tail_elements == 2_000_000
    sm = wl_mod.get_workload("smoke")
    assert [(s.rows, s.cols) for s in sm.matrices] == [(128, 256)] and sm.tail == (1024,)


def test_alg_flop_totals():
    tf = {n: wl_mod.workload_alg_flops(wl_mod.get_workload(n)) / 1e12
          for n in ("gpt2l", "llama8b", "spectrum", "share32b")}
    assert abs(tf["gpt2l"] - 15.10) < 0.01
    assert abs(tf["llama8b"] - 471.8) < 0.1
    assert abs(tf["spectrum"] - 40.4) < 0.1
    assert abs(tf["share32b"] - 160.7) < 0.1
    assert wl_mod.ns_alg_flops(128, 256) == 5 * (3 * 128 * 128 * 256 + 128 ** 3)
    assert wl_mod.ns_alg_flops(256, 128) == wl_mod.ns_alg_flops(128, 256)


def test_generation_is_seeded_and_per_matrix():
    wl = wl_mod.custom_workload([(5, 7), (9, 3)])
    a = wl_mod.host_matrix(wl, 1)
    b = wl_mod.host_matrix(wl, 1)
    for x, y in zip(a, b):
        assert x.dtype == y.dtype and bool((x == y).all())
    W, G, V = a
    assert tuple(W.shape) == (9, 3) and str(G.dtype) == "torch.bfloat16" and float(V.abs().sum()) == 0.0
    c = wl_mod.host_matrix(wl, 0)
    assert tuple(c[0].shape) == (5, 7)


def test_structured_spectrum_generation():
    wl = wl_mod.get_workload("spectrum")
    # use a reduced copy of the recipe so the test stays fast
    small = wl_mod.Workload("spec_small", 3, (wl_mod.MatrixSpec(64, 96, "w", "haar"),
                                              wl_mod.MatrixSpec(96, 64, "t", "haar"),
                                              wl_mod.MatrixSpec(16, 64, "o", "orthorows")), (),
                            0.02, 1.0, 0.02, 1e-3)
    for i in range(2):
        u, s, vt = wl_mod.spectral_factors(small, i)
        k = min(small.matrices[i].rows, small.matrices[i].cols)
        np.testing.assert_allclose(u.T @ u, np.eye(k), atol=1e-12)
        np.testing.assert_allclose(vt @ vt.T, np.eye(k), atol=1e-12)
        assert s.min() >= 1e-4 and s.max() <= 1.0
        G = wl_mod.exact_matrix(small, i)
        np.testing.assert_allclose(np.linalg.svd(G, compute_uv=False), np.sort(s)[::-1], rtol=1e-10)
    for i in range(3):
        assert all(t.is_contiguous() for t in wl_mod.host_matrix(small, i))
    G = wl_mod.exact_matrix(small, 2)
    gram = G @ G.T
    np.testing.assert_allclose(gram - np.diag(np.diag(gram)), 0, atol=1e-12)
