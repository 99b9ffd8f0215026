"""Pins for the oracle's RMNP and AdamW.

RMNP ("Optimizers In A Sharded World", sections 1 and 5): checked against the
library row normalisation, against the exact polar factor when the Gram matrix
is diagonal (section 1: the two directions coincide then), and for exact
equality between row-sharded and unsharded evaluation (section 5, appendix
exactness check: 512 x 384, seed 7, max |diff| = 0).

AdamW ("MatrixFSDP", sections 3 and 5.1): checked against torch.optim.AdamW in
float64 and against closed forms."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import (adamw_step, rmnp_direction, rmnp_matrix_step, rmnp_row_sharded, shape_scale)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_printed_values.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = (t.strip() for t in line.split("=", 1))
            out[k] = float(v)
    return out


def test_rmnp_matches_library_normalize():
    rng = np.random.default_rng(1)
    V = rng.standard_normal((37, 53)) * rng.uniform(0.01, 10, size=(37, 1))
    ref = torch.nn.functional.normalize(torch.from_numpy(V), p=2, dim=-1).numpy()
    np.testing.assert_allclose(rmnp_direction(V), ref, rtol=1e-14, atol=0)
    assert np.allclose(np.linalg.norm(rmnp_direction(V), axis=1), 1.0, atol=1e-14)


def test_rmnp_zero_row_clamped():
    V = np.zeros((2, 4))
    V[1] = [1.0, 0, 0, 0]
    D = rmnp_direction(V)
    assert np.all(D[0] == 0) and np.array_equal(D[1], [1.0, 0, 0, 0])


def test_rmnp_nan_row_like_library_normalize():
    """A NaN anywhere in a row makes that whole row NaN and leaves the other
    rows alone, as F.normalize (whose clamp keeps NaN) does."""
    rng = np.random.default_rng(4)
    V = rng.standard_normal((5, 9))
    V[2, 6] = np.nan
    ref = torch.nn.functional.normalize(torch.from_numpy(V), p=2, dim=-1).numpy()
    D = rmnp_direction(V)
    assert np.isnan(ref[2]).all() and np.isnan(D[2]).all()
    keep = [0, 1, 3, 4]
    np.testing.assert_allclose(D[keep], ref[keep], rtol=1e-14, atol=0)


def test_rmnp_equals_polar_for_diagonal_gram():
    rng = np.random.default_rng(2)
    q, _ = np.linalg.qr(rng.standard_normal((96, 24)))
    d = rng.normal(1.0, 0.3, size=24) ** 2
    V = d[:, None] * q.T                                 # 24 x 96, V V^T diagonal
    w, E = np.linalg.eigh(V @ V.T)
    polar = E @ np.diag(w ** -0.5) @ E.T @ V            # (V V^T)^{-1/2} V
    np.testing.assert_allclose(rmnp_direction(V), polar, atol=1e-12)


def test_rmnp_row_sharded_is_exact():
    g = golden()
    m, n, shards = int(g["rmnp_exactness_rows"]), int(g["rmnp_exactness_cols"]), int(g["rmnp_exactness_shards"])
    V = torch.randn(m, n, generator=torch.Generator().manual_seed(7)).double().numpy()
    diff = np.abs(rmnp_row_sharded(V, shards) - rmnp_direction(V)).max()
    assert diff == g["rmnp_sharded_vs_full_max_abs_diff"]


def test_rmnp_step_update():
    rng = np.random.default_rng(3)
    W, G, V = (rng.standard_normal((8, 4)) for _ in range(3))
    Wn, Vn, D = rmnp_matrix_step(W, G, V, lr=0.1, wd=0.5, mu=0.9)
    np.testing.assert_allclose(Vn, 0.9 * V + G, rtol=1e-15)
    np.testing.assert_allclose(Wn, W * 0.95 - 0.1 * math.sqrt(2.0) * D, rtol=1e-14)


@pytest.mark.parametrize("betas", [(0.9, 0.95), (0.9, 0.999)])
def test_adamw_matches_library_optimizer(betas):
    rng = np.random.default_rng(4)
    p0 = rng.standard_normal(257)
    lr, wd, eps = 1e-3, 1e-2, 1e-8
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=lr, betas=betas, eps=eps, weight_decay=wd, foreach=False)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    for t in range(1, 7):
        g = rng.standard_normal(257) * (10.0 ** rng.uniform(-4, 1))
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
        p, m, v = adamw_step(p, g, m, v, lr=lr, wd=wd, beta1=betas[0], beta2=betas[1], eps=eps, step=t)
        np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-13, atol=1e-16)
        st = opt.state[tp]
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-300)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-300)


def test_adamw_closed_forms():
    g = np.array([2.0, -3.0, 0.0, 1e-9])
    p = np.array([1.0, 1.0, 1.0, 1.0])
    lr, wd, eps = 1e-3, 1e-2, 1e-8
    # first step from zero state: update is lr * g / (|g| + eps) after decay
    p1, m1, v1 = adamw_step(p, g, np.zeros(4), np.zeros(4), lr=lr, wd=wd, eps=eps, step=1)
    np.testing.assert_allclose(p1, p * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-15)
    assert p1[2] == 1.0 * (1 - lr * wd)                  # zero gradient: decay only
    # constant gradient: bias-corrected moments equal g and g^2 at every step
    p, m, v = p.copy(), np.zeros(4), np.zeros(4)
    for t in range(1, 10):
        prev = p
        p, m, v = adamw_step(p, g, m, v, lr=lr, wd=wd, eps=eps, step=t)
        np.testing.assert_allclose(p, prev * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-12)
    with pytest.raises(ValueError):
        adamw_step(p, g, m, v, step=0)


def test_colcut_rmnp_equals_unsharded_rows():
    """Cutting every row into column shards and adding the per-row partial
    sums gives the same row norms (the page: a row's squared norm is the sum
    of its shards' squared norms); only the clamp differs (1e-7)."""
    from oracle import rmnp_colcut_direction
    rng = np.random.default_rng(12)
    V = rng.standard_normal((40, 384)) * rng.uniform(0.1, 3, size=(40, 1))
    for cuts in ([384], [160] * 2 + [64], [48] * 8, [1, 383]):
        edges = np.cumsum([0] + cuts)
        shards = [V[:, a:b] for a, b in zip(edges[:-1], edges[1:])]
        D = np.concatenate(rmnp_colcut_direction(shards), axis=1)
        np.testing.assert_allclose(D, rmnp_direction(V), rtol=1e-14, atol=0)
    Z = np.zeros((3, 10))
    Z[1, 4] = 1e-9        # norm below the column-cut clamp
    D = np.concatenate(rmnp_colcut_direction([Z[:, :6], Z[:, 6:]]), axis=1)
    assert np.all(D[0] == 0) and D[1, 4] == pytest.approx(1e-9 / 1e-7, rel=1e-15)


def test_htrmnp_reading_special_cases():
    """HTRMNP ("Optimizers In A Sharded World", section 7) has no printed
    formula; these pin the reading D_i = V_i / max(||V_i||, eps)^(1 - p) at
    its special cases only (parity unpinned): p = 0 is RMNP exactly, p = 1 is
    the identity, and the direction is homogeneous of degree p in each row."""
    from oracle import htrmnp_direction, HTRMNP_POWER
    assert HTRMNP_POWER == 0.125
    rng = np.random.default_rng(31)
    V = rng.standard_normal((23, 41)) * rng.uniform(0.01, 5, size=(23, 1))
    assert np.array_equal(htrmnp_direction(V, power=0.0), rmnp_direction(V))
    np.testing.assert_allclose(htrmnp_direction(V, power=1.0), V, rtol=1e-15)
    c = rng.uniform(0.1, 10, size=(23, 1))
    np.testing.assert_allclose(htrmnp_direction(c * V), c ** 0.125 * htrmnp_direction(V), rtol=1e-13)
    norms = np.linalg.norm(htrmnp_direction(V), axis=1)
    np.testing.assert_allclose(norms, np.linalg.norm(V, axis=1) ** 0.125, rtol=1e-13)
    Z = np.zeros((2, 5))
    assert np.all(htrmnp_direction(Z) == 0)
