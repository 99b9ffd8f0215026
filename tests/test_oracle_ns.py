"""Pins for the oracle's Muon arithmetic (momentum, Frobenius normalisation,
quintic Newton-Schulz, update).

Newton-Schulz maps each singular value of the normalised input through the
scalar quintic phi(x) = a x + b x^3 + c x^5 while keeping the singular vectors
("Optimizers In A Sharded World", section 1: the iteration approximates
(V V^T)^{-1/2} V). The scalar map is computed here by a plain scalar loop, so a
wrong coefficient, a dropped term, a swapped product order or a lost transpose
in the matrix code fails these tests."""
import math

import numpy as np
import pytest

from oracle import (NS_COEFFS, bf16_round, decoupled_update, frobenius_normalize, momentum,
                    muon_matrix_step, newton_schulz, newton_schulz_pages_form, shape_scale)


def phi_iterated(x: float, steps=5, coeffs=NS_COEFFS) -> float:
    a, b, c = coeffs
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def haar(rng, n, k):
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


def structured(rng, m, n, s):
    k = min(m, n)
    return (haar(rng, m, k) * s) @ haar(rng, n, k).T


@pytest.mark.parametrize("shape", [(12, 20), (20, 12), (16, 16), (1, 9), (9, 1), (33, 65)])
@pytest.mark.parametrize("steps", [1, 2, 5])
def test_spectral_map_closed_form(shape, steps):
    rng = np.random.default_rng(hash(shape) % 1000 + steps)
    m, n = shape
    k = min(m, n)
    U, V = haar(rng, m, k), haar(rng, n, k)
    s = np.exp(rng.uniform(np.log(1e-3), 0, size=k))
    G = (U * s) @ V.T
    X0 = frobenius_normalize(G, eps=0.0)
    out = newton_schulz(X0, steps=steps)
    shat = s / np.linalg.norm(s)
    expect = (U * np.array([phi_iterated(x, steps) for x in shat])) @ V.T
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-11 * max(1, np.abs(expect).max()))


def test_phi5_known_values_and_rank_one():
    a = NS_COEFFS[0]
    assert abs(phi_iterated(1.0) - 0.6964364094697522) < 1e-15
    # slope at zero after five iterations is a^5
    assert abs(phi_iterated(1e-12) / 1e-12 - a ** 5) / a ** 5 < 1e-9
    rng = np.random.default_rng(2)
    u = rng.standard_normal(7)
    v = rng.standard_normal(11)
    u /= np.linalg.norm(u)
    v /= np.linalg.norm(v)
    G = 3.7 * np.outer(u, v)
    out = newton_schulz(frobenius_normalize(G, eps=0.0))
    np.testing.assert_allclose(out, phi_iterated(1.0) * np.outer(u, v), atol=1e-13)


def test_two_algebraic_forms_agree():
    rng = np.random.default_rng(3)
    for shape in [(10, 30), (30, 10), (17, 17)]:
        X0 = frobenius_normalize(rng.standard_normal(shape))
        np.testing.assert_allclose(newton_schulz(X0), newton_schulz_pages_form(X0), rtol=0, atol=1e-12)


def test_invariances():
    rng = np.random.default_rng(4)
    G = rng.standard_normal((9, 14))
    X0 = frobenius_normalize(G)
    base = newton_schulz(X0)
    Q1, Q2 = haar(rng, 9, 9), haar(rng, 14, 14)
    np.testing.assert_allclose(newton_schulz(frobenius_normalize(Q1 @ G @ Q2)), Q1 @ base @ Q2, atol=1e-11)
    np.testing.assert_allclose(newton_schulz(X0.T), base.T, atol=1e-13)
    # positive scaling: exact with eps = 0 (eps only perturbs at the 1e-8 level)
    base0 = newton_schulz(frobenius_normalize(G, eps=0.0))
    np.testing.assert_allclose(newton_schulz(frobenius_normalize(123.0 * G, eps=0.0)), base0, atol=1e-12)


@pytest.mark.parametrize("shape", [(4, 7), (16, 16), (33, 65), (65, 33)])
def test_brute_force_polar_within_polynomial_spread(shape):
    """The exact polar factor U V^T (from an SVD) differs from the iteration's
    output by at most max_i |phi^5(sigma_i) - 1| in spectral norm."""
    rng = np.random.default_rng(sum(shape))
    G = rng.standard_normal(shape)
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    polar = U @ Vt
    out = newton_schulz(frobenius_normalize(G, eps=0.0))
    spread = max(abs(phi_iterated(x) - 1.0) for x in s / np.linalg.norm(s))
    err = np.linalg.norm(out - polar, 2)
    assert err <= spread + 1e-9
    # the spread itself is bounded on [0.0015, 1] by the scalar map's range
    xs = np.linspace(0.0015, 1.0, 20001)
    ys = np.array([phi_iterated(x) for x in xs])
    assert 0.679 < ys.min() and ys.max() < 1.21


def test_zero_input_is_zero():
    X0 = frobenius_normalize(np.zeros((5, 8)))
    assert np.all(X0 == 0)
    assert np.all(newton_schulz(X0, round_bf16=True) == 0)


def test_rounded_path_stores_bf16_and_stays_close():
    rng = np.random.default_rng(6)
    for shape in [(48, 80), (80, 48)]:
        X0 = frobenius_normalize(rng.standard_normal(shape))
        trace = []
        out_r = newton_schulz(X0, round_bf16=True, trace=trace)
        out_e = newton_schulz(X0, round_bf16=False)
        names = [n for n, _ in trace]
        assert names[0] == "X0" and len(names) == 1 + 3 * 5
        for name, arr in trace[:-1]:
            np.testing.assert_array_equal(bf16_round(arr), arr, err_msg=name)
        final = trace[-1][1]
        assert not np.array_equal(bf16_round(final), final)   # last iterate is unrounded
        rel = np.linalg.norm(out_r - out_e) / np.linalg.norm(out_e)
        assert rel < 2e-2, rel


def test_rounded_path_close_to_library_bf16_iteration():
    """torch's Muon helper runs the same B = bA + cAA form natively in bf16
    (it casts first, then normalises); the emulated-bf16 oracle must land
    within bf16-level distance of it."""
    torch = pytest.importorskip("torch")
    muon = pytest.importorskip("torch.optim._muon")
    rng = np.random.default_rng(8)
    for shape in [(64, 96), (96, 64)]:
        G = rng.standard_normal(shape)
        ref = muon._zeropower_via_newtonschulz(torch.from_numpy(G).float(), NS_COEFFS, 5, 1e-7)
        ref = ref.double().numpy()
        got = newton_schulz(frobenius_normalize(G), round_bf16=True)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 3e-2, rel


def test_momentum_closed_form():
    rng = np.random.default_rng(9)
    G = rng.standard_normal((3, 5))
    V = np.zeros_like(G)
    mu = 0.95
    for t in range(1, 8):
        V = momentum(V, G, mu)
        np.testing.assert_allclose(V, G * (1 - mu ** t) / (1 - mu), rtol=1e-14)


def test_frobenius_normalize_by_hand():
    X = frobenius_normalize(np.array([[3.0, 4.0]]), eps=1e-7)
    np.testing.assert_allclose(X, np.array([[3.0, 4.0]]) / (5.0 + 1e-7), rtol=0, atol=0)


def test_shape_scale_and_update():
    assert shape_scale(3840, 1280) == math.sqrt(3.0)
    assert shape_scale(1280, 5120) == 1.0
    assert shape_scale(7, 7) == 1.0
    W = np.array([[1.0, -2.0]])
    D = np.array([[0.5, 0.25]])
    np.testing.assert_allclose(decoupled_update(W, D, 0.1, 0.2, 2.0),
                               np.array([[1.0 * 0.98 - 0.1, -2.0 * 0.98 - 0.05]]), rtol=1e-15)


def test_muon_zero_gradient_is_pure_decay():
    rng = np.random.default_rng(10)
    W = rng.standard_normal((6, 4))
    Wn, Vn, O = muon_matrix_step(W, np.zeros_like(W), np.zeros_like(W), lr=0.02, wd=0.01)
    assert np.all(O == 0) and np.all(Vn == 0)
    np.testing.assert_array_equal(Wn, W * (1 - 0.02 * 0.01))


def test_muon_step_structured_and_transposed():
    rng = np.random.default_rng(11)
    s = np.exp(rng.uniform(np.log(1e-2), 0, size=12))
    G = structured(rng, 12, 30, s)
    W = rng.standard_normal((12, 30))
    Wn, Vn, O = muon_matrix_step(W, G, np.zeros_like(G), mu=0.9, round_bf16=False)
    X0 = frobenius_normalize(G)
    np.testing.assert_allclose(O, newton_schulz(X0), atol=1e-14)
    np.testing.assert_allclose(Wn, W * (1 - 0.02 * 0.01) - 0.02 * O, atol=1e-14)
    # tall matrix: the step on G^T is the transpose of the step on G (the
    # iteration runs in the wide orientation either way) -- bit-identical
    WnT, _, OT = muon_matrix_step(W.T, G.T, np.zeros_like(G.T), mu=0.9, round_bf16=True)
    _, _, Or = muon_matrix_step(W, G, np.zeros_like(G), mu=0.9, round_bf16=True)
    np.testing.assert_array_equal(OT, Or.T)
    np.testing.assert_allclose(WnT, W.T * (1 - 2e-4) - 0.02 * math.sqrt(30 / 12) * Or.T, atol=1e-14)
