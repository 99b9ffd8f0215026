"""Pins for the oracle's Muon variants.

* The appendix algebraic form of the iteration ("Optimizers In A Sharded
  World", appendix "The Code That Ran") with bf16 storage: equal to the
  Gram-polynomial form up to bf16 rounding, with every stored intermediate
  bf16-representable.
* Nesterov look-ahead and the match_rms_adamw learning-rate adjustment
  ("MatrixFSDP", section 5.1, which runs torch.optim.Muon): checked against
  torch.optim.Muon itself on the CPU. torch.optim.Muon orthogonalises in bf16,
  so the comparison is at bf16 tolerance; each test also shows that the wrong
  variant misses by far more than that tolerance."""
import numpy as np
import pytest
import torch

from oracle import (bf16_round, frobenius_normalize, match_rms_adamw_scale, muon_matrix_step,
                    newton_schulz, newton_schulz_pages_form, shape_scale)


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / np.linalg.norm(np.asarray(b)))


@pytest.mark.parametrize("shape", [(40, 72), (72, 40), (64, 64)])
def test_pages_form_rounded_close_to_gram_form(shape):
    rng = np.random.default_rng(21)
    X0 = frobenius_normalize(rng.standard_normal(shape))
    exact = newton_schulz(X0)
    np.testing.assert_allclose(newton_schulz_pages_form(X0), exact, rtol=0, atol=1e-12)
    trace = []
    r = newton_schulz_pages_form(X0, round_bf16=True, trace=trace)
    assert r.shape == shape
    assert rel(r, exact) < 2e-2
    assert rel(r, newton_schulz(X0, round_bf16=True)) < 3e-2
    m = min(shape)
    for name, M in trace[:-1]:            # the final iterate stays unrounded
        assert np.array_equal(bf16_round(M), M), name
        if name.startswith("A"):
            assert M.shape == (m, m) and np.array_equal(M, M.T)
        elif name.startswith("B"):
            assert M.shape == (m, max(shape))     # B = A X is m x n in this form


def _torch_muon_delta(W, grads, **kw):
    p = torch.nn.Parameter(torch.from_numpy(W.astype(np.float32)))
    opt = torch.optim.Muon([p], **kw)
    for g in grads:
        before = p.detach().double().numpy().copy()
        p.grad = torch.from_numpy(g.astype(np.float32))
        opt.step()
    after = p.detach().double().numpy()
    return before, after


@pytest.mark.parametrize("nesterov", [False, True])
@pytest.mark.parametrize("lr_adjust", ["original", "match_rms_adamw"])
@pytest.mark.parametrize("shape", [(48, 96), (96, 48)])
def test_variants_match_torch_muon(nesterov, lr_adjust, shape):
    rng = np.random.default_rng(5)
    W = rng.standard_normal(shape) * 0.02
    grads = [rng.standard_normal(shape) * s for s in (1.0, 0.3, 2.0)]
    lr, wd, mu, steps = 0.05, 1e-2, 0.5, 2
    before, after = _torch_muon_delta(W, grads, lr=lr, weight_decay=wd, momentum=mu, nesterov=nesterov,
                                      ns_steps=steps, eps=1e-7, adjust_lr_fn=lr_adjust)
    # replay the same three steps in the oracle (float64, bf16-emulated NS)
    Wc, V = W.astype(np.float32).astype(np.float64), np.zeros(shape)
    for g in grads:
        Wprev, Vprev = Wc, V
        g32 = g.astype(np.float32).astype(np.float64)
        Wc, V, _ = muon_matrix_step(Wc, g32, V, lr=lr, wd=wd, mu=mu, ns_steps=steps, nesterov=nesterov,
                                    lr_adjust=lr_adjust)
    ours = Wc - Wprev * (1 - lr * wd)
    theirs = after - before * (1 - lr * wd)
    assert rel(ours, theirs) < 3e-2
    # the wrong Nesterov setting or the wrong scale misses by far more
    _, _, O_other = muon_matrix_step(Wprev, g32, Vprev, lr=lr, wd=wd, mu=mu, ns_steps=steps,
                                     nesterov=not nesterov, lr_adjust=lr_adjust)
    scale = match_rms_adamw_scale(*shape) if lr_adjust == "match_rms_adamw" else shape_scale(*shape)
    assert rel(-lr * scale * O_other, theirs) > 0.1
    other = "original" if lr_adjust == "match_rms_adamw" else "match_rms_adamw"
    oscale = match_rms_adamw_scale(*shape) if other == "match_rms_adamw" else shape_scale(*shape)
    assert rel(ours * (oscale / scale), theirs) > 0.25


def test_match_rms_scale_values():
    # 0.2 sqrt(max(rows, cols)) is symmetric in the shape, unlike sqrt(max(1, rows/cols))
    assert match_rms_adamw_scale(1280, 5120) == pytest.approx(0.2 * 71.55417527999327, rel=1e-15)
    assert match_rms_adamw_scale(5120, 1280) == match_rms_adamw_scale(1280, 5120)
    assert shape_scale(5120, 1280) == 2.0 and shape_scale(1280, 5120) == 1.0


def test_variant_arguments_rejected():
    W = np.zeros((4, 8))
    with pytest.raises(ValueError):
        muon_matrix_step(W, W + 1, W, ns_form="cubic")
    with pytest.raises(ValueError):
        muon_matrix_step(W, W + 1, W, lr_adjust="sqrt")
