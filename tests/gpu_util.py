"""Helpers for the GPU parity tests: device upload of seeded inputs, the
library call, and the comparison metrics with the tolerances of the
specification (Newton-Schulz output: relative Frobenius error <= 1e-2; fp32
AdamW and RMNP: max |gpu - ref| / max |ref| <= 1e-5)."""
import math

import numpy as np

NS_REL_FROB_TOL = 1e-2
FP32_MAX_REL_TOL = 1e-5


def rel_frob(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def max_rel(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max() if ref.size else 0.0
    return float(np.abs(got - ref).max() / den) if den > 0 else float(np.abs(got).max() if got.size else 0.0)


def f64(t) -> np.ndarray:
    """A torch tensor (any device, fp32 or bf16) as a float64 numpy array."""
    return t.detach().float().cpu().double().numpy()


def to_device(host_mats, device):
    return [(W.to(device), G.to(device), V.to(device)) for (W, G, V) in host_mats]


def shape_scale(rows, cols):
    return math.sqrt(max(1.0, rows / cols))


def extract_update(W0, W1, lr, wd, rows, cols, scale=None):
    """Recovers the applied direction O from W1 = W0 (1 - lr wd) - lr s O
    (s = sqrt(max(1, rows/cols)) unless given)."""
    s = shape_scale(rows, cols) if scale is None else scale
    return (np.asarray(W0, np.float64) * (1.0 - lr * wd) - np.asarray(W1, np.float64)) / (lr * s)
