"""CPU oracle for the owner-local optimizer step (TEST INFRASTRUCTURE ONLY).

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this module. The library never calls it, and it shares no code with the
CUDA path: it is plain NumPy in float64, written to be checked by eye against
the pages it cites.

Sources (cited by page title and section):
  [MFSDP]  "MatrixFSDP: communication-free matrix optimizers under ZeRO-3
           parameter sharding" (arXiv 2607.05895v1).
           Section 3 (owner placement: the owner runs Muon on the whole 2D
           matrix, the tail owner runs AdamW), section 4.4 (optimizer routing),
           section 5.1 (hyperparameters: Muon lr 1e-3, wd 1e-2; AdamW betas,
           eps 1e-8, decoupled weight decay as in Loshchilov and Hutter).
  [SHARD]  "Optimizers In A Sharded World: Muon's O(mn) Vs RMNP's Zero".
           Section 1 (momentum V_t = mu V_{t-1} + G_t; Muon's target direction
           (V V^T)^{-1/2} V approximated by five Newton-Schulz iterations of
           three products each; RMNP direction V_i / ||V_i||_2 per row), and
           the appendix "The Code That Ran" (the quintic iteration with
           coefficients (3.4445, -4.7750, 2.0315) and eps 1e-7 added to the
           Frobenius norm, the transpose when rows > cols, the shape scale
           sqrt(max(1, rows/cols)), the row-normalisation with fp32 sums and
           the 1e-12 clamp of F.normalize).

Readings where the pages are silent:
  * The iteration is written as A = X X^T, B = b A + c A A, X' = a X + B X.
    The appendix script writes it as A = X X^T, B = A X, X' = a X + b B + c A B;
    the two are equal in exact arithmetic (a self-check pins this). The
    appendix form is kept as a selectable variant.
  * Nesterov momentum (torch.optim.Muon's default, used by [MFSDP] section
    5.1) is an option, off by default: the appendix script updates with the
    plain momentum.
  * The Frobenius norm is taken of the fp32 momentum; X0 = bf16(V / (||V|| + eps)).
  * Weight decay is decoupled and multiplicative for Muon and RMNP, with the
    same learning rate: W <- W (1 - lr wd) - lr s D.
  * The last iterate is not rounded to bf16 before the weight update.
  * AdamW: bias-corrected moments, eps outside the square root, step t >= 1.

bf16 emulation: with `round_bf16=True` every matrix the GPU stores in bf16 as a
GEMM operand (X between iterations, A and B) is rounded to nearest-even bf16
directly from float64; accumulation stays float64.

Parity status: every function below is pinned by the CPU tests against
closed forms, library routines or invariants, except htrmnp_direction and
htrmnp_matrix_step: their formula is a reading of one sentence of the pages
(parity unpinned; see their docstrings).
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

# default quintic coefficients ([SHARD] appendix)
NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_EPS = 1e-7            # added to the Frobenius norm ([SHARD] appendix)
RMNP_EPS = 1e-12         # F.normalize clamp ([SHARD] appendix, row-sharded RMNP)

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
_BF16_MIN_QUANTUM_EXP = -133   # quantum of bf16 subnormals: 2^-126 * 2^-7


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned
    as float64. bf16 keeps 8 significant bits, the fp32 exponent range and
    gradual underflow; values beyond the largest finite bf16 become +-inf."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    fin = np.isfinite(x)
    xf = x[fin]
    _, e = np.frexp(xf)                      # xf = f * 2^e with 0.5 <= |f| < 1
    q = np.maximum(e - 8, _BF16_MIN_QUANTUM_EXP)
    y = np.ldexp(np.rint(np.ldexp(xf, -q)), q)   # np.rint rounds halves to even
    y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, xf), y)
    out[fin] = y
    return out


def _identity(x):
    return x


# ---------------------------------------------------------------------------
# Muon ([SHARD] section 1 and appendix; [MFSDP] sections 3, 4.4)
# ---------------------------------------------------------------------------

def momentum(V: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """Heavy-ball momentum V_t = mu V_{t-1} + G_t ([SHARD] section 1)."""
    return mu * np.asarray(V, np.float64) + np.asarray(G, np.float64)


def frobenius_normalize(V: np.ndarray, eps: float = NS_EPS) -> np.ndarray:
    """X = V / (||V||_F + eps) ([SHARD] appendix, first lines of the quintic
    iteration)."""
    V = np.asarray(V, np.float64)
    return V / (math.sqrt(float(np.sum(V * V))) + eps)


def newton_schulz(X0: np.ndarray, coeffs: Sequence[float] = NS_COEFFS, steps: int = 5,
                  round_bf16: bool = False, trace: Optional[list] = None) -> np.ndarray:
    """Quintic Newton-Schulz iteration ([SHARD] section 1: five iterations of
    three matrix products approximating (X X^T)^{-1/2} X; appendix: the
    coefficients and the transpose to the wide orientation).

    X0 is already normalised. If X0 has more rows than columns the iteration
    runs on X0^T and the result is transposed back. Per iteration:
        A  = X X^T
        B  = b A + c A A
        X' = a X + B X
    With round_bf16, X (before every iteration), A and B are rounded to bf16;
    the final iterate is returned unrounded. `trace`, if given, receives
    (name, array) pairs of every stored intermediate."""
    a, b, c = (float(t) for t in coeffs)
    q = bf16_round if round_bf16 else _identity
    X = np.asarray(X0, np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = q(X)
    if trace is not None:
        trace.append(("X0", X))
    for k in range(steps):
        A = q(X @ X.T)
        B = q(b * A + c * (A @ A))
        Xn = a * X + B @ X
        X = q(Xn) if k < steps - 1 else Xn
        if trace is not None:
            trace.extend([(f"A{k}", A), (f"B{k}", B), (f"X{k + 1}", X)])
    return X.T if tall else X


def newton_schulz_pages_form(X0: np.ndarray, coeffs: Sequence[float] = NS_COEFFS,
                             steps: int = 5, round_bf16: bool = False,
                             trace: Optional[list] = None) -> np.ndarray:
    """The same iteration in the algebraic form of the appendix script
    ([SHARD] appendix "The Code That Ran", the quintic iteration):
        A  = X X^T
        B  = A X            (m x n, unlike the m x m B of newton_schulz)
        X' = a X + b B + c A B
    With round_bf16, X (before every iteration), A and B are rounded to bf16
    (the matrices the GPU stores between products); a X + b B + c A B is
    combined unrounded and the final iterate is returned unrounded."""
    a, b, c = (float(t) for t in coeffs)
    q = bf16_round if round_bf16 else _identity
    X = np.asarray(X0, np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = q(X)
    if trace is not None:
        trace.append(("X0", X))
    for k in range(steps):
        A = q(X @ X.T)
        B = q(A @ X)
        Xn = a * X + b * B + c * (A @ B)
        X = q(Xn) if k < steps - 1 else Xn
        if trace is not None:
            trace.extend([(f"A{k}", A), (f"B{k}", B), (f"X{k + 1}", X)])
    return X.T if tall else X


def shape_scale(rows: int, cols: int) -> float:
    """sqrt(max(1, rows/cols)) on the stored [out, in] shape ([SHARD]
    appendix, scale of the Muon and RMNP updates)."""
    return math.sqrt(max(1.0, rows / cols))


def match_rms_adamw_scale(rows: int, cols: int) -> float:
    """0.2 sqrt(max(rows, cols)): the learning-rate adjustment named
    match_rms_adamw in the convergence settings of [MFSDP] section 5.1, as
    torch.optim.Muon (which that section uses) defines it: it brings the RMS
    of the orthogonalised update to that of a typical AdamW update."""
    return 0.2 * math.sqrt(max(rows, cols))


def nesterov_direction(V_new: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """Nesterov look-ahead G_t + mu V_t. [MFSDP] section 5.1 runs
    torch.optim.Muon, whose default update is the Nesterov one; with the
    momentum written V_t = mu V_{t-1} + G_t ([SHARD] section 1) that update is
    (1 - mu)(G_t + mu V_t), and the positive factor cancels in the Frobenius
    normalisation (up to eps)."""
    return np.asarray(G, np.float64) + mu * np.asarray(V_new, np.float64)


def decoupled_update(W: np.ndarray, D: np.ndarray, lr: float, wd: float, scale: float) -> np.ndarray:
    """W <- W (1 - lr wd) - lr scale D (decoupled weight decay, [MFSDP]
    section 5.1 gives wd; the multiplicative form is the reading taken)."""
    return np.asarray(W, np.float64) * (1.0 - lr * wd) - (lr * scale) * np.asarray(D, np.float64)


def muon_matrix_step(W, G, V, lr=0.02, wd=0.01, mu=0.95, coeffs=NS_COEFFS, eps=NS_EPS,
                     ns_steps=5, round_bf16=True, nesterov=False, lr_adjust="original",
                     ns_form="gram"):
    """One owner-local Muon step on a whole 2D matrix ([MFSDP] section 3: the
    owner holds the full gradient; [SHARD] section 1 and appendix for the
    arithmetic). Returns (W_new, V_new, O) where O is the Newton-Schulz output
    in the stored orientation.

    Variants: nesterov=True orthogonalises G + mu V_new instead of V_new;
    lr_adjust="match_rms_adamw" replaces the shape scale by
    0.2 sqrt(max(rows, cols)); ns_form="appendix" runs the iteration in the
    appendix script's algebraic form (newton_schulz_pages_form)."""
    R, C = np.shape(W)
    Vn = momentum(V, G, mu)
    U = nesterov_direction(Vn, G, mu) if nesterov else Vn
    X0 = frobenius_normalize(U, eps)
    if ns_form == "gram":
        O = newton_schulz(X0, coeffs, ns_steps, round_bf16=round_bf16)
    elif ns_form == "appendix":
        O = newton_schulz_pages_form(X0, coeffs, ns_steps, round_bf16=round_bf16)
    else:
        raise ValueError(f"unknown ns_form {ns_form!r}")
    if lr_adjust == "original":
        scale = shape_scale(R, C)
    elif lr_adjust == "match_rms_adamw":
        scale = match_rms_adamw_scale(R, C)
    else:
        raise ValueError(f"unknown lr_adjust {lr_adjust!r}")
    Wn = decoupled_update(W, O, lr, wd, scale)
    return Wn, Vn, O


# ---------------------------------------------------------------------------
# RMNP ([SHARD] sections 1 and 5, appendix rmnp_local)
# ---------------------------------------------------------------------------

def rmnp_direction(V: np.ndarray, eps: float = RMNP_EPS) -> np.ndarray:
    """D_i = V_i / max(||V_i||_2, eps) for every stored row i ([SHARD]
    section 1; the clamp is F.normalize's, as used in the appendix)."""
    V = np.asarray(V, np.float64)
    norms = np.sqrt(np.sum(V * V, axis=1))
    return V / np.maximum(norms, eps)[:, None]


def rmnp_matrix_step(W, G, V, lr=0.02, wd=0.01, mu=0.95, eps=RMNP_EPS):
    """One RMNP step: momentum, row normalisation, shape-scaled decoupled
    update. Returns (W_new, V_new, D)."""
    R, C = np.shape(W)
    Vn = momentum(V, G, mu)
    D = rmnp_direction(Vn, eps)
    Wn = decoupled_update(W, D, lr, wd, shape_scale(R, C))
    return Wn, Vn, D


HTRMNP_POWER = 0.125     # default power of the row norm ([SHARD] section 7)


def htrmnp_direction(V: np.ndarray, power: float = HTRMNP_POWER, eps: float = RMNP_EPS) -> np.ndarray:
    """HTRMNP direction. [SHARD] section 7 says only that HTRMNP scales RMNP's
    row-normalised direction with a power of the row norm (p = 0.125 by
    default); no formula is printed. Reading taken here: the row direction
    keeps the fraction p of its norm,
        D_i = V_i / max(||V_i||_2, eps)^(1 - p),
    so p = 0 is RMNP and p = 1 leaves V unchanged. PARITY UNPINNED: the pages
    fix neither the formula nor a value of it; the tests pin this reading's
    special cases (p = 0, p = 1, degree-p homogeneity) only."""
    V = np.asarray(V, np.float64)
    norms = np.sqrt(np.sum(V * V, axis=1))
    return V / (np.maximum(norms, eps) ** (1.0 - power))[:, None]


def htrmnp_matrix_step(W, G, V, lr=0.02, wd=0.01, mu=0.95, power=HTRMNP_POWER, eps=RMNP_EPS):
    """One HTRMNP step: momentum, the power-scaled row direction above, and
    RMNP's shape-scaled decoupled update. Returns (W_new, V_new, D)."""
    R, C = np.shape(W)
    Vn = momentum(V, G, mu)
    D = htrmnp_direction(Vn, power, eps)
    Wn = decoupled_update(W, D, lr, wd, shape_scale(R, C))
    return Wn, Vn, D


def rmnp_row_sharded(V: np.ndarray, shards: int, eps: float = RMNP_EPS) -> np.ndarray:
    """RMNP computed shard by shard over contiguous row blocks and
    concatenated ([SHARD] section 5: each rank normalises its own complete
    rows)."""
    V = np.asarray(V, np.float64)
    m = V.shape[0]
    parts = [rmnp_direction(V[r * m // shards:(r + 1) * m // shards], eps) for r in range(shards)]
    return np.concatenate(parts, axis=0)


RMNP_COLCUT_EPS = 1e-7   # clamp of the column-cut scheme ([SHARD] appendix)


def rmnp_colcut_direction(V_shards: Sequence[np.ndarray], eps: float = RMNP_COLCUT_EPS) -> List[np.ndarray]:
    """RMNP when each row is cut into column shards ([SHARD] section 3,
    column-cut tensor parallelism; appendix rmnp_colcut): every shard
    contributes the sum of squares of its part of each row, the per-row
    partial sums are added over the shards (the page's all-reduce), and each
    shard divides its part by max(sqrt(total), eps)."""
    shards = [np.asarray(v, np.float64) for v in V_shards]
    total = np.zeros(shards[0].shape[0])
    for v in shards:
        total = total + np.sum(v * v, axis=1)
    norm = np.maximum(np.sqrt(total), eps)
    return [v / norm[:, None] for v in shards]


def rmnp_colcut_matrix_step(W_shards, G_shards, V_shards, rows: int, cols: int, lr=0.02, wd=0.01, mu=0.95,
                            eps=RMNP_COLCUT_EPS):
    """Column-cut RMNP step over the shards of one [rows, cols] matrix:
    momentum per shard, the cut-row normalisation above, and the same
    shape-scaled decoupled update as unsharded RMNP (scale of the whole
    matrix). Returns (W_new_shards, V_new_shards, D_shards)."""
    Vn = [momentum(V, G, mu) for V, G in zip(V_shards, G_shards)]
    D = rmnp_colcut_direction(Vn, eps)
    s = shape_scale(rows, cols)
    Wn = [decoupled_update(W, d, lr, wd, s) for W, d in zip(W_shards, D)]
    return Wn, Vn, D


# ---------------------------------------------------------------------------
# AdamW on the packed non-matrix tail ([MFSDP] sections 3, 4.4, 5.1)
# ---------------------------------------------------------------------------

def adamw_step(p, g, m, v, lr=1e-3, wd=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, step=1):
    """Decoupled AdamW with bias correction (the tail owner's optimizer,
    [MFSDP] section 3; hyperparameters section 5.1). `step` is t after the
    increment (t >= 1). Returns (p_new, m_new, v_new)."""
    if step < 1:
        raise ValueError("step must be >= 1")
    p = np.asarray(p, np.float64)
    g = np.asarray(g, np.float64)
    m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64)
    p = p * (1.0 - lr * wd)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** step)
    v_hat = v / (1.0 - beta2 ** step)
    p = p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v


# ---------------------------------------------------------------------------
# whole-table helpers
# ---------------------------------------------------------------------------

def muon_table_step(mats: List[Tuple[np.ndarray, np.ndarray, np.ndarray]], **kw):
    """Muon over an owner's shape table: the matrices are independent, so the
    table step is the per-matrix step applied to each ([MFSDP] section 4.4)."""
    return [muon_matrix_step(W, G, V, **kw) for (W, G, V) in mats]


def rmnp_table_step(mats, **kw):
    return [rmnp_matrix_step(W, G, V, **kw) for (W, G, V) in mats]
