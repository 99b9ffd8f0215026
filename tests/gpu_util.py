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


def fp32_accumulation_noise(X0, O_ref, coeffs, steps):
    """Relative Frobenius distance between the oracle's rounded iteration O_ref
    and the same iteration (bf16 at the same points) with fp32 instead of fp64
    accumulation, computed with NumPy float32 products. It measures how far
    the bf16 rounding decisions alone move a correct fp32-accumulating
    implementation from the oracle on this input (a rounding boundary that
    fp32 and fp64 sums fall on different sides of flips one bf16 value, and
    the iteration amplifies small singular directions)."""
    import oracle
    a, b, c = (np.float32(t) for t in coeffs)
    X = np.asarray(X0, np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = oracle.bf16_round(X).astype(np.float32)
    for k in range(steps):
        A = oracle.bf16_round((X @ X.T).astype(np.float64)).astype(np.float32)
        B = oracle.bf16_round((b * A + c * (A @ A)).astype(np.float64)).astype(np.float32)
        Xn = a * X + B @ X
        X = oracle.bf16_round(Xn.astype(np.float64)).astype(np.float32) if k < steps - 1 else Xn
    X = X.astype(np.float64)
    return rel_frob(X.T if tall else X, O_ref)


# ---------------------------------------------------------------- oracle checks in worker processes

def oracle_muon_errors(W0, G0, V0, W1, V1, opts, scale):
    """(max relative momentum error, relative Frobenius error of the
    Newton-Schulz direction) of one GPU Muon step: W0/G0/V0 the inputs, W1/V1
    the GPU's outputs (float32 arrays; G0 holds the bf16 values exactly),
    `opts` the oracle's keyword arguments, `scale` the update's shape scale."""
    import oracle
    W0, G0, V0 = (np.asarray(x, np.float64) for x in (W0, G0, V0))
    R, C = W0.shape
    _, Vn, O = oracle.muon_matrix_step(W0, G0, V0, **opts)
    O_gpu = extract_update(W0, W1, opts["lr"], opts["wd"], R, C, scale)
    return max_rel(V1, Vn), rel_frob(O_gpu, O)


class OraclePool:
    """Worker processes (spawned, so a CUDA context in the parent is never
    forked) that run CPU oracle checks of large matrices side by side while
    the GPU part of a test goes on. The oracle's elementwise bf16 emulation is
    single-threaded, so several workers with a share of the BLAS threads each
    finish a batch of matrices ~2.5x sooner than one process. A worker that
    dies makes every pending result raise instead of waiting."""

    def __init__(self, workers: int = 4):
        import concurrent.futures as cf
        import multiprocessing as mp
        import os
        import oracle_worker
        cores = len(os.sched_getaffinity(0))
        workers = max(1, min(workers, cores))
        self.ex = cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn"),
                                         initializer=oracle_worker.init, initargs=(max(1, cores // workers),))

    def muon_errors(self, *args):
        """A future of oracle_muon_errors(*args) run in a worker."""
        import oracle_worker
        return self.ex.submit(oracle_worker.muon_errors, *args)

    def close(self):
        self.ex.shutdown(wait=True, cancel_futures=True)
