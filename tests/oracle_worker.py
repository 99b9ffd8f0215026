"""Worker-process side of the oracle pool of the full-table GPU tests. It
imports nothing heavy at module import, so that the pool's initializer can
set the BLAS thread count before numpy loads in the worker."""
import os

THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def init(threads: int) -> None:
    for k in THREAD_VARS:
        os.environ[k] = str(threads)


def muon_errors(*args):
    from gpu_util import oracle_muon_errors
    return oracle_muon_errors(*args)
