"""The C ABI used from plain C: tests/c/abi_from_c.c includes only
include/mo.h, is compiled as C11 with warnings as errors, links the in-tree
libmo.so and checks the host-only entry points and the argument validation
(no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from matrix_optimizers_zero_gb300 import build as mo_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_abi_from_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = mo_build.build()
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(mo_build._nvcc()))), "include")
    exe = str(tmp_path / "abi_from_c")
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
                    "-L", os.path.dirname(lib), "-lmo", "-Wl,-rpath," + os.path.dirname(lib), "-o", exe],
                   check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"
