"""The C ABI from a plain C99 program (tests/c/abi_check.c): no Python or PyTorch in the
process that calls the library.  The CPU test builds it and runs its host-side checks;
the GPU test runs a chunked prefill through gdn_chunk_prefill and steps the same tokens
one at a time through gdn_recurrent_decode, all from C, and compares the two."""
import os
import shutil
import subprocess

import pytest

from gated_deltanet_linear_11_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def abi_check(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(_lib.LIB_PATH):
        pytest.skip("libgdn.so not built")
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("abi") / "abi_check")
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "c", "abi_check.c"),
           "-L", libdir, "-lgdn", "-Wl,-rpath," + libdir,
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64"),
           "-lm", "-o", exe]
    p = subprocess.run(cmd, capture_output=True, text=True)
    assert p.returncode == 0, p.stdout + p.stderr
    return exe


def test_c_program_host_checks(abi_check):
    p = subprocess.run([abi_check, "cpu"], capture_output=True, text=True, timeout=60)
    assert p.returncode == 0 and p.stdout.strip().endswith("ok"), p.stdout + p.stderr


@pytest.mark.gpu
def test_c_program_prefill_matches_recurrent_decode(abi_check):
    p = subprocess.run([abi_check, "gpu"], capture_output=True, text=True, timeout=300)
    print(p.stdout)
    assert p.returncode == 0 and p.stdout.strip().endswith("ok"), p.stdout + p.stderr
