"""The C ABI from a plain C program (tests/c/abi_demo.c): compiled with gcc
against include/w4a16.h, linked with the library, the CUDA runtime and the
oracle, and run without Python in the process.  It packs a seeded layer on the
device, runs w4a16_linear and checks the packed words bit for bit and y within
the linear's rule against the oracle.
"""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_uses_the_abi(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    from weight_only_int4_w4a16_gb300.build import LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    oracle_lib = oracle.build()
    exe = str(tmp_path / "abi_demo")
    libdirs = [os.path.dirname(LIB), os.path.dirname(oracle_lib), os.path.join(cuda, "lib64")]
    cmd = [cc, "-O2", "-std=c11", os.path.join(ROOT, "tests", "c", "abi_demo.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), "-o", exe]
    for d in libdirs:
        cmd += ["-L", d, f"-Wl,-rpath,{d}"]
    cmd += ["-l:" + os.path.basename(LIB), "-l:" + os.path.basename(oracle_lib), "-lcudart", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "c abi ok" in run.stdout
